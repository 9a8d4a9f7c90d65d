// Parameters and launcher of the acceptance-statistics update (internal header).
#pragma once

#include "common.cuh"

namespace spec {

constexpr int kAcceptStatsMaxGamma = 1024;

struct AcceptStatsParams {
  int R, gamma, bucket, n_buckets, min_count;
  double beta;
  const int32_t* ell;
  const int32_t* accept_len;
  double* ema;
  long long* count;
  double* estimate;
  uint32_t* status;
};

cudaError_t launch_accept_stats(const AcceptStatsParams& p, cudaStream_t stream);

}  // namespace spec
