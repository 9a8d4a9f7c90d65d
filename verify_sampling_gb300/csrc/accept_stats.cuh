// Parameters and launchers of the runtime statistics: acceptance EMA per
// length and the calibration diagram (internal header).
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

constexpr int kCalibrationMaxBins = 1024;

struct CalibrationParams {
  int R, gamma, n_bins;
  const float* c;
  const int32_t* ell;
  const int32_t* accept_len;
  long long* count;
  double* sum_c;
  long long* sum_acc;
  double* ece;
  uint32_t* status;
};

cudaError_t launch_calibration(const CalibrationParams& p, cudaStream_t stream);

}  // namespace spec
