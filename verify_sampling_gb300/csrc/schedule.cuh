// Parameters and launcher of the single-block prefix scheduler (internal header).
#pragma once

#include "common.cuh"

namespace spec {

constexpr int kSchedMaxCandidates = 8192;  // R * gamma, one thread block

struct SchedParams {
  int R, gamma, n_sps, K, mode, npad;
  double b_lo, b_step;
  double threshold;  // SPEC_SCHED_THRESHOLD: admit survivals >= threshold
  bool unit_grid;  // b_step == 1 and b_lo integral: SPS(B) is a table entry
  long b_lo_int;
  const float* a;
  const float* sps;
  int32_t* ell;
  int32_t* row_off;
  double* stats;
  int32_t* order;
  const int32_t* K_dev;  // nullable: cap = min(K, max(*K_dev, 0)), read on the device
  int32_t* n_free;       // nullable: the rule's n with no cap
  uint32_t* status;
};

size_t schedule_smem_bytes(int R, int gamma);
cudaError_t launch_schedule(SchedParams p, cudaStream_t stream);

}  // namespace spec
