// RNN sequential head: the per-request state update that runs between two
// draft positions (internal header).
#pragma once

#include "common.cuh"

namespace spec {

struct RnnStateParams {
  int R, gamma, V, rank, k;  // k: the position whose state s_k is computed (1-based)
  int nsplit;                // > 0: first merge the fused kernel's split partials of position k-1
  const Partial* part;       // [R, nsplit] those partials (reference in log2 units)
  const int32_t* x0;
  int32_t* x;       // x_{k-1}: read (nsplit == 0) or merged and written (nsplit > 0)
  float* q_tok;     // written with x when merging
  float* lse_q;
  const void* A;    // [gamma, V, rank]
  const void* W;    // [gamma, rank, rank]
  void* S;          // [R, gamma, rank]: reads s_{k-1}, writes s_k
  uint32_t* status;
};

// One launch: s_k for every request.  fac_f32 selects fp32 factors and states
// (else bf16); pdl launches it as a programmatic dependent of the previous
// kernel (which must then trigger it, or simply finish).
cudaError_t launch_rnn_state(const RnnStateParams& p, bool fac_f32, bool pdl, cudaStream_t stream);

}  // namespace spec
