// Parameters and launchers of the draft-stage kernels (internal header).
#pragma once

#include <algorithm>

#include "common.cuh"

namespace spec {

constexpr int kDraftThreads = 256;
constexpr int kConfThreads = 512;
constexpr int kMaxRank = 256;
constexpr int kMaxGamma = 64;

struct DraftStepParams {
  int R, gamma, V, rank, k, nsplit;
  uint32_t rid_base;
  PhiloxKey key;
  const void* U;
  const void* A;
  const void* Ct;
  const void* W;  // RNN head: recurrence [gamma, rank, rank] (null: Markov head)
  void* S;        // RNN head: states [R, gamma, rank] (null: Markov head)
  const int32_t* x0;
  const float* draft_temp;
  int32_t* x;
  float* q_tok;
  float* lse_q;
  float* P_out;
  Partial* partials;  // [R, nsplit]
  unsigned* counters; // [R], zero on entry
  uint32_t* status;
};

struct ConfParams {
  int R, gamma, V, d, e;
  const int32_t* x0;
  const int32_t* x;
  const void* h;
  const void* W1;
  const void* w;
  const float* sts_temp;
  float* c;
  float* a;
  uint32_t* status;
  bool vec;  // h, W1 and w rows are 16-byte aligned: 16-byte loads
};

// Number of vocabulary splits per draft row: enough CTAs to cover the GPU
// several times over, never fewer than 1024 vocabulary entries per CTA.
inline int draft_nsplit(int R, int V) {
  const int target_ctas = 4 * 152 * 2;
  const int max_split = std::max(1, (V + 1023) / 1024);
  return std::max(1, std::min(max_split, (target_ctas + R - 1) / R));
}

// gamma generic sampling steps, then (want_probs) the P_out pass; probs_only
// skips the sampling steps (their outputs came from the fused kernel).
cudaError_t launch_draft_steps(const DraftStepParams& p, int logit_dtype, int fac_dtype,
                               bool want_probs, cudaStream_t stream, bool probs_only = false);
cudaError_t launch_confidence(const ConfParams& p, int conf_dtype, cudaStream_t stream);

}  // namespace spec
