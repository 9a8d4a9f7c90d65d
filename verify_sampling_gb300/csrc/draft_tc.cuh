// Fused tensor-core draft step (internal header).
#pragma once

#include "common.cuh"

namespace spec {

// Upper bound on the SM count the workspace is sized for.
constexpr int kMaxDeviceSms = 256;

struct DraftTCParams {
  int R, gamma, V, rank, k, nsplit, mtiles, ntiles, stages;
  uint32_t rid_base;
  PhiloxKey key;
  PhiloxRoundKeys rk;  // round keys of `key` (filled by launch_draft_tc)
  const int32_t* x0;
  const float* draft_temp;
  const void* A;  // bf16 [gamma, V, rank]
  const void* W;  // RNN head: bf16 [gamma, rank, rank] (null: Markov head)
  void* S;        // RNN head: bf16 states [R, gamma, rank], 16-byte aligned (null: Markov head)
  int32_t* x;
  float* q_tok;
  float* lse_q;
  Partial* partials;   // [2][R, nsplit]: slot k % 2 holds position k's split partials
  unsigned* counters;  // [mtiles], zero on entry
  unsigned* row_best;  // [gamma, R] best race score per row over all CTAs (ordered keys), zero on entry
  uint32_t* status;
};

// Vocabulary splits per 128-request tile for a device with `device_sms` SMs.
int draft_tc_nsplit(int R, int V, int device_sms);

// gamma dependent launches (one per position) of the fused kernel; with the RNN
// head each is preceded by the state kernel of its position.
cudaError_t launch_draft_tc(const DraftTCParams& p, int logit_dtype, const void* U, const void* Ct,
                            cudaStream_t stream);

}  // namespace spec
