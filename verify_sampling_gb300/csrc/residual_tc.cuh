// Fused tensor-core residual resample (internal header).
#pragma once

#include "common.cuh"

namespace spec {

struct ResidTCParams {
  int R, gamma, V, rank, smem_bytes, ntiles, max_mtiles;
  uint32_t rid_base;
  PhiloxKey key;
  PhiloxRoundKeys rk;  // round keys of `key` (kept in the parameter bank)
  float inv_target_temp;
  const int32_t* x0;
  const int32_t* x;
  const float* draft_temp;
  const void* A;  // bf16 [gamma, V, rank]
  const void* S;  // RNN head: bf16 states [R, gamma, rank], 16-byte aligned (null: Markov head)
  const float* lse_q;
  const int32_t* tgt_row_off;
  const float* row_m;       // [R, gamma + 1] target-row softmax reference (log2 units)
  const float* row_s;       // [R, gamma + 1] target-row softmax sum
  const int* res_cnt;       // [gamma] requests whose first rejection is at j = k
  const int* res_list;      // [gamma, R] those requests
  Partial* partials;        // [max_mtiles, kResTileRows, nsplit]
  unsigned* counters;       // [max_mtiles], zero on entry
  unsigned* row_best;       // [R] shared race bounds, zero on entry
  int32_t* out_tok;         // [R, gamma + 1]
  int* fallback;            // [R] position whose residual was zero everywhere (0: none)
  float* c_star;            // c* mode: [R, gamma] sums of min(p, q), zero on entry
  uint32_t* status;
};

// Requests per tile of the residual kernel: few enough that every row copy
// can span several 64-column tiles and the rows replicate over all four TMEM
// lane quadrants.
constexpr int kResTileRows = 16;

// Request tiles the residual kernel may need: sum_k ceil(cnt_k / kResTileRows).
inline int resid_tc_max_mtiles(int R, int gamma) {
  return (R + kResTileRows - 1) / kResTileRows + gamma;
}

bool resid_tc_supported(int tgt_dtype, int logit_dtype, int fac_dtype, int rank, int V,
                        const void* tgt, const void* U, const void* A, const void* Ct);

// cstar = false: the residual resample of the rows in res_list.  cstar = true:
// sum_v min(p_v, q_v) of every row in res_list, added into c_star.
cudaError_t launch_resid_tc(const ResidTCParams& p, int tgt_dtype, int logit_dtype, const void* tgt,
                            const void* U, const void* Ct, int grid, bool cstar,
                            cudaStream_t stream);

}  // namespace spec
