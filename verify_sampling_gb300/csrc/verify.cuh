// Parameters and launchers of the verify-stage kernels (internal header).
#pragma once

#include <algorithm>

#include "common.cuh"

namespace spec {

constexpr int kVerifyThreads = 256;
constexpr int kRowChunk = 8192;  // vocabulary entries per row-pass work unit
constexpr int kPlanThreads = 1024;

// Per-call scratch carved out of the caller's workspace.
struct VerifyScratch {
  Partial* row_part;  // [R, gamma + 1, nsplit]
  Partial* res_part;  // [R, nsplit] (two races per record)
  float* row_m;       // [R, gamma + 1] softmax reference of L / T_t, log2 units
  float* row_s;       // [R, gamma + 1] softmax sum of 2^(L log2e / T_t - row_m)
  int* row_res;       // [R, gamma + 1] accept bit (sample) / argmax (greedy) / bonus token
  int* req_jstar;     // [R] residual position (0: none)
  int* res_list;      // [gamma, R] requests per rejected position (fused residual)
  int* row_list;      // [R * (gamma + 1)] scheduled rows r * (gamma + 1) + j - 1, packed
  int* n_rows;        // [1] number of scheduled rows
  Partial* rt_part;   // [max_mtiles, 128, kMaxDeviceSms] fused-residual partials
  unsigned* row_cnt;  // [R, gamma + 1]   } zeroed together
  unsigned* req_cnt;  // [R]              } at the start
  unsigned* res_cnt;  // [R]              } of every call
  int* res_num;       // [gamma]          }
  unsigned* rt_cnt;   // [max_mtiles]     }
  unsigned* rt_best;  // [R]              }
  int* fallback;      // [R]              }
  unsigned long long* unit_cnt;  // [1] row-pass work counter }
  unsigned long long* done_mask;  // [R] rows finished, bit j-1 }
  unsigned long long* term_mask;  // [R] rows that end the request (reject, mismatch, last) }
};

struct VerifyParams {
  int mode, R, gamma, V, nsplit, rank;
  uint32_t rid_base;
  PhiloxKey key;
  PhiloxRoundKeys rk;  // round keys of `key`
  float inv_target_temp;
  const void* tgt;
  const int32_t* tgt_row_off;
  const int32_t* ell;
  const int32_t* x;
  const float* q_tok;
  const float* lse_q;
  // residual recompute of q at row j*
  const void* U;
  const void* A;
  const void* Ct;
  const void* S;  // RNN head: states [R, gamma, rank] in the factor dtype (null: Markov head)
  const int32_t* x0;
  const float* draft_temp;
  int32_t* accept_len;
  int32_t* out_tok;
  int32_t* n_out;
  float* p_tok;
  float* lse_t;
  float* c_star;  // [R, gamma] sum_v min(p, q) of the verified draft rows (nullable)
  uint32_t* status;
  bool tc_residual;      // residual on the fused tensor-core kernel
  bool row_ring;         // row pass: per-warp bulk-copy rings in dynamic shared memory
  bool skip_dead;        // rows in position order; rows past a request's end are skipped
  int device_sms;
  VerifyScratch ws;
};

// Row-pass work units per row (vocabulary chunks of kRowChunk entries).
inline int verify_nsplit(int R, int gamma, int V) {
  (void)R;
  (void)gamma;
  return std::max(1, (V + kRowChunk - 1) / kRowChunk);
}

inline int residual_nsplit(int R, int V) {
  const int target_ctas = 4 * 152 * 2;
  const int max_split = std::max(1, (V + 1023) / 1024);
  return std::max(1, std::min(max_split, (target_ctas + R - 1) / R));
}

size_t verify_scratch_bytes(int R, int gamma, int V);
VerifyScratch verify_scratch_carve(void* base, int R, int gamma, int V, size_t* counters_offset,
                                   size_t* counters_bytes);

cudaError_t launch_verify(const VerifyParams& p, int tgt_dtype, int logit_dtype, int fac_dtype,
                          cudaStream_t stream);

}  // namespace spec
