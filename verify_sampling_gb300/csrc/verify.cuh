// Parameters and launchers of the verify-stage kernels (internal header).
#pragma once

#include <algorithm>

#include "common.cuh"

namespace spec {

constexpr int kVerifyThreads = 256;

// Per-call scratch carved out of the caller's workspace.
struct VerifyScratch {
  Partial* row_part;  // [R, gamma + 1, nsplit]
  Partial* res_part;  // [R, nsplit] (two races per record)
  float* row_m;       // [R, gamma + 1] softmax max of L / T_t
  float* row_s;       // [R, gamma + 1] softmax sum
  int* row_res;       // [R, gamma + 1] accept bit (sample) / argmax (greedy) / bonus token
  int* req_jstar;     // [R] residual position (0: none)
  int* res_list;      // [gamma, R] requests per rejected position (fused residual)
  Partial* rt_part;   // [max_mtiles, 128, kMaxDeviceSms] fused-residual partials
  unsigned* row_cnt;  // [R, gamma + 1]   } zeroed together
  unsigned* req_cnt;  // [R]              } at the start
  unsigned* res_cnt;  // [R]              } of every call
  int* res_num;       // [gamma]          }
  unsigned* rt_cnt;   // [max_mtiles]     }
  unsigned* rt_best;  // [R]              }
  int* fallback;      // [R]              }
};

struct VerifyParams {
  int mode, R, gamma, V, nsplit, rank;
  uint32_t rid_base;
  PhiloxKey key;
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
  const int32_t* x0;
  const float* draft_temp;
  int32_t* accept_len;
  int32_t* out_tok;
  int32_t* n_out;
  float* p_tok;
  float* lse_t;
  uint32_t* status;
  bool tc_residual;      // residual on the fused tensor-core kernel
  int device_sms;
  VerifyScratch ws;
};

inline int verify_nsplit(int R, int gamma, int V) {
  const long rows = (long)R * (gamma + 1);
  const int target_ctas = 4 * 152 * 2;
  const int max_split = std::max(1, (V + 2047) / 2048);
  return (int)std::max<long>(1, std::min<long>(max_split, (target_ctas + rows - 1) / rows));
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
