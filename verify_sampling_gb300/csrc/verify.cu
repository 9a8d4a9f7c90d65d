// Verify stage: rejection-sampling verification with residual resampling and
// bonus token, or greedy argmax matching.
//
// History article, "1.1运行机制": accept x_j if p >= q, otherwise with
// probability p/q; after the first rejection the rest of the draft is void.
// DSpark summary, Figure 1: the rejected position is regenerated -- from
// norm(max(0, p - q)), which keeps the output distribution equal to the
// target's ("数学上的美感").  A fully accepted prefix earns one bonus token from
// the next target row (the "1 +" of B in DSpark "2.2").
//
// Kernel 1 (rows): grid (nsplit, gamma + 1, R); CTAs of rows j > l_r + 1 exit
// at once.  Each CTA reduces its vocabulary slice of row (r, j); the last CTA
// of the row finishes the row (lse, accept test, bonus/argmax token); the last
// row of the request resolves the request (first rejection, outputs).
// Kernel 2 (residual): grid (nsplit, R); only requests with a rejection work:
// they recompute q at j* and draw the residual Gumbel-max.
#include "verify.cuh"

#include "draft_tc.cuh"
#include "residual_tc.cuh"

namespace spec {

namespace {

__device__ __forceinline__ int clamp_ell(const VerifyParams& p, int r) {
  int l = p.ell[r];
  if (l < 0 || l > p.gamma) {
    if (threadIdx.x == 0) set_status(p.status, SPEC_STATUS_BAD_ELL);
    l = l < 0 ? 0 : p.gamma;
  }
  return l;
}

__device__ __forceinline__ size_t target_row(const VerifyParams& p, int r, int j) {
  long row = (long)p.tgt_row_off[r] + (j - 1);
  if (row < 0) {
    if (threadIdx.x == 0) set_status(p.status, SPEC_STATUS_BAD_ROW);
    row = 0;
  }
  return (size_t)row;
}

// Resolve request r once all its rows are finished (thread 0 only).
__device__ void resolve_request(const VerifyParams& p, int r, int l) {
  const VerifyScratch& ws = p.ws;
  const int G1 = p.gamma + 1;
  const int32_t* xr = p.x + (size_t)r * p.gamma;
  const int* res = ws.row_res + (size_t)r * G1;
  int jstar = 0;
  for (int j = 1; j <= l; ++j) {
    const int rj = __ldcg(res + (j - 1));
    const bool accepted = (p.mode == SPEC_VERIFY_GREEDY) ? (xr[j - 1] == rj) : (rj != 0);
    if (!accepted) {
      jstar = j;
      break;
    }
  }
  int y;
  if (p.mode == SPEC_VERIFY_GREEDY)
    y = __ldcg(res + (jstar ? jstar - 1 : l));
  else
    y = jstar ? -1 : __ldcg(res + l);  // -1: filled in by the residual kernel
  const int acc = jstar ? jstar - 1 : l;
  int32_t* out = p.out_tok + (size_t)r * G1;
  for (int i = 0; i < G1; ++i) out[i] = (i < acc) ? xr[i] : (i == acc ? y : -1);
  p.accept_len[r] = acc;
  p.n_out[r] = acc + 1;
  ws.req_jstar[r] = (p.mode == SPEC_VERIFY_SAMPLE) ? jstar : 0;
  if (p.tc_residual && p.mode == SPEC_VERIFY_SAMPLE && jstar > 0) {
    const int pos = atomicAdd(ws.res_num + (jstar - 1), 1);
    ws.res_list[(size_t)(jstar - 1) * p.R + pos] = r;
  }
}

}  // namespace

template <typename TT>
__global__ void __launch_bounds__(kVerifyThreads) verify_rows_kernel(VerifyParams p) {
  __shared__ Race red[kVerifyThreads / 32];
  const int r = blockIdx.z, j = blockIdx.y + 1, split = blockIdx.x;
  const int l = clamp_ell(p, r);
  if (j > l + 1) return;
  const int V = p.V, G1 = p.gamma + 1;
  const uint32_t rid = p.rid_base + (uint32_t)r;
  const size_t row = target_row(p, r, j);
  const TT* L = reinterpret_cast<const TT*>(p.tgt) + row * (size_t)V;
  const bool bonus = (j == l + 1);
  const int nvb = (V + 3) / 4;
  const int per = (nvb + p.nsplit - 1) / p.nsplit;
  const int vb_begin = split * per, vb_end = min(nvb, vb_begin + per);
  const float inv_t = p.inv_target_temp;
  Partial* part = p.ws.row_part + ((size_t)r * G1 + (j - 1)) * p.nsplit;

  if (p.mode == SPEC_VERIFY_GREEDY) {
    ArgMax st = argmax_empty();
    for (int vb = vb_begin + threadIdx.x; vb < vb_end; vb += blockDim.x)
#pragma unroll
      for (int lane = 0; lane < 4; ++lane) {
        const int v = vb * 4 + lane;
        if (v < V) argmax_push(st, ld_f(L, (size_t)v), v);
      }
    ArgMax* am_red = reinterpret_cast<ArgMax*>(red);
    st = block_reduce(
        st, am_red,
        [](const ArgMax& a, int off) {
          return ArgMax{__shfl_down_sync(0xffffffffu, a.val, off),
                        __shfl_down_sync(0xffffffffu, a.idx, off)};
        },
        [](const ArgMax& a, const ArgMax& b) { return argmax_merge(a, b); });
    if (threadIdx.x == 0) {
      Partial w{};
      w.f0 = st.val;
      w.i0 = st.idx;
      part[split] = w;
    }
  } else if (bonus) {
    Race st = race_empty();
    const PhiloxKey key = p.key;
    for (int vb = vb_begin + threadIdx.x; vb < vb_end; vb += blockDim.x) {
      const uint4 bits = philox((uint32_t)vb, (uint32_t)j, rid, kPurposeBonus, key);
#pragma unroll
      for (int lane = 0; lane < 4; ++lane) {
        const int v = vb * 4 + lane;
        if (v < V) race_push(st, ld_f(L, (size_t)v) * inv_t, neg_log_uniform(word_of(bits, lane)), v);
      }
    }
    st = block_reduce(
        st, red, [](const Race& a, int off) { return race_shfl_down(a, off); },
        [](const Race& a, const Race& b) { return race_merge(a, b); });
    if (threadIdx.x == 0) {
      Partial w{};
      w.f0 = st.m;
      w.f1 = st.s;
      w.f2 = st.be;
      w.f3 = st.bE;
      w.i0 = st.idx;
      part[split] = w;
    }
  } else {
    Soft st = soft_empty();
    for (int vb = vb_begin + threadIdx.x; vb < vb_end; vb += blockDim.x)
#pragma unroll
      for (int lane = 0; lane < 4; ++lane) {
        const int v = vb * 4 + lane;
        if (v < V) soft_push(st, ld_f(L, (size_t)v) * inv_t);
      }
    Soft* s_red = reinterpret_cast<Soft*>(red);
    st = block_reduce(
        st, s_red,
        [](const Soft& a, int off) {
          return Soft{__shfl_down_sync(0xffffffffu, a.m, off), __shfl_down_sync(0xffffffffu, a.s, off)};
        },
        [](const Soft& a, const Soft& b) { return soft_merge(a, b); });
    if (threadIdx.x == 0) {
      Partial w{};
      w.f0 = st.m;
      w.f1 = st.s;
      part[split] = w;
    }
  }

  const size_t rj = (size_t)r * G1 + (j - 1);
  if (!last_block_arrives(p.ws.row_cnt + rj, (unsigned)p.nsplit)) return;

  // Last CTA of row (r, j): finish the row.
  __shared__ bool request_done;
  if (threadIdx.x == 0) {
    if (p.mode == SPEC_VERIFY_GREEDY) {
      ArgMax acc = argmax_empty();
      for (int s = 0; s < p.nsplit; ++s) {
        const Partial w = load_partial(part + s);
        acc = argmax_merge(acc, ArgMax{w.f0, w.i0});
      }
      p.ws.row_res[rj] = acc.idx;
    } else {
      float m, s;
      int token = 0;
      if (bonus) {
        Race acc = race_empty();
        for (int t = 0; t < p.nsplit; ++t) {
          const Partial w = load_partial(part + t);
          acc = race_merge(acc, Race{w.f0, w.f1, w.f2, w.f3, w.i0});
        }
        m = acc.m;
        s = acc.s;
        token = acc.idx;
      } else {
        Soft acc = soft_empty();
        for (int t = 0; t < p.nsplit; ++t) {
          const Partial w = load_partial(part + t);
          acc = soft_merge(acc, Soft{w.f0, w.f1});
        }
        m = acc.m;
        s = acc.s;
        int xj = p.x[(size_t)r * p.gamma + (j - 1)];
        if (xj < 0 || xj >= V) {
          set_status(p.status, SPEC_STATUS_BAD_TOKEN);
          xj = 0;
        }
        // p(x_j) = exp(L[x_j]/T - m) / s; accept iff u < p / q (q <= 0: accept).
        const float px = expf(ld_f(L, (size_t)xj) * inv_t - m) / s;
        const float q = p.q_tok[(size_t)r * p.gamma + (j - 1)];
        const float u = uniform_from_word(philox(0u, (uint32_t)j, rid, kPurposeAccept, p.key).x);
        token = (q <= 0.f || u < px / q) ? 1 : 0;
        if (p.p_tok) p.p_tok[(size_t)r * p.gamma + (j - 1)] = px;
      }
      p.ws.row_m[rj] = m;
      p.ws.row_s[rj] = s;
      p.ws.row_res[rj] = token;
      if (p.lse_t) p.lse_t[rj] = m + logf(s);
    }
    __threadfence();
    const unsigned prev = atomicAdd(p.ws.req_cnt + r, 1u);
    request_done = (prev == (unsigned)l);
    if (request_done) {
      p.ws.req_cnt[r] = 0u;
      __threadfence();
      resolve_request(p, r, l);
    }
  }
}

// Generic residual (any dtype, FFMA bias).  `gate[r]` is the rejected position
// of request r (0: nothing to do): every rejected request when the fused
// kernel is not used, else only those whose fused residual was zero everywhere.
template <typename TT, typename TL, typename TF>
__global__ void __launch_bounds__(kVerifyThreads) residual_kernel(VerifyParams p, const int* gate) {
  __shared__ float arow[256];
  __shared__ WRace red[kVerifyThreads / 32];
  const int r = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int jstar = gate[r];
  if (jstar == 0) return;
  const int V = p.V, G1 = p.gamma + 1, rank = p.rank;
  const uint32_t rid = p.rid_base + (uint32_t)r;
  const size_t rj = (size_t)r * G1 + (jstar - 1);
  const float m_t = p.ws.row_m[rj], s_t = p.ws.row_s[rj];
  const float inv_s_t = 1.0f / s_t;
  const TT* L = reinterpret_cast<const TT*>(p.tgt) + target_row(p, r, jstar) * (size_t)V;
  const int k = jstar;
  int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * p.gamma + (k - 2)];
  if (x_prev < 0 || x_prev >= V) x_prev = 0;
  const TF* A = reinterpret_cast<const TF*>(p.A) + (size_t)(k - 1) * V * rank;
  const TF* Ct = reinterpret_cast<const TF*>(p.Ct) + (size_t)(k - 1) * V * rank;
  for (int i = threadIdx.x; i < rank; i += blockDim.x) arow[i] = ld_f(A, (size_t)x_prev * rank + i);
  __syncthreads();
  const TL* U = reinterpret_cast<const TL*>(p.U) + ((size_t)r * p.gamma + (k - 1)) * V;
  const float inv_tq = 1.0f / p.draft_temp[k - 1];
  const float lse_q = p.lse_q[(size_t)r * p.gamma + (k - 1)];
  const float inv_tt = p.inv_target_temp;
  const int nvb = (V + 3) / 4;
  const int per = (nvb + nsplit - 1) / nsplit;
  const int vb_begin = split * per, vb_end = min(nvb, vb_begin + per);

  WRace res = wrace_empty(), pr = wrace_empty();
  for (int vb = vb_begin + threadIdx.x; vb < vb_end; vb += blockDim.x) {
    const uint4 bits = philox((uint32_t)vb, (uint32_t)jstar, rid, kPurposeResidual, p.key);
#pragma unroll
    for (int lane = 0; lane < 4; ++lane) {
      const int v = vb * 4 + lane;
      if (v < V) {
        float bias = 0.f;
        for (int i = 0; i < rank; ++i) bias = fmaf(arow[i], ld_f(Ct, (size_t)v * rank + i), bias);
        const float zq = (ld_f(U, (size_t)v) + bias) * inv_tq;
        const float et = expf(ld_f(L, (size_t)v) * inv_tt - m_t);
        const float pv = et * inv_s_t;
        const float qv = expf(zq - lse_q);
        const float E = neg_log_uniform(word_of(bits, lane));
        wrace_push(res, pv - qv, E, v);
        wrace_push(pr, et, E, v);
      }
    }
  }
  auto shfl = [](const WRace& a, int off) {
    return WRace{__shfl_down_sync(0xffffffffu, a.bw, off), __shfl_down_sync(0xffffffffu, a.bE, off),
                 __shfl_down_sync(0xffffffffu, a.idx, off)};
  };
  auto merge = [](const WRace& a, const WRace& b) { return wrace_merge(a, b); };
  res = block_reduce(res, red, shfl, merge);
  __syncthreads();
  pr = block_reduce(pr, red, shfl, merge);
  Partial* part = p.ws.res_part + (size_t)r * nsplit;
  if (threadIdx.x == 0) {
    Partial w{};
    w.f0 = res.bw;
    w.f1 = res.bE;
    w.i0 = res.idx;
    w.f4 = pr.bw;
    w.f5 = pr.bE;
    w.i1 = pr.idx;
    part[split] = w;
  }
  if (!last_block_arrives(p.ws.res_cnt + r, (unsigned)nsplit)) return;
  if (threadIdx.x == 0) {
    WRace a = wrace_empty(), b = wrace_empty();
    for (int s = 0; s < nsplit; ++s) {
      const Partial w = load_partial(part + s);
      a = wrace_merge(a, WRace{w.f0, w.f1, w.i0});
      b = wrace_merge(b, WRace{w.f4, w.f5, w.i1});
    }
    const int y = (a.idx >= 0) ? a.idx : b.idx;
    p.out_tok[(size_t)r * G1 + (jstar - 1)] = y;
  }
}

// ------------------------------------------------------------- scratch ----
static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Scratch layout: arrays that need no initialisation first, then the
// counters and flags that every call zeroes in one memset.
enum { kRowPart, kResPart, kRowM, kRowS, kRowRes, kReqJstar, kResList, kRtPart,
       kRowCnt, kReqCnt, kResCnt, kResNum, kRtCnt, kRtBest, kFallback, kLayoutN };

static size_t layout(int R, int gamma, int V, size_t off[kLayoutN]) {
  const size_t rows = (size_t)R * (gamma + 1);
  const size_t ns = (size_t)verify_nsplit(R, gamma, V), nr = (size_t)residual_nsplit(R, V);
  const size_t mt = (size_t)resid_tc_max_mtiles(R, gamma);
  const size_t sizes[kLayoutN] = {rows * ns * sizeof(Partial), (size_t)R * nr * sizeof(Partial),
                                  rows * sizeof(float), rows * sizeof(float), rows * sizeof(int),
                                  (size_t)R * sizeof(int), (size_t)gamma * R * sizeof(int),
                                  mt * 128 * kMaxDeviceSms * sizeof(Partial),
                                  rows * sizeof(unsigned), (size_t)R * sizeof(unsigned),
                                  (size_t)R * sizeof(unsigned), (size_t)gamma * sizeof(int),
                                  mt * sizeof(unsigned), (size_t)R * sizeof(unsigned),
                                  (size_t)R * sizeof(int)};
  size_t o = 0;
  for (int i = 0; i < kLayoutN; ++i) {
    off[i] = o;
    o = (i < kRowCnt) ? align_up(o + sizes[i]) : o + sizes[i];
  }
  return align_up(o);
}

size_t verify_scratch_bytes(int R, int gamma, int V) {
  size_t off[kLayoutN];
  return layout(R, gamma, V, off);
}

VerifyScratch verify_scratch_carve(void* base, int R, int gamma, int V, size_t* counters_offset,
                                   size_t* counters_bytes) {
  size_t off[kLayoutN];
  const size_t total = layout(R, gamma, V, off);
  char* b = static_cast<char*>(base);
  VerifyScratch s;
  s.row_part = reinterpret_cast<Partial*>(b + off[kRowPart]);
  s.res_part = reinterpret_cast<Partial*>(b + off[kResPart]);
  s.row_m = reinterpret_cast<float*>(b + off[kRowM]);
  s.row_s = reinterpret_cast<float*>(b + off[kRowS]);
  s.row_res = reinterpret_cast<int*>(b + off[kRowRes]);
  s.req_jstar = reinterpret_cast<int*>(b + off[kReqJstar]);
  s.res_list = reinterpret_cast<int*>(b + off[kResList]);
  s.rt_part = reinterpret_cast<Partial*>(b + off[kRtPart]);
  s.row_cnt = reinterpret_cast<unsigned*>(b + off[kRowCnt]);
  s.req_cnt = reinterpret_cast<unsigned*>(b + off[kReqCnt]);
  s.res_cnt = reinterpret_cast<unsigned*>(b + off[kResCnt]);
  s.res_num = reinterpret_cast<int*>(b + off[kResNum]);
  s.rt_cnt = reinterpret_cast<unsigned*>(b + off[kRtCnt]);
  s.rt_best = reinterpret_cast<unsigned*>(b + off[kRtBest]);
  s.fallback = reinterpret_cast<int*>(b + off[kFallback]);
  *counters_offset = off[kRowCnt];
  *counters_bytes = total - off[kRowCnt];
  return s;
}

// ------------------------------------------------------------ launchers ---
template <typename TT, typename TL, typename TF>
static cudaError_t launch_typed(const VerifyParams& p, int tgt_dtype, int logit_dtype,
                                cudaStream_t stream) {
  const dim3 g1((unsigned)p.nsplit, (unsigned)(p.gamma + 1), (unsigned)p.R);
  verify_rows_kernel<TT><<<g1, kVerifyThreads, 0, stream>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || p.mode == SPEC_VERIFY_GREEDY) return err;
  const dim3 g2((unsigned)residual_nsplit(p.R, p.V), (unsigned)p.R);
  if (!p.tc_residual) {
    residual_kernel<TT, TL, TF><<<g2, kVerifyThreads, 0, stream>>>(p, p.ws.req_jstar);
    return cudaGetLastError();
  }
  ResidTCParams t{};
  t.R = p.R;
  t.gamma = p.gamma;
  t.V = p.V;
  t.rank = p.rank;
  t.ntiles = (p.V + 63) / 64;
  t.max_mtiles = resid_tc_max_mtiles(p.R, p.gamma);
  t.rid_base = p.rid_base;
  t.key = p.key;
  t.inv_target_temp = p.inv_target_temp;
  t.x0 = p.x0;
  t.x = p.x;
  t.draft_temp = p.draft_temp;
  t.A = p.A;
  t.lse_q = p.lse_q;
  t.tgt_row_off = p.tgt_row_off;
  t.row_m = p.ws.row_m;
  t.row_s = p.ws.row_s;
  t.res_cnt = p.ws.res_num;
  t.res_list = p.ws.res_list;
  t.partials = p.ws.rt_part;
  t.counters = p.ws.rt_cnt;
  t.row_best = p.ws.rt_best;
  t.out_tok = p.out_tok;
  t.fallback = p.ws.fallback;
  t.status = p.status;
  const int grid = std::max(p.device_sms, t.max_mtiles);
  err = launch_resid_tc(t, tgt_dtype, logit_dtype, p.tgt, p.U, p.Ct, grid, stream);
  if (err != cudaSuccess) return err;
  // requests whose residual was zero everywhere (fp32 rounding only): the
  // generic kernel redoes them, sampling from p if its residual is zero too
  residual_kernel<TT, TL, TF><<<g2, kVerifyThreads, 0, stream>>>(p, p.ws.fallback);
  return cudaGetLastError();
}

template <typename TT>
static cudaError_t launch_tgt(const VerifyParams& p, int tgt_dtype, int logit_dtype, int fac_dtype,
                              cudaStream_t stream) {
  if (logit_dtype == SPEC_F32 && fac_dtype == SPEC_F32)
    return launch_typed<TT, float, float>(p, tgt_dtype, logit_dtype, stream);
  if (logit_dtype == SPEC_F32)
    return launch_typed<TT, float, __nv_bfloat16>(p, tgt_dtype, logit_dtype, stream);
  if (fac_dtype == SPEC_F32)
    return launch_typed<TT, __nv_bfloat16, float>(p, tgt_dtype, logit_dtype, stream);
  return launch_typed<TT, __nv_bfloat16, __nv_bfloat16>(p, tgt_dtype, logit_dtype, stream);
}

cudaError_t launch_verify(const VerifyParams& p, int tgt_dtype, int logit_dtype, int fac_dtype,
                          cudaStream_t stream) {
  if (tgt_dtype == SPEC_F32) return launch_tgt<float>(p, tgt_dtype, logit_dtype, fac_dtype, stream);
  return launch_tgt<__nv_bfloat16>(p, tgt_dtype, logit_dtype, fac_dtype, stream);
}

}  // namespace spec
