// Draft stage kernels: sequential-head sampling step, full-distribution output
// and the confidence head with survival products.
//
// DSpark summary, "第二阶段：轻量顺序头": P_k = softmax((U_k + B_k(x_{k-1})) / T_k)
// with the low-rank bias B_k(x) = A_k[x, :] C_k (history article, "杀招一");
// DSpark summary, "2.1 置信度头": c_k = sigmoid(w . [h_k ; W1[x_{k-1}]] / tau_k);
// history article, "杀招二": a_j = prod_{i<=j} c_i.
#include <type_traits>

#include "draft.cuh"
#include "rnn.cuh"

namespace spec {

// ------------------------------------------------------------ draft step --
// One launch per position k.  Grid (nsplit, R): CTA (s, r) streams vocabulary
// blocks [vb_begin, vb_end) of row (r, k), 4 entries per Philox block, keeps a
// Gumbel race + online softmax per thread, reduces it over the CTA and publishes
// a partial; the last CTA of the row merges the partials into x_k, q_tok, lse.
// The bias row is A_k[x_{k-1}] (Markov head) or the state s_k (RNN head, written
// by the state kernel launched just before).
template <typename TL, typename TF>
__global__ void __launch_bounds__(kDraftThreads)
    draft_step_kernel(DraftStepParams p) {
  __shared__ float arow[kMaxRank];
  __shared__ Race red[kDraftThreads / 32];
  const int r = blockIdx.y, split = blockIdx.x;
  const int k = p.k;  // 1-based position
  const int V = p.V, rank = p.rank, gamma = p.gamma;
  const uint32_t rid = p.rid_base + (uint32_t)r;

  int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * gamma + (k - 2)];
  if (x_prev < 0 || x_prev >= V) {
    if (threadIdx.x == 0) set_status(p.status, SPEC_STATUS_BAD_TOKEN);
    x_prev = 0;
  }
  const TF* brow = bias_row<TF>(p.A, p.S, V, rank, gamma, k, r, x_prev);
  const TF* Ct = reinterpret_cast<const TF*>(p.Ct) + (size_t)(k - 1) * V * rank;
  for (int i = threadIdx.x; i < rank; i += blockDim.x) arow[i] = ld_f(brow, (size_t)i);
  __syncthreads();

  const TL* U = reinterpret_cast<const TL*>(p.U) + ((size_t)r * gamma + (k - 1)) * V;
  const float inv_t = 1.0f / p.draft_temp[k - 1];
  const int nvb = (V + 3) / 4;
  const int per = (nvb + p.nsplit - 1) / p.nsplit;
  const int vb_begin = split * per, vb_end = min(nvb, vb_begin + per);
  const PhiloxKey key = p.key;

  Race st = race_empty();
  for (int vb = vb_begin + threadIdx.x; vb < vb_end; vb += blockDim.x) {
    const uint4 bits = philox((uint32_t)vb, (uint32_t)k, rid, kPurposeDraft, key);
#pragma unroll
    for (int lane = 0; lane < 4; ++lane) {
      const int v = vb * 4 + lane;
      if (v < V) {
        float bias = 0.f;
        const size_t crow = (size_t)v * rank;
        for (int i = 0; i < rank; ++i) bias = fmaf(arow[i], ld_f(Ct, crow + i), bias);
        const float z = (ld_f(U, (size_t)v) + bias) * inv_t;
        race_push(st, z, neg_log_uniform(word_of(bits, lane)), v);
      }
    }
  }
  st = block_reduce(
      st, red, [](const Race& a, int off) { return race_shfl_down(a, off); },
      [](const Race& a, const Race& b) { return race_merge(a, b); });

  Partial* part = p.partials + (size_t)r * p.nsplit;
  if (threadIdx.x == 0) {
    Partial w;
    w.f0 = st.m;
    w.f1 = st.s;
    w.f2 = st.be;
    w.f3 = st.bE;
    w.i0 = st.idx;
    part[split] = w;
  }
  if (!last_block_arrives(p.counters + r, (unsigned)p.nsplit)) return;

  // Last CTA of the row: merge all partials (thread 0; nsplit is small).
  if (threadIdx.x == 0) {
    Race acc = race_empty();
    for (int s = 0; s < p.nsplit; ++s) {
      const Partial w = load_partial(part + s);
      Race o{w.f0, w.f1, w.f2, w.f3, w.i0};
      acc = race_merge(acc, o);
    }
    const size_t o = (size_t)r * gamma + (k - 1);
    p.x[o] = acc.idx;
    p.q_tok[o] = acc.be / acc.s;
    p.lse_q[o] = acc.m + logf(acc.s);
  }
}

// Full draft distributions P[r, k, v] = exp(z_v - lse) (optional output).
template <typename TL, typename TF>
__global__ void __launch_bounds__(256) draft_probs_kernel(DraftStepParams p) {
  __shared__ float arow[kMaxRank];
  const int r = blockIdx.z, k = blockIdx.y + 1;
  const int V = p.V, rank = p.rank, gamma = p.gamma;
  int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * gamma + (k - 2)];
  if (x_prev < 0 || x_prev >= V) x_prev = 0;
  const TF* brow = bias_row<TF>(p.A, p.S, V, rank, gamma, k, r, x_prev);
  const TF* Ct = reinterpret_cast<const TF*>(p.Ct) + (size_t)(k - 1) * V * rank;
  for (int i = threadIdx.x; i < rank; i += blockDim.x) arow[i] = ld_f(brow, (size_t)i);
  __syncthreads();
  const size_t o = (size_t)r * gamma + (k - 1);
  const TL* U = reinterpret_cast<const TL*>(p.U) + o * V;
  const float inv_t = 1.0f / p.draft_temp[k - 1];
  const float lse = p.lse_q[o];
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
    float bias = 0.f;
    for (int i = 0; i < rank; ++i) bias = fmaf(arow[i], ld_f(Ct, (size_t)v * rank + i), bias);
    const float z = (ld_f(U, (size_t)v) + bias) * inv_t;
    p.P_out[o * V + v] = expf(z - lse);
  }
}

// ------------------------------------------------------------ confidence --
// Lane's share of sum_i a[i] * b[i] over n entries (n a multiple of 16 bytes,
// both rows 16-byte aligned), added to s.
__device__ __forceinline__ float dot16(const float* a, const float* b, int n, int lane, float s) {
  for (int i = 4 * lane; i < n; i += 128) {
    const float4 x = *reinterpret_cast<const float4*>(a + i);
    const float4 y = *reinterpret_cast<const float4*>(b + i);
    s = fmaf(x.x, y.x, s);
    s = fmaf(x.y, y.y, s);
    s = fmaf(x.z, y.z, s);
    s = fmaf(x.w, y.w, s);
  }
  return s;
}
__device__ __forceinline__ float dot16(const __nv_bfloat16* a, const __nv_bfloat16* b, int n, int lane,
                                       float s) {
  for (int i = 8 * lane; i < n; i += 256) {
    const uint4 x = *reinterpret_cast<const uint4*>(a + i);
    const uint4 y = *reinterpret_cast<const uint4*>(b + i);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // bf16 -> fp32 is exact: the bits shifted into place
      s = fmaf(__uint_as_float(xs[j] << 16), __uint_as_float(ys[j] << 16), s);
      s = fmaf(__uint_as_float(xs[j] & 0xffff0000u), __uint_as_float(ys[j] & 0xffff0000u), s);
    }
  }
  return s;
}

// One CTA per request, one warp per position (looping when gamma > warps).
template <typename TC>
__global__ void __launch_bounds__(kConfThreads) confidence_kernel(ConfParams p) {
  __shared__ float cs[kMaxGamma];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int gamma = p.gamma, d = p.d, e = p.e;
  const TC* w = reinterpret_cast<const TC*>(p.w);
  for (int k = 1 + warp; k <= gamma; k += nwarps) {
    int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * gamma + (k - 2)];
    if (x_prev < 0 || x_prev >= p.V) {
      if (lane == 0) set_status(p.status, SPEC_STATUS_BAD_TOKEN);
      x_prev = 0;
    }
    const TC* h = reinterpret_cast<const TC*>(p.h) + ((size_t)r * gamma + (k - 1)) * d;
    const TC* emb = reinterpret_cast<const TC*>(p.W1) + (size_t)x_prev * e;
    float s = 0.f;
    if (p.vec) {  // 16-byte loads: eight bf16 or four fp32 per lane and step
      s = dot16(w, h, d, lane, s);
      s = dot16(w + d, emb, e, lane, s);
    } else {
      for (int i = lane; i < d; i += 32) s = fmaf(ld_f(w, i), ld_f(h, i), s);
      for (int i = lane; i < e; i += 32) s = fmaf(ld_f(w, (size_t)d + i), ld_f(emb, i), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_down_sync(0xffffffffu, s, off);
    if (lane == 0) cs[k - 1] = 1.0f / (1.0f + expf(-s / p.sts_temp[k - 1]));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float surv = 1.0f;
    for (int k = 0; k < gamma; ++k) {
      surv *= cs[k];
      p.c[(size_t)r * gamma + k] = cs[k];
      p.a[(size_t)r * gamma + k] = surv;
    }
  }
}

// ------------------------------------------------------------- launchers --
static RnnStateParams rnn_params(const DraftStepParams& p, int k) {
  RnnStateParams q{};
  q.R = p.R;
  q.gamma = p.gamma;
  q.V = p.V;
  q.rank = p.rank;
  q.k = k;
  q.x0 = p.x0;
  q.x = p.x;
  q.A = p.A;
  q.W = p.W;
  q.S = p.S;
  q.status = p.status;
  return q;
}

template <typename TL, typename TF>
static cudaError_t launch_draft_typed(const DraftStepParams& base, bool want_probs,
                                      bool probs_only, cudaStream_t stream) {
  DraftStepParams p = base;
  const dim3 grid((unsigned)p.nsplit, (unsigned)p.R);
  for (int k = 1; k <= p.gamma && !probs_only; ++k) {
    p.k = k;
    if (p.S) {  // RNN head: s_k from x_{k-1} (final: the previous step merged it)
      cudaError_t err = launch_rnn_state(rnn_params(p, k), std::is_same<TF, float>::value, false, stream);
      if (err != cudaSuccess) return err;
    }
    draft_step_kernel<TL, TF><<<grid, kDraftThreads, 0, stream>>>(p);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (want_probs) {
    const unsigned bx = (unsigned)std::min(64, (p.V + 255) / 256);
    draft_probs_kernel<TL, TF><<<dim3(bx, p.gamma, p.R), 256, 0, stream>>>(p);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_draft_steps(const DraftStepParams& p, int logit_dtype, int fac_dtype,
                               bool want_probs, cudaStream_t stream, bool probs_only) {
  if (logit_dtype == SPEC_F32 && fac_dtype == SPEC_F32)
    return launch_draft_typed<float, float>(p, want_probs, probs_only, stream);
  if (logit_dtype == SPEC_F32 && fac_dtype == SPEC_BF16)
    return launch_draft_typed<float, __nv_bfloat16>(p, want_probs, probs_only, stream);
  if (logit_dtype == SPEC_BF16 && fac_dtype == SPEC_F32)
    return launch_draft_typed<__nv_bfloat16, float>(p, want_probs, probs_only, stream);
  return launch_draft_typed<__nv_bfloat16, __nv_bfloat16>(p, want_probs, probs_only, stream);
}

cudaError_t launch_confidence(const ConfParams& base, int conf_dtype, cudaStream_t stream) {
  ConfParams p = base;
  const size_t es = conf_dtype == SPEC_F32 ? 4 : 2;
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  p.vec = al16(p.h) && al16(p.W1) && al16(p.w) && ((size_t)p.d * es) % 16 == 0 &&
          ((size_t)p.e * es) % 16 == 0;
  const int threads = std::min(kConfThreads, 32 * std::max(1, p.gamma));
  if (conf_dtype == SPEC_F32)
    confidence_kernel<float><<<p.R, threads, 0, stream>>>(p);
  else
    confidence_kernel<__nv_bfloat16><<<p.R, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
