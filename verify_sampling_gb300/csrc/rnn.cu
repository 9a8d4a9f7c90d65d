// RNN sequential head: state update between draft positions.
//
// DSpark summary, "第二阶段：轻量顺序头", names a recurrent (RNN) variant of the
// sequential head that keeps a longer dependency than the Markov head's
// previous token, without giving its formula.  The library's reading:
//     s_0 = 0,  s_k = store(tanh(A_k[x_{k-1}, :] + s_{k-1} W_k)),  B_k = s_k C_k,
// so the draft kernels take the bias row from s_k where the Markov head takes
// A_k[x_{k-1}].  The pre-activation is summed in fp32, A_k first and then
// i = 0..r-1 in order; store() rounds to the factor dtype.
//
// One launch per position, between the draft grids of positions k-1 and k.  A
// CTA takes kRnnRows requests, one warp each for the per-request part: on the
// fused tensor-core path the warp first merges the split partials of position
// k-1 (that path's draft grid leaves them unmerged) and writes x, q_tok and
// lse_q there; it stages s_{k-1} (loaded before the merge) and the row
// A_k[x_{k-1}] in shared memory.  The r x r product
// runs with one thread per output column j for all the CTA's requests, so each
// W_k[i][j] is loaded once per CTA (coalesced over j) and used kRnnRows times.
#include "draft.cuh"
#include "fused_tc.cuh"
#include "rnn.cuh"
#include "tc.cuh"

namespace spec {

namespace {

constexpr int kRnnRows = 4;
constexpr int kRnnThreads = 32 * kRnnRows;
constexpr int kBatch = 16;
constexpr size_t kMaxStagedBytes = 64 * 1024;  // W_k staged in shared memory up to this size

__device__ __forceinline__ void store_state(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_state(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// kStaged: W_k (a weight, not written by the previous grid) is copied into
// shared memory before the wait on the previous grid, so its loads overlap
// that grid's tail; otherwise it is read from global memory in batches.
template <typename TF, bool kStaged>
__global__ void __launch_bounds__(kRnnThreads) rnn_state_kernel(RnnStateParams p) {
  __shared__ float s_prev[kRnnRows][kMaxRank];
  __shared__ float s_arow[kRnnRows][kMaxRank];  // A_k[x_{k-1}] of each request
  extern __shared__ uint4 s_w[];  // kStaged: W_k [rank, rank]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kRnnRows, k = p.k, rank = p.rank, G = p.gamma, V = p.V;
  const int m = r0 + warp;
  const TF* S = reinterpret_cast<const TF*>(p.S);
  const TF* Wk = reinterpret_cast<const TF*>(p.W) + (size_t)(k - 1) * rank * rank;
  if (kStaged && k > 1) {
    const uint4* src = reinterpret_cast<const uint4*>(Wk);
    const int n16 = (int)((size_t)rank * rank * sizeof(TF) / 16);
    for (int t = threadIdx.x; t < n16; t += kRnnThreads) s_w[t] = __ldg(src + t);
  }
  // Programmatic launch: wait for the previous draft grid (its tokens or
  // partials and s_{k-1}); then let the next draft grid start its prologue and
  // its first U / C loads (it waits for this grid before reading s_k).
  tc::grid_dep_wait();
  tc::grid_dep_launch();
  if (m < p.R) {
    // s_{k-1} is loaded before the merge, so the two round trips overlap
    constexpr int kPerLane = kMaxRank / 32;
    float sv[kPerLane];
    if (k > 1) {
      const TF* prev = S + ((size_t)m * G + (k - 2)) * rank;
#pragma unroll
      for (int q = 0; q < kPerLane; ++q) sv[q] = lane + 32 * q < rank ? ld_f(prev, (size_t)(lane + 32 * q)) : 0.f;
    }
    int xp;
    if (k == 1) {
      xp = p.x0[m];
    } else if (p.nsplit > 0) {
      Race acc = race_empty();
      const Partial* src = p.part + (size_t)m * p.nsplit;
      for (int s = lane; s < p.nsplit; s += 32) {
        const Partial w = load_partial(src + s);
        acc = fused::race_merge2(acc, Race{w.f0, w.f1, w.f2, w.f3, w.i0});
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc = fused::race_merge2(acc, fused::race_shfl_xor(acc, off));
      if (lane == 0) fused::store_race(p.x, p.q_tok, p.lse_q, (size_t)m * G + (k - 2), acc);
      xp = acc.idx;
    } else {
      xp = p.x[(size_t)m * G + (k - 2)];
    }
    if (xp < 0 || xp >= V) {
      if (lane == 0) set_status(p.status, SPEC_STATUS_BAD_TOKEN);
      xp = 0;
    }
    const TF* arow = reinterpret_cast<const TF*>(p.A) + ((size_t)(k - 1) * V + xp) * rank;
    for (int i = lane; i < rank; i += 32) s_arow[warp][i] = ld_f(arow, (size_t)i);
    if (k > 1) {
#pragma unroll
      for (int q = 0; q < kPerLane; ++q)
        if (lane + 32 * q < rank) s_prev[warp][lane + 32 * q] = sv[q];
    }
  }
  __syncthreads();
  const int nrows = min(kRnnRows, p.R - r0);
  const TF* sW = reinterpret_cast<const TF*>(s_w);
  TF* out = reinterpret_cast<TF*>(p.S);
  for (int j = threadIdx.x; j < rank; j += kRnnThreads) {
    float acc[kRnnRows];
#pragma unroll
    for (int w = 0; w < kRnnRows; ++w) acc[w] = w < nrows ? s_arow[w][j] : 0.f;
    if (kStaged && k > 1) {  // s_0 = 0: the product vanishes at k = 1
      for (int i = 0; i < rank; ++i) {
        const float wij = ld_f(sW, (size_t)i * rank + j);
#pragma unroll
        for (int w = 0; w < kRnnRows; ++w) acc[w] = fmaf(s_prev[w][i], wij, acc[w]);
      }
    } else if (k > 1) {
      // W_k[i][j] in batches of kBatch rows, every load of a batch in flight
      // before its multiply-adds (the order over i stays ascending)
      for (int i0 = 0; i0 < rank; i0 += kBatch) {
        float wv[kBatch];
#pragma unroll
        for (int t = 0; t < kBatch; ++t) wv[t] = i0 + t < rank ? ld_f(Wk, (size_t)(i0 + t) * rank + j) : 0.f;
#pragma unroll
        for (int t = 0; t < kBatch; ++t)
          if (i0 + t < rank) {
#pragma unroll
            for (int w = 0; w < kRnnRows; ++w) acc[w] = fmaf(s_prev[w][i0 + t], wv[t], acc[w]);
          }
      }
    }
#pragma unroll
    for (int w = 0; w < kRnnRows; ++w)
      if (w < nrows) store_state(out + ((size_t)(r0 + w) * G + (k - 1)) * rank + j, tanhf(acc[w]));
  }
}

template <typename TF>
cudaError_t launch_typed(const RnnStateParams& p, bool pdl, cudaStream_t stream) {
  const size_t wbytes = (size_t)p.rank * p.rank * sizeof(TF);
  const bool staged = wbytes <= kMaxStagedBytes && wbytes % 16 == 0 && ((uintptr_t)p.W & 15) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.R + kRnnRows - 1) / kRnnRows));
  cfg.blockDim = dim3(kRnnThreads);
  cfg.dynamicSmemBytes = staged ? wbytes : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (!staged) return cudaLaunchKernelEx(&cfg, rnn_state_kernel<TF, false>, p);
  auto kern = rnn_state_kernel<TF, true>;
  const cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxStagedBytes);
  if (err != cudaSuccess) return err;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_rnn_state(const RnnStateParams& p, bool fac_f32, bool pdl, cudaStream_t stream) {
  return fac_f32 ? launch_typed<float>(p, pdl, stream) : launch_typed<__nv_bfloat16>(p, pdl, stream);
}

}  // namespace spec
