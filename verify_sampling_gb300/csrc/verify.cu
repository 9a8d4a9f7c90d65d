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
// Kernel 1 (rows): persistent CTAs over (request, vocabulary chunk) units,
// reading only the scheduled rows; the last chunk of a row finishes the row
// (lse, accept test, bonus/argmax token); the last row of the request resolves
// the request (first rejection, outputs).
// Kernel 2 (residual): grid (nsplit, R); only requests with a rejection work:
// they recompute q at j* and draw the residual Gumbel-max.
// Optional diagnostic (c_star): DSpark summary, "2.1 置信度头" -- the confidence
// head's target c* = 1 - TV(p, q) = sum_v min(p_v, q_v) of every verified
// draft row, from a plan of the rows per position and the tensor-core residual
// pass in its summing form (or a generic FFMA kernel).
#include "verify.cuh"

#include "draft_tc.cuh"
#include "fused_tc.cuh"
#include "residual_tc.cuh"

namespace spec {

namespace {

__device__ __forceinline__ int clamp_ell(const VerifyParams& p, int r) {
  int l = p.ell[r];
  if (l < 0 || l > p.gamma) {
    if ((threadIdx.x & 31) == 0) set_status(p.status, SPEC_STATUS_BAD_ELL);
    l = l < 0 ? 0 : p.gamma;
  }
  return l;
}

__device__ __forceinline__ size_t target_row(const VerifyParams& p, int r, int j) {
  long row = (long)p.tgt_row_off[r] + (j - 1);
  if (row < 0) {
    if ((threadIdx.x & 31) == 0) set_status(p.status, SPEC_STATUS_BAD_ROW);
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

// ----------------------------------------------------------- row pass ----
// Warp-level persistent work: a unit is one chunk (kRowChunk entries) of one
// row (r, j); units run over (r, j, chunk) with the chunk fastest.  A warp
// claims 32 consecutive units with one atomic, keeps those of scheduled rows
// (j <= l_r + 1; a ballot over the claimed range) and streams each in batches
// of 32 entries per lane (four groups of 8 consecutive entries, 16-byte
// streaming loads); the other warps of the SM keep their loads in flight
// meanwhile.  No block-wide barrier is used.  Log2 units: e = 2^(L log2e / T
// - ref), the reference fixed at the lane's first batch maximum (moved if a
// later batch overflows the sum).
//   j <= l_r (sample): softmax partial;
//   j == l_r + 1 (sample): softmax plus the bonus Gumbel race (purpose 3): each
//     lane seeds its race with its first batch maximum, the warp shares the best
//     seed, and only elements with 1 - u <= e * bE / be take the logarithm;
//   greedy: argmax (lowest index on ties).
// The warp that completes a row's last chunk merges the row's partials and
// finishes the row; the one that finishes a request's last row resolves it.

constexpr int kBatch = 32 * 32;  // entries per warp batch
constexpr int kRingStages = 3;   // bulk-copy batches in flight per warp

// Eight consecutive entries from v0 (a multiple of 8) as floats; entries at or
// past V read as -inf.  `vec`: whole 16-byte pieces inside the row may be
// loaded at once (16-byte aligned rows).
__device__ __forceinline__ void load8(const float* L, long v0, long V, bool vec, float (&x)[8]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long b = v0 + 4 * h;
    if (vec && b + 4 <= V) {
      const float4 f = __ldcs(reinterpret_cast<const float4*>(L + b));
      x[4 * h] = f.x;
      x[4 * h + 1] = f.y;
      x[4 * h + 2] = f.z;
      x[4 * h + 3] = f.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) x[4 * h + i] = (b + i < V) ? __ldcs(L + b + i) : -CUDART_INF_F;
    }
  }
}
__device__ __forceinline__ void load8(const __nv_bfloat16* L, long v0, long V, bool vec, float (&x)[8]) {
  if (vec && v0 + 8 <= V) {
    const uint4 q = __ldcs(reinterpret_cast<const uint4*>(L + v0));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[2 * h] = __uint_as_float(w[h] << 16);
      x[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (v0 + i < V) ? __bfloat162float(L[v0 + i]) : -CUDART_INF_F;
  }
}

// The same from a shared-memory batch: entry `off` (a multiple of 8) of a
// stage holding n valid entries; entries past n read as -inf.
template <typename TT>
__device__ __forceinline__ void load8s_t(const unsigned char* sx, int off, int n, float (&x)[8]);
template <>
__device__ __forceinline__ void load8s_t<float>(const unsigned char* sx, int off, int n, float (&x)[8]) {
  const float* f = reinterpret_cast<const float*>(sx) + off;
  if (off + 8 <= n) {
    const float4 a = *reinterpret_cast<const float4*>(f), b = *reinterpret_cast<const float4*>(f + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (off + i < n) ? f[i] : -CUDART_INF_F;
  }
}
template <>
__device__ __forceinline__ void load8s_t<__nv_bfloat16>(const unsigned char* sx, int off, int n, float (&x)[8]) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(sx) + off;
  if (off + 8 <= n) {
    const uint4 q = *reinterpret_cast<const uint4*>(h);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (off + i < n) ? __uint_as_float((uint32_t)h[i] << 16) : -CUDART_INF_F;
  }
}

// Merge of row partials in log2 units: the softmax parts always, the race
// parts (idx < 0: none) by the race rule.
__device__ __forceinline__ Race row_merge(const Race& a, const Race& b) {
  if (!(b.m > -CUDART_INF_F)) return a;
  if (!(a.m > -CUDART_INF_F)) return b;
  const float m = fmaxf(a.m, b.m);
  const float sa = tc::ex2(a.m - m), sb = tc::ex2(b.m - m);
  Race o;
  o.m = m;
  o.s = a.s * sa + b.s * sb;
  const float ea = a.be * sa, eb = b.be * sb;
  if (race_beats(ea, a.bE, a.idx, eb, b.bE, b.idx)) {
    o.be = ea;
    o.bE = a.bE;
    o.idx = a.idx;
  } else {
    o.be = eb;
    o.bE = b.bE;
    o.idx = b.idx;
  }
  return o;
}
__device__ __forceinline__ Race row_shfl_xor(const Race& st, int mask) {
  return Race{__shfl_xor_sync(0xffffffffu, st.m, mask), __shfl_xor_sync(0xffffffffu, st.s, mask),
              __shfl_xor_sync(0xffffffffu, st.be, mask), __shfl_xor_sync(0xffffffffu, st.bE, mask),
              __shfl_xor_sync(0xffffffffu, st.idx, mask)};
}
__device__ __forceinline__ ArgMax argmax_shfl_xor(const ArgMax& a, int mask) {
  return ArgMax{__shfl_xor_sync(0xffffffffu, a.val, mask), __shfl_xor_sync(0xffffffffu, a.idx, mask)};
}

// Finish row (r, j) from its merged state (lane 0 of the finishing warp).
__device__ void finish_row(const VerifyParams& p, int r, int j, int l, const Race& acc, float ks,
                           const void* Lrow, bool bf16, bool bonus) {
  const size_t rj = (size_t)r * (p.gamma + 1) + (j - 1);
  int token = 0;
  if (bonus) {
    token = acc.idx;
  } else {
    int xj = p.x[(size_t)r * p.gamma + (j - 1)];
    if (xj < 0 || xj >= p.V) {
      set_status(p.status, SPEC_STATUS_BAD_TOKEN);
      xj = 0;
    }
    const float lx = bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(Lrow)[xj])
                          : reinterpret_cast<const float*>(Lrow)[xj];
    // p(x_j) = 2^(L[x_j] log2e / T - m) / s; accept iff u < p / q (q <= 0: accept)
    const float px = tc::ex2(fmaf(lx, ks, -acc.m)) / acc.s;
    const float q = p.q_tok[(size_t)r * p.gamma + (j - 1)];
    const float u = uniform_from_word(philox(0u, (uint32_t)j, p.rid_base + (uint32_t)r, kPurposeAccept, p.key).x);
    token = (q <= 0.f || u < px / q) ? 1 : 0;
    if (p.p_tok) p.p_tok[(size_t)r * p.gamma + (j - 1)] = px;
  }
  p.ws.row_m[rj] = acc.m;
  p.ws.row_s[rj] = acc.s;
  p.ws.row_res[rj] = token;
  if (p.lse_t) {  // ln s = (k - 1) ln 2 + ln f with s = 2^k (f / 2), f in [1, 2)
    int kx;
    const float f = 2.f * frexpf(acc.s, &kx);
    p.lse_t[rj] = (float)fma((double)acc.m + (double)(kx - 1), 0.6931471805599453, (double)logf(f));
  }
  (void)l;
}

// Plan: the packed list of scheduled rows, codes r * (gamma + 1) + j - 1 for
// j = 1 .. l_r + 1, and their number B (one CTA).  Request order; with
// skip_dead, position order (every request's row 1, then every row 2, ...),
// so that a request's earlier rows are mostly finished before its later rows
// are claimed and the rows past its end can be skipped.
__global__ void __launch_bounds__(kPlanThreads) verify_plan_kernel(VerifyParams p) {
  __shared__ int warp_sum[kPlanThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = p.gamma + 1;
  if (tid == 0) carry = 0;
  __syncthreads();
  const int passes = p.skip_dead ? G1 : 1;
  for (int pass = 0; pass < passes; ++pass) {
    for (int r0 = 0; r0 < p.R; r0 += kPlanThreads) {  // uniform trip count
      const int r = r0 + tid;
      const int rows_r = (r < p.R) ? clamp_ell(p, r) + 1 : 0;
      // request order: all rows of r; position order: row pass + 1 if scheduled
      const int n = p.skip_dead ? (pass < rows_r ? 1 : 0) : rows_r;
      int incl = n;  // inclusive warp scan
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) warp_sum[warp] = incl;
      __syncthreads();
      int before = carry;
      for (int w = 0; w < warp; ++w) before += warp_sum[w];
      const int start = before + incl - n;
      for (int q = 0; q < n; ++q) p.ws.row_list[start + q] = r * G1 + (p.skip_dead ? pass : q);
      __syncthreads();
      if (tid == kPlanThreads - 1) carry = start + n;
      __syncthreads();
    }
  }
  if (tid == 0) *p.ws.n_rows = carry;
}

template <typename TT, bool kGreedy>
__global__ void __launch_bounds__(kVerifyThreads, 2) verify_rows_kernel(VerifyParams p) {
  extern __shared__ __align__(128) unsigned char ring_smem[];
  __shared__ __align__(8) uint64_t ring_bar[kVerifyThreads / 32][kRingStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long V = p.V;
  const int G1 = p.gamma + 1, cpr = p.nsplit;
  const float ks = fused::kLog2e * p.inv_target_temp;  // log2 units per logit
  constexpr bool greedy = kGreedy;
  const bool vec = ((size_t)V * sizeof(TT)) % 16 == 0 && (reinterpret_cast<uintptr_t>(p.tgt) & 15) == 0;

  // Aligned rows are read through a ring of kRingStages bulk copies per warp
  // (lane 0 keeps up to kRingStages batches in flight, across unit borders);
  // otherwise straight from global memory.
  constexpr uint32_t kStageB = kBatch * sizeof(TT);
  const bool bulk = vec && p.row_ring;
  unsigned char* ring = ring_smem + (size_t)warp * kRingStages * kStageB;
  if (bulk && lane == 0) {
    for (int i = 0; i < kRingStages; ++i) tc::mbar_init(&ring_bar[warp][i], 1);
    tc::fence_barrier_init();
  }
  __syncwarp();

  const unsigned long long units = (unsigned long long)(*p.ws.n_rows) * cpr;
  // A work unit: chunk c of row (r, j); row pointer L, entries [c0, c1).
  struct Unit {
    int ok, c, r, j, l, c0, c1, dead;
    const TT* L;
  };
  // per warp: the current unit, the one after it, and lane 0's issue state
  __shared__ Unit s_cur[kVerifyThreads / 32], s_next[kVerifyThreads / 32];
  __shared__ uint32_t s_iss[kVerifyThreads / 32];
  __shared__ int s_iss_cur[kVerifyThreads / 32], s_ib0[kVerifyThreads / 32];
  auto describe = [&](unsigned long long u) {
    Unit d{};
    d.ok = u < units;
    if (d.ok) {
      d.c = (int)(u % (unsigned long long)cpr);
      const int code = p.ws.row_list[u / (unsigned long long)cpr];
      d.r = code / G1;
      d.j = code % G1 + 1;
      d.l = clamp_ell(p, d.r);
      d.L = reinterpret_cast<const TT*>(p.tgt) + target_row(p, d.r, d.j) * (size_t)V;
      d.c0 = d.c * kRowChunk;
      d.c1 = (long)d.c0 + kRowChunk < V ? d.c0 + kRowChunk : (int)V;
      // a row past an end already found (a rejection, a mismatch) is not
      // needed: its chunk is skipped (an empty range issues no copies)
      if (p.skip_dead && (__ldcg(p.ws.term_mask + d.r) & ((1ull << (d.j - 1)) - 1ull))) {
        d.dead = 1;
        d.c1 = d.c0;
      }
    }
    return d;
  };
  auto claim_next = [&]() {  // lane 0 claims and describes the next unit
    if (lane == 0) s_next[warp] = describe(atomicAdd(p.ws.unit_cnt, 1ull));
    __syncwarp();
  };
  if (lane == 0) {
    s_cur[warp] = describe(atomicAdd(p.ws.unit_cnt, 1ull));
    s_iss[warp] = 0u;
    s_iss_cur[warp] = 1;
    s_ib0[warp] = s_cur[warp].c0;
  }
  __syncwarp();
  claim_next();
  uint32_t con = 0;  // ring batches consumed
  // lane 0: keep up to kRingStages batches in flight, from the current unit,
  // then from the next one
  auto issue_some = [&]() {
    uint32_t iss = s_iss[warp];
    int iss_cur = s_iss_cur[warp], ib0 = s_ib0[warp];
    while (iss - con < (uint32_t)kRingStages) {
      const Unit& d = iss_cur ? s_cur[warp] : s_next[warp];
      if (!d.ok) break;
      if (ib0 >= d.c1) {
        if (!iss_cur) break;
        iss_cur = 0;
        ib0 = s_next[warp].c0;
        continue;
      }
      const int slot = (int)(iss % kRingStages);
      const int n = d.c1 - ib0 < kBatch ? d.c1 - ib0 : kBatch;
      const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(TT);
      tc::fence_proxy_async();  // the stage's earlier reads come before the async write
      tc::mbar_expect_tx(&ring_bar[warp][slot], bytes);
      tc::bulk_load(ring + (size_t)slot * kStageB, d.L + ib0, bytes, &ring_bar[warp][slot]);
      ib0 += kBatch;
      ++iss;
    }
    s_iss[warp] = iss;
    s_iss_cur[warp] = iss_cur;
    s_ib0[warp] = ib0;
  };
  if (bulk && lane == 0) issue_some();
  bool failed = false;
  while (s_cur[warp].ok) {
    {
      const int c = s_cur[warp].c, r = s_cur[warp].r, j = s_cur[warp].j, l = s_cur[warp].l;
      const uint32_t rid = p.rid_base + (uint32_t)r;
      const bool bonus = !greedy && j == l + 1;
      const TT* L = s_cur[warp].L;
      const int c0 = s_cur[warp].c0, c1 = s_cur[warp].c1;

      Race st = race_empty();  // log2 units; be, bE, idx: bonus race
      ArgMax am = argmax_empty();
      float c_own = CUDART_INF_F;  // bonus: filter factor bE / be (with slack)
      PhiloxRow prow{};
      if (bonus) prow = philox_row((uint32_t)j, rid, kPurposeBonus, p.rk);
      // one batch of 32 entries per lane: x from the ring stage (bulk) or from
      // global memory; `fetch` may be called again by the overflow path
      auto batch = [&](int b0, const unsigned char* sx) {
        // eight consecutive entries of group g (from the stage, or global memory)
        auto get = [&](int g, float (&x)[8]) {
          const int off = g * 256 + lane * 8;
          if (sx) load8s_t<TT>(sx, off, c1 - b0, x);
          else load8(L, (long)b0 + off, c1, vec, x);
        };
        if (greedy) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float x[8];
            get(g, x);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int v = b0 + g * 256 + lane * 8 + q;
              if (v < c1 && (am.idx < 0 || x[q] > am.val)) {
                am.val = x[q];
                am.idx = v;
              }
            }
          }
          return;
        }
        // First finite entries of this lane: fix the reference at this batch's
        // maximum (log2 units) and, in the bonus row, seed the race with it.
        if (!(st.m > -CUDART_INF_F)) {
          float mx = -CUDART_INF_F;
          int im = 0;
#pragma unroll 1
          for (int g = 0; g < 4; ++g) {
            float x[8];
            get(g, x);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (x[q] > mx) {
                mx = x[q];
                im = g * 8 + q;
              }
          }
          if (mx > -CUDART_INF_F) {
            st.m = mx * ks;
            if (bonus) {  // its e is computed exactly as in the pass below
              const int vm = b0 + (im >> 3) * 256 + lane * 8 + (im & 7);
              const uint4 bm = philox_in_row((uint32_t)(vm >> 2), prow, p.rk);
              st.be = tc::ex2(fmaf(mx, ks, -st.m));
              st.bE = -logf(uniform_from_word(word_of(bm, vm & 3)));
              st.idx = vm;
              c_own = (st.bE / st.be) * fused::kFilterUp;
            }
          }
        }
        // Lanes without a finite entry yet (e.g. past V in a tail chunk) take
        // part in the warp-wide steps but contribute nothing; the batch is
        // skipped only when the whole warp has nothing.
        const bool have = st.m > -CUDART_INF_F;
        if (!__any_sync(0xffffffffu, have)) return;
        // bonus: the warp's best lowered score bounds every lane's filter
        float gbest = -CUDART_INF_F;
        if (bonus) {
          gbest = (st.idx >= 0) ? st.m + fused::lg2(st.be) - fused::lg2(st.bE) - fused::kPublishMargin
                                : -CUDART_INF_F;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) gbest = fmaxf(gbest, __shfl_xor_sync(0xffffffffu, gbest, off));
        }
        if (!have) return;
        float cf = fminf(c_own, tc::ex2(st.m - gbest) * fused::kFilterUp);
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          float x[8];
          get(g, x);
          float2 e[4];
          float ts;
          {
            const float2 ks2 = make_float2(ks, ks), nref2 = make_float2(-st.m, -st.m);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 a = __ffma2_rn(make_float2(x[2 * q], x[2 * q + 1]), ks2, nref2);
              e[q] = make_float2(tc::ex2(a.x), tc::ex2(a.y));
            }
            const float2 t = __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
            ts = t.x + t.y;
          }
          if (!(ts <= 1e37f) || st.s + ts > 1e30f) {  // rare: one test for both guards below
            if (!(ts <= 1e37f)) {  // a logit far above the reference (or a NaN): re-reference
              float mz = x[0];
#pragma unroll
              for (int q = 1; q < 8; ++q) mz = fmaxf(mz, x[q]);
              const float mnew = fmaxf(mz * ks, st.m);
              const float sc = tc::ex2(st.m - mnew);
              st.s *= sc;
              st.be *= sc;
              st.m = mnew;
              if (st.be > 0.f) c_own = (st.bE / st.be) * fused::kFilterUp;
              cf = fminf(c_own, tc::ex2(st.m - gbest) * fused::kFilterUp);
              ts = 0.f;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                e[q] = make_float2(tc::ex2(fmaf(x[2 * q], ks, -st.m)), tc::ex2(fmaf(x[2 * q + 1], ks, -st.m)));
                ts += e[q].x + e[q].y;
              }
            }
            st.s += ts;
            if (st.s > 1e30f) {  // keep the sum far from overflow: exact rescale by 2^-64
              st.s *= 0x1p-64f;
              st.be *= 0x1p-64f;
              st.m += 64.f;
              if (st.be > 0.f) c_own = (st.bE / st.be) * fused::kFilterUp;
              cf = fminf(c_own, tc::ex2(st.m - gbest) * fused::kFilterUp);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                e[q].x *= 0x1p-64f;
                e[q].y *= 0x1p-64f;
              }
            }
          } else {
            st.s += ts;
          }
          if (!bonus) continue;
          // ---- bonus race over this group ----
          const int v0 = b0 + g * 256 + lane * 8;
          uint32_t words[8];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 bb = philox_in_row((uint32_t)(v0 >> 2) + q, prow, p.rk);
            words[4 * q] = bb.x;
            words[4 * q + 1] = bb.y;
            words[4 * q + 2] = bb.z;
            words[4 * q + 3] = bb.w;
          }
          const float2 cf2 = make_float2(cf, cf), one2 = make_float2(1.f, 1.f);
          uint32_t all_neg = 0xffffffffu;
          float2 d[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            d[q] = __fadd2_rn(__ffma2_rn(e[q], cf2, one2),
                              make_float2(neg_one_plus_w(words[2 * q]), neg_one_plus_w(words[2 * q + 1])));
            all_neg &= __float_as_uint(d[q].x) & __float_as_uint(d[q].y);
          }
          if (!(all_neg >> 31)) {  // rare: exact race test in index order
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float dq = (q & 1) ? d[q >> 1].y : d[q >> 1].x;
              const float eq = (q & 1) ? e[q >> 1].y : e[q >> 1].x;
              if (!(__float_as_uint(dq) >> 31) && eq > 0.f && v0 + q < c1) {
                const float E = -logf(uniform_from_word(words[q]));
                if (race_beats(eq, E, v0 + q, st.be, st.bE, st.idx)) {
                  st.be = eq;
                  st.bE = E;
                  st.idx = v0 + q;
                  c_own = (st.bE / st.be) * fused::kFilterUp;
                  cf = fminf(cf, c_own);
                }
              }
            }
          }
        }
      };
      for (int b0 = c0; b0 < c1; b0 += kBatch) {
        // one call site, so that the batch code is inlined once
        const unsigned char* sx = nullptr;
        int slot = 0;
        if (bulk) {
          slot = (int)(con % kRingStages);
          if (!tc::mbar_wait(&ring_bar[warp][slot], (uint32_t)(con / kRingStages) & 1u, fused::kWaitNs)) {
            failed = true;
            break;
          }
          sx = ring + (size_t)slot * kStageB;
        }
        batch(b0, sx);
        if (bulk) {
          __syncwarp();  // every lane is done with the stage
          ++con;
          if (lane == 0) issue_some();
        }
      }
      if (__any_sync(0xffffffffu, failed)) break;
      if (s_cur[warp].dead) goto next_unit;
      // warp merge of the unit, partial, and the row / request completion
      Partial w{};
      if (greedy) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) am = argmax_merge(am, argmax_shfl_xor(am, off));
        w.f0 = am.val;
        w.i0 = am.idx;
      } else {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) st = row_merge(st, row_shfl_xor(st, off));
        w.f0 = st.m;
        w.f1 = st.s;
        w.f2 = st.be;
        w.f3 = st.bE;
        w.i0 = st.idx;
      }
      const size_t rj = (size_t)r * G1 + (j - 1);
      Partial* part = p.ws.row_part + rj * cpr;
      bool last = false;
      if (lane == 0) {
        part[c] = w;
        __threadfence();
        last = atomicAdd(p.ws.row_cnt + rj, 1u) == (unsigned)(cpr - 1);
        if (last) __threadfence();
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
      if (lane == 0) p.ws.row_cnt[rj] = 0u;
      if (greedy) {
        ArgMax acc = argmax_empty();
        for (int s = lane; s < cpr; s += 32) {
          const Partial q = load_partial(part + s);
          acc = argmax_merge(acc, ArgMax{q.f0, q.i0});
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc = argmax_merge(acc, argmax_shfl_xor(acc, off));
        if (lane == 0) p.ws.row_res[rj] = acc.idx;
      } else {
        Race acc = race_empty();
        for (int s = lane; s < cpr; s += 32) {
          const Partial q = load_partial(part + s);
          acc = row_merge(acc, Race{q.f0, q.f1, q.f2, q.f3, q.i0});
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc = row_merge(acc, row_shfl_xor(acc, off));
        if (lane == 0) finish_row(p, r, j, l, acc, ks, L, sizeof(TT) == 2, bonus);
      }
      if (lane == 0) {
        if (p.skip_dead) {
          // The request ends at its first row that rejects (mismatches) or at
          // row l + 1; it is resolved once every row up to that end is finished.
          const unsigned long long bit = 1ull << (j - 1);
          const int res = p.ws.row_res[rj];
          const bool ends = (j == l + 1) || (greedy ? p.x[(size_t)r * p.gamma + (j - 1)] != res : res == 0);
          if (ends) atomicOr(p.ws.term_mask + r, bit);
          __threadfence();
          const unsigned long long done = atomicOr(p.ws.done_mask + r, bit) | bit;
          __threadfence();
          const unsigned long long term = atomicOr(p.ws.term_mask + r, 0ull);
          const int jend = __ffsll((long long)term);  // lowest ending row, 0: none yet
          const unsigned long long need = jend >= 64 ? ~0ull : (1ull << jend) - 1ull;
          if (jend > 0 && (done & need) == need && atomicExch(p.ws.req_cnt + r, 1u) == 0u) {
            __threadfence();
            resolve_request(p, r, l);
          }
        } else {
          __threadfence();
          const unsigned prev = atomicAdd(p.ws.req_cnt + r, 1u);
          if (prev == (unsigned)l) {
            p.ws.req_cnt[r] = 0u;
            __threadfence();
            resolve_request(p, r, l);
          }
        }
      }
      }
    }
  next_unit:
    // next unit; lane 0 moves its issue position into it
    __syncwarp();
    if (lane == 0) {
      s_cur[warp] = s_next[warp];
      if (s_iss_cur[warp]) s_ib0[warp] = s_cur[warp].c0;  // the finished unit was issued in full
      s_iss_cur[warp] = 1;
    }
    __syncwarp();
    claim_next();
    if (bulk && lane == 0) issue_some();
  }
  if (failed && bulk && lane == 0) {
    // a ring wait gave up: let the copies still in flight land before exiting
    set_status(p.status, SPEC_STATUS_TIMEOUT);
    for (uint32_t n = con; n != s_iss[warp]; ++n)
      tc::mbar_wait(&ring_bar[warp][n % kRingStages], (uint32_t)(n / kRingStages) & 1u, fused::kWaitNs);
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
  const float m_t = p.ws.row_m[rj], s_t = p.ws.row_s[rj];  // m_t in log2 units
  const float inv_s_t = 1.0f / s_t;
  const TT* L = reinterpret_cast<const TT*>(p.tgt) + target_row(p, r, jstar) * (size_t)V;
  const int k = jstar;
  int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * p.gamma + (k - 2)];
  if (x_prev < 0 || x_prev >= V) x_prev = 0;
  const TF* brow = bias_row<TF>(p.A, p.S, V, rank, p.gamma, k, r, x_prev);
  const TF* Ct = reinterpret_cast<const TF*>(p.Ct) + (size_t)(k - 1) * V * rank;
  for (int i = threadIdx.x; i < rank; i += blockDim.x) arow[i] = ld_f(brow, (size_t)i);
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
        const float et = exp2f(fmaf(ld_f(L, (size_t)v), inv_tt * fused::kLog2e, -m_t));
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

// c* plan (one CTA): per position k, the requests with l_r >= k in request
// order (res_list[k-1][.], res_num[k-1]), and c_star set to 0 on the verified
// rows (the passes add into it) and NaN past l_r.
__global__ void __launch_bounds__(kPlanThreads) cstar_plan_kernel(VerifyParams p) {
  __shared__ int warp_sum[kPlanThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.gamma;
  for (int i = tid; i < p.R * G; i += kPlanThreads) {
    int l = p.ell[i / G];
    l = l < 0 ? 0 : (l > G ? G : l);
    p.c_star[i] = (i % G) < l ? 0.f : __int_as_float(0x7fc00000);  // quiet NaN
  }
  for (int k = 1; k <= G; ++k) {
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int r0 = 0; r0 < p.R; r0 += kPlanThreads) {  // uniform trip count
      const int r = r0 + tid;
      int l = (r < p.R) ? p.ell[r] : 0;
      l = l < 0 ? 0 : (l > G ? G : l);
      const bool take = r < p.R && l >= k;
      const unsigned bal = __ballot_sync(0xffffffffu, take);
      if (lane == 0) warp_sum[warp] = __popc(bal);
      __syncthreads();
      int before = carry;
      for (int w = 0; w < warp; ++w) before += warp_sum[w];
      if (take) p.ws.res_list[(size_t)(k - 1) * p.R + before + __popc(bal & ((1u << lane) - 1u))] = r;
      __syncthreads();
      if (tid == kPlanThreads - 1) carry = before + __popc(bal);
      __syncthreads();
    }
    if (tid == 0) p.ws.res_num[k - 1] = carry;
    __syncthreads();
  }
}

// Generic c* pass (any dtype, FFMA bias): grid (nsplit, R, gamma); block
// (s, r, k) adds sum min(p_v, q_v) over its vocabulary slice of row (r, k),
// k <= l_r, into c_star[r, k].
template <typename TT, typename TL, typename TF>
__global__ void __launch_bounds__(kVerifyThreads) cstar_kernel(VerifyParams p) {
  __shared__ float arow[256];
  __shared__ float red[kVerifyThreads / 32];
  const int r = blockIdx.y, k = blockIdx.z + 1, split = blockIdx.x, nsplit = gridDim.x;
  const int G = p.gamma, G1 = G + 1, V = p.V, rank = p.rank;
  int l = p.ell[r];
  l = l < 0 ? 0 : (l > G ? G : l);
  if (k > l) return;  // uniform across the block
  const size_t rj = (size_t)r * G1 + (k - 1);
  const float m_t = p.ws.row_m[rj], inv_s_t = 1.0f / p.ws.row_s[rj];  // m_t in log2 units
  const TT* L = reinterpret_cast<const TT*>(p.tgt) + target_row(p, r, k) * (size_t)V;
  int x_prev = (k == 1) ? p.x0[r] : p.x[(size_t)r * G + (k - 2)];
  if (x_prev < 0 || x_prev >= V) x_prev = 0;
  const TF* brow = bias_row<TF>(p.A, p.S, V, rank, p.gamma, k, r, x_prev);
  const TF* Ct = reinterpret_cast<const TF*>(p.Ct) + (size_t)(k - 1) * V * rank;
  for (int i = threadIdx.x; i < rank; i += blockDim.x) arow[i] = ld_f(brow, (size_t)i);
  __syncthreads();
  const TL* U = reinterpret_cast<const TL*>(p.U) + ((size_t)r * G + (k - 1)) * V;
  const float inv_tq = 1.0f / p.draft_temp[k - 1];
  const float lse_q = p.lse_q[(size_t)r * G + (k - 1)];
  const float kt = p.inv_target_temp * fused::kLog2e;
  const int per = (V + nsplit - 1) / nsplit;
  const int v_begin = split * per, v_end = min(V, v_begin + per);
  float sum = 0.f;
  for (int v = v_begin + threadIdx.x; v < v_end; v += blockDim.x) {
    float bias = 0.f;
    for (int i = 0; i < rank; ++i) bias = fmaf(arow[i], ld_f(Ct, (size_t)v * rank + i), bias);
    const float zq = (ld_f(U, (size_t)v) + bias) * inv_tq;
    const float pv = exp2f(fmaf(ld_f(L, (size_t)v), kt, -m_t)) * inv_s_t;
    sum += fminf(pv, expf(zq - lse_q));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_down_sync(0xffffffffu, sum, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kVerifyThreads / 32; ++w) t += red[w];
    atomicAdd(&p.c_star[(size_t)r * G + (k - 1)], t);
  }
}

// ------------------------------------------------------------- scratch ----
static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

// Scratch layout: arrays that need no initialisation first, then the
// counters and flags that every call zeroes in one memset.
enum { kRowPart, kResPart, kRowM, kRowS, kRowRes, kReqJstar, kResList, kRtPart, kRowList, kNRows,
       kUnitCnt, kDoneMask, kTermMask, kRowCnt, kReqCnt, kResCnt, kResNum, kRtCnt, kRtBest, kFallback,
       kLayoutN };

static size_t layout(int R, int gamma, int V, size_t off[kLayoutN]) {
  const size_t rows = (size_t)R * (gamma + 1);
  const size_t ns = (size_t)verify_nsplit(R, gamma, V), nr = (size_t)residual_nsplit(R, V);
  const size_t mt = (size_t)resid_tc_max_mtiles(R, gamma);
  const size_t sizes[kLayoutN] = {rows * ns * sizeof(Partial), (size_t)R * nr * sizeof(Partial),
                                  rows * sizeof(float), rows * sizeof(float), rows * sizeof(int),
                                  (size_t)R * sizeof(int), (size_t)gamma * R * sizeof(int),
                                  mt * kResTileRows * kMaxDeviceSms * sizeof(Partial), rows * sizeof(int),
                                  sizeof(int), sizeof(unsigned long long),
                                  (size_t)R * sizeof(unsigned long long), (size_t)R * sizeof(unsigned long long),
                                  rows * sizeof(unsigned), (size_t)R * sizeof(unsigned),
                                  (size_t)R * sizeof(unsigned), (size_t)gamma * sizeof(int),
                                  mt * sizeof(unsigned), (size_t)R * sizeof(unsigned),
                                  (size_t)R * sizeof(int)};
  size_t o = 0;
  for (int i = 0; i < kLayoutN; ++i) {
    off[i] = o;
    o = (i < kUnitCnt) ? align_up(o + sizes[i]) : o + sizes[i];  // counters packed after
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
  s.row_list = reinterpret_cast<int*>(b + off[kRowList]);
  s.n_rows = reinterpret_cast<int*>(b + off[kNRows]);
  s.row_cnt = reinterpret_cast<unsigned*>(b + off[kRowCnt]);
  s.req_cnt = reinterpret_cast<unsigned*>(b + off[kReqCnt]);
  s.res_cnt = reinterpret_cast<unsigned*>(b + off[kResCnt]);
  s.res_num = reinterpret_cast<int*>(b + off[kResNum]);
  s.rt_cnt = reinterpret_cast<unsigned*>(b + off[kRtCnt]);
  s.rt_best = reinterpret_cast<unsigned*>(b + off[kRtBest]);
  s.fallback = reinterpret_cast<int*>(b + off[kFallback]);
  s.unit_cnt = reinterpret_cast<unsigned long long*>(b + off[kUnitCnt]);
  s.done_mask = reinterpret_cast<unsigned long long*>(b + off[kDoneMask]);
  s.term_mask = reinterpret_cast<unsigned long long*>(b + off[kTermMask]);
  *counters_offset = off[kUnitCnt];
  *counters_bytes = total - off[kUnitCnt];  // the counter block, to the end
  return s;
}

// ------------------------------------------------------------ launchers ---
template <typename TT, typename TL, typename TF>
static cudaError_t launch_typed(const VerifyParams& p, int tgt_dtype, int logit_dtype,
                                cudaStream_t stream) {
  verify_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  const unsigned g1 = (unsigned)(2 * std::max(1, p.device_sms));
  // per-warp rings of bulk-copied batches
  const size_t ring = (size_t)(kVerifyThreads / 32) * kRingStages * kBatch * sizeof(TT);
  VerifyParams pr = p;
  auto kern = p.mode == SPEC_VERIFY_GREEDY ? verify_rows_kernel<TT, true> : verify_rows_kernel<TT, false>;
  pr.row_ring = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring) == cudaSuccess;
  if (!pr.row_ring) (void)cudaGetLastError();
  kern<<<g1, kVerifyThreads, pr.row_ring ? ring : 0, stream>>>(pr);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || p.mode == SPEC_VERIFY_GREEDY) return err;
  const dim3 g2((unsigned)residual_nsplit(p.R, p.V), (unsigned)p.R);
  if (!p.tc_residual) {
    residual_kernel<TT, TL, TF><<<g2, kVerifyThreads, 0, stream>>>(p, p.ws.req_jstar);
    err = cudaGetLastError();
    if (err != cudaSuccess || !p.c_star) return err;
    cstar_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    const int rows = std::max(1, p.R * p.gamma);
    const int ns = std::max(1, std::min((p.V + 1023) / 1024, (4 * 152 * 2 + rows - 1) / rows));
    cstar_kernel<TT, TL, TF>
        <<<dim3((unsigned)ns, (unsigned)p.R, (unsigned)p.gamma), kVerifyThreads, 0, stream>>>(p);
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
  t.rk = p.rk;
  t.inv_target_temp = p.inv_target_temp;
  t.x0 = p.x0;
  t.x = p.x;
  t.draft_temp = p.draft_temp;
  t.A = p.A;
  t.S = p.S;
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
  err = launch_resid_tc(t, tgt_dtype, logit_dtype, p.tgt, p.U, p.Ct, grid, false, stream);
  if (err != cudaSuccess) return err;
  // requests whose residual was zero everywhere (fp32 rounding only): the
  // generic kernel redoes them, sampling from p if its residual is zero too
  residual_kernel<TT, TL, TF><<<g2, kVerifyThreads, 0, stream>>>(p, p.ws.fallback);
  err = cudaGetLastError();
  if (err != cudaSuccess || !p.c_star) return err;
  // c*: every verified row, grouped by position (the residual lists are free now)
  cstar_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  t.c_star = p.c_star;
  const int cgrid = std::max(p.device_sms, p.gamma * ((p.R + kResTileRows - 1) / kResTileRows));
  return launch_resid_tc(t, tgt_dtype, logit_dtype, p.tgt, p.U, p.Ct, cgrid, true, stream);
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
