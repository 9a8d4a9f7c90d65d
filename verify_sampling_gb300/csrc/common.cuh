// Device building blocks shared by the sm_103a kernels of libspec.
//
//  * Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
//    32x32->64 multiplies of words 0 and 2, with a Weyl key schedule.
//  * Gumbel-max in "exponential race" form: argmax_v (z_v + G_v) with
//    G_v = -ln(E_v), E_v = -ln(u_v), equals argmax_v exp(z_v - m) / E_v for any
//    shift m.  The kernels keep exp(z - m) (already needed for the softmax sum)
//    and compare candidates by cross-multiplication, so no second logarithm and
//    no division appear in the streaming loop.
//  * Online softmax state (running max m, sum s of exp(z - m)).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "spec.h"

namespace spec {

constexpr uint32_t kPurposeDraft = 0;
constexpr uint32_t kPurposeAccept = 1;
constexpr uint32_t kPurposeResidual = 2;
constexpr uint32_t kPurposeBonus = 3;

// ----------------------------------------------------------------- Philox --
struct PhiloxKey {
  uint32_t lo, hi;
};

__host__ __device__ inline PhiloxKey philox_key(uint64_t seed) {
  return PhiloxKey{(uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32)};
}

// Round keys of the Weyl schedule: round i uses (key.lo + i*W0, key.hi + i*W1).
struct PhiloxRoundKeys {
  uint32_t k0[10], k1[10];
};

__host__ __device__ inline PhiloxRoundKeys philox_round_keys(PhiloxKey key) {
  PhiloxRoundKeys rk;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    rk.k0[i] = key.lo + (uint32_t)i * 0x9E3779B9u;
    rk.k1[i] = key.hi + (uint32_t)i * 0xBB67AE85u;
  }
  return rk;
}

// One Philox-4x32-10 block for counter (w0, w1, w2, w3).  Each round takes the
// two 32x32 -> 64-bit products of words 0 and 2 (one wide multiply each).
__device__ __forceinline__ uint4 philox(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                        const PhiloxRoundKeys& rk) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * w0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * w2;
    w0 = (uint32_t)(p1 >> 32) ^ w1 ^ rk.k0[round];
    w1 = (uint32_t)p1;
    w2 = (uint32_t)(p0 >> 32) ^ w3 ^ rk.k1[round];
    w3 = (uint32_t)p0;
  }
  return make_uint4(w0, w1, w2, w3);
}

__device__ __forceinline__ uint4 philox(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                        PhiloxKey key) {
  return philox(w0, w1, w2, w3, philox_round_keys(key));
}

// Philox along one row of the stream: counter words 1-3 (position j, request
// id, purpose) are fixed and only word 0 (the vocabulary block) varies.  The
// parts of the first two rounds that depend only on the fixed words are
// computed once per row, so a block costs 18 wide multiplies instead of 20.
// With counter (c, j, rid, purpose):
//   round 1: w0 = hi(M1 rid) ^ j ^ k0[0] (fixed), w1 = lo(M1 rid) (fixed),
//            w2 = hi(M0 c) ^ purpose ^ k1[0], w3 = lo(M0 c);
//   round 2: w0 = hi(M1 w2) ^ (w1 ^ k0[1]), w1 = lo(M1 w2),
//            w2 = (hi(M0 w0) ^ k1[1]) ^ lo(M0 c), w3 = lo(M0 w0) (fixed).
struct PhiloxRow {
  uint32_t b0;  // purpose ^ k1[0]
  uint32_t x0;  // lo(M1 rid) ^ k0[1]
  uint32_t x2;  // hi(M0 w0) ^ k1[1], w0 of round 1
  uint32_t w3;  // lo(M0 w0)
};

__host__ __device__ inline PhiloxRow philox_row(uint32_t j, uint32_t rid, uint32_t purpose,
                                                const PhiloxRoundKeys& rk) {
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * rid;
  const uint32_t w0 = (uint32_t)(p1 >> 32) ^ j ^ rk.k0[0];
  const uint64_t p0 = (uint64_t)0xD2511F53u * w0;
  return PhiloxRow{purpose ^ rk.k1[0], (uint32_t)p1 ^ rk.k0[1], (uint32_t)(p0 >> 32) ^ rk.k1[1],
                   (uint32_t)p0};
}

// The block with counter word 0 = c of the row `row` (round keys: pass kernel
// parameters so that they stay in the constant bank).
__device__ __forceinline__ uint4 philox_in_row(uint32_t c, const PhiloxRow& row,
                                               const PhiloxRoundKeys& rk) {
  const uint64_t q0 = (uint64_t)0xD2511F53u * c;
  const uint64_t q1 = (uint64_t)0xCD9E8D57u * ((uint32_t)(q0 >> 32) ^ row.b0);
  uint32_t w0 = (uint32_t)(q1 >> 32) ^ row.x0, w1 = (uint32_t)q1;
  uint32_t w2 = row.x2 ^ (uint32_t)q0, w3 = row.w3;
#pragma unroll
  for (int round = 2; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * w0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * w2;
    w0 = (uint32_t)(p1 >> 32) ^ w1 ^ rk.k0[round];
    w1 = (uint32_t)p1;
    w2 = (uint32_t)(p0 >> 32) ^ w3 ^ rk.k1[round];
    w3 = (uint32_t)p0;
  }
  return make_uint4(w0, w1, w2, w3);
}

__device__ __forceinline__ uint32_t word_of(uint4 b, int lane) {
  return lane == 0 ? b.x : lane == 1 ? b.y : lane == 2 ? b.z : b.w;
}

// Uniform (2*m+1) * 2^-24 in (0,1) with m = the low 23 bits of the word: the bit
// pattern 1.m is 1 + m*2^-23; subtracting 1 - 2^-24 leaves (2m+1)*2^-24, which
// is representable, so the subtraction is exact.
__device__ __forceinline__ float uniform_from_word(uint32_t x) {
  return __uint_as_float(0x3f800000u | (x & 0x7fffffu)) - 0.99999994f;
}

// 1 + (1 - u) - 2^-24 as a float (exact): the pattern 1.m' of the complemented
// low bits m' = 2^23 - 1 - m.  One logic operation.
__device__ __forceinline__ float one_plus_w(uint32_t x) {
  return __uint_as_float(0x3f800000u | (~x & 0x7fffffu));
}
// -(1 + (1 - u) - 2^-24): the same value negated (one logic operation).
__device__ __forceinline__ float neg_one_plus_w(uint32_t x) {
  return __uint_as_float(0xbf800000u | (~x & 0x7fffffu));
}

// E = -ln(u) > 0, an Exp(1) variate.  logf is accurate to about one ulp of its
// result, which keeps E accurate relative to itself even for u near 1 (u - 1
// is exact there).
__device__ __forceinline__ float neg_log_uniform(uint32_t x) { return -logf(uniform_from_word(x)); }

// ------------------------------------------------------------ races/state --
// Gumbel race + online softmax over a stream of logits z.
struct Race {
  float m;   // running max of z
  float s;   // sum of exp(z - m)
  float be;  // exp(z_best - m)
  float bE;  // E of the best candidate
  int idx;   // best candidate (-1: none yet)
};

__device__ __forceinline__ Race race_empty() { return Race{-CUDART_INF_F, 0.f, 0.f, 1.f, -1}; }

// Does candidate (e1/E1, i1) beat (e2/E2, i2)?  Lower index wins exact ties.
__device__ __forceinline__ bool race_beats(float e1, float E1, int i1, float e2, float E2, int i2) {
  if (i1 < 0) return false;
  if (i2 < 0) return true;
  const float l = e1 * E2, r = e2 * E1;
  return l > r || (l == r && i1 < i2);
}

__device__ __forceinline__ void race_push(Race& st, float z, float E, int v) {
  if (!(z > -CUDART_INF_F)) return;  // -inf (masked) or NaN never wins
  if (z > st.m) {
    const float sc = expf(st.m - z);
    st.s *= sc;
    st.be *= sc;
    st.m = z;
  }
  const float e = expf(z - st.m);
  st.s += e;
  if (race_beats(e, E, v, st.be, st.bE, st.idx)) {
    st.be = e;
    st.bE = E;
    st.idx = v;
  }
}

__device__ __forceinline__ Race race_merge(const Race& a, const Race& b) {
  if (b.idx < 0) return a;
  if (a.idx < 0) return b;
  const float m = fmaxf(a.m, b.m);
  const float sa = expf(a.m - m), sb = expf(b.m - m);
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

__device__ __forceinline__ Race race_shfl_down(const Race& st, int off) {
  Race o;
  o.m = __shfl_down_sync(0xffffffffu, st.m, off);
  o.s = __shfl_down_sync(0xffffffffu, st.s, off);
  o.be = __shfl_down_sync(0xffffffffu, st.be, off);
  o.bE = __shfl_down_sync(0xffffffffu, st.bE, off);
  o.idx = __shfl_down_sync(0xffffffffu, st.idx, off);
  return o;
}

// Online softmax only (m, s).
struct Soft {
  float m, s;
};
__device__ __forceinline__ Soft soft_empty() { return Soft{-CUDART_INF_F, 0.f}; }
__device__ __forceinline__ void soft_push(Soft& st, float z) {
  if (!(z > -CUDART_INF_F)) return;
  if (z > st.m) {
    st.s *= expf(st.m - z);
    st.m = z;
  }
  st.s += expf(z - st.m);
}
__device__ __forceinline__ Soft soft_merge(const Soft& a, const Soft& b) {
  if (!(b.m > -CUDART_INF_F)) return a;
  if (!(a.m > -CUDART_INF_F)) return b;
  const float m = fmaxf(a.m, b.m);
  return Soft{m, a.s * expf(a.m - m) + b.s * expf(b.m - m)};
}

// Weighted race without a softmax: argmax_v w_v / E_v over w_v > 0.
struct WRace {
  float bw, bE;
  int idx;
};
__device__ __forceinline__ WRace wrace_empty() { return WRace{0.f, 1.f, -1}; }
__device__ __forceinline__ void wrace_push(WRace& st, float w, float E, int v) {
  if (!(w > 0.f)) return;
  if (race_beats(w, E, v, st.bw, st.bE, st.idx)) {
    st.bw = w;
    st.bE = E;
    st.idx = v;
  }
}
__device__ __forceinline__ WRace wrace_merge(const WRace& a, const WRace& b) {
  return race_beats(b.bw, b.bE, b.idx, a.bw, a.bE, a.idx) ? b : a;
}

// Argmax with lowest index on ties.
struct ArgMax {
  float val;
  int idx;
};
__device__ __forceinline__ ArgMax argmax_empty() { return ArgMax{-CUDART_INF_F, -1}; }
__device__ __forceinline__ void argmax_push(ArgMax& st, float v, int i) {
  if (st.idx < 0 || v > st.val || (v == st.val && i < st.idx)) {
    st.val = v;
    st.idx = i;
  }
}
__device__ __forceinline__ ArgMax argmax_merge(const ArgMax& a, const ArgMax& b) {
  if (b.idx < 0) return a;
  if (a.idx < 0) return b;
  if (b.val > a.val || (b.val == a.val && b.idx < a.idx)) return b;
  return a;
}

// Workspace record for one partial result (32 bytes).
struct alignas(32) Partial {
  float f0, f1, f2, f3;
  int i0;
  float f4, f5;
  int i1;
};

// Read a partial published by another CTA (L2, bypassing L1).
__device__ __forceinline__ Partial load_partial(const Partial* p) {
  const int4* q = reinterpret_cast<const int4*>(p);
  int4 a = __ldcg(q), b = __ldcg(q + 1);
  Partial o;
  o.f0 = __int_as_float(a.x);
  o.f1 = __int_as_float(a.y);
  o.f2 = __int_as_float(a.z);
  o.f3 = __int_as_float(a.w);
  o.i0 = b.x;
  o.f4 = __int_as_float(b.y);
  o.f5 = __int_as_float(b.z);
  o.i1 = b.w;
  return o;
}

// ----------------------------------------------------------------- loads ---
__device__ __forceinline__ float ld_f(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// Row of the bias factor for position k (1-based) of request r: the Markov
// head's A_k[x_prev] or, when the RNN head's state array S [R, gamma, rank] is
// given, the stored state s_k = S[r][k - 1].
template <typename TF>
__device__ __forceinline__ const TF* bias_row(const void* A, const void* S, int V, int rank, int gamma,
                                              int k, int r, int x_prev) {
  if (S) return reinterpret_cast<const TF*>(S) + ((size_t)r * gamma + (k - 1)) * rank;
  return reinterpret_cast<const TF*>(A) + ((size_t)(k - 1) * V + x_prev) * rank;
}

// ---------------------------------------------------------- block helpers --
// Block-wide merge of per-thread states; the result is valid in thread 0.
template <typename S, typename ShflFn, typename MergeFn>
__device__ __forceinline__ S block_reduce(S st, S* smem, ShflFn shfl, MergeFn merge) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) st = merge(st, shfl(st, off));
  if (lane == 0) smem[warp] = st;
  __syncthreads();
  if (warp == 0) {
    st = smem[lane < nwarps ? lane : 0];
    if (lane >= nwarps) st = smem[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      S o = shfl(st, off);
      if (lane + off < nwarps) st = merge(st, o);
    }
  }
  return st;
}

// Last-block-done protocol: returns true in exactly one CTA of the group that
// shares `counter`, after all of the group's CTAs have published their
// partials (each CTA calls this once, after writing its partial).  The winning
// CTA resets the counter for the next use.
__device__ __forceinline__ bool last_block_arrives(unsigned* counter, unsigned expected) {
  __shared__ bool is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(counter, 1u);
    is_last = (prev == expected - 1);
    if (is_last) *counter = 0u;
  }
  __syncthreads();
  if (is_last) __threadfence();
  return is_last;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace spec
