// Shared pieces of the fused tensor-core kernels (draft step and residual
// resample): CTA layout constants, ring counters, U/target tile loaders for
// the 128-byte swizzle layout the TMA writes, race helpers in log2 units and
// the tensor-map encoder.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace spec {
namespace fused {

constexpr int kNT = 64;        // vocabulary columns per tile (MMA N)
constexpr int kEpiWarps = 16;  // 4 TMEM lane quadrants x 4 column groups
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = (kEpiWarps + 2) * 32;
constexpr int kTmemBufs = 4;
constexpr uint32_t kTmemCols = kTmemBufs * kNT;
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFilterUp = 1.0f + 1.0f / 262144.0f;  // 1 + 2^-18
constexpr float kPublishMargin = 1.0f / 4096.0f;      // log2 units
constexpr size_t kSmemBudget = 227 * 1024 - 1024;     // dynamic smem per CTA

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Order-preserving map float -> uint32 (0 sorts below every float).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {  // NaN for key 0
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Merge of two race states whose reference `m` is in log2 units.
__device__ __forceinline__ Race race_merge2(const Race& a, const Race& b) {
  if (b.idx < 0) return a;
  if (a.idx < 0) return b;
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

// Writes the outputs of a merged race (reference m in log2 units) at index o:
// the token, q = e_best / s and lse = ln(sum_v exp(z_v / T)) = m ln 2 + ln s.
// With s = 2^k f, f in [1, 2), lse = (m + k) ln 2 + ln f: only a small
// logarithm is taken and one fp64 multiply-add keeps m + k exact.
__device__ __forceinline__ void store_race(int32_t* x, float* q_tok, float* lse_q, size_t o,
                                           const Race& acc) {
  x[o] = acc.idx;
  q_tok[o] = acc.be / acc.s;
  int ks;
  const float f = 2.f * frexpf(acc.s, &ks);
  lse_q[o] = (float)fma((double)acc.m + (double)(ks - 1), 0.6931471805599453, (double)logf(f));
}

__device__ __forceinline__ Race race_shfl_xor(const Race& st, int mask) {
  Race o;
  o.m = __shfl_xor_sync(0xffffffffu, st.m, mask);
  o.s = __shfl_xor_sync(0xffffffffu, st.s, mask);
  o.be = __shfl_xor_sync(0xffffffffu, st.be, mask);
  o.bE = __shfl_xor_sync(0xffffffffu, st.bE, mask);
  o.idx = __shfl_xor_sync(0xffffffffu, st.idx, mask);
  return o;
}

__device__ __forceinline__ WRace wrace_shfl_xor(const WRace& st, int mask) {
  return WRace{__shfl_xor_sync(0xffffffffu, st.bw, mask), __shfl_xor_sync(0xffffffffu, st.bE, mask),
               __shfl_xor_sync(0xffffffffu, st.idx, mask)};
}

template <typename TL>
struct UTile {
  static constexpr int kBoxCols = 128 / (int)sizeof(TL);  // 128-byte rows
  static constexpr int kBoxes = kNT / kBoxCols;
  static constexpr uint32_t kBytes = 128u * kNT * sizeof(TL);
};

// Byte offsets, inside a [128 x 64] tile, of the 16-byte chunks holding the 16
// logits of `row` from column 16*grp (fp32: two 32-column boxes; bf16: one
// 64-column box), in the 128-byte swizzle layout the TMA writes.
__device__ __forceinline__ void u_offsets(int row, int grp, uint32_t (&off)[4], float) {
  const int box = grp >> 1, c0 = (grp & 1) * 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) off[j] = box * 16384 + row * 128 + (((c0 + j) ^ (row & 7)) << 4);
}
__device__ __forceinline__ void u_offsets(int row, int grp, uint32_t (&off)[4], __nv_bfloat16) {
#pragma unroll
  for (int j = 0; j < 2; ++j) off[j] = row * 128 + (((grp * 2 + j) ^ (row & 7)) << 4);
  off[2] = off[3] = 0;
}
__device__ __forceinline__ void load_u16(const unsigned char* tile, const uint32_t (&off)[4],
                                         float (&u)[16], float) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 f = tc::lds128(tile + off[j]);
    u[4 * j] = __uint_as_float(f.x);
    u[4 * j + 1] = __uint_as_float(f.y);
    u[4 * j + 2] = __uint_as_float(f.z);
    u[4 * j + 3] = __uint_as_float(f.w);
  }
}
__device__ __forceinline__ void load_u16(const unsigned char* tile, const uint32_t (&off)[4],
                                         float (&u)[16], __nv_bfloat16) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 q = tc::lds128(tile + off[j]);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      u[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
      u[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
    }
  }
}

// Ring position with incremental phase (no division by the runtime depth).
struct Ring {
  int idx;
  uint32_t phase;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Host: cuTensorMapEncodeTiled for a 2-D or 3-D row-major tensor with the
// 128-byte swizzle (dims innermost first; `es` bytes per element).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, size_t es, const void* base, int rank,
                  const uint64_t* dims, const uint32_t* box);

}  // namespace fused
}  // namespace spec
