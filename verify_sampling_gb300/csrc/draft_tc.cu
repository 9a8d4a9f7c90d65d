// Fused draft step on the 5th-generation tensor cores (sm_100 family).
//
// One launch per draft position k computes, for a tile of 128 requests and a
// range of the vocabulary,
//     bias[m, v] = A_k[x_{m,k-1}, :] . C_k[:, v]          (tcgen05.mma, bf16 -> f32 in TMEM)
//     z[m, v]    = (U[m, k, v] + bias[m, v]) / T_k
// and folds every z into a per-request online softmax (sum of exp) and a
// Gumbel race with the purpose-0 Philox stream; no z is ever written to
// memory.  DSpark summary, "第二阶段：轻量顺序头" and the history article,
// "杀招一": P_k = softmax(U_k + B_k(x_{k-1})), B_k low-rank.
//
// CTA layout (576 threads, one CTA per SM):
//   warps 0-15  epilogue: warp w reads TMEM lane quadrant w % 4 (32 requests)
//               and column group w / 4 (32 of the 128 columns of a tile, as
//               two 16-column halves)
//   warp 16     TMA producer: per 128-column tile, the C_k tile [128 x r] and
//               the U tile as two [128 x 64] stages
//   warp 17     tensor-memory owner and single-thread MMA issuer (N = 128)
// Pipelines: a ring of C_k tiles (freed by the MMA's commit), a ring of
// `stages` U stages (each freed by the 8 warps that read it) and four
// 128-column TMEM accumulators (full/empty mbarriers).  The gathered A rows
// (128 x r bf16) are written once per launch in the 128-byte swizzle layout.
// Every wait is bounded; on a timeout the CTA sets SPEC_STATUS_TIMEOUT, drains
// what it issued and returns.
//
// Gumbel race (see common.cuh): the winner maximises z_v - ln E_v with
// E_v = -ln u_v.  Each thread keeps e = 2^(z log2e / T - ref) and the best
// (e, E); the logarithm E is computed only for candidates, selected by an exact
// filter: since E >= 1 - u, an element can reach a score g only if
// 1 - u <= e * 2^(ref - g).  The bound g is the larger of the thread's own best
// and the best score any thread of the same row has published so far: a
// shared-memory word per row, raised with atomicMax, into which one thread per
// row copies the row's global word (raised by new CTA-level bests) every
// tile.  Published scores
// are real scores lowered by a margin, so the row's winner always passes; the
// filter only decides which elements need the exact comparison.  The race
// starts from the first tile's largest element, so the first tile does not
// send every element through the exact test.
#include "draft.cuh"
#include "draft_tc.cuh"
#include "fused_tc.cuh"
#include "rnn.cuh"
#include "tc.cuh"

namespace spec {

namespace {

using namespace fused;

// The 512 epilogue threads merge the split partials of position `kpos` for
// the tile's 128 requests, four threads per request with all of a thread's
// loads in flight (one round trip up to 48 splits).  Writes x, q_tok and lse_q
// of that position when `write`, and the token into s_x (nullable).
__device__ __forceinline__ void merge_position(const DraftTCParams& p, const Partial* part, int m0,
                                               int kpos, bool write, int* s_x) {
  const int row = threadIdx.x >> 2, lp = threadIdx.x & 3, m = m0 + row;
  Race acc = race_empty();
  if (m < p.R) {
    const Partial* src = part + (size_t)m * p.nsplit;
    for (int s0 = lp; s0 < p.nsplit; s0 += 48) {
      Partial w[12];
#pragma unroll
      for (int q = 0; q < 12; ++q)
        if (s0 + 4 * q < p.nsplit) w[q] = load_partial(src + s0 + 4 * q);
#pragma unroll
      for (int q = 0; q < 12; ++q)
        if (s0 + 4 * q < p.nsplit) acc = race_merge2(acc, Race{w[q].f0, w[q].f1, w[q].f2, w[q].f3, w[q].i0});
    }
  }
  acc = race_merge2(acc, race_shfl_xor(acc, 1));
  acc = race_merge2(acc, race_shfl_xor(acc, 2));
  if (lp != 0) return;
  if (s_x) s_x[row] = m < p.R ? acc.idx : -1;
  if (write && m < p.R) store_race(p.x, p.q_tok, p.lse_q, (size_t)m * p.gamma + (kpos - 1), acc);
}

// Split partials of position kpos: two slots, alternating with the position.
__device__ __forceinline__ Partial* partial_slot(const DraftTCParams& p, int kpos) {
  return p.partials + (size_t)(kpos & 1) * p.R * p.nsplit;
}

// Cold path: exact race test of one filtered element; on a new best, publish
// the row's score to the CTA (and, when it raises the CTA's bound, to the
// row's word in global memory) and return true.
__device__ __forceinline__ bool race_candidate(Race& st, float e, uint32_t word, int v,
                                               uint32_t* row_best, uint32_t shared_seen,
                                               unsigned* global_best) {
  if (!(e > 0.f)) return false;  // an underflowed (or NaN) weight never wins
  const float E = -logf(uniform_from_word(word));
  if (!race_beats(e, E, v, st.be, st.bE, st.idx)) return false;
  st.be = e;
  st.bE = E;
  st.idx = v;
  // score in log2 units: ref + log2(e) - log2(E), lowered by a margin that
  // covers the approximate logarithms
  const float score = st.m + lg2(e) - lg2(E) - kPublishMargin;
  const uint32_t key = ordered_key(score);
  if (key > shared_seen) {
    atomicMax(row_best, key);  // shared memory
    atomicMax(global_best, key);
  }
  return true;
}

// Vocabulary columns per MMA tile (N); each epilogue warp takes 32 of them
// as two 16-column halves.  U arrives in 64-column stages (two per tile), C
// in 128-column tiles through a ring of its own.
constexpr int kDNT = 128;
constexpr uint32_t kDTmemCols = kTmemBufs * kDNT;
// C_k ring depth: two 128-column tiles, one when the rank is 192 or 256 (the
// U ring then keeps at least two stages).
__host__ __device__ constexpr int c_stages(int KC) { return KC >= 3 ? 1 : 2; }

}  // namespace

using namespace fused;

// kIdleWarps: R is not a multiple of 128, so a lane quadrant of the last
// request tile may lie wholly past R (such a warp only keeps the pipeline
// going).  576 threads per CTA leave at most 96 registers per thread.
template <typename TL, int KC, bool kIdleWarps>
__global__ void __launch_bounds__(kThreads, 1)
    draft_tc_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_c,
                    DraftTCParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kSc = c_stages(KC);
  constexpr uint32_t kCBytes = KC * kDNT * 128;  // C_k tile [128 columns x r]
  constexpr uint32_t kUBytes = UTile<TL>::kBytes;  // U stage [128 requests x 64 columns]
  unsigned char* sA = smem;
  unsigned char* sC = smem + KC * 16384;
  unsigned char* sU = sC + kSc * kCBytes;

  __shared__ __align__(8) uint64_t full_c[2], empty_c[2], full_u[kMaxStages], empty_u[kMaxStages];
  __shared__ __align__(8) uint64_t tfull[kTmemBufs], tempty[kTmemBufs];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t s_best[128];  // per tile row: best race score so far (ordered key, 0 = none)
  __shared__ int s_x[128];          // x_{k-1} of the tile's requests, merged here
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x % p.mtiles, split = blockIdx.x / p.mtiles;
  const int m0 = mtile * 128;
  const int t_begin = (int)((long)split * p.ntiles / p.nsplit);
  const int t_end = (int)((long)(split + 1) * p.ntiles / p.nsplit);
  const int T = t_end - t_begin;
  const int S = p.stages;
  const int k = p.k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSc; ++s) {
      tc::mbar_init(&full_c[s], 1);
      tc::mbar_init(&empty_c[s], 1);  // the MMA's commit
    }
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full_u[s], 1);
      tc::mbar_init(&empty_u[s], kEpiWarps / 2);  // the 8 warps reading that 64-column half
    }
    for (int b = 0; b < kTmemBufs; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kEpiWarps);
    }
    abort_flag = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, kDTmemCols);
  if (warp == kProducerWarp && lane == 0) {
    tc::tma_prefetch_desc(&tm_u);
    tc::tma_prefetch_desc(&tm_c);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // The next position's grid may start its prologue and its U / C loads on SMs
  // that this grid frees; it waits (griddepcontrol.wait) before reading x.
  tc::grid_dep_launch();

  auto fail = [&]() {
    abort_flag = 1;
    set_status(p.status, SPEC_STATUS_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int issued_c = 0, issued_u = 0;
      Ring rc{0, 0u}, ru{0, 0u};
      for (int t = 0; t < T && !abort_flag; ++t, rc.next(kSc)) {
        if (!tc::mbar_wait(&empty_c[rc.idx], rc.phase ^ 1u, kWaitNs)) {
          fail();
          break;
        }
        const int n0 = (t_begin + t) * kDNT;
        tc::mbar_expect_tx(&full_c[rc.idx], kCBytes);
#pragma unroll
        for (int kc = 0; kc < KC; ++kc)
          tc::tma_load_3d(sC + rc.idx * kCBytes + kc * 16384, &tm_c, &full_c[rc.idx], kc * 64, n0, k - 1);
        issued_c = t + 1;
        bool ok = true;
        for (int h = 0; h < 2; ++h, ru.next(S)) {
          if (!tc::mbar_wait(&empty_u[ru.idx], ru.phase ^ 1u, kWaitNs)) {
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&full_u[ru.idx], kUBytes);
#pragma unroll
          for (int bx = 0; bx < UTile<TL>::kBoxes; ++bx)
            tc::tma_load_3d(sU + ru.idx * kUBytes + bx * 16384, &tm_u, &full_u[ru.idx],
                            n0 + h * kNT + bx * UTile<TL>::kBoxCols, k - 1, m0);
          ++issued_u;
        }
        if (!ok) {
          fail();
          break;
        }
      }
      if (abort_flag) {
        // drain: the last load issued into each stage must land before exit
        for (int t = (issued_c > kSc ? issued_c - kSc : 0); t < issued_c; ++t)
          tc::mbar_wait(&full_c[t % kSc], (uint32_t)(t / kSc) & 1u, kWaitNs);
        for (int u = (issued_u > S ? issued_u - S : 0); u < issued_u; ++u)
          tc::mbar_wait(&full_u[u % S], (uint32_t)(u / S) & 1u, kWaitNs);
      }
    }
  } else if (warp == kMmaWarp) {
    named_bar_sync(1, (kEpiWarps + 1) * 32);  // gathered A rows are in shared memory
    if (lane == 0) {
      constexpr uint32_t idesc = tc::bf16_idesc(128, kDNT);
      int last = -1;
      Ring r{0, 0u}, rb{0, 0u};
      const uint32_t a_base = tc::smem_u32(sA);
      for (int t = 0; t < T && !abort_flag; ++t, r.next(kSc), rb.next(kTmemBufs)) {
        if (!tc::mbar_wait(&full_c[r.idx], r.phase, kWaitNs) ||
            !tc::mbar_wait(&tempty[rb.idx], rb.phase ^ 1u, kWaitNs)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const uint32_t b_base = tc::smem_u32(sC + r.idx * kCBytes);
#pragma unroll
        for (int kk = 0; kk < KC * 4; ++kk) {
          const int kc = kk >> 2, ko = (kk & 3) * 32;
          tc::mma_bf16(tmem + (uint32_t)(rb.idx * kDNT), tc::sw128_desc(a_base + kc * 16384 + ko),
                       tc::sw128_desc(b_base + kc * 16384 + ko), idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&tfull[rb.idx]);
        tc::mma_commit(&empty_c[r.idx]);
        last = t;
      }
      if (abort_flag && last >= 0)  // in-flight MMAs must finish before TMEM is freed
        tc::mbar_wait(&tfull[last % kTmemBufs], (uint32_t)(last / kTmemBufs) & 1u, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quad = warp & 3, grp = warp >> 2;
    const int row = quad * 32 + lane, m = m0 + row;
    const bool valid = m < p.R;
    const int V = p.V, rank = p.rank;

    tc::grid_dep_wait();  // the previous position's partials (or states) are written
    // x_{k-1}: every CTA of the tile merges the previous position's split
    // partials itself (the previous grid ends without a merge on its critical
    // path); the CTA of split 0 also writes that position's outputs.  With the
    // RNN head the state kernel between the two grids has merged them.
    const bool rnn = p.S != nullptr;
    if (k > 1 && !rnn) {
      merge_position(p, partial_slot(p, k - 1), m0, k - 1, split == 0, s_x);
      named_bar_sync(2, kEpiWarps * 32);
    }
    // Gather the bias rows of the tile's 128 requests -- A_k[x_{k-1}], or the
    // RNN head's states s_k -- 128 x r bf16 in 16-byte chunks, 2*KC per thread,
    // all loads in flight before the stores.
    const __nv_bfloat16* Ak = reinterpret_cast<const __nv_bfloat16*>(p.A) + (size_t)(k - 1) * V * rank;
    const __nv_bfloat16* Sk = reinterpret_cast<const __nv_bfloat16*>(p.S) + (size_t)(k - 1) * rank;
    if (rnn) {
      constexpr int kPer = 128 * KC * 8 / (kEpiWarps * 32);
      uint4 val[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = threadIdx.x + j * kEpiWarps * 32, c = idx % (KC * 8), mm = m0 + idx / (KC * 8);
        val[j] = mm < p.R ? *reinterpret_cast<const uint4*>(Sk + (size_t)mm * p.gamma * rank + c * 8)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = threadIdx.x + j * kEpiWarps * 32, i = idx / (KC * 8), c = idx % (KC * 8);
        const int kc = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sA + kc * 16384 + i * 128 + ((cc ^ (i & 7)) << 4)) = val[j];
      }
    } else {
      constexpr int kPer = 128 * KC * 8 / (kEpiWarps * 32);
      int xp[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = threadIdx.x + j * kEpiWarps * 32, mm = m0 + idx / (KC * 8);
        xp[j] = mm < p.R ? ((k == 1) ? p.x0[mm] : s_x[idx / (KC * 8)]) : -1;
      }
      uint4 val[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = threadIdx.x + j * kEpiWarps * 32, c = idx % (KC * 8), mm = m0 + idx / (KC * 8);
        val[j] = make_uint4(0, 0, 0, 0);
        if (mm < p.R) {
          int x = xp[j];
          if (x < 0 || x >= V) {
            if (c == 0) set_status(p.status, SPEC_STATUS_BAD_TOKEN);
            x = 0;
          }
          val[j] = *reinterpret_cast<const uint4*>(Ak + (size_t)x * rank + c * 8);
        }
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = threadIdx.x + j * kEpiWarps * 32, i = idx / (KC * 8), c = idx % (KC * 8);
        const int kc = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sA + kc * 16384 + i * 128 + ((cc ^ (i & 7)) << 4)) = val[j];
      }
    }
    if (threadIdx.x < 128) s_best[threadIdx.x] = 0;
    tc::fence_proxy_async();
    named_bar_sync(1, (kEpiWarps + 1) * 32);

    // Race state in log2 units: e = 2^(z log2e / T - st.m).  The reference
    // st.m is fixed at the first tile of the row (its maximum) and moves only
    // when a tile's sum overflows, or by exact powers of two when the running
    // sum grows large -- no per-element maximum is needed.
    Race st = race_empty();
    // c_own = (bE / be) * (1 + 2^-18): the filter factor of the thread's own
    // best; the shared best adds c_shared = 2^(ref - g).  The test
    // f <= e*c + 1 with f = 1 + (1 - u) - 2^-24 is 1 - u <= e*c with a safe
    // margin (e*c + 1 rounds by at most 2^-24, covered by the 2^-24 in f and
    // the slack in c).
    float c_own = CUDART_INF_F;
    const float kscale = kLog2e / p.draft_temp[k - 1];
    const float2 kscale2 = make_float2(kscale, kscale);
    float nref = 0.f;  // -st.m once the reference is set
    const PhiloxRow prow = philox_row((uint32_t)k, p.rid_base + (uint32_t)m, kPurposeDraft, p.rk);
    uint32_t* row_best = &s_best[row];
    // rows past R race on zeros like any other row (their results are never
    // written); their publications go to their own shared word only
    unsigned* global_best = valid ? p.row_best + (size_t)(k - 1) * p.R + m : row_best;
    uint32_t global_seen = 0;  // one thread per row imports the global bound, one tile late
    // The warp's 64-column U stage of each tile (the tile's U stages are
    // numbered 2t and 2t + 1) and its 32 columns in the TMEM tile.
    const int hw = grp >> 1;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(grp * 32);
    Ring ru{hw, 0u}, rb{0, 0u};
    // (no abort test in these loops: every wait is bounded, and a failed one
    // ends the loop)
    bool warp_idle = false;
    if constexpr (kIdleWarps) {
      warp_idle = !__any_sync(0xffffffffu, valid);
      for (int t = 0; warp_idle && t < T; ++t, ru.next(S), ru.next(S), rb.next(kTmemBufs)) {
        if (!tc::mbar_wait(&tfull[rb.idx], rb.phase, kWaitNs) ||
            !tc::mbar_wait(&full_u[ru.idx], ru.phase, kWaitNs)) {
          fail();
          break;
        }
        __syncwarp();
        tc::mbar_arrive2_if(&tempty[rb.idx], &empty_u[ru.idx], lane == 0);
      }
    }
    for (int t = 0; !warp_idle && t < T; ++t, ru.next(S), ru.next(S), rb.next(kTmemBufs)) {
      if (grp == 0 && valid) {  // the row's bound from the other CTAs (loaded last tile)
        if (global_seen) atomicMax(row_best, global_seen);
        global_seen = __ldcg(global_best);
      }
      if (!tc::mbar_wait(&tfull[rb.idx], rb.phase, kWaitNs) ||
          !tc::mbar_wait(&full_u[ru.idx], ru.phase, kWaitNs)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      // two 16-column halves; the tile's TMEM and U stage are released once
      // the second half is loaded
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t uoff[4];
        u_offsets(row, (grp & 1) * 2 + h, uoff, TL());
        uint32_t braw[16];
        tc::tmem_ld16(t_lane + (uint32_t)(rb.idx * kDNT + h * 16), braw);
        float u[16];
        load_u16(sU + ru.idx * kUBytes, uoff, u, TL());
        tc::tmem_ld_wait();
        if (h == 1) {
          tc::fence_before_sync();
          __syncwarp();
          tc::mbar_arrive2_if(&tempty[rb.idx], &empty_u[ru.idx], lane == 0);
        }
        const int colbase = (t_begin + t) * kDNT + grp * 32 + h * 16;
        float2 z[8];  // U + bias (the temperature is folded into kscale)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          z[i] = __fadd2_rn(make_float2(u[2 * i], u[2 * i + 1]),
                            make_float2(__uint_as_float(braw[2 * i]), __uint_as_float(braw[2 * i + 1])));
        if (colbase + 16 > V) {  // vocabulary tail (last tile only)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (colbase + 2 * i >= V) z[i].x = -CUDART_INF_F;
            if (colbase + 2 * i + 1 >= V) z[i].y = -CUDART_INF_F;
          }
        }
        // e = 2^(z kscale - ref) for the 16 columns and their sum (a tree)
        float2 e[8];
        {
          const float2 nref2 = make_float2(nref, nref);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 a = __ffma2_rn(z[i], kscale2, nref2);
            e[i] = make_float2(tc::ex2(a.x), tc::ex2(a.y));
          }
        }
        float2 s4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) s4[i] = __fadd2_rn(e[2 * i], e[2 * i + 1]);
        const float2 s2 = __fadd2_rn(__fadd2_rn(s4[0], s4[1]), __fadd2_rn(s4[2], s4[3]));
        float ts = s2.x + s2.y;
        // Rare: the row's first tile (no reference yet: the weights above were
        // taken against 0 and are redone), a logit far above the reference, or
        // a running sum about to grow too large; one test for all three.
        if (!(st.m > -CUDART_INF_F) || !(ts <= 1e37f) || st.s + ts > 1e30f) {
          if (!(st.m > -CUDART_INF_F)) {
            // First tile of the row: fix the reference at the tile's maximum and
            // seed the race with that element (without a bound every element of
            // the first tile would take the exact test).  Its e is computed
            // exactly as the tile's weights are.
            float mz = z[0].x;
            int im = 0;
#pragma unroll
            for (int j = 1; j < 16; ++j) {
              const float zj = (j & 1) ? z[j >> 1].y : z[j >> 1].x;
              if (zj > mz) {
                mz = zj;
                im = j;
              }
            }
            if (!(mz > -CUDART_INF_F)) continue;
            st.m = mz * kscale;
            nref = -st.m;
            const uint4 bits = philox_in_row((uint32_t)(colbase >> 2) + (uint32_t)(im >> 2), prow, p.rk);
            if (race_candidate(st, tc::ex2(fmaf(mz, kscale, nref)), word_of(bits, im & 3), colbase + im,
                               row_best, *reinterpret_cast<volatile uint32_t*>(row_best), global_best))
              c_own = __fdividef(st.bE, st.be) * kFilterUp;
            // the tile's weights and their sum against the new reference
            ts = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              e[i] = make_float2(tc::ex2(fmaf(z[i].x, kscale, nref)), tc::ex2(fmaf(z[i].y, kscale, nref)));
              ts += e[i].x + e[i].y;
            }
          } else if (!(ts <= 1e37f)) {  // a logit far above the reference (or a NaN): re-reference
            float mz = fmaxf(z[0].x, z[0].y);
#pragma unroll
            for (int i = 1; i < 8; ++i) mz = fmaxf(mz, fmaxf(z[i].x, z[i].y));
            const float mnew = fmaxf(mz * kscale, st.m);
            const float sc = tc::ex2(st.m - mnew);
            st.s *= sc;
            st.be *= sc;
            st.m = mnew;
            nref = -mnew;
            c_own = st.be > 0.f ? (st.bE / st.be) * kFilterUp : CUDART_INF_F;
            ts = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              e[i] = make_float2(tc::ex2(fmaf(z[i].x, kscale, nref)), tc::ex2(fmaf(z[i].y, kscale, nref)));
              ts += e[i].x + e[i].y;
            }
          }
          st.s += ts;
          if (st.s > 1e30f) {  // keep the sum far from overflow: exact rescale by 2^-64
            st.s *= 0x1p-64f;
            st.be *= 0x1p-64f;
            st.m += 64.f;
            nref -= 64.f;
            c_own = st.be > 0.f ? (st.bE / st.be) * kFilterUp : CUDART_INF_F;
            // the tile's weights move to the new reference too: the filter and the
            // exact tests below compare them with the rescaled best
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = make_float2(e[i].x * 0x1p-64f, e[i].y * 0x1p-64f);
          }
        } else {
          st.s += ts;
        }
        // Filter factor for the tile: the tighter of the thread's own best and
        // the best any thread of this row in the CTA has published.  An element
        // passes when f <= e c + 1, f = 1 + (1 - u) - 2^-24; with g = e c + 1 >= 1
        // and f in [1, 2) the difference g - f is exact, so its sign decides.
        float2 cf2;
        cf2.x = fminf(c_own, tc::ex2(st.m - key_value(*reinterpret_cast<volatile uint32_t*>(row_best))) *
                                 kFilterUp);
        cf2.y = cf2.x;
        const float2 one2 = make_float2(1.f, 1.f);
        // All four Philox blocks and the filter of the 16 columns in one
        // straight-line block (the compiler interleaves the chains with the
        // arithmetic); one branch to the rare exact tests.
        uint32_t words[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 bits = philox_in_row((uint32_t)(colbase >> 2) + q, prow, p.rk);
          words[4 * q] = bits.x;
          words[4 * q + 1] = bits.y;
          words[4 * q + 2] = bits.z;
          words[4 * q + 3] = bits.w;
        }
        uint32_t all_neg = 0xffffffffu;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 d = __fadd2_rn(__ffma2_rn(e[i], cf2, one2),
                                      make_float2(neg_one_plus_w(words[2 * i]), neg_one_plus_w(words[2 * i + 1])));
          all_neg &= __float_as_uint(d.x) & __float_as_uint(d.y);
        }
        if (!(all_neg >> 31)) {  // rare: elements that could beat the best, in index order
          uint32_t mask = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 d = __fadd2_rn(__ffma2_rn(e[i], cf2, one2),
                                        make_float2(neg_one_plus_w(words[2 * i]), neg_one_plus_w(words[2 * i + 1])));
            mask |= ((__float_as_uint(d.x) >> 31) ^ 1u) << (2 * i);
            mask |= ((__float_as_uint(d.y) >> 31) ^ 1u) << (2 * i + 1);
          }
          if (colbase + 16 > V) mask &= (V > colbase) ? (1u << (V - colbase)) - 1u : 0u;
          while (mask) {
            const int i = __ffs(mask) - 1;
            mask &= mask - 1u;
            // column i's weight and word by a select tree on the bits of i
            float e8[8], e4[4], e2[2];
            uint32_t w8[8], w4[4], w2[2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              e8[j] = (i & 1) ? e[j].y : e[j].x;
              w8[j] = (i & 1) ? words[2 * j + 1] : words[2 * j];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              e4[j] = (i & 2) ? e8[2 * j + 1] : e8[2 * j];
              w4[j] = (i & 2) ? w8[2 * j + 1] : w8[2 * j];
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              e2[j] = (i & 4) ? e4[2 * j + 1] : e4[2 * j];
              w2[j] = (i & 4) ? w4[2 * j + 1] : w4[2 * j];
            }
            const float ei = (i & 8) ? e2[1] : e2[0];
            const uint32_t wi = (i & 8) ? w2[1] : w2[0];
            if (race_candidate(st, ei, wi, colbase + i, row_best, *reinterpret_cast<volatile uint32_t*>(row_best),
                               global_best)) {
              c_own = __fdividef(st.bE, st.be) * kFilterUp;
              cf2.x = fminf(cf2.x, c_own);
              cf2.y = cf2.x;
            }
          }
        }
      }
    }
    // Merge the four column groups of each row inside the CTA, through the
    // stage buffers (every issued load has been consumed once all epilogue
    // warps reach the barrier).
    Race* grp_state = reinterpret_cast<Race*>(sU);  // [3][128]
    named_bar_sync(2, kEpiWarps * 32);
    if (grp > 0) grp_state[(grp - 1) * 128 + row] = st;
    named_bar_sync(2, kEpiWarps * 32);
    if (grp == 0 && valid) {
#pragma unroll
      for (int g = 0; g < 3; ++g) st = race_merge2(st, grp_state[g * 128 + row]);
      Partial w{};
      w.f0 = st.m;
      w.f1 = st.s;
      w.f2 = st.be;
      w.f3 = st.bE;
      w.i0 = st.idx;
      partial_slot(p, k)[(size_t)m * p.nsplit + split] = w;
    }
  }

  // ----------------------------------------------------------- teardown --
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kDTmemCols);
  }
  // Positions before the last are merged by the next position's grid.
  if (k < p.gamma) return;
  if (!last_block_arrives(p.counters + mtile, (unsigned)p.nsplit)) return;

  // Last CTA of this request tile at the last position: merge its partials.
  if (threadIdx.x < kEpiWarps * 32) merge_position(p, partial_slot(p, k), m0, k, true, nullptr);
}

// ------------------------------------------------------------------ host --
namespace {

template <typename TL, int KC>
size_t smem_bytes(int stages) {
  return 1024 + (size_t)KC * 16384 + (size_t)c_stages(KC) * KC * kDNT * 128 + (size_t)stages * UTile<TL>::kBytes;
}

template <typename TL, int KC>
int pick_stages() {
  const size_t budget = kSmemBudget;
  int s = kMaxStages;
  while (s > 2 && smem_bytes<TL, KC>(s) > budget) --s;
  return s;
}

template <typename TL, int KC>
cudaError_t launch_typed(const DraftTCParams& base, const void* U, const void* Ct,
                         cudaStream_t stream) {
  DraftTCParams p = base;
  CUtensorMap tm_u, tm_c;
  const CUtensorMapDataType udt =
      sizeof(TL) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t udims[3] = {(uint64_t)p.V, (uint64_t)p.gamma, (uint64_t)p.R};
  const uint32_t ubox[3] = {(uint32_t)UTile<TL>::kBoxCols, 1, 128};
  const uint64_t cdims[3] = {(uint64_t)p.rank, (uint64_t)p.V, (uint64_t)p.gamma};
  const uint32_t cbox[3] = {64, (uint32_t)kDNT, 1};
  if (!encode_tiled(&tm_u, udt, sizeof(TL), U, 3, udims, ubox) ||
      !encode_tiled(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ct, 3, cdims, cbox))
    return cudaErrorInvalidValue;
  p.rk = philox_round_keys(p.key);
  p.ntiles = (p.V + kDNT - 1) / kDNT;
  p.stages = pick_stages<TL, KC>();
  const size_t smem = smem_bytes<TL, KC>(p.stages);
  auto kern = (p.R % 128 != 0) ? draft_tc_kernel<TL, KC, true> : draft_tc_kernel<TL, KC, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.mtiles * p.nsplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  RnnStateParams q{};
  if (p.S) {
    q.R = p.R;
    q.gamma = p.gamma;
    q.V = p.V;
    q.rank = p.rank;
    q.x0 = p.x0;
    q.x = p.x;
    q.q_tok = p.q_tok;
    q.lse_q = p.lse_q;
    q.A = p.A;
    q.W = p.W;
    q.S = p.S;
    q.status = p.status;
  }
  for (int k = 1; k <= p.gamma; ++k) {
    p.k = k;
    if (p.S) {  // RNN head: merge position k-1, then s_k, before the grid of position k
      q.k = k;
      q.nsplit = k > 1 ? p.nsplit : 0;
      q.part = p.partials + (size_t)((k - 1) & 1) * p.R * p.nsplit;
      err = launch_rnn_state(q, /*fac_f32=*/false, /*pdl=*/true, stream);
      if (err != cudaSuccess) return err;
    }
    err = cudaLaunchKernelEx(&cfg, kern, tm_u, tm_c, p);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace

int draft_tc_nsplit(int R, int V, int device_sms) {
  const int mtiles = (R + 127) / 128;
  const int ntiles = (V + kDNT - 1) / kDNT;
  int ns = std::max(1, device_sms / mtiles);
  return std::max(1, std::min(ns, ntiles));
}

cudaError_t launch_draft_tc(const DraftTCParams& p, int logit_dtype, const void* U, const void* Ct,
                            cudaStream_t stream) {
  const int KC = p.rank / 64;
  if (logit_dtype == SPEC_F32) {
    switch (KC) {
      case 1: return launch_typed<float, 1>(p, U, Ct, stream);
      case 2: return launch_typed<float, 2>(p, U, Ct, stream);
      case 3: return launch_typed<float, 3>(p, U, Ct, stream);
      case 4: return launch_typed<float, 4>(p, U, Ct, stream);
    }
  } else {
    switch (KC) {
      case 1: return launch_typed<__nv_bfloat16, 1>(p, U, Ct, stream);
      case 2: return launch_typed<__nv_bfloat16, 2>(p, U, Ct, stream);
      case 3: return launch_typed<__nv_bfloat16, 3>(p, U, Ct, stream);
      case 4: return launch_typed<__nv_bfloat16, 4>(p, U, Ct, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace spec
