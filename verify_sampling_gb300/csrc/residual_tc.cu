// Fused residual resample on the tensor cores (sm_100 family).
//
// For every request whose first rejection is at position j* = k the target
// token is regenerated from norm(max(0, p - q)) at row k (history article,
// "1.1运行机制"; DSpark summary, Figure 1): Gumbel-max over
// log(max(0, p_v - q_v)) + G_v with the purpose-2 stream, i.e. argmax of
// res_v / E_v in race form; if no residual is positive, the same race over
// p_v.  q_v = exp(z_v - lse_q) with z the draft logits of row k:
//     z[m, v] = (U[m, k, v] + A_k[x_{m,k-1}, :] . C_k[:, v]) / T_k,
// so the bias is again a rank-r GEMM: the requests of one position form the
// M dimension (gathered, up to kResTileRows per tile and replicated to the
// 128 rows of the MMA), the vocabulary the N dimension.
// p_v = 2^(L_v log2e / T_t - m_t) / s_t uses the softmax reference/sum of the target row
// that the verify row pass stored.
//
// The same pass, instantiated with kCStar, sums min(p_v, q_v) over the
// vocabulary for every verified draft row instead (DSpark summary, "2.1
// 置信度头": c* = 1 - TV(p, q), the confidence head's calibration target).
//
// Layout and pipelines follow the fused draft kernel (fused_tc.cuh): one CTA
// per SM, 16 epilogue warps, a TMA producer warp and an MMA warp.  Two rings:
// the C_k tiles (one per 64-column tile, freed by the MMA) and the gathered
// rows (U row and target row of every request of the tile, w consecutive
// 64-column tiles per stage, one bulk copy per request and operand, freed by
// the epilogue after its w-th tile).  w is chosen per CTA from the number of
// gathered rows: with few rows each copy spans up to 512 columns, since the
// cost of a gather is the number of copies, not their bytes.  Work split: the
// request tiles of all positions are counted on the device; CTA b takes tile
// b % M and vocabulary split b / M.
#include "fused_tc.cuh"
#include "draft_tc.cuh"
#include "residual_tc.cuh"
#include "tc.cuh"

namespace spec {

namespace {

using namespace fused;

__device__ __forceinline__ WRace wrace_merge_(const WRace& a, const WRace& b) {
  return race_beats(b.bw, b.bE, b.idx, a.bw, a.bE, a.idx) ? b : a;
}

// Gathered rows are copied linearly, w 64-column segments per request, with a
// 16-byte pad per row (pitch = w * 64 * size + 16, 16 modulo 128) so that
// eight consecutive rows reading the same 16-byte chunk hit eight different
// bank groups.
template <typename T>
__host__ __device__ constexpr uint32_t row_pitch(int w) {
  return (uint32_t)w * kNT * sizeof(T) + 16u;
}

// 8 consecutive values of `row` from column `col` of a gathered block.
__device__ __forceinline__ void load_row8(const unsigned char* blk, uint32_t pitch, int row, int col,
                                          float (&v)[8], float) {
  const unsigned char* base = blk + row * pitch + col * 4;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float4 f = *reinterpret_cast<const float4*>(base + 16 * j);
    v[4 * j] = f.x;
    v[4 * j + 1] = f.y;
    v[4 * j + 2] = f.z;
    v[4 * j + 3] = f.w;
  }
}
__device__ __forceinline__ void load_row8(const unsigned char* blk, uint32_t pitch, int row, int col,
                                          float (&v)[8], __nv_bfloat16) {
  const uint4 q = *reinterpret_cast<const uint4*>(blk + row * pitch + col * 2);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    v[2 * h] = __uint_as_float(w[h] << 16);
    v[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
  }
}

}  // namespace

using namespace fused;

// 576 threads per CTA leave at most 96 registers per thread.
template <typename TT, typename TL, int KC, bool kCStar>
__global__ void __launch_bounds__(kThreads, 1)
    resid_tc_kernel(const __grid_constant__ CUtensorMap tm_c, const TL* __restrict__ U,
                    const TT* __restrict__ tgt, ResidTCParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kCBytes = KC * kNT * 128;
  unsigned char* sA = smem;
  unsigned char* sC = smem + KC * 16384;  // C ring, then the row ring

  __shared__ __align__(8) uint64_t full_c[kMaxStages], empty_c[kMaxStages];
  __shared__ __align__(8) uint64_t full_r[kMaxStages], empty_r[kMaxStages];
  __shared__ __align__(8) uint64_t tfull[kTmemBufs], tempty[kTmemBufs];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int s_tile[5];  // M, k, first list index, rows, splits
  __shared__ int s_req[128];
  __shared__ uint32_t s_rbest[kResTileRows];  // per request slot: best published score (ordered key)
  __shared__ int s_trow[128];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.gamma;

  // ---- work assignment (identical in every CTA) -------------------------
  if (threadIdx.x == 0) {
    int M = 0;
    for (int kk = 0; kk < G; ++kk) M += (p.res_cnt[kk] + kResTileRows - 1) / kResTileRows;
    int nsplit = M > 0 ? max(1, (int)gridDim.x / M) : 1;
    nsplit = min(min(nsplit, p.ntiles), kMaxDeviceSms);
    int mt = M > 0 ? (int)blockIdx.x % M : 0, split = M > 0 ? (int)blockIdx.x / M : 0;
    int k = 0, i0 = 0, rows = 0;
    if (M > 0 && split < nsplit) {
      int acc = 0;
      for (int kk = 0; kk < G; ++kk) {
        const int n = (p.res_cnt[kk] + kResTileRows - 1) / kResTileRows;
        if (mt < acc + n) {
          k = kk + 1;
          i0 = (mt - acc) * kResTileRows;
          rows = min(kResTileRows, p.res_cnt[kk] - i0);
          break;
        }
        acc += n;
      }
    }
    s_tile[0] = (rows > 0) ? M : 0;
    s_tile[1] = k;
    s_tile[2] = i0;
    s_tile[3] = rows;
    s_tile[4] = nsplit;
  }
  __syncthreads();
  const int M = s_tile[0];
  if (M == 0) return;  // nothing to do (uniform across the CTA)
  const int nsplit = s_tile[4];
  const int k = s_tile[1], i0 = s_tile[2], nrows = s_tile[3];
  const int mt = (int)blockIdx.x % M, split = (int)blockIdx.x / M;
  const int t_begin = (int)((long)split * p.ntiles / nsplit);
  const int t_end = (int)((long)(split + 1) * p.ntiles / nsplit);
  const int T = t_end - t_begin;
  const int G1 = G + 1;
  // Ring sizes for this tile's gathered rows (at most kResTileRows): the
  // widest row stage (gw tiles) of which three fit next to three C stages,
  // then as many C stages as leave room for three row stages (up to six), and
  // the rest for row stages.  The host checks that two C stages and one row
  // stage of gw = 1 always fit.
  const uint32_t avail0 = (uint32_t)p.smem_bytes - 1024u - KC * 16384u;
  int gw = 1;  // 64-column tiles per row stage
  uint32_t pitch_u = row_pitch<TL>(1), pitch_t = row_pitch<TT>(1);
  uint32_t rstage = ((uint32_t)nrows * (pitch_u + pitch_t) + 127u) & ~127u;
  for (int cand = 8; cand > 1; cand >>= 1) {
    const uint32_t pu = row_pitch<TL>(cand), pt = row_pitch<TT>(cand);
    const uint32_t bytes = ((uint32_t)nrows * (pu + pt) + 127u) & ~127u;
    if (3u * bytes + 3u * kCBytes <= avail0) {
      gw = cand;
      pitch_u = pu;
      pitch_t = pt;
      rstage = bytes;
      break;
    }
  }
  int Sc = 2;
  while (Sc < 6 && (uint32_t)(Sc + 1) * kCBytes + 3u * rstage <= avail0) ++Sc;
  const uint32_t fit = (avail0 - (uint32_t)Sc * kCBytes) / rstage;
  const int Sr = (int)(fit < (uint32_t)kMaxStages ? fit : (uint32_t)kMaxStages);
  unsigned char* sRow = sC + Sc * kCBytes;
  const uint32_t u_block = (uint32_t)nrows * pitch_u;  // target rows follow the U rows
  // Sixteen requests fill half of one TMEM lane quadrant, so the A tile holds
  // them eight times (row i holds request slot i % 16).  In every quadrant,
  // lanes 16-31 repeat the requests of lanes 0-15 and take the other half of
  // the warp's columns, and quadrant g takes the tiles t with t % 4 == g: all
  // 512 epilogue lanes work.
  static_assert(kResTileRows == 16, "the replication assumes 16-request tiles");
  constexpr int kSlots = 16;
  for (int i = threadIdx.x; i < 128; i += blockDim.x) {
    int r = -1, trow = 0;
    if (i < nrows) {
      r = p.res_list[(size_t)(k - 1) * p.R + i0 + i];
      trow = p.tgt_row_off[r] + (k - 1);
    }
    s_req[i] = r;
    s_trow[i] = trow;
    if (i < kResTileRows) s_rbest[i] = 0u;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < Sc; ++s) {
      tc::mbar_init(&full_c[s], 1);
      tc::mbar_init(&empty_c[s], 1);
    }
    for (int s = 0; s < Sr; ++s) {
      tc::mbar_init(&full_r[s], 1);
      tc::mbar_init(&empty_r[s], kEpiWarps);
    }
    for (int b = 0; b < kTmemBufs; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);  // the four warps of the tile's quadrant
    }
    abort_flag = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);
  if (warp == kProducerWarp && lane == 0) tc::tma_prefetch_desc(&tm_c);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  auto fail = [&]() {
    abort_flag = 1;
    set_status(p.status, SPEC_STATUS_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // Lane 0 loads the C tiles and arms the barriers; all 32 lanes issue the
    // row copies of a group (one per request and operand, w tiles wide).
    int issued_c = 0, issued_g = 0;
    Ring rc{0, 0u}, rr{0, 0u};
    for (int t = 0; t < T && !abort_flag; ++t, rc.next(Sc)) {
      const int n0 = (t_begin + t) * kNT;
      if (t % gw == 0) {
        bool ok = true;
        if (lane == 0) ok = tc::mbar_wait(&empty_r[rr.idx], rr.phase ^ 1u, kWaitNs);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          if (lane == 0) fail();
          break;
        }
        unsigned char* st = sRow + rr.idx * rstage;
        // columns of this group inside the split and the vocabulary (a
        // multiple of 16 bytes in both dtypes, because V times the element
        // size is)
        const int seg = min(min(gw, T - t) * kNT, p.V - n0);
        const uint32_t ub = (uint32_t)seg * sizeof(TL), tb = (uint32_t)seg * sizeof(TT);
        if (lane == 0) tc::mbar_expect_tx(&full_r[rr.idx], (uint32_t)nrows * (ub + tb));
        __syncwarp();
        for (int i = lane; i < nrows; i += 32) {
          const size_t urow = (size_t)s_req[i] * p.gamma + (k - 1);
          tc::bulk_load(st + i * pitch_u, U + urow * p.V + n0, ub, &full_r[rr.idx]);
          tc::bulk_load(st + u_block + i * pitch_t, tgt + (size_t)s_trow[i] * p.V + n0, tb,
                        &full_r[rr.idx]);
        }
        issued_g += 1;
        rr.next(Sr);
      }
      bool ok = true;
      if (lane == 0) ok = tc::mbar_wait(&empty_c[rc.idx], rc.phase ^ 1u, kWaitNs);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      if (lane == 0) {
        unsigned char* st = sC + rc.idx * kCBytes;
        tc::mbar_expect_tx(&full_c[rc.idx], kCBytes);
#pragma unroll
        for (int kc = 0; kc < KC; ++kc)
          tc::tma_load_3d(st + kc * 8192, &tm_c, &full_c[rc.idx], kc * 64, n0, k - 1);
      }
      __syncwarp();
      issued_c = t + 1;
    }
    if (abort_flag && lane == 0) {
      // the copies still in flight must land before the CTA exits
      for (int t = (issued_c > Sc ? issued_c - Sc : 0); t < issued_c; ++t)
        tc::mbar_wait(&full_c[t % Sc], (uint32_t)(t / Sc) & 1u, kWaitNs);
      for (int g = (issued_g > Sr ? issued_g - Sr : 0); g < issued_g; ++g)
        tc::mbar_wait(&full_r[g % Sr], (uint32_t)(g / Sr) & 1u, kWaitNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    named_bar_sync(1, (kEpiWarps + 1) * 32);
    if (lane == 0) {
      constexpr uint32_t idesc = tc::bf16_idesc(128, kNT);
      int last = -1;
      Ring r{0, 0u}, rb{0, 0u};
      const uint32_t a_base = tc::smem_u32(sA);
      for (int t = 0; t < T && !abort_flag; ++t, r.next(Sc), rb.next(kTmemBufs)) {
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
          tc::mma_bf16(tmem + (uint32_t)(rb.idx * kNT), tc::sw128_desc(a_base + kc * 16384 + ko),
                       tc::sw128_desc(b_base + kc * 8192 + ko), idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&tfull[rb.idx]);
        tc::mma_commit(&empty_c[r.idx]);
        last = t;
      }
      if (abort_flag && last >= 0)
        tc::mbar_wait(&tfull[last % kTmemBufs], (uint32_t)(last / kTmemBufs) & 1u, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quad = warp & 3, grp = warp >> 2;
    const int slot = lane & (kSlots - 1), half = lane >> 4;  // request slot, column half
    const bool valid = slot < nrows;
    // the stages hold exactly nrows rows: lanes past them read row 0 (unused)
    const int lrow = valid ? slot : 0;
    const int V = p.V, rank = p.rank;
    for (int idx = threadIdx.x; idx < 128 * KC * 8; idx += kEpiWarps * 32) {
      const int i = idx / (KC * 8), c = idx % (KC * 8);
      uint4 val = make_uint4(0, 0, 0, 0);
      if (i % kSlots < nrows) {
        const int req = s_req[i % kSlots];
        int xp = (k == 1) ? p.x0[req] : p.x[(size_t)req * G + (k - 2)];
        if (xp < 0 || xp >= V) xp = 0;
        val = *reinterpret_cast<const uint4*>(bias_row<__nv_bfloat16>(p.A, p.S, V, rank, G, k, req, xp) +
                                              c * 8);
      }
      const int kc = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(sA + kc * 16384 + i * 128 + ((cc ^ (i & 7)) << 4)) = val;
    }
    tc::fence_proxy_async();
    named_bar_sync(1, (kEpiWarps + 1) * 32);

    // Per-request constants (log2 units): q = 2^(z kq + nlq), p = 2^(L kt + nt) / s_t.
    const int req = valid ? s_req[slot] : 0;
    const uint32_t rid = p.rid_base + (uint32_t)req;
    const size_t rk1 = (size_t)req * G + (k - 1);
    const size_t rj = (size_t)req * G1 + (k - 1);
    const float kq = kLog2e / p.draft_temp[k - 1];
    const float nlq = valid ? -p.lse_q[rk1] * kLog2e : 0.f;
    const float kt = kLog2e * p.inv_target_temp;
    const float nt = valid ? -p.row_m[rj] : 0.f;  // row_m is in log2 units
    const float inv_s = valid ? 1.0f / p.row_s[rj] : 0.f;
    unsigned* row_best = p.row_best + req;
    // the row-constant parts of the first two Philox rounds, once per thread
    const PhiloxRow prow = philox_row((uint32_t)k, rid, kPurposeResidual, p.rk);
    // Race on the residual: an element can beat a best (bw, bE) only if
    // 1 - u <= res * bE / bw (filter as in the draft kernel, with the shared
    // per-request bound).  Requests with no positive residual anywhere are
    // flagged by the final combine and served by the fallback kernel.
    WRace rres = wrace_empty();
    float csum = 0.f;  // kCStar: this thread's sum of min(p, q)
    float c_res = CUDART_INF_F;
    uint32_t shared_key = 0;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(grp * 16);
    Ring rr{0, 0u}, rb{0, 0u};
    for (int t = 0; t < T; ++t, rb.next(kTmemBufs)) {
      if (abort_flag) break;
      const bool group_done = (t % gw == gw - 1) || (t == T - 1);
      // Every warp waits for each row group (so none runs a ring lap ahead)
      // and releases it after the group's last tile; only the tile's quadrant
      // waits for the accumulator and computes.
      const bool own = (t & 3) == quad;
      if ((t % gw == 0 || own) && !tc::mbar_wait(&full_r[rr.idx], rr.phase, kWaitNs)) {
        fail();
        break;
      }
      if (!own) {
        __syncwarp();
        if (group_done) {
          if (lane == 0) tc::mbar_arrive(&empty_r[rr.idx]);
          rr.next(Sr);
        }
        continue;
      }
      // the request's bound: the CTA's own best so far (shared memory, every
      // candidate of the tile's 32 thread streams raises it at once) and the
      // best of all CTAs (global, read one own tile late)
      const uint32_t shared_now = max(shared_key, *reinterpret_cast<volatile uint32_t*>(&s_rbest[slot]));
      if (!kCStar && valid) shared_key = __ldcg(row_best);
      if (!tc::mbar_wait(&tfull[rb.idx], rb.phase, kWaitNs)) {
        fail();
        break;
      }
      tc::fence_after_sync();
      const unsigned char* sr = sRow + rr.idx * rstage;
      const int col = (t % gw) * kNT + grp * 16 + 8 * half;
      // q first (frees the bias and U registers), then the target row: the
      // lane's 8 columns of the warp's 16.
      float qv[8], L[8];
      {
        uint32_t braw[16];
        float u[8];
        tc::tmem_ld16(t_lane + (uint32_t)(rb.idx * kNT), braw);
        load_row8(sr, pitch_u, lrow, col, u, TL());
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float b = __uint_as_float(half ? braw[8 + c] : braw[c]);
          qv[c] = tc::ex2(fmaf(u[c] + b, kq, nlq));
        }
      }
      load_row8(sr + u_block, pitch_t, lrow, col, L, TT());
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&tempty[rb.idx]);
        if (group_done) tc::mbar_arrive(&empty_r[rr.idx]);
      }
      if (group_done) rr.next(Sr);
      if (!valid) continue;
      const int colbase = (t_begin + t) * kNT + grp * 16 + 8 * half;
      if constexpr (kCStar) {
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (colbase + c < V) part += fminf(tc::ex2(fmaf(L[c], kt, nt)) * inv_s, qv[c]);
        csum += part;
      } else {
        float res[8];  // p - q of the 8 columns
#pragma unroll
        for (int i = 0; i < 8; ++i) res[i] = tc::ex2(fmaf(L[i], kt, nt)) * inv_s - qv[i];
        // Both Philox blocks and the filter of the 8 columns in one straight-line
        // block; one branch to the rare exact tests.
        uint32_t words[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 bits = philox_in_row((uint32_t)((colbase >> 2) + q), prow, p.rk);
          words[4 * q] = bits.x;
          words[4 * q + 1] = bits.y;
          words[4 * q + 2] = bits.z;
          words[4 * q + 3] = bits.w;
        }
        if (!(c_res < CUDART_INF_F)) {
          // No own candidate yet: seed the race with the largest positive residual
          // of these 8 columns (one exact test), so that the filter has a bound
          // from the first tile on instead of sending every element of it to the
          // exact test.  The seed is an element of the race like any other.
          float rm = 0.f;
          int im = -1;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (res[i] > rm && colbase + i < V) {
              rm = res[i];
              im = i;
            }
          if (im >= 0) {
            uint32_t wm = words[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) wm = (im == j) ? words[j] : wm;
            const float E = -logf(uniform_from_word(wm));
            if (race_beats(rm, E, colbase + im, rres.bw, rres.bE, rres.idx)) {
              rres = WRace{rm, E, colbase + im};
              c_res = __fdividef(E, rm) * kFilterUp;
              const uint32_t key = ordered_key(lg2(rm) - lg2(E) - kPublishMargin);
              atomicMax(&s_rbest[slot], key);
              atomicMax(row_best, key);
            }
          }
        }
        const float cr = fminf(c_res, tc::ex2(-key_value(shared_now)) * kFilterUp);  // NaN: none yet
        uint32_t mask = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mask |= (one_plus_w(words[i]) <= fmaf(res[i], cr, 1.0f) && res[i] > 0.f) ? (1u << i) : 0u;
        if (mask) {  // rare: exact race tests, in index order
          if (colbase + 8 > V) mask &= (V > colbase) ? (1u << (V - colbase)) - 1u : 0u;
          while (mask) {
            const int i = __ffs(mask) - 1;
            mask &= mask - 1u;
            float ri = res[0];
            uint32_t wi = words[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) {
              ri = (i == j) ? res[j] : ri;
              wi = (i == j) ? words[j] : wi;
            }
            const float E = -logf(uniform_from_word(wi));
            if (race_beats(ri, E, colbase + i, rres.bw, rres.bE, rres.idx)) {
              rres = WRace{ri, E, colbase + i};
              c_res = __fdividef(E, ri) * kFilterUp;
              const uint32_t key = ordered_key(lg2(ri) - lg2(E) - kPublishMargin);
              atomicMax(&s_rbest[slot], key);
              atomicMax(row_best, key);
            }
          }
        }
      }
    }
    if constexpr (kCStar) {
      // quadrants, column groups, halves and splits all add into the row's sum
      if (valid && !abort_flag) atomicAdd(&p.c_star[rk1], csum);
    } else {
      // merge the 32 states of each request (quadrant, column group, column
      // half) through shared memory: [32][16]
      WRace* st_all = reinterpret_cast<WRace*>(sC);
      constexpr int kStates = 32;
      named_bar_sync(2, kEpiWarps * 32);
      if (valid) st_all[((quad * 4 + grp) * 2 + half) * kSlots + slot] = rres;
      named_bar_sync(2, kEpiWarps * 32);
      if (valid && quad == 0 && grp == 0 && half == 0) {
        for (int g = 1; g < kStates; ++g) rres = wrace_merge_(rres, st_all[g * kSlots + slot]);
        Partial pw{};
        pw.f0 = rres.bw;
        pw.f1 = rres.bE;
        pw.i0 = rres.idx;
        p.partials[((size_t)mt * kResTileRows + slot) * nsplit + split] = pw;
      }
    }
  }

  // ----------------------------------------------------------- teardown --
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (kCStar) return;
  if (!last_block_arrives(p.counters + mt, (unsigned)nsplit)) return;

  static_assert(kEpiWarps * 32 / 16 >= kResTileRows, "sixteen merge threads per request");
  // Last CTA of this request tile: merge the splits, sixteen threads per
  // request with all their loads in flight (one round trip up to 128 splits).
  if (threadIdx.x < kEpiWarps * 32) {
    const int row = threadIdx.x >> 4, part = threadIdx.x & 15;
    WRace a = wrace_empty();
    if (row < nrows) {
      const Partial* src = p.partials + ((size_t)mt * kResTileRows + row) * nsplit;
      for (int s0 = part; s0 < nsplit; s0 += 16 * 8) {
        Partial w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (s0 + 16 * q < nsplit) w[q] = load_partial(src + s0 + 16 * q);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (s0 + 16 * q < nsplit) a = wrace_merge_(a, WRace{w[q].f0, w[q].f1, w[q].i0});
      }
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) a = wrace_merge_(a, wrace_shfl_xor(a, off));
    if (part == 0 && row < nrows) {
      const int req = s_req[row];
      if (a.idx >= 0)
        p.out_tok[(size_t)req * G1 + (k - 1)] = a.idx;
      else
        p.fallback[req] = k;  // no positive residual: sample from p instead
    }
  }
}

// ------------------------------------------------------------------ host --
namespace {

// The kernel splits whatever shared memory it gets into rings sized for its
// rows; two C stages and one row stage of a full tile must fit.
template <typename TT, typename TL, int KC>
size_t min_smem_bytes() {
  const size_t row1 = kResTileRows * (size_t)(row_pitch<TL>(1) + row_pitch<TT>(1));
  return 1024 + (size_t)KC * 16384 + 2 * (size_t)KC * kNT * 128 + ((row1 + 127) & ~(size_t)127);
}

template <typename TT, typename TL, int KC>
cudaError_t launch_typed(const ResidTCParams& base, const void* tgt, const void* U, const void* Ct,
                         int grid, bool cstar, cudaStream_t stream) {
  ResidTCParams p = base;
  CUtensorMap tm_c;
  const uint64_t cdims[3] = {(uint64_t)p.rank, (uint64_t)p.V, (uint64_t)p.gamma};
  const uint32_t cbox[3] = {64, (uint32_t)kNT, 1};
  if (!encode_tiled(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ct, 3, cdims, cbox))
    return cudaErrorInvalidValue;
  // all of the per-CTA shared memory but 4 KB left for the static arrays
  const size_t smem = 227 * 1024 - 4096;
  if (min_smem_bytes<TT, TL, KC>() > smem) return cudaErrorInvalidValue;
  p.smem_bytes = (int)smem;
  auto kern = cstar ? resid_tc_kernel<TT, TL, KC, true> : resid_tc_kernel<TT, TL, KC, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, smem, stream>>>(tm_c, static_cast<const TL*>(U), static_cast<const TT*>(tgt), p);
  return cudaGetLastError();
}

template <typename TT, typename TL>
cudaError_t launch_kc(const ResidTCParams& p, const void* tgt, const void* U, const void* Ct,
                      int grid, bool cstar, cudaStream_t stream) {
  switch (p.rank / 64) {
    case 1: return launch_typed<TT, TL, 1>(p, tgt, U, Ct, grid, cstar, stream);
    case 2: return launch_typed<TT, TL, 2>(p, tgt, U, Ct, grid, cstar, stream);
    case 3: return launch_typed<TT, TL, 3>(p, tgt, U, Ct, grid, cstar, stream);
    case 4: return launch_typed<TT, TL, 4>(p, tgt, U, Ct, grid, cstar, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool resid_tc_supported(int tgt_dtype, int logit_dtype, int fac_dtype, int rank, int V,
                        const void* tgt, const void* U, const void* A, const void* Ct) {
  auto es = [](int d) { return d == SPEC_F32 ? (size_t)4 : (size_t)2; };
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  return fac_dtype == SPEC_BF16 && rank % 64 == 0 && rank <= 256 &&
         ((size_t)V * es(logit_dtype)) % 16 == 0 && ((size_t)V * es(tgt_dtype)) % 16 == 0 &&
         al16(tgt) && al16(U) && al16(A) && al16(Ct);
}

cudaError_t launch_resid_tc(const ResidTCParams& p, int tgt_dtype, int logit_dtype, const void* tgt,
                            const void* U, const void* Ct, int grid, bool cstar,
                            cudaStream_t stream) {
  if (tgt_dtype == SPEC_F32) {
    if (logit_dtype == SPEC_F32) return launch_kc<float, float>(p, tgt, U, Ct, grid, cstar, stream);
    return launch_kc<float, __nv_bfloat16>(p, tgt, U, Ct, grid, cstar, stream);
  }
  if (logit_dtype == SPEC_F32)
    return launch_kc<__nv_bfloat16, float>(p, tgt, U, Ct, grid, cstar, stream);
  return launch_kc<__nv_bfloat16, __nv_bfloat16>(p, tgt, U, Ct, grid, cstar, stream);
}

}  // namespace spec
