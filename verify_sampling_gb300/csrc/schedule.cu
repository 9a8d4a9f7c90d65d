// Hardware-aware prefix scheduler: one thread block.
//
// DSpark summary, "2.2 硬件感知前缀调度器": maximise Theta = tau * SPS(B) with
// B = sum_r (1 + l_r) and tau = sum_r sum_{j<=l_r} a_{r,j}, by sorting all
// survivals in descending order and admitting them while Theta rises; "挑战2"
// adds the top-K cap and the global search.  History article, "杀招三": the
// same rule walked through.
//
// Layout of the work: the N = R * gamma keys ~bits(a) are radix-sorted
// ascending (stable, so a descending with ties by id = r * gamma + j - 1
// ascending: request, then position) in shared memory.  tau_n is an fp64
// inclusive scan of the sorted survivals, Theta_n = tau_n * SPS(R + n); the
// early-stop index is the first n with Theta_{n+1} <= Theta_n and the global
// index the smallest argmax.  DSpark summary, comparison table (SpecDec++) and
// Figure 5: the threshold index is the first sorted n whose survival is below
// a static threshold.
#include "schedule.cuh"

namespace spec {

namespace {

constexpr int kThreads = 1024;
constexpr int kHistCells = 32 * 257;  // radix digit histograms, [warp][257]

__device__ __forceinline__ double sps_at(const float* sps, int n_sps, double b_lo, double b_step,
                                         double B) {
  // Same operation order as the definition: t = (B - b_lo) / b_step, linear
  // interpolation (1 - f) * s_i + f * s_{i+1}, clamped to the end values.
  const double t = __ddiv_rn(__dsub_rn(B, b_lo), b_step);
  if (t <= 0.0) return (double)sps[0];
  if (t >= (double)(n_sps - 1)) return (double)sps[n_sps - 1];
  const double fi = floor(t);
  const int i = (int)fi;
  const double f = __dsub_rn(t, fi);
  return __dadd_rn(__dmul_rn(__dsub_rn(1.0, f), (double)sps[i]), __dmul_rn(f, (double)sps[i + 1]));
}

// Lanes of the warp whose digit d (8 bits) equals this lane's, among the
// lanes with `valid` set: one ballot per bit.
__device__ __forceinline__ unsigned digit_peers(uint32_t d, bool valid) {
  unsigned peers = __ballot_sync(0xffffffffu, valid);
  if (!valid) peers = ~peers;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const bool bit = (d >> b) & 1u;
    const unsigned bal = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? bal : ~bal;
  }
  return peers;
}

__device__ __forceinline__ int warp_incl_scan_int(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kThreads) schedule_kernel(SchedParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int N = p.R * p.gamma, Np = p.npad;
  // [Np] each, in this order: keyA, valA, keyB, valB (keyB and valB together
  // hold Theta once the sort is done)
  uint32_t* keyA = reinterpret_cast<uint32_t*>(smem_raw);
  int* valA = reinterpret_cast<int*>(keyA + Np);
  uint32_t* keyB = reinterpret_cast<uint32_t*>(valA + Np);
  int* valB = reinterpret_cast<int*>(keyB + Np);
  int* hist = valB + Np;         // [32 warps][257]: digit d of warp w at w * 257 + d
  int* ell_s = hist + kHistCells;  // [R]
  double* theta = reinterpret_cast<double*>(keyB);  // after the sort: [nmax + 1] over keyB, valB
  __shared__ unsigned long long seg_q[kThreads];
  __shared__ int warp_itot[32];
  __shared__ int nstar_s;
  __shared__ double best_s[32];
  __shared__ int bestn_s[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 1. keys: ~bits(a) ascending is a descending (float bits are monotone for
  // a >= 0); the sort below is stable, so equal a keep id order (request, then
  // position).
  for (int i = tid; i < N; i += kThreads) {
    float a = p.a[i];
    if (!(a >= 0.f) || isinf(a)) {  // negative, NaN or inf
      set_status(p.status, SPEC_STATUS_BAD_SURVIVAL);
      a = 0.f;
    }
    keyA[i] = ~__float_as_uint(a + 0.0f);  // -0 -> +0
    valA[i] = i;
  }
  __syncthreads();

  // 2. stable LSD radix sort, 8-bit digits, 4 passes.  Warp w owns a
  // contiguous segment of the array; ranks inside a warp step come from
  // per-bit ballots, offsets from a scan of the per-warp digit histograms in
  // (digit, warp) order, which keeps equal digits in array order.
  {
    const int seg = (((N + 31) / 32) + 31) & ~31;  // per-warp segment, multiple of 32
    const int wb = warp * seg;
    uint32_t *ks = keyA, *kd = keyB;
    int *vs = valA, *vd = valB;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 8 * pass;
      for (int i = tid; i < kHistCells; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int s0 = 0; s0 < seg; s0 += 32) {
        const int idx = wb + s0 + lane;
        const bool valid = idx < N;
        const uint32_t d = valid ? (ks[idx] >> shift) & 255u : 0u;
        const unsigned peers = digit_peers(d, valid);
        if (valid && lane == __ffs(peers) - 1) hist[warp * 257 + d] += __popc(peers);
      }
      __syncthreads();
      {
        // cells in (digit, warp) order: cell c = d * 32 + w, eight per thread
        int loc[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = tid * 8 + q;
          loc[q] = hist[(c & 31) * 257 + (c >> 5)];
          sum += loc[q];
        }
        const int incl = warp_incl_scan_int(sum);
        if (lane == 31) warp_itot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
          const int wt = warp_itot[lane];
          warp_itot[lane] = warp_incl_scan_int(wt) - wt;
        }
        __syncthreads();
        int run = warp_itot[warp] + incl - sum;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = tid * 8 + q;
          hist[(c & 31) * 257 + (c >> 5)] = run;
          run += loc[q];
        }
      }
      __syncthreads();
      for (int s0 = 0; s0 < seg; s0 += 32) {
        const int idx = wb + s0 + lane;
        const bool valid = idx < N;
        uint32_t key = 0u, d = 0u;
        int val = 0;
        if (valid) {
          key = ks[idx];
          val = vs[idx];
          d = (key >> shift) & 255u;
        }
        const unsigned peers = digit_peers(d, valid);
        const int base = valid ? hist[warp * 257 + d] : 0;
        __syncwarp();
        if (valid) {
          const int pos = base + __popc(peers & ((1u << lane) - 1u));
          kd[pos] = key;
          vd[pos] = val;
          if (lane == __ffs(peers) - 1) hist[warp * 257 + d] = base + __popc(peers);
        }
        __syncwarp();
      }
      __syncthreads();
      uint32_t* tk = ks;
      ks = kd;
      kd = tk;
      int* tv = vs;
      vs = vd;
      vd = tv;
    }
  }
  // four passes: the sorted keys and ids are back in keyA / valA

  // 3. zero the per-request counts; SPS(R + n) for every admissible n, in
  // parallel (theta[n] holds it until step 4 multiplies in tau_n).
  // The cap: K, lowered by the device word K_dev when given (asynchronous cap).
  // With n_free requested, Theta is formed for every n so that the uncapped
  // decision can be taken too.
  const int kcap = p.K_dev ? min(p.K, max(*p.K_dev, 0)) : p.K;
  const int nmax = min(kcap, N);
  const int ntheta = p.n_free ? N : nmax;
  for (int i = tid; i < p.R; i += kThreads) ell_s[i] = 0;
  for (int n = tid; n <= ntheta; n += kThreads) {
    double v = 0.0;
    if (n > 0) {
      if (p.unit_grid) {
        // b_step = 1 and integral b_lo: t = B - b_lo is an integer, so the
        // interpolation weight is 0 and the value is the table entry itself
        const long t = (long)(p.R + n) - p.b_lo_int;
        v = (double)p.sps[t <= 0 ? 0 : (t >= p.n_sps - 1 ? p.n_sps - 1 : t)];
      } else {
        v = sps_at(p.sps, p.n_sps, p.b_lo, p.b_step, (double)(p.R + n));
      }
    }
    theta[n] = v;
  }
  __syncthreads();

  // 4. tau_n, Theta_n = tau_n * SPS(R + n).  tau is an exact prefix sum in
  // 64-bit fixed point scaled to the largest survival a_1 (the first sorted
  // entry): each a_k is truncated to a multiple of 2^-shift with
  // a_1 * 2^shift < 2^49, so the 8192-term sums stay below 2^62 and the total
  // truncation is below 2^-36 a_1 <= 2^-36 tau_n.  One conversion to fp64 per
  // position.  Thread t owns sorted positions [t*per, (t+1)*per).
  const int per = (N + kThreads - 1) / kThreads;
  const int lo = tid * per, hi = min(N, lo + per);
  const int cnt = hi - lo;
  // From the bits: a = m * 2^(E' - 150) with E' = max(E, 1) and m the
  // significand (hidden bit for E > 0); a_1 < 2^(E1' - 126).  So
  // a * 2^shift = m * 2^(E' - E1' + 25) for shift = 175 - E1'.
  const int e1 = max((int)((~keyA[0] >> 23) & 0xffu), 1);
  auto fixed = [&](uint32_t bits) -> unsigned long long {
    const int E = (int)((bits >> 23) & 0xffu);
    const unsigned long long m = (bits & 0x7fffffu) | (E > 0 ? 0x800000u : 0u);
    const int sh = max(E, 1) - e1 + 25;  // <= 25 since a <= a_1
    if (sh >= 0) return m << sh;
    return sh > -64 ? (m >> (-sh)) : 0ull;
  };
  unsigned long long qv[kSchedMaxCandidates / kThreads];
  unsigned long long local = 0ull;
#pragma unroll
  for (int i = 0; i < kSchedMaxCandidates / kThreads; ++i) {
    qv[i] = (i < cnt) ? fixed(~keyA[lo + i]) : 0ull;
    local += qv[i];
  }
  unsigned long long incl = local;  // inclusive warp scan
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __shared__ unsigned long long warp_q[32];
  if (lane == 31) warp_q[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long wt = warp_q[lane];
    unsigned long long wi = wt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_q[lane] = wi - wt;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const double unit = ldexp(1.0, e1 - 175);  // 2^-shift, exact
  {
    unsigned long long run = warp_q[warp] + incl - local;
#pragma unroll
    for (int i = 0; i < kSchedMaxCandidates / kThreads; ++i)
      if (i < cnt) {
        run += qv[i];
        const int n = lo + i + 1;
        if (n <= ntheta) theta[n] = __dmul_rn(__dmul_rn((double)run, unit), theta[n]);
      }
    seg_q[tid] = warp_q[warp] + incl - local;
  }
  __syncthreads();
  // 5. choose n*.
  if (p.mode != SPEC_SCHED_GLOBAL) {
    // first sorted position that stops the admission
    // The first stop over all of [0, ntheta); the capped n* is min(first, nmax).
    const bool thr = p.mode == SPEC_SCHED_THRESHOLD;
    int first = ntheta;
    for (int n = tid; n < ntheta; n += kThreads) {
      const bool stop = thr ? !((double)__uint_as_float(~keyA[n]) >= p.threshold)
                            : !(theta[n + 1] > theta[n]);
      if (stop) first = min(first, n);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) first = min(first, __shfl_down_sync(0xffffffffu, first, off));
    if (lane == 0) bestn_s[warp] = first;
    __syncthreads();
    if (tid == 0) {
      int f = ntheta;
      for (int w = 0; w < kThreads / 32; ++w) f = min(f, bestn_s[w]);
      nstar_s = min(f, nmax);
      if (p.n_free) *p.n_free = f;
    }
  } else {
    // smallest argmax of Theta over n <= lim, block-wide (result in thread 0)
    auto argmax_upto = [&](int lim) -> int {
      double best = -1.0;
      int bn = 0;
      for (int n = tid; n <= lim; n += kThreads)
        if (theta[n] > best) {
          best = theta[n];
          bn = n;
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const double ob = __shfl_down_sync(0xffffffffu, best, off);
        const int on = __shfl_down_sync(0xffffffffu, bn, off);
        if (ob > best || (ob == best && on < bn)) {
          best = ob;
          bn = on;
        }
      }
      if (lane == 0) {
        best_s[warp] = best;
        bestn_s[warp] = bn;
      }
      __syncthreads();
      int n = 0;
      if (tid == 0) {
        double b = -1.0;
        for (int w = 0; w < kThreads / 32; ++w)
          if (best_s[w] > b || (best_s[w] == b && bestn_s[w] < n)) {
            b = best_s[w];
            n = bestn_s[w];
          }
      }
      __syncthreads();  // best_s may be reused by the next call
      return n;
    };
    const int n_cap = argmax_upto(nmax);
    if (tid == 0) nstar_s = n_cap;
    if (p.n_free) {
      const int n_all = argmax_upto(ntheta);
      if (tid == 0) *p.n_free = n_all;
    }
  }
  __syncthreads();
  const int nstar = nstar_s;

  // 6. l_r, row offsets, stats, order.
  for (int n = tid; n < nstar; n += kThreads) atomicAdd(&ell_s[valA[n] / p.gamma], 1);
  __syncthreads();
  {
    // exclusive scan of (1 + l_r) over R entries, per-thread segments
    const int perR = (p.R + kThreads - 1) / kThreads;
    const int rlo = tid * perR, rhi = min(p.R, rlo + perR);
    int loc = 0;
    for (int i = rlo; i < rhi; ++i) loc += 1 + ell_s[i];
    int inc = warp_incl_scan_int(loc);
    if (lane == 31) warp_itot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int wt = warp_itot[lane];
      warp_itot[lane] = warp_incl_scan_int(wt) - wt;
    }
    __syncthreads();
    int run = warp_itot[warp] + inc - loc;
    for (int i = rlo; i < rhi; ++i) {
      p.row_off[i] = run;
      p.ell[i] = ell_s[i];
      run += 1 + ell_s[i];
    }
    if (rhi == p.R && rlo < rhi) p.row_off[p.R] = run;
    if (p.R == 0 && tid == 0) p.row_off[0] = 0;
  }
  if (p.order)
    for (int i = tid; i < N; i += kThreads) p.order[i] = valA[i];
  // tau at n*: the owner of sorted position n* - 1 sums its prefix again.
  if (nstar == 0) {
    if (tid == 0) {
      p.stats[0] = 0.0;
      p.stats[1] = (double)p.R;
      p.stats[2] = 0.0;
      p.stats[3] = 0.0;
    }
  } else if (nstar - 1 >= lo && nstar - 1 < hi) {
    unsigned long long run = seg_q[tid];
    for (int i = lo; i < nstar; ++i) run += fixed(~keyA[i]);
    p.stats[0] = (double)nstar;
    p.stats[1] = (double)(p.R + nstar);
    p.stats[2] = __dmul_rn((double)run, unit);
    p.stats[3] = theta[nstar];
  }
}

// keys and ids twice (radix ping-pong; the second pair later holds Theta as
// doubles: Np >= N + 1), the digit histograms and the per-request counts.
static int sched_npad(int R, int gamma) { return ((R * gamma + 1) + 31) & ~31; }

size_t schedule_smem_bytes(int R, int gamma) {
  const size_t Np = (size_t)sched_npad(R, gamma);
  return sizeof(uint32_t) * 4 * Np + sizeof(int) * ((size_t)kHistCells + (size_t)R);
}

cudaError_t launch_schedule(SchedParams p, cudaStream_t stream) {
  p.npad = sched_npad(p.R, p.gamma);
  p.unit_grid = p.b_step == 1.0 && p.b_lo == floor(p.b_lo) && fabs(p.b_lo) < 1e9;
  p.b_lo_int = p.unit_grid ? (long)p.b_lo : 0;
  const size_t smem = schedule_smem_bytes(p.R, p.gamma);
  cudaError_t err =
      cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  schedule_kernel<<<1, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
