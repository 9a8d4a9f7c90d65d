// Hardware-aware prefix scheduler: one thread block.
//
// DSpark summary, "2.2 硬件感知前缀调度器": maximise Theta = tau * SPS(B) with
// B = sum_r (1 + l_r) and tau = sum_r sum_{j<=l_r} a_{r,j}, by sorting all
// survivals in descending order and admitting them while Theta rises; "挑战2"
// adds the top-K cap and the global search.  History article, "杀招三": the
// same rule walked through.
//
// Layout of the work: N = R * gamma 64-bit keys (~bits(a) << 32 | id) are
// bitonic-sorted ascending in shared memory, which orders a descending and ties
// by id = r * gamma + j - 1 ascending (request, then position).  tau_n is an
// fp64 inclusive scan of the sorted survivals, Theta_n = tau_n * SPS(R + n);
// the early-stop index is the first n with Theta_{n+1} <= Theta_n and the
// global index the smallest argmax.
#include "schedule.cuh"

namespace spec {

namespace {

constexpr int kThreads = 1024;

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

__device__ __forceinline__ double warp_incl_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v = __dadd_rn(v, o);
  }
  return v;
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
  const int N = p.R * p.gamma;
  const int npow2 = p.npow2;
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem_raw);                 // [npow2 + 8]
  double* theta = reinterpret_cast<double*>(smem_raw);                     // aliases keys
  int* ids = reinterpret_cast<int*>(smem_raw + sizeof(uint64_t) * (npow2 + 8));  // [N]
  int* ell_s = ids + N;                                                    // [R]
  __shared__ double seg_sum[kThreads];
  __shared__ double warp_tot[32];
  __shared__ int warp_itot[32];
  __shared__ int nstar_s;
  __shared__ double best_s[32];
  __shared__ int bestn_s[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 1. keys: a >= 0 as float bits (monotone for non-negative floats).
  for (int i = tid; i < npow2; i += kThreads) {
    uint64_t key = ~0ull;
    if (i < N) {
      float a = p.a[i];
      if (!(a >= 0.f) || isinf(a)) {  // negative, NaN or inf
        set_status(p.status, SPEC_STATUS_BAD_SURVIVAL);
        a = 0.f;
      }
      const uint32_t bits = __float_as_uint(a + 0.0f);  // -0 -> +0
      key = ((uint64_t)(~bits) << 32) | (uint32_t)i;
    }
    keys[i] = key;
  }
  __syncthreads();

  // 2. bitonic sort, ascending.
  for (int kk = 2; kk <= npow2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npow2; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool up = (i & kk) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }

  // 3. ids and sorted survivals; zero the per-request counts.
  for (int i = tid; i < N; i += kThreads) ids[i] = (int)(keys[i] & 0xffffffffu);
  for (int i = tid; i < p.R; i += kThreads) ell_s[i] = 0;
  __syncthreads();

  // 4. tau_n, Theta_n (fp64).  Thread t owns sorted positions [t*per, (t+1)*per).
  const int nmax = min(p.K, N);
  const int per = (N + kThreads - 1) / kThreads;
  const int lo = tid * per, hi = min(N, lo + per);
  double local = 0.0;
  for (int i = lo; i < hi; ++i) local = __dadd_rn(local, (double)__uint_as_float(~(uint32_t)(keys[i] >> 32)));
  double incl = warp_incl_scan(local);
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double wt = warp_tot[lane];
    double wi = warp_incl_scan(wt);
    warp_tot[lane] = __dsub_rn(wi, wt);  // exclusive prefix of warp totals
  }
  __syncthreads();
  const double excl = __dadd_rn(warp_tot[warp], __dsub_rn(incl, local));
  seg_sum[tid] = excl;
  // Sorted survivals of my segment before theta overwrites the keys.
  float mine[16];
  const int cnt = hi - lo;
  for (int i = 0; i < cnt && i < 16; ++i) mine[i] = __uint_as_float(~(uint32_t)(keys[lo + i] >> 32));
  __syncthreads();
  {
    double tau = excl;
    if (tid == 0) theta[0] = 0.0;
    for (int i = 0; i < cnt; ++i) {
      tau = __dadd_rn(tau, (double)mine[i]);
      const int n = lo + i + 1;
      if (n <= nmax)
        theta[n] = __dmul_rn(tau, sps_at(p.sps, p.n_sps, p.b_lo, p.b_step, (double)(p.R + n)));
    }
  }
  __syncthreads();

  // 5. choose n*.
  if (p.mode == SPEC_SCHED_EARLY_STOP) {
    int first = nmax;
    for (int n = tid; n < nmax; n += kThreads)
      if (!(theta[n + 1] > theta[n])) first = min(first, n);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) first = min(first, __shfl_down_sync(0xffffffffu, first, off));
    if (lane == 0) bestn_s[warp] = first;
    __syncthreads();
    if (tid == 0) {
      int f = nmax;
      for (int w = 0; w < kThreads / 32; ++w) f = min(f, bestn_s[w]);
      nstar_s = f;
    }
  } else {
    double best = -1.0;
    int bn = 0;
    for (int n = tid; n <= nmax; n += kThreads)
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
    if (tid == 0) {
      double b = -1.0;
      int n = 0;
      for (int w = 0; w < kThreads / 32; ++w)
        if (best_s[w] > b || (best_s[w] == b && bestn_s[w] < n)) {
          b = best_s[w];
          n = bestn_s[w];
        }
      nstar_s = n;
    }
  }
  __syncthreads();
  const int nstar = nstar_s;

  // 6. l_r, row offsets, stats, order.
  for (int n = tid; n < nstar; n += kThreads) atomicAdd(&ell_s[ids[n] / p.gamma], 1);
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
    for (int i = tid; i < N; i += kThreads) p.order[i] = ids[i];
  // tau at n*: the owner of sorted position n* - 1 recomputes its prefix.
  if (nstar == 0) {
    if (tid == 0) {
      p.stats[0] = 0.0;
      p.stats[1] = (double)p.R;
      p.stats[2] = 0.0;
      p.stats[3] = 0.0;
    }
  } else if (nstar - 1 >= lo && nstar - 1 < hi) {
    double tau = seg_sum[tid];
    for (int i = 0; i < nstar - lo; ++i) tau = __dadd_rn(tau, (double)mine[i]);
    p.stats[0] = (double)nstar;
    p.stats[1] = (double)(p.R + nstar);
    p.stats[2] = tau;
    p.stats[3] = theta[nstar];
  }
}

size_t schedule_smem_bytes(int R, int gamma) {
  const int N = R * gamma;
  int npow2 = 2;
  while (npow2 < N) npow2 <<= 1;
  return sizeof(uint64_t) * (size_t)(npow2 + 8) + sizeof(int) * (size_t)(N + R);
}

cudaError_t launch_schedule(SchedParams p, cudaStream_t stream) {
  const int N = p.R * p.gamma;
  int npow2 = 2;
  while (npow2 < N) npow2 <<= 1;
  p.npow2 = npow2;
  const size_t smem = schedule_smem_bytes(p.R, p.gamma);
  cudaError_t err =
      cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  schedule_kernel<<<1, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
