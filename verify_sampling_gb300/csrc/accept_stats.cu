// Acceptance-rate statistics per MTP length: one thread block.
//
// LightSpec article, "无需额外训练，基于运行时统计的动态调度": the runtime keeps,
// per request-scale / batch-size class and per MTP length, an exponential
// moving average of the acceptance rate, updated every round, and estimates a
// length with too few samples by interpolating over the other lengths.
//
// Per round: the per-length request counts n_L and accepted sums S_L are exact
// 64-bit integer sums in shared memory; each length then takes
// m_L = S_L / (L n_L) and ema = fma(beta, m_L - ema, ema) (the first sample
// sets ema), every step one correctly rounded fp64 operation, so the table is
// reproducible bit for bit.  The estimate of a length without enough samples
// is the straight line between the nearest usable lengths on either side.
#include "accept_stats.cuh"

namespace spec {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) accept_stats_kernel(AcceptStatsParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int G = p.gamma;
  unsigned long long* n_s = reinterpret_cast<unsigned long long*>(smem_raw);  // [G + 1]
  unsigned long long* acc_s = n_s + (G + 1);                                   // [G + 1]
  double* e_s = reinterpret_cast<double*>(acc_s + (G + 1));                    // [G]
  long long* c_s = reinterpret_cast<long long*>(e_s + G);                      // [G]
  const int tid = threadIdx.x;

  for (int i = tid; i <= G; i += kThreads) {
    n_s[i] = 0ull;
    acc_s[i] = 0ull;
  }
  __syncthreads();

  // 1. exact per-length sums; requests without a draft carry no statistic
  bool bad = false;
  for (int r = tid; r < p.R; r += kThreads) {
    const int l = p.ell[r], acc = p.accept_len[r];
    if (l < 0 || l > G || acc < 0 || acc > l) {
      bad = true;
      continue;
    }
    if (l == 0) continue;
    atomicAdd(&n_s[l], 1ull);
    atomicAdd(&acc_s[l], (unsigned long long)acc);
  }
  if (bad) set_status(p.status, SPEC_STATUS_BAD_ELL);
  __syncthreads();

  // 2. moving averages of class `bucket`
  double* ema = p.ema + (size_t)p.bucket * G;
  long long* cnt = p.count + (size_t)p.bucket * G;
  for (int L = 1 + tid; L <= G; L += kThreads) {
    double e = ema[L - 1];
    long long c = cnt[L - 1];
    const unsigned long long n = n_s[L];
    if (n > 0) {
      const double m = __ddiv_rn((double)acc_s[L], __dmul_rn((double)L, (double)n));
      e = (c == 0) ? m : __fma_rn(p.beta, __dsub_rn(m, e), e);
      c += (long long)n;
      ema[L - 1] = e;
      cnt[L - 1] = c;
    }
    e_s[L - 1] = e;
    c_s[L - 1] = c;
  }
  if (!p.estimate) return;
  __syncthreads();

  // 3. estimates: the entry itself, or the line between the nearest usable
  // lengths below and above, or the nearest one, or NaN
  const long long need = p.min_count > 1 ? (long long)p.min_count : 1ll;
  for (int L = 1 + tid; L <= G; L += kThreads) {
    double v;
    if (c_s[L - 1] >= need) {
      v = e_s[L - 1];
    } else {
      int lo = 0, hi = 0;
      for (int q = L - 1; q >= 1; --q)
        if (c_s[q - 1] >= need) {
          lo = q;
          break;
        }
      for (int q = L + 1; q <= G; ++q)
        if (c_s[q - 1] >= need) {
          hi = q;
          break;
        }
      if (lo && hi) {
        const double w = __ddiv_rn((double)(L - lo), (double)(hi - lo));
        v = __fma_rn(w, __dsub_rn(e_s[hi - 1], e_s[lo - 1]), e_s[lo - 1]);
      } else if (lo) {
        v = e_s[lo - 1];
      } else if (hi) {
        v = e_s[hi - 1];
      } else {
        v = __longlong_as_double(0x7ff8000000000000ll);  // quiet NaN
      }
    }
    p.estimate[L - 1] = v;
  }
}

}  // namespace

cudaError_t launch_accept_stats(const AcceptStatsParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)(p.gamma + 1) * 16 + (size_t)p.gamma * 16;
  accept_stats_kernel<<<1, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
