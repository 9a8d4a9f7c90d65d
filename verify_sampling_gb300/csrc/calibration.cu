// Reliability diagram and expected calibration error of the confidences: one
// thread block.
//
// DSpark summary, Figure 6 and "2.1 置信度头": the confidence head's outputs
// (after sequential temperature scaling) are compared with the acceptance the
// verifier realises, bin by bin over [0, 1]; the ECE is the count-weighted
// mean gap between a bin's mean confidence and its acceptance rate.
//
// A thread takes one request at a time and walks the positions the verifier
// ruled on (up to the first rejection); bin sums gather in shared memory
// (64-bit integer counts, fp64 confidence sums) and are then added to the
// caller's tables, which accumulate over rounds.
#include "accept_stats.cuh"

namespace spec {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) calibration_kernel(CalibrationParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int nb = p.n_bins, G = p.gamma;
  unsigned long long* n_s = reinterpret_cast<unsigned long long*>(smem_raw);  // [nb]
  unsigned long long* a_s = n_s + nb;                                         // [nb]
  double* c_s = reinterpret_cast<double*>(a_s + nb);                           // [nb]
  const int tid = threadIdx.x;
  for (int b = tid; b < nb; b += kThreads) {
    n_s[b] = 0ull;
    a_s[b] = 0ull;
    c_s[b] = 0.0;
  }
  __syncthreads();

  bool bad_len = false, bad_c = false;
  for (int r = tid; r < p.R; r += kThreads) {
    const int l = p.ell[r], acc = p.accept_len[r];
    if (l < 0 || l > G || acc < 0 || acc > l) {
      bad_len = true;
      continue;
    }
    const int tested = min(l, acc + 1);
    for (int j = 1; j <= tested; ++j) {
      const float cj = p.c[(size_t)r * G + (j - 1)];
      if (!(cj >= 0.f && cj <= 1.f)) {
        bad_c = true;
        continue;
      }
      const int b = min((int)floor(__dmul_rn((double)cj, (double)nb)), nb - 1);
      atomicAdd(&n_s[b], 1ull);
      atomicAdd(&c_s[b], (double)cj);
      if (j <= acc) atomicAdd(&a_s[b], 1ull);
    }
  }
  if (bad_len) set_status(p.status, SPEC_STATUS_BAD_ELL);
  if (bad_c) set_status(p.status, SPEC_STATUS_BAD_SURVIVAL);
  __syncthreads();

  for (int b = tid; b < nb; b += kThreads) {
    if (n_s[b] == 0ull) continue;
    p.count[b] += (long long)n_s[b];
    p.sum_acc[b] += (long long)a_s[b];
    p.sum_c[b] = __dadd_rn(p.sum_c[b], c_s[b]);
  }
  if (!p.ece) return;
  __syncthreads();
  if (tid == 0) {
    long long N = 0;
    double dev = 0.0;
    for (int b = 0; b < nb; ++b) {
      N += p.count[b];
      dev = __dadd_rn(dev, fabs(__dsub_rn((double)p.sum_acc[b], p.sum_c[b])));
    }
    *p.ece = N > 0 ? __ddiv_rn(dev, (double)N) : __longlong_as_double(0x7ff8000000000000ll);
  }
}

}  // namespace

cudaError_t launch_calibration(const CalibrationParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)p.n_bins * 24;
  calibration_kernel<<<1, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
