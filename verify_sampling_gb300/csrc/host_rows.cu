// Gather of the scheduled target rows straight from page-locked host memory.
//
// In a round the target model produces logits only for the rows the schedule
// admits: rows 1 .. l_r + 1 of each request (DSpark summary, "2.2 硬件感知前缀
// 调度器": B = sum_r (1 + l_r)).  A caller that holds every candidate row on
// the host, padded [R, gamma + 1, V], therefore needs only those B rows on the
// device.  Their positions are known only on the device (the schedule's
// row_off), so instead of a host round trip the copy is a kernel: one CTA per
// (request, row) reads the row through the device's mapping of the host
// buffer and writes it at its packed position.  The link's throughput is the
// same for copy-engine copies and for SM loads of mapped host memory, and the
// other B rows never cross it.
#include "host_rows.cuh"

namespace spec {

namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(GatherRowsParams p) {
  const int r = blockIdx.y, j0 = blockIdx.x;  // j0 = j - 1
  const int lo = p.row_off[r], len = p.row_off[r + 1] - lo;
  const long total = (long)p.R * p.G1;
  if (len < 1 || len > p.G1 || lo < 0 || (long)lo + len > total) {
    if (j0 == 0 && threadIdx.x == 0) set_status(p.status, SPEC_STATUS_BAD_ROW);
    return;
  }
  if (j0 >= len) return;
  const unsigned char* s = p.src + ((size_t)r * p.G1 + j0) * p.row_bytes;
  unsigned char* d = p.dst + ((size_t)lo + j0) * p.row_bytes;
  const bool vec = ((p.row_bytes | (uintptr_t)s | (uintptr_t)d) & 15) == 0;
  if (vec) {
    const uint4* s4 = reinterpret_cast<const uint4*>(s);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    const size_t n = p.row_bytes / 16;
    const size_t step = (size_t)kGatherThreads * kGatherUnroll;
    for (size_t i0 = threadIdx.x; i0 < n; i0 += step) {
      uint4 v[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const size_t i = i0 + (size_t)u * kGatherThreads;
        if (i < n) v[u] = s4[i];
      }
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const size_t i = i0 + (size_t)u * kGatherThreads;
        if (i < n) d4[i] = v[u];
      }
    }
  } else {
    for (size_t i = threadIdx.x; i < p.row_bytes; i += kGatherThreads) d[i] = s[i];
  }
}

}  // namespace

cudaError_t launch_gather_rows(const GatherRowsParams& p, cudaStream_t stream) {
  const dim3 grid((unsigned)p.G1, (unsigned)p.R);
  gather_rows_kernel<<<grid, kGatherThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace spec
