// The library's counter-based random stream, exposed for reproduction and
// audit: the same Philox-4x32-10 blocks and uniform / -ln(u) mappings that the
// sampling kernels use (common.cuh).  Also the self-test of the bounded
// pipeline wait (tc.cuh).
#include "common.cuh"
#include "tc.cuh"

namespace spec {

__global__ void stream_uniforms_kernel(PhiloxKey key, uint32_t j, uint32_t rid, uint32_t purpose,
                                       int V, float* u_out, float* e_out) {
  const int vb = blockIdx.x * blockDim.x + threadIdx.x;
  if (vb * 4 >= V) return;
  const uint4 bits = philox((uint32_t)vb, j, rid, purpose, key);
#pragma unroll
  for (int lane = 0; lane < 4; ++lane) {
    const int v = vb * 4 + lane;
    if (v < V) {
      const uint32_t w = word_of(bits, lane);
      u_out[v] = uniform_from_word(w);
      if (e_out) e_out[v] = neg_log_uniform(w);
    }
  }
}

// One thread waits on a fresh mbarrier (expected arrivals: 1) for phase 0,
// which nothing completes; the bounded wait gives up after limit_ns.
__global__ void wait_selftest_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  tc::fence_barrier_init();
  if (!tc::mbar_wait(&bar, 0u, limit_ns)) set_status(status, SPEC_STATUS_TIMEOUT);
}

}  // namespace spec

extern "C" int spec_wait_selftest(uint64_t limit_ns, uint32_t* status, spec_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000ull || !status) return SPEC_ERR_INVALID_ARG;
  if ((uintptr_t)status & 3) return SPEC_ERR_ALIGNMENT;
  spec::wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, status);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_stream_uniforms(uint64_t seed, uint32_t j, uint32_t rid, uint32_t purpose,
                                    int V, float* u_out, float* e_out, spec_stream_t stream) {
  if (V < 1 || V >= (1 << 30) || !u_out) return SPEC_ERR_INVALID_ARG;
  if (((uintptr_t)u_out & 3) || ((uintptr_t)e_out & 3)) return SPEC_ERR_ALIGNMENT;
  const int nvb = (V + 3) / 4;
  const int threads = 256;
  spec::stream_uniforms_kernel<<<(nvb + threads - 1) / threads, threads, 0,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(
      spec::philox_key(seed), j, rid, purpose, V, u_out, e_out);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
