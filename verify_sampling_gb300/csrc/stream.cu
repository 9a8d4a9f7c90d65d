// The library's counter-based random stream, exposed for reproduction and
// audit: the same Philox-4x32-10 blocks and uniform / -ln(u) mappings that the
// sampling kernels use (common.cuh).
#include "common.cuh"

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

}  // namespace spec

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
