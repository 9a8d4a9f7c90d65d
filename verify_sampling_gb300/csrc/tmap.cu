// Host-side tensor-map encoding for the fused kernels' TMA loads.
#include "fused_tc.cuh"

namespace spec {
namespace fused {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver entry point, resolved once through the runtime (no -lcuda link).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, size_t es, const void* base, int rank,
                  const uint64_t* dims, const uint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 2 || rank > 3) return false;
  cuuint64_t gdims[3], strides[2];
  cuuint32_t gbox[3], estr[3] = {1, 1, 1};
  uint64_t stride = es;
  for (int i = 0; i < rank; ++i) {
    gdims[i] = dims[i];
    gbox[i] = box[i];
    if (i > 0) strides[i - 1] = stride;
    stride *= dims[i];
  }
  return enc(map, dt, (cuuint32_t)rank, const_cast<void*>(base), gdims, strides, gbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fused
}  // namespace spec
