// spec_draft_sample_static: the draft stage with its scratch memory in a
// fixed device array of this library instead of a caller-provided workspace.
//
// For callers that cannot allocate device memory at the point of the call --
// for example code running inside an allocator, a runtime that forbids
// cudaMalloc during serving, or an embedding that owns all device memory
// itself.  The array (kStaticScratchBytes) is a file-scope __device__ object:
// every GPU that loads the library holds it until the process exits.
//
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it; make that first call before any stream
// capture.  The cache is keyed by the device's current context as well: a
// context that is destroyed and created again (cudaDeviceReset, or a primary
// context released and retained) loads the module again, the array can move,
// and the next call looks the address up anew.  All calls share the one array
// and it keeps the last call's contents: the counters are cleared at the
// start of every call, and two calls that overlap on the GPU (different
// streams, or different host threads on one stream without ordering) race on
// it and give wrong results.
#include <cuda.h>

#include <mutex>

#include "draft.cuh"
#include "draft_run.cuh"
#include "draft_tc.cuh"

namespace {

using namespace spec;

// 2 MiB.  The need is 32 * R * s + 4 * R * (1 + gamma) bytes (the first term
// rounded up to 256): s = 2 * splits on the tensor-core path, with splits =
// SMs / ceil(R / 128) capped by the 64-column vocabulary tiles, and the
// generic kernel's split count otherwise.  On a 152-SM GB300 the tensor-core
// path at gamma = 16 fits up to about 15000 requests (4096 need 1.33 MB).
constexpr size_t kStaticScratchBytes = 2u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_draft_scratch[kStaticScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(ptr);
}

// Unique id of the calling thread's current context (0 if there is none yet).
bool current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_draft_scratch on device `dev` in its current context.
void* scratch_address(int dev) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) return nullptr;
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;  // the lookup also makes the primary context current
    if (cudaGetSymbolAddress(&p, g_draft_scratch) != cudaSuccess) return nullptr;
    if (!current_context_id(&ctx) || ctx == 0) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" int spec_draft_sample_static(const spec_draft_args* args, uint64_t seed,
                                        spec_stream_t stream) {
  // The same argument rules as spec_draft_sample (the workspace fields are ignored).
  const int rc = check_draft_args(args);
  if (rc != SPEC_OK) return rc;
  const spec_draft_args& a = *args;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  int sms = 0;
  const int tc_sms = draft_tc_ok(a, &sms) ? sms : 0;

  // Exact scratch for the path taken: partials [R, splits] (two slots on the
  // fused path), then counters [R] and the race bounds [gamma, R].
  const size_t part_bytes = round256((size_t)a.R *
                                     (tc_sms ? 2 * draft_tc_nsplit(a.R, a.V, tc_sms) : draft_nsplit(a.R, a.V)) *
                                     sizeof(Partial));
  const size_t cnt_bytes = (size_t)a.R * (1 + a.gamma) * sizeof(unsigned);
  if (part_bytes + cnt_bytes > kStaticScratchBytes) return SPEC_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(scratch_address(dev));
  if (!ws) return SPEC_ERR_CUDA;
  return run_draft(a, seed, reinterpret_cast<Partial*>(ws), reinterpret_cast<unsigned*>(ws + part_bytes),
                   tc_sms, reinterpret_cast<cudaStream_t>(stream));
}
