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
// capture.  All calls share the one array and it keeps the last call's
// contents: the counters are cleared at the start of every call, and two calls
// that overlap on the GPU (different streams, or different host threads on
// one stream without ordering) race on it and give wrong results.
#include <mutex>

#include "draft.cuh"
#include "draft_run.cuh"
#include "draft_tc.cuh"

namespace {

using namespace spec;

constexpr size_t kStaticScratchBytes = 2u << 20;  // 2 MiB: about 58000 requests
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_draft_scratch[kStaticScratchBytes];

// Device address of g_draft_scratch on device `dev` (looked up once).
void* scratch_address(int dev) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_draft_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
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
