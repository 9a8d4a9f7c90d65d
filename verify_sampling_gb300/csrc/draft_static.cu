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
  if (!args) return SPEC_ERR_INVALID_ARG;
  const spec_draft_args& a = *args;
  // The same argument rules as spec_draft_sample (the workspace fields are ignored).
  if (a.R < 1 || a.R > 65535 || a.gamma < 1 || a.gamma > kMaxGamma || a.V < 1 || a.V >= (1 << 30) ||
      a.r < 1 || a.r > kMaxRank || a.d < 0 || a.e < 0 || (double)a.R * a.gamma * a.V >= 1099511627776.0)
    return SPEC_ERR_INVALID_ARG;
  if ((a.logit_dtype != SPEC_F32 && a.logit_dtype != SPEC_BF16) ||
      (a.fac_dtype != SPEC_F32 && a.fac_dtype != SPEC_BF16) ||
      (a.conf_dtype != SPEC_F32 && a.conf_dtype != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  if (!a.U || !a.A || !a.Ct || !a.x0 || !a.draft_temp || !a.x || !a.q_tok || !a.lse_q || !a.sts_temp ||
      !a.c || !a.a || (a.d > 0 && !a.h) || (a.e > 0 && !a.W1) || (a.d + a.e > 0 && !a.w))
    return SPEC_ERR_INVALID_ARG;
  const bool rnn = a.head == SPEC_HEAD_RNN;
  if ((a.head != SPEC_HEAD_MARKOV && !rnn) || (rnn && (!a.Wrnn || !a.S))) return SPEC_ERR_INVALID_ARG;
  auto al = [](const void* q, size_t n) { return ((uintptr_t)q % n) == 0; };
  const size_t ls = a.logit_dtype == SPEC_F32 ? 4 : 2, fs = a.fac_dtype == SPEC_F32 ? 4 : 2,
               cs = a.conf_dtype == SPEC_F32 ? 4 : 2;
  if (!al(a.U, ls) || !al(a.A, fs) || !al(a.Ct, fs) || !al(a.x0, 4) || !al(a.draft_temp, 4) ||
      !al(a.x, 4) || !al(a.q_tok, 4) || !al(a.lse_q, 4) || !al(a.sts_temp, 4) || !al(a.c, 4) ||
      !al(a.a, 4) || !al(a.P_out, 4) || !al(a.h, cs) || !al(a.W1, cs) || !al(a.w, cs) ||
      !al(a.status, 4) || (rnn && (!al(a.Wrnn, fs) || !al(a.S, fs))))
    return SPEC_ERR_ALIGNMENT;

  int dev = 0, major = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const bool tc = a.fac_dtype == SPEC_BF16 && a.r % 64 == 0 && ((size_t)a.V * ls) % 16 == 0 &&
                  al(a.U, 16) && al(a.A, 16) && al(a.Ct, 16) && (!rnn || al(a.S, 16)) && major == 10 && sms >= 1 &&
                  sms <= kMaxDeviceSms;

  // Exact scratch for the path taken: partials [R, splits], then counters [R]
  // and the race bounds [gamma, R].
  const int nsplit_generic = draft_nsplit(a.R, a.V);
  const int nsplit_tc = tc ? draft_tc_nsplit(a.R, a.V, sms) : 0;
  const size_t part_bytes =
      round256((size_t)a.R * (tc ? 2 * nsplit_tc : nsplit_generic) * sizeof(Partial));
  const size_t cnt_bytes = (size_t)a.R * (1 + a.gamma) * sizeof(unsigned);
  if (part_bytes + cnt_bytes > kStaticScratchBytes) return SPEC_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(scratch_address(dev));
  if (!ws) return SPEC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  DraftStepParams p{};
  p.R = a.R;
  p.gamma = a.gamma;
  p.V = a.V;
  p.rank = a.r;
  p.nsplit = nsplit_generic;
  p.rid_base = a.request_id_base;
  p.key = philox_key(seed);
  p.U = a.U;
  p.A = a.A;
  p.Ct = a.Ct;
  if (rnn) {
    p.W = a.Wrnn;
    p.S = a.S;
  }
  p.x0 = a.x0;
  p.draft_temp = a.draft_temp;
  p.x = a.x;
  p.q_tok = a.q_tok;
  p.lse_q = a.lse_q;
  p.P_out = a.P_out;
  p.partials = reinterpret_cast<Partial*>(ws);
  p.counters = reinterpret_cast<unsigned*>(ws + part_bytes);
  p.status = a.status;
  if (cudaMemsetAsync(p.counters, 0, cnt_bytes, s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (tc) {
    DraftTCParams t{};
    t.R = a.R;
    t.gamma = a.gamma;
    t.V = a.V;
    t.rank = a.r;
    t.mtiles = (a.R + 127) / 128;
    t.ntiles = (a.V + 63) / 64;
    t.nsplit = nsplit_tc;
    t.rid_base = a.request_id_base;
    t.key = p.key;
    t.x0 = a.x0;
    t.draft_temp = a.draft_temp;
    t.A = a.A;
    t.W = p.W;
    t.S = p.S;
    t.x = a.x;
    t.q_tok = a.q_tok;
    t.lse_q = a.lse_q;
    t.partials = p.partials;
    t.counters = p.counters;
    t.row_best = p.counters + a.R;
    t.status = a.status;
    if (launch_draft_tc(t, a.logit_dtype, a.U, a.Ct, s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (a.P_out && launch_draft_steps(p, a.logit_dtype, a.fac_dtype, true, s, true) != cudaSuccess)
      return SPEC_ERR_CUDA;
  } else if (launch_draft_steps(p, a.logit_dtype, a.fac_dtype, a.P_out != nullptr, s) != cudaSuccess) {
    return SPEC_ERR_CUDA;
  }
  ConfParams c{};
  c.R = a.R;
  c.gamma = a.gamma;
  c.V = a.V;
  c.d = a.d;
  c.e = a.e;
  c.x0 = a.x0;
  c.x = a.x;
  c.h = a.h;
  c.W1 = a.W1;
  c.w = a.w;
  c.sts_temp = a.sts_temp;
  c.c = a.c;
  c.a = a.a;
  c.status = a.status;
  return launch_confidence(c, a.conf_dtype, s) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
