// C-ABI entry points of libspec: argument validation, workspace carving and
// kernel launches.  Every check happens on the host before anything is
// launched; no call synchronises the host or allocates device memory.
#include <cstdint>

#include "draft.cuh"
#include "draft_run.cuh"
#include "draft_tc.cuh"
#include "host_rows.cuh"
#include "schedule.cuh"
#include "accept_stats.cuh"
#include "residual_tc.cuh"
#include "verify.cuh"

namespace {

using namespace spec;

constexpr int kMaxGridY = 65535;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool valid_dtype(int d) { return d == SPEC_F32 || d == SPEC_BF16; }
size_t dtype_size(int d) { return d == SPEC_F32 ? 4 : 2; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Partials: the larger of the generic kernel's [R, nsplit] and the fused
// kernel's two slots of [R, splits <= kMaxDeviceSms] (positions alternate, so
// a position's partials survive until the next position's grid has merged
// them); counters: one per request (generic) or per 128-request tile (fused).
size_t draft_partials_bytes(int R, int V) {
  const size_t ns = (size_t)std::max(draft_nsplit(R, V), 2 * kMaxDeviceSms);
  return align256((size_t)R * ns * sizeof(Partial));
}
size_t draft_scratch_bytes(int R, int gamma, int V) {
  return draft_partials_bytes(R, V) + align256((size_t)R * (1 + gamma) * sizeof(unsigned));
}

bool draft_sizes_ok(int R, int gamma, int V, int r) {
  return R >= 1 && R <= kMaxGridY && gamma >= 1 && gamma <= kMaxGamma && V >= 1 &&
         V < (1 << 30) && r >= 1 && r <= kMaxRank &&
         (double)R * gamma * V < 1099511627776.0;  // 2^40
}

bool verify_sizes_ok(int R, int gamma, int V) {
  return R >= 1 && R <= kMaxGridY && gamma >= 1 && gamma + 1 <= kMaxGridY && V >= 1 &&
         V < (1 << 30) && (double)R * (gamma + 1) * V < 1099511627776.0;
}

int check_workspace(void* ws, size_t have, size_t need) {
  if (need == 0) return SPEC_OK;
  if (!ws || have < need) return SPEC_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return SPEC_ERR_ALIGNMENT;
  return SPEC_OK;
}

}  // namespace

// ------------------------------------------------- shared by the two draft
// entry points (spec_draft_sample and spec_draft_sample_static)
namespace spec {

// The fused tensor-core path needs bf16 factors with r a multiple of 64, 16-byte
// aligned rows of U (V * element size a multiple of 16) and an sm_100-family GPU.
bool draft_tc_ok(const spec_draft_args& a, int* sms) {
  if (a.fac_dtype != SPEC_BF16 || a.r % 64 != 0 || a.r > 256) return false;
  if (((size_t)a.V * dtype_size(a.logit_dtype)) % 16 != 0) return false;
  if (!aligned(a.U, 16) || !aligned(a.A, 16) || !aligned(a.Ct, 16)) return false;
  if (a.head == SPEC_HEAD_RNN && !aligned(a.S, 16)) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return major == 10 && *sms >= 1 && *sms <= kMaxDeviceSms;
}

int check_draft_args(const spec_draft_args* a) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  if (!draft_sizes_ok(a->R, a->gamma, a->V, a->r) || a->d < 0 || a->e < 0)
    return SPEC_ERR_INVALID_ARG;
  if (!valid_dtype(a->logit_dtype) || !valid_dtype(a->fac_dtype) || !valid_dtype(a->conf_dtype))
    return SPEC_ERR_INVALID_ARG;
  if (!a->U || !a->A || !a->Ct || !a->x0 || !a->draft_temp || !a->x || !a->q_tok || !a->lse_q)
    return SPEC_ERR_INVALID_ARG;
  if (!a->sts_temp || !a->c || !a->a) return SPEC_ERR_INVALID_ARG;
  if (a->head != SPEC_HEAD_MARKOV && a->head != SPEC_HEAD_RNN) return SPEC_ERR_INVALID_ARG;
  if (a->head == SPEC_HEAD_RNN && (!a->Wrnn || !a->S)) return SPEC_ERR_INVALID_ARG;
  if ((a->d > 0 && !a->h) || (a->e > 0 && !a->W1) || (a->d + a->e > 0 && !a->w))
    return SPEC_ERR_INVALID_ARG;
  const size_t ls = dtype_size(a->logit_dtype), fs = dtype_size(a->fac_dtype),
               cs = dtype_size(a->conf_dtype);
  if (!aligned(a->U, ls) || !aligned(a->A, fs) || !aligned(a->Ct, fs) || !aligned(a->x0, 4) ||
      !aligned(a->draft_temp, 4) || !aligned(a->x, 4) || !aligned(a->q_tok, 4) ||
      !aligned(a->lse_q, 4) || !aligned(a->sts_temp, 4) || !aligned(a->c, 4) ||
      !aligned(a->a, 4) || !aligned(a->P_out, 4) || !aligned(a->h, cs) || !aligned(a->W1, cs) ||
      !aligned(a->w, cs) || !aligned(a->status, 4))
    return SPEC_ERR_ALIGNMENT;
  if (a->head == SPEC_HEAD_RNN && (!aligned(a->Wrnn, fs) || !aligned(a->S, fs)))
    return SPEC_ERR_ALIGNMENT;
  return SPEC_OK;
}

int run_draft(const spec_draft_args& a, uint64_t seed, Partial* partials, unsigned* counters,
              int tc_sms, cudaStream_t s) {
  DraftStepParams p{};
  p.R = a.R;
  p.gamma = a.gamma;
  p.V = a.V;
  p.rank = a.r;
  p.nsplit = draft_nsplit(a.R, a.V);
  p.rid_base = a.request_id_base;
  p.key = philox_key(seed);
  p.U = a.U;
  p.A = a.A;
  p.Ct = a.Ct;
  if (a.head == SPEC_HEAD_RNN) {
    p.W = a.Wrnn;
    p.S = a.S;
  }
  p.x0 = a.x0;
  p.draft_temp = a.draft_temp;
  p.x = a.x;
  p.q_tok = a.q_tok;
  p.lse_q = a.lse_q;
  p.P_out = a.P_out;
  p.partials = partials;
  p.counters = counters;
  p.status = a.status;
  // counters [R] and the fused kernel's shared race bounds [gamma, R], zeroed together
  if (cudaMemsetAsync(p.counters, 0, (size_t)a.R * (1 + a.gamma) * sizeof(unsigned), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (tc_sms > 0) {
    DraftTCParams t{};
    t.R = a.R;
    t.gamma = a.gamma;
    t.V = a.V;
    t.rank = a.r;
    t.mtiles = (a.R + 127) / 128;
    t.ntiles = (a.V + 63) / 64;
    t.nsplit = draft_tc_nsplit(a.R, a.V, tc_sms);
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
    if (a.P_out && launch_draft_steps(p, a.logit_dtype, a.fac_dtype, true, s, /*probs_only=*/true) !=
                       cudaSuccess)
      return SPEC_ERR_CUDA;
  } else if (launch_draft_steps(p, a.logit_dtype, a.fac_dtype, a.P_out != nullptr, s) !=
             cudaSuccess) {
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

}  // namespace spec

extern "C" {

int spec_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* spec_error_string(int code) {
  switch (code) {
    case SPEC_OK: return "success";
    case SPEC_ERR_INVALID_ARG: return "invalid argument (null pointer, size or enum value)";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case SPEC_ERR_ALIGNMENT: return "pointer not aligned as required";
    case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status code";
  }
}

size_t spec_workspace_bytes(int stage, int R, int gamma, int V, int r) {
  switch (stage) {
    case SPEC_STAGE_DRAFT:
      return draft_sizes_ok(R, gamma, V, r) ? draft_scratch_bytes(R, gamma, V) : 0;
    case SPEC_STAGE_SCHEDULE:
      return 0;
    case SPEC_STAGE_VERIFY:
      return verify_sizes_ok(R, gamma, V) ? verify_scratch_bytes(R, gamma, V) : 0;
    default:
      return 0;
  }
}

int spec_draft_sample(const spec_draft_args* args, uint64_t seed, spec_stream_t stream) {
  int rc = check_draft_args(args);
  if (rc != SPEC_OK) return rc;
  const spec_draft_args& a = *args;
  const size_t need = draft_scratch_bytes(a.R, a.gamma, a.V);
  rc = check_workspace(a.workspace, a.workspace_bytes, need);
  if (rc != SPEC_OK) return rc;
  char* ws = static_cast<char*>(a.workspace);
  int sms = 0;
  const int tc_sms = draft_tc_ok(a, &sms) ? sms : 0;
  // partials first, the counters after the larger of the two paths' partials
  return run_draft(a, seed, reinterpret_cast<Partial*>(ws),
                   reinterpret_cast<unsigned*>(ws + draft_partials_bytes(a.R, a.V)), tc_sms,
                   reinterpret_cast<cudaStream_t>(stream));
}

int spec_schedule(const spec_sched_args* args, spec_stream_t stream) {
  if (!args) return SPEC_ERR_INVALID_ARG;
  const spec_sched_args& a = *args;
  if (a.R < 1 || a.gamma < 1 || a.n_sps < 1 || a.K < 0 ||
      (a.mode != SPEC_SCHED_EARLY_STOP && a.mode != SPEC_SCHED_GLOBAL &&
       a.mode != SPEC_SCHED_THRESHOLD) ||
      (a.mode == SPEC_SCHED_THRESHOLD && a.threshold != a.threshold) || !(a.b_step > 0.0) ||
      !(a.b_step < 1e300) || !(a.b_lo > -1e300 && a.b_lo < 1e300))
    return SPEC_ERR_INVALID_ARG;
  if (!a.a || !a.sps || !a.ell || !a.row_off || !a.stats) return SPEC_ERR_INVALID_ARG;
  if ((long)a.R * a.gamma > kSchedMaxCandidates) return SPEC_ERR_UNSUPPORTED;
  if (!aligned(a.a, 4) || !aligned(a.sps, 4) || !aligned(a.ell, 4) || !aligned(a.row_off, 4) ||
      !aligned(a.stats, 8) || !aligned(a.order, 4) || !aligned(a.status, 4) ||
      !aligned(a.K_dev, 4) || !aligned(a.n_free, 4))
    return SPEC_ERR_ALIGNMENT;
  SchedParams p{};
  p.R = a.R;
  p.gamma = a.gamma;
  p.n_sps = a.n_sps;
  p.K = a.K;
  p.mode = a.mode;
  p.b_lo = a.b_lo;
  p.b_step = a.b_step;
  p.threshold = a.threshold;
  p.a = a.a;
  p.sps = a.sps;
  p.ell = a.ell;
  p.row_off = a.row_off;
  p.stats = a.stats;
  p.order = a.order;
  p.K_dev = a.K_dev;
  p.n_free = a.n_free;
  p.status = a.status;
  return launch_schedule(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK
                                                                                    : SPEC_ERR_CUDA;
}

int spec_verify(const spec_verify_args* args, uint64_t seed, spec_stream_t stream) {
  if (!args) return SPEC_ERR_INVALID_ARG;
  const spec_verify_args& a = *args;
  if (a.mode != SPEC_VERIFY_SAMPLE && a.mode != SPEC_VERIFY_GREEDY) return SPEC_ERR_INVALID_ARG;
  if (!verify_sizes_ok(a.R, a.gamma, a.V) || !valid_dtype(a.tgt_dtype)) return SPEC_ERR_INVALID_ARG;
  if (!a.tgt || !a.tgt_row_off || !a.ell || !a.x || !a.accept_len || !a.out_tok || !a.n_out)
    return SPEC_ERR_INVALID_ARG;
  const bool sample = a.mode == SPEC_VERIFY_SAMPLE;
  if (a.c_star && !sample) return SPEC_ERR_INVALID_ARG;  // c* needs the draft rows
  if (!aligned(a.c_star, 4)) return SPEC_ERR_ALIGNMENT;
  int fac_dtype = SPEC_BF16, logit_dtype = SPEC_BF16, rank = 1;
  if (sample) {
    if (!a.q_tok || !a.lse_q || !a.draft || !(a.target_temp > 0.f) || !(a.target_temp < 1e30f))
      return SPEC_ERR_INVALID_ARG;
    const spec_draft_args& d = *a.draft;
    if (d.R != a.R || d.gamma != a.gamma || d.V != a.V || d.r < 1 || d.r > kMaxRank ||
        !valid_dtype(d.logit_dtype) || !valid_dtype(d.fac_dtype) || !d.U || !d.A || !d.Ct ||
        !d.x0 || !d.draft_temp)
      return SPEC_ERR_INVALID_ARG;
    if (d.request_id_base != a.request_id_base) return SPEC_ERR_INVALID_ARG;
    if (d.head != SPEC_HEAD_MARKOV && d.head != SPEC_HEAD_RNN) return SPEC_ERR_INVALID_ARG;
    if (d.head == SPEC_HEAD_RNN && !d.S) return SPEC_ERR_INVALID_ARG;
    fac_dtype = d.fac_dtype;
    logit_dtype = d.logit_dtype;
    rank = d.r;
    if (!aligned(d.U, dtype_size(logit_dtype)) || !aligned(d.A, dtype_size(fac_dtype)) ||
        !aligned(d.Ct, dtype_size(fac_dtype)) || !aligned(d.x0, 4) || !aligned(d.draft_temp, 4) ||
        !aligned(a.q_tok, 4) || !aligned(a.lse_q, 4) ||
        (d.head == SPEC_HEAD_RNN && !aligned(d.S, dtype_size(fac_dtype))))
      return SPEC_ERR_ALIGNMENT;
  }
  if (!aligned(a.tgt, dtype_size(a.tgt_dtype)) || !aligned(a.tgt_row_off, 4) || !aligned(a.ell, 4) ||
      !aligned(a.x, 4) || !aligned(a.accept_len, 4) || !aligned(a.out_tok, 4) ||
      !aligned(a.n_out, 4) || !aligned(a.p_tok, 4) || !aligned(a.lse_t, 4) || !aligned(a.status, 4))
    return SPEC_ERR_ALIGNMENT;
  const size_t need = verify_scratch_bytes(a.R, a.gamma, a.V);
  int rc = check_workspace(a.workspace, a.workspace_bytes, need);
  if (rc != SPEC_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  VerifyParams p{};
  p.mode = a.mode;
  p.R = a.R;
  p.gamma = a.gamma;
  p.V = a.V;
  p.nsplit = verify_nsplit(a.R, a.gamma, a.V);
  p.rank = rank;
  p.rid_base = a.request_id_base;
  p.key = philox_key(seed);
  p.rk = philox_round_keys(p.key);
  p.inv_target_temp = sample ? 1.0f / a.target_temp : 1.0f;
  p.tgt = a.tgt;
  p.tgt_row_off = a.tgt_row_off;
  p.ell = a.ell;
  p.x = a.x;
  p.q_tok = a.q_tok;
  p.lse_q = a.lse_q;
  if (sample) {
    p.U = a.draft->U;
    p.A = a.draft->A;
    p.Ct = a.draft->Ct;
    if (a.draft->head == SPEC_HEAD_RNN) p.S = a.draft->S;
    p.x0 = a.draft->x0;
    p.draft_temp = a.draft->draft_temp;
  }
  p.accept_len = a.accept_len;
  p.out_tok = a.out_tok;
  p.n_out = a.n_out;
  p.p_tok = a.p_tok;
  p.lse_t = a.lse_t;
  p.c_star = a.c_star;
  p.status = a.status;
  // Greedy mode: rows after a request's first mismatch influence no output.
  // (In sample mode the position order measured slower than the request order
  // at c5 -- its bonus-row races form the tail -- so it keeps request order.)
  p.skip_dead = !sample && a.gamma + 1 <= 64;
  {
    int dev = 0, major = 0, sms = 0;
    const bool dev_ok =
        cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    if (!dev_ok) return SPEC_ERR_CUDA;
    p.tc_residual = sample && major == 10 && sms >= 1 && sms <= kMaxDeviceSms &&
                    resid_tc_supported(a.tgt_dtype, logit_dtype, fac_dtype, rank, a.V, a.tgt, p.U, p.A, p.Ct) &&
                    aligned(p.S, 16);
    p.device_sms = sms;
  }
  size_t cnt_off = 0, cnt_bytes = 0;
  p.ws = verify_scratch_carve(a.workspace, a.R, a.gamma, a.V, &cnt_off, &cnt_bytes);
  if (cudaMemsetAsync(static_cast<char*>(a.workspace) + cnt_off, 0, cnt_bytes, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (a.p_tok && cudaMemsetAsync(a.p_tok, 0, (size_t)a.R * a.gamma * sizeof(float), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (a.lse_t &&
      cudaMemsetAsync(a.lse_t, 0, (size_t)a.R * (a.gamma + 1) * sizeof(float), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (launch_verify(p, a.tgt_dtype, logit_dtype, fac_dtype, s) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int spec_accept_stats(const spec_accept_stats_args* args, spec_stream_t stream) {
  if (!args) return SPEC_ERR_INVALID_ARG;
  const spec_accept_stats_args& a = *args;
  if (a.R < 0 || a.gamma < 1 || a.n_buckets < 1 || a.bucket < 0 || a.bucket >= a.n_buckets ||
      !(a.beta > 0.0 && a.beta <= 1.0))
    return SPEC_ERR_INVALID_ARG;
  if (!a.ema || !a.count || (a.R > 0 && (!a.ell || !a.accept_len))) return SPEC_ERR_INVALID_ARG;
  if (a.gamma > kAcceptStatsMaxGamma) return SPEC_ERR_UNSUPPORTED;
  if (!aligned(a.ell, 4) || !aligned(a.accept_len, 4) || !aligned(a.ema, 8) ||
      !aligned(a.count, 8) || !aligned(a.estimate, 8) || !aligned(a.status, 4))
    return SPEC_ERR_ALIGNMENT;
  AcceptStatsParams p{};
  p.R = a.R;
  p.gamma = a.gamma;
  p.bucket = a.bucket;
  p.n_buckets = a.n_buckets;
  p.min_count = a.min_count;
  p.beta = a.beta;
  p.ell = a.ell;
  p.accept_len = a.accept_len;
  p.ema = a.ema;
  p.count = reinterpret_cast<long long*>(a.count);
  p.estimate = a.estimate;
  p.status = a.status;
  return launch_accept_stats(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

int spec_calibration(const spec_calibration_args* args, spec_stream_t stream) {
  if (!args) return SPEC_ERR_INVALID_ARG;
  const spec_calibration_args& a = *args;
  if (a.R < 0 || a.gamma < 1 || a.n_bins < 1) return SPEC_ERR_INVALID_ARG;
  if (!a.count || !a.sum_c || !a.sum_acc || (a.R > 0 && (!a.c || !a.ell || !a.accept_len)))
    return SPEC_ERR_INVALID_ARG;
  if (a.n_bins > kCalibrationMaxBins) return SPEC_ERR_UNSUPPORTED;
  if (!aligned(a.c, 4) || !aligned(a.ell, 4) || !aligned(a.accept_len, 4) ||
      !aligned(a.count, 8) || !aligned(a.sum_c, 8) || !aligned(a.sum_acc, 8) ||
      !aligned(a.ece, 8) || !aligned(a.status, 4))
    return SPEC_ERR_ALIGNMENT;
  CalibrationParams p{};
  p.R = a.R;
  p.gamma = a.gamma;
  p.n_bins = a.n_bins;
  p.c = a.c;
  p.ell = a.ell;
  p.accept_len = a.accept_len;
  p.count = reinterpret_cast<long long*>(a.count);
  p.sum_c = a.sum_c;
  p.sum_acc = reinterpret_cast<long long*>(a.sum_acc);
  p.ece = a.ece;
  p.status = a.status;
  return launch_calibration(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

int spec_round_host(const spec_round_host_args* args, uint64_t seed, spec_stream_t stream) {
  if (!args || !args->draft || !args->sched || !args->verify) return SPEC_ERR_INVALID_ARG;
  const spec_draft_args& d = *args->draft;
  const spec_sched_args& sc = *args->sched;
  const spec_verify_args& v = *args->verify;
  // the stages must be chained through the same device buffers
  if (sc.R != d.R || sc.gamma != d.gamma || v.R != d.R || v.gamma != d.gamma || v.V != d.V ||
      v.mode != SPEC_VERIFY_SAMPLE || sc.a != d.a || v.ell != sc.ell || v.x != d.x ||
      v.q_tok != d.q_tok || v.lse_q != d.lse_q || !v.draft || v.draft->U != d.U ||
      v.draft->A != d.A || v.draft->Ct != d.Ct || v.draft->x0 != d.x0 ||
      v.draft->head != d.head || (d.head == SPEC_HEAD_RNN && v.draft->S != d.S))
    return SPEC_ERR_INVALID_ARG;
  if (!valid_dtype(d.logit_dtype) || !valid_dtype(d.conf_dtype) || !valid_dtype(v.tgt_dtype) ||
      d.R < 1 || d.gamma < 1 || d.V < 1 || d.d < 0)
    return SPEC_ERR_INVALID_ARG;
  const bool packed = args->tgt_scheduled_only != 0;
  const void* tgt_dev_view = nullptr;  // the device's address of tgt_host (packed mode)
  if (packed) {
    if (!args->tgt_host || v.tgt_row_off != sc.row_off || !v.tgt) return SPEC_ERR_INVALID_ARG;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, args->tgt_host) != cudaSuccess) {
      cudaGetLastError();  // clear this (non-sticky) error so later launch checks do not see it
      return SPEC_ERR_UNSUPPORTED;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return SPEC_ERR_UNSUPPORTED;
    tgt_dev_view = attr.devicePointer;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto h2d = [&](const void* dst, const void* src, size_t bytes) {
    if (!src || bytes == 0) return true;
    if (!dst) return false;
    return cudaMemcpyAsync(const_cast<void*>(dst), src, bytes, cudaMemcpyHostToDevice, s) ==
           cudaSuccess;
  };
  const size_t RG = (size_t)d.R * d.gamma;
  if (!h2d(d.U, args->U_host, RG * d.V * dtype_size(d.logit_dtype)) ||
      !h2d(d.h, args->h_host, RG * d.d * dtype_size(d.conf_dtype)) ||
      !h2d(d.x0, args->x0_host, (size_t)d.R * sizeof(int32_t)) ||
      (!packed && !h2d(v.tgt, args->tgt_host, args->tgt_rows * d.V * dtype_size(v.tgt_dtype))))
    return SPEC_ERR_CUDA;
  int rc = spec_draft_sample(args->draft, seed, stream);
  if (rc != SPEC_OK) return rc;
  rc = spec_schedule(args->sched, stream);
  if (rc != SPEC_OK) return rc;
  if (packed) {
    GatherRowsParams g{};
    g.R = d.R;
    g.G1 = d.gamma + 1;
    g.row_bytes = (size_t)d.V * dtype_size(v.tgt_dtype);
    g.src = static_cast<const unsigned char*>(tgt_dev_view);
    g.dst = static_cast<unsigned char*>(const_cast<void*>(v.tgt));
    g.row_off = sc.row_off;
    g.status = v.status;
    if (launch_gather_rows(g, s) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  rc = spec_verify(args->verify, seed, stream);
  if (rc != SPEC_OK) return rc;
  auto d2h = [&](void* dst, const void* src, size_t bytes) {
    if (!dst) return true;
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  };
  if (!d2h(args->out_tok_host, v.out_tok, (size_t)d.R * (d.gamma + 1) * sizeof(int32_t)) ||
      !d2h(args->accept_len_host, v.accept_len, (size_t)d.R * sizeof(int32_t)) ||
      !d2h(args->n_out_host, v.n_out, (size_t)d.R * sizeof(int32_t)) ||
      !d2h(args->stats_host, sc.stats, 4 * sizeof(double)))
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // extern "C"



