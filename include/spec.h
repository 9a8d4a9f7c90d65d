/*
 * spec.h -- C ABI of the GB300 speculative-decoding round library (libspec.so).
 *
 * One speculative round for R concurrent requests and a draft block of gamma
 * positions over a vocabulary of V tokens, in three stages:
 *
 *   spec_draft_sample  semi-autoregressive draft head (Markov, or RNN with a
 *                      recurrent state), sampling, confidence head with
 *                      sequential temperature scaling and survival products
 *   spec_schedule      hardware-aware prefix scheduler (sorted survivals,
 *                      greedy admission while tau * SPS(B) rises, top-K cap)
 *   spec_verify        lossless rejection-sampling verification (residual
 *                      resample, bonus token) or greedy argmax matching
 *
 * Sources: "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation" (summary article, adg.csdn.net) and the
 * speculative-decoding history article (wzjinhao.cn/news/15713); the citations
 * at each entry point name the section.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers to caller-owned memory, row-major,
 *    index order (request, position, vocabulary).  Positions j are 1-based in
 *    the text and 0-based in memory (slot j-1).
 *  - Argument structs are HOST memory, read only during the call.
 *  - Every call is asynchronous on `stream`; none synchronises the host and
 *    none allocates device memory.  Scratch memory is the caller's `workspace`
 *    buffer of at least spec_workspace_bytes(...) bytes, 256-byte aligned; two
 *    calls that run at the same time need separate workspaces.
 *  - Return value: SPEC_OK or an SPEC_ERR_* code.  Argument errors are found
 *    on the host before anything is launched.  SPEC_ERR_CUDA reports a launch
 *    error (cudaGetLastError) -- the stream may hold a partial round then.
 *  - Data errors found on the device (a token id outside [0, V), an l_r outside
 *    [0, gamma], a non-finite survival) set bits in the optional device word
 *    `status` (OR-ed, never cleared by the library); the kernels clamp the bad
 *    value and carry on, so a bad input never faults the GPU.
 *  - Randomness: one counter-based Philox-4x32-10 stream (Salmon et al., SC'11).
 *    Counter = (v / 4, position j, request_id_base + r, purpose), key = (seed
 *    low 32 bits, seed high 32 bits); vocabulary entry v uses output word v % 4,
 *    mapped to the uniform (2 * (word & 0x7FFFFF) + 1) * 2^-24 in (0, 1).  Purposes:
 *    0 draft Gumbel, 1 accept test (word 0 of block 0), 2 residual Gumbel,
 *    3 bonus Gumbel.  Results depend only on (seed, global request id,
 *    position), so a batch split into pieces with matching request_id_base
 *    gives identical results.
 *  - The library keeps no global state, with one exception: the scratch array
 *    of spec_draft_sample_static (below) and its cached device address.
 *    Calls are thread-safe, except that calls of that entry point which
 *    overlap on the GPU share its scratch.
 */
#ifndef SPEC_H
#define SPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *spec_stream_t;

enum spec_status_code {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* null pointer, bad size or enum value          */
  SPEC_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement  */
  SPEC_ERR_ALIGNMENT = 3,   /* a pointer is not aligned as documented        */
  SPEC_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required    */
  SPEC_ERR_CUDA = 5         /* a CUDA runtime call or launch failed          */
};

enum spec_dtype { SPEC_F32 = 0, SPEC_BF16 = 1 };
enum spec_verify_mode { SPEC_VERIFY_SAMPLE = 0, SPEC_VERIFY_GREEDY = 1 };
enum spec_sched_mode { SPEC_SCHED_EARLY_STOP = 0, SPEC_SCHED_GLOBAL = 1, SPEC_SCHED_THRESHOLD = 2 };
enum spec_stage { SPEC_STAGE_DRAFT = 0, SPEC_STAGE_SCHEDULE = 1, SPEC_STAGE_VERIFY = 2 };
enum spec_head { SPEC_HEAD_MARKOV = 0, SPEC_HEAD_RNN = 1 };

/* Bits of the device status word. */
#define SPEC_STATUS_BAD_TOKEN 0x1u    /* a token id was outside [0, V)          */
#define SPEC_STATUS_BAD_ELL 0x2u      /* an l_r was outside [0, gamma]          */
#define SPEC_STATUS_BAD_SURVIVAL 0x4u /* a survival was negative or not finite  */
#define SPEC_STATUS_BAD_ROW 0x8u      /* a target row index was negative        */
#define SPEC_STATUS_TIMEOUT 0x10u     /* an internal pipeline wait gave up after
                                         2 s (never expected): the call's
                                         outputs are invalid                     */

/* ------------------------------------------------------------------ draft -
 * DSpark summary, "第二阶段：轻量顺序头" (sequential Markov head) and the
 * history article, "杀招一": for k = 1..gamma, sequentially,
 *     z_k = (U_k + B_k(x_{k-1})) / T_k,   B_k(x) = A_k[x, :] C_k,
 *     P_k = softmax(z_k),  x_k ~ P_k  (Gumbel-max with the purpose-0 stream),
 * x_0 = the anchor token x0[r].  DSpark summary, "2.1 置信度头": the
 * confidence c_k = sigmoid((w . [h_k ; W1[x_{k-1}]]) / tau_k) with the
 * per-position temperature tau_k of sequential temperature scaling, and the
 * history article, "杀招二": survival a_{r,j} = prod_{i<=j} c_{r,i}.
 *
 * Layouts (dtype in brackets):
 *   U      [R, gamma, V]   logit_dtype   parallel-backbone logits U_k
 *   A      [gamma, V, r]   fac_dtype     left factor, row x = A_k[x, :]
 *   Ct     [gamma, V, r]   fac_dtype     right factor C_k stored TRANSPOSED
 *                                        (vocabulary-major): Ct[k][v][i] = C_k[i][v]
 *   x0     [R] int32       anchor tokens
 *   draft_temp [gamma] f32 T_k (> 0)
 *   h      [R, gamma, d]   conf_dtype    backbone hidden states h_k
 *   W1     [V, e]          conf_dtype    Markov embedding table
 *   w      [d + e]         conf_dtype    confidence-head weights (no bias)
 *   sts_temp [gamma] f32   tau_k (> 0)
 * Outputs (f32 unless noted):
 *   x [R, gamma] int32 sampled tokens; q_tok = P_k[x_k]; lse_q = log sum exp z_k;
 *   c, a [R, gamma]; P_out [R, gamma, V] (nullable) the full draft distributions.
 * Sizes: R >= 1, 1 <= gamma <= 64, 1 <= V < 2^30, 1 <= r <= 256, d >= 0, e >= 0,
 * R * gamma * V < 2^40.  Alignment: every pointer aligned to its element size.
 *
 * Sequential head.  The same passage names two heads, a Markov head and an RNN
 * head that keeps a longer dependency, and gives no formula for the second.
 * head = SPEC_HEAD_MARKOV (0, the default of a zeroed struct) is the bias
 * above.  head = SPEC_HEAD_RNN keeps one state vector per request:
 *     s_0 = 0,  s_k = store(tanh(A_k[x_{k-1}, :] + s_{k-1} W_k)),  B_k = s_k C_k,
 * the pre-activation summed in fp32 (A_k first, then i = 0..r-1 ascending) and
 * store() rounding to fac_dtype (bf16: round to nearest even; f32: as is).
 *   Wrnn   [gamma, r, r]   fac_dtype     W_k[i][j] maps s_{k-1}[i] to column j
 *   S      [R, gamma, r]   fac_dtype     out: s_k of (r, k) at S[r][k-1]; spec_verify
 *                                        reads it back (through args->draft) for the
 *                                        residual and c*, so keep it until then
 * Wrnn and S are ignored (may be NULL) for the Markov head; for the RNN head
 * both are required and aligned to the element size.  Any other head value is
 * SPEC_ERR_INVALID_ARG.
 */
typedef struct spec_draft_args {
  int R, gamma, V, r, d, e;
  int logit_dtype; /* spec_dtype of U                 */
  int fac_dtype;   /* spec_dtype of A and Ct          */
  int conf_dtype;  /* spec_dtype of h, W1 and w       */
  uint32_t request_id_base;
  const void *U;
  const void *A;
  const void *Ct;
  const int32_t *x0;
  const float *draft_temp;
  const void *h;
  const void *W1;
  const void *w;
  const float *sts_temp;
  int32_t *x;
  float *q_tok;
  float *lse_q;
  float *c;
  float *a;
  float *P_out;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *status; /* nullable device word */
  int head;         /* spec_head */
  const void *Wrnn;
  void *S;
} spec_draft_args;

int spec_draft_sample(const spec_draft_args *args, uint64_t seed, spec_stream_t stream);

/* Same as spec_draft_sample, for callers that cannot allocate device memory
 * (code inside an allocator, runtimes that forbid cudaMalloc while serving,
 * embeddings that own all device memory).  The pages have no counterpart: this
 * is a property of the library, not of the method.  It ignores
 * args->workspace and uses a 2 MiB scratch array that the library keeps in
 * device memory (held by every GPU that loads the library until exit); it
 * calls no cudaMalloc or cudaFree.  Returns SPEC_ERR_UNSUPPORTED when the
 * sizes need more scratch than that (the need is about
 * 64 * R * splits + 4 * R * (1 + gamma) bytes on the tensor-core path, two
 * slots of split partials, with at most 152 splits per 128 requests on a
 * GB300, and 32 * R * splits + 4 * R * (1 + gamma) on the generic one; for
 * example 4096 requests at gamma = 16 on the tensor-core path need 1.33 MB).
 * The first call on each device resolves the array's device address
 * (cudaGetSymbolAddress) and caches it per context; make it before any stream
 * capture.  A context that is destroyed and created again (cudaDeviceReset)
 * gets a fresh lookup on its next call.  All calls share the array: calls
 * that overlap on the GPU race and give wrong results. */
int spec_draft_sample_static(const spec_draft_args *args, uint64_t seed, spec_stream_t stream);

/* --------------------------------------------------------------- schedule -
 * DSpark summary, "2.2 硬件感知前缀调度器": maximise Theta = tau * SPS(B),
 * B = sum_r (1 + l_r), tau = sum_r sum_{j<=l_r} a_{r,j}, by sorting all
 * R * gamma survivals in descending order and admitting them one at a time
 * while Theta rises (early stop), cost O(gamma R log gamma R); the history
 * article, "杀招三", walks through the same rule.  DSpark summary, "挑战2":
 * the number admitted is capped by K (top-K from older confidences) and a
 * global search over all sorted prefixes may replace the early stop.
 *
 *   a       [R, gamma] f32  survivals (>= 0; non-increasing in j for a
 *                            prefix-closed result)
 *   sps     [n_sps] f32     SPS(B) at B_i = b_lo + i * b_step (b_step > 0);
 *                            linear interpolation inside, clamped outside
 *   K       cap on sum_r l_r (>= 0)
 *   mode    SPEC_SCHED_EARLY_STOP: admit while Theta_{n+1} > Theta_n (strict),
 *           Theta_0 = 0;  SPEC_SCHED_GLOBAL: n = smallest argmax_n Theta_n;
 *           SPEC_SCHED_THRESHOLD: a static confidence threshold (DSpark
 *           summary, comparison table: SpecDec++; Figure 5 sweeps it) -- n =
 *           the number of survivals with a >= threshold (compared in fp64,
 *           exactly), capped by K; SPS only enters the reported Theta
 *   threshold  used by SPEC_SCHED_THRESHOLD only; NaN is an argument error
 * Sort order: a descending, then request ascending, then position ascending.
 * tau and Theta are computed in fp64.
 * Outputs: ell [R] int32; row_off [R + 1] int32 with row_off[r + 1] = row_off[r]
 * + 1 + l_r (the packed verify layout); stats [4] f64 = {n, B, tau, Theta};
 * order [R * gamma] int32 (nullable) = candidate ids r * gamma + j - 1 in
 * sorted order.  Sizes: R * gamma <= 8192 (one thread block).
 *
 * Asynchronous cap (DSpark summary, "挑战2"): the verification capacity of a
 * round is capped from the confidences of two rounds earlier, while the
 * candidates themselves are ranked by the newest survivals; the history
 * article, "杀招三", adds that the scheduler uses the previous batch's estimate
 * so the GPU never waits for the host.  Reading: K_t = the number the same
 * rule admits on round t-2's survivals with no cap.  Both ends stay on the
 * device:
 *   n_free  (nullable) receives that uncapped number for this round's a;
 *   K_dev   (nullable) is read on the device: the cap becomes
 *           min(K, max(K_dev[0], 0)).
 * A caller keeps two int32 words, passes word t % 2 as both K_dev and n_free
 * in round t (the kernel reads K_dev before it writes n_free), and fills both
 * with K before the first round.  With both NULL the call is as above.
 */
typedef struct spec_sched_args {
  int R, gamma;
  const float *a;
  const float *sps;
  int n_sps;
  double b_lo, b_step;
  int K;
  int mode;
  int32_t *ell;
  int32_t *row_off;
  double *stats;
  int32_t *order;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *status;
  double threshold;
  const int32_t *K_dev; /* nullable device word: cap = min(K, max(K_dev[0], 0)) */
  int32_t *n_free;      /* nullable device word: n the same rule admits with no cap */
} spec_sched_args;

int spec_schedule(const spec_sched_args *args, spec_stream_t stream);

/* ----------------------------------------------------- acceptance stats -
 * LightSpec article, "无需额外训练，基于运行时统计的动态调度": acceptance rates are
 * kept per request-scale / batch-size class and per MTP length as exponential
 * moving averages updated every round, and a length with too few samples is
 * estimated by interpolating over the other lengths.  One call folds a
 * verified round into class `bucket` (one thread block, no workspace):
 *   n_L = #{r : ell[r] = L}, S_L = sum of their accept_len, for L = 1..gamma;
 *   where n_L > 0:  m_L = S_L / (L * n_L)  (fp64, correctly rounded);
 *                   ema = m_L if count == 0, else fma(beta, m_L - ema, ema);
 *                   count += n_L.
 * Requests with ell = 0 carry no draft and are skipped.  An ell outside
 * [0, gamma] or an accept_len outside [0, ell] is skipped and sets
 * SPEC_STATUS_BAD_ELL.
 *   ell, accept_len  [R] int32 device (spec_schedule / spec_verify outputs)
 *   ema    [n_buckets, gamma] f64 device, in/out (zero it before the first call)
 *   count  [n_buckets, gamma] int64 device, in/out (zero before the first call)
 *   estimate [gamma] f64 device, nullable: rates of class `bucket` after the
 *          update -- the entry where count >= max(min_count, 1), else linear
 *          interpolation in L between the nearest such lengths below and
 *          above (fma(w, e_hi - e_lo, e_lo), w = (L - lo) / (hi - lo)), the
 *          nearest one when only one side has any, NaN when none has
 *   beta   in (0, 1];  0 <= bucket < n_buckets;  gamma <= 1024;  R >= 0
 * Every operation is the fp64 one written above, so results are
 * reproducible bit for bit.
 */
typedef struct spec_accept_stats_args {
  int R, gamma;
  const int32_t *ell;
  const int32_t *accept_len;
  int bucket, n_buckets;
  double beta;
  int min_count;
  double *ema;
  int64_t *count;
  double *estimate;
  uint32_t *status;
} spec_accept_stats_args;

int spec_accept_stats(const spec_accept_stats_args *args, spec_stream_t stream);

/* ---------------------------------------------------------- calibration -
 * DSpark summary, Figure 6 and "2.1 置信度头": the confidences c_{r,j} (after
 * sequential temperature scaling) are judged by a reliability diagram and the
 * expected calibration error (ECE) against realised acceptance.  One call
 * folds a verified round into an equal-width diagram of n_bins bins over
 * [0, 1] (one thread block, no workspace):
 *   tested positions of request r: j = 1..min(l_r, accept_len_r + 1), the
 *   ones the verifier ruled on; position j counts as accepted iff
 *   j <= accept_len_r;  bin b = min(floor(c * n_bins), n_bins - 1) (fp64);
 *   count[b] += 1, sum_c[b] += c, sum_acc[b] += accepted.
 *   ece (nullable) = sum_b |sum_acc_b - sum_c_b| / sum_b count_b after the
 *   update, i.e. sum_b (n_b / N) |acc_b - conf_b|; NaN when N = 0.
 *   c [R, gamma] f32 device (spec_draft_sample's c);  ell, accept_len [R] int32
 *   count, sum_acc [n_bins] int64 and sum_c [n_bins] f64 device, in/out (zero
 *   them before the first call);  ece [1] f64 device;  1 <= n_bins <= 1024
 * Counts are exact; sum_c adds in an unspecified order (fp64 rounding only).
 * An ell outside [0, gamma] or accept_len outside [0, ell] sets
 * SPEC_STATUS_BAD_ELL, a c outside [0, 1] or NaN SPEC_STATUS_BAD_SURVIVAL; the
 * entry is skipped.
 */
typedef struct spec_calibration_args {
  int R, gamma;
  const float *c;
  const int32_t *ell;
  const int32_t *accept_len;
  int n_bins;
  int64_t *count;
  double *sum_c;
  int64_t *sum_acc;
  double *ece;
  uint32_t *status;
} spec_calibration_args;

int spec_calibration(const spec_calibration_args *args, spec_stream_t stream);

/* ----------------------------------------------------------------- verify -
 * History article, "1.1运行机制" (rejection sampling): accept x_j with
 * probability min(1, p(x_j) / q(x_j)) -- the test is u < p/q with u from the
 * purpose-1 stream -- and discard the rest of the draft after the first
 * rejection; DSpark summary, Figure 1: the rejected position j* is
 * regenerated, here from norm(max(0, p - q)) (Gumbel-max over the residual,
 * purpose 2; from p itself if the residual is zero everywhere), which makes
 * the round lossless ("数学上的美感").  When all l_r admitted positions are
 * accepted, one bonus token is sampled from target row l_r + 1 (purpose 3),
 * the "1 +" of B in DSpark "2.2".  SPEC_VERIFY_GREEDY accepts while x_j is the
 * target argmax (lowest index on ties) and emits the target argmax of the
 * first mismatching row (or of row l_r + 1).
 *
 *   tgt      target logits rows [*, V] (tgt_dtype); the row of (r, j),
 *            j = 1..l_r + 1, is tgt_row_off[r] + j - 1.  This fits a packed
 *            [B, V] batch (tgt_row_off = row_off of spec_schedule) and a padded
 *            [R, gamma + 1, V] layout (tgt_row_off[r] = r * (gamma + 1)).
 *   ell [R], x [R, gamma] int32; q_tok, lse_q [R, gamma] f32 (from the draft)
 *   p = softmax(L / target_temp)  (target_temp > 0; unused in greedy mode)
 *   draft    the draft call's arguments (U, A, Ct, x0, draft_temp, r, dtypes):
 *            the residual recomputes q at row j*.  May be NULL in greedy mode.
 * Outputs: accept_len [R]; out_tok [R, gamma + 1] = accepted draft tokens, then
 * the regenerated or bonus token, then -1; n_out [R] = accept_len + 1.
 * Optional (nullable): p_tok [R, gamma] = p(x_j) for j <= l_r (others 0),
 * lse_t [R, gamma + 1] = log sum exp(L_j / target_temp) of the rows read
 * (sample mode; others 0).
 * c_star [R, gamma] f32 (nullable; sample mode only, else SPEC_ERR_INVALID_ARG):
 * the calibration target of the confidence head, DSpark summary "2.1 置信度头":
 * c* = 1 - TV(p, q) = sum_v min(p_v, q_v) for every verified draft row
 * j <= l_r (q recomputed from the draft arguments), NaN past l_r.  A
 * diagnostic: it costs one more pass over the admitted target and draft rows.
 * Rows read: greedy mode needs a request's rows only up to its first
 * mismatch or row l_r + 1.  With gamma <= 63 its rows are taken in position
 * order and a row past a request's end already found is skipped (rows in
 * flight when the end is found are still read).  Sample mode reads every
 * scheduled row.
 */
typedef struct spec_verify_args {
  int mode;
  int R, gamma, V;
  int tgt_dtype;
  uint32_t request_id_base;
  const void *tgt;
  const int32_t *tgt_row_off;
  const int32_t *ell;
  const int32_t *x;
  const float *q_tok;
  const float *lse_q;
  float target_temp;
  const spec_draft_args *draft;
  int32_t *accept_len;
  int32_t *out_tok;
  int32_t *n_out;
  float *p_tok;
  float *lse_t;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *status;
  float *c_star;
} spec_verify_args;

int spec_verify(const spec_verify_args *args, uint64_t seed, spec_stream_t stream);

/* --------------------------------------------------- one round, host I/O -
 * DSpark summary, Figure 1 (one round: draft, schedule, verify) as a single
 * call on host buffers.  The per-round inputs are copied from host memory
 * into the device buffers the stage arguments name.  The three stages then
 * run as spec_draft_sample, spec_schedule and spec_verify, and the per-round
 * results are copied back.  Everything is asynchronous on `stream`, one
 * cudaMemcpyAsync per buffer.  Page-locked host buffers keep the copies
 * asynchronous; pageable ones make them synchronous.  The weights (A, Ct, W1,
 * w, the temperatures, the SPS table) stay in device memory across rounds.
 *   draft, sched, verify  as for the three calls.  draft->U, draft->h,
 *     draft->x0 and verify->tgt are the destinations of the input copies.
 *     The stages must be chained (checked): sched->a is draft->a;
 *     verify->ell is sched->ell; verify->x, q_tok and lse_q are draft's x,
 *     q_tok and lse_q; the sizes agree; and verify runs in sample mode with
 *     verify->draft the same draft arguments.
 *   U_host [R, gamma, V] (draft logit dtype), h_host [R, gamma, d] (confidence
 *     dtype), x0_host [R] int32, tgt_host [tgt_rows, V] (target dtype):
 *     per-round inputs; each is nullable, and then the device buffer is used
 *     as it stands.
 *   out_tok_host [R, gamma + 1], accept_len_host [R], n_out_host [R] int32
 *     and stats_host [4] f64 (the schedule's {n, B, tau, Theta}): per-round
 *     outputs, each nullable.
 *   tgt_scheduled_only  nonzero: tgt_host holds every candidate row of every
 *     request, padded [R, gamma + 1, V], and only the rows the schedule
 *     admits -- rows 1 .. l_r + 1 of request r, B in all, the rows a target
 *     model computes for the round -- cross the link: after the schedule a
 *     kernel reads them through the device's mapping of tgt_host and writes
 *     them to verify->tgt in the packed layout of sched->row_off, with no
 *     host synchronisation.  Then verify->tgt_row_off must be sched->row_off,
 *     verify->tgt must hold R * (gamma + 1) rows, tgt_rows is ignored, and
 *     tgt_host must be page-locked memory the device can address
 *     (cudaHostAlloc, cudaHostRegister): SPEC_ERR_UNSUPPORTED otherwise.
 *     Zero: tgt_host's tgt_rows rows are copied as they are, before the draft.
 * Returns the first stage's error, or SPEC_ERR_CUDA when a copy fails to
 * enqueue.
 */
typedef struct spec_round_host_args {
  const spec_draft_args *draft;
  const spec_sched_args *sched;
  const spec_verify_args *verify;
  const void *U_host;
  const void *h_host;
  const int32_t *x0_host;
  const void *tgt_host;
  size_t tgt_rows;
  int32_t *out_tok_host;
  int32_t *accept_len_host;
  int32_t *n_out_host;
  double *stats_host;
  int tgt_scheduled_only;
} spec_round_host_args;

int spec_round_host(const spec_round_host_args *args, uint64_t seed, spec_stream_t stream);

/* ------------------------------------------------------------ stream ----
 * The library's random stream, as the kernels draw it (see "Randomness" above):
 * u_out[v] = uniform of vocabulary entry v at (position j, global request id
 * rid, purpose) for v < V, and e_out[v] (nullable) = -ln(u_out[v]) as the
 * sampling kernels compute it (an Exp(1) variate; Gumbel noise is -ln e).
 * Lets a caller reproduce or audit any draw.  V >= 1; outputs are device f32.
 */
int spec_stream_uniforms(uint64_t seed, uint32_t j, uint32_t rid, uint32_t purpose, int V,
                         float *u_out, float *e_out, spec_stream_t stream);

/* ------------------------------------------------------- wait self-test -
 * Exercises the bounded wait that every pipeline wait of the tensor-core
 * kernels uses (an mbarrier try-wait that gives up after a time limit): one
 * thread waits on a barrier that nothing will ever complete, gives up after
 * limit_ns nanoseconds (measured on the GPU's global timer), sets
 * SPEC_STATUS_TIMEOUT in *status (device word, required) and returns.  No
 * copy or tensor-memory operation is in flight, so the context stays usable.
 * 1 <= limit_ns <= 2e9 (SPEC_ERR_INVALID_ARG otherwise). */
int spec_wait_selftest(uint64_t limit_ns, uint32_t *status, spec_stream_t stream);

/* Workspace bytes a stage needs for these sizes (0 if the sizes are invalid).
 * `stage` is a spec_stage; r is ignored by SCHEDULE and VERIFY-greedy. */
size_t spec_workspace_bytes(int stage, int R, int gamma, int V, int r);

/* Static, NUL-terminated text for a status code. */
const char *spec_error_string(int code);

/* Library version, MAJOR * 10000 + MINOR * 100 + PATCH. */
int spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_H */
