/*
 * One speculative round through the C ABI alone (no Python): draft, schedule
 * and verify for R = 4 requests, gamma = 3 draft positions and V = 1000
 * tokens, on inputs drawn from a fixed 64-bit LCG.  Prints the admitted
 * lengths, the accept lengths and the emitted tokens.
 *
 * Build (next to an in-tree libspec.so):
 *   gcc -std=c99 -O2 -I include -I /usr/local/cuda/include examples/round.c \
 *       -L verify_sampling_gb300 -Wl,-rpath,$PWD/verify_sampling_gb300 -lspec \
 *       -L /usr/local/cuda/lib64 -lcudart -o round
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "spec.h"

enum { R = 4, G = 3, V = 1000, RANK = 8, D = 16, E = 8, NSPS = R * (G + 1) + 1 };

static uint64_t lcg_state = 0x2545F4914F6CDD1Dull;

/* uniform in [-1, 1) from the top 53 bits of a 64-bit LCG (Knuth's MMIX constants) */
static float lcg(void) {
  lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
  return (float)((double)(lcg_state >> 11) * (1.0 / 9007199254740992.0) * 2.0 - 1.0);
}

static void fill(float *x, size_t n, float scale) {
  for (size_t i = 0; i < n; ++i) x[i] = scale * lcg();
}

#define CHECK_CUDA(call)                                                         \
  do {                                                                           \
    cudaError_t e_ = (call);                                                     \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      return 1;                                                                  \
    }                                                                            \
  } while (0)
#define CHECK_SPEC(call)                                                         \
  do {                                                                           \
    int s_ = (call);                                                             \
    if (s_ != SPEC_OK) {                                                         \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, spec_error_string(s_));  \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

/* device copy of n bytes of host data */
static void *to_device(const void *h, size_t n) {
  void *d = NULL;
  if (cudaMalloc(&d, n) != cudaSuccess) return NULL;
  if (h && cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(void) {
  /* ---- inputs (host) ---- */
  static float U[R * G * V], A[G * V * RANK], Ct[G * V * RANK], h[R * G * D], W1[V * E], w[D + E];
  static float tgt[R * (G + 1) * V], sps[NSPS];
  float draft_temp[G], sts_temp[G];
  int32_t x0[R], row_off[R];
  fill(U, sizeof U / sizeof *U, 2.0f);
  fill(A, sizeof A / sizeof *A, 0.3f);
  fill(Ct, sizeof Ct / sizeof *Ct, 0.5f);
  fill(h, sizeof h / sizeof *h, 1.0f);
  fill(W1, sizeof W1 / sizeof *W1, 1.0f);
  fill(w, sizeof w / sizeof *w, 0.2f);
  for (int r = 0; r < R; ++r)
    for (int j = 0; j <= G; ++j)
      for (int v = 0; v < V; ++v)  /* target row j + 1 of request r: near the draft logits */
        tgt[(r * (G + 1) + j) * V + v] = U[(r * G + (j < G ? j : G - 1)) * V + v] + 0.5f * lcg();
  for (int i = 0; i < NSPS; ++i) sps[i] = 1000.0f - 10.0f * (float)i; /* SPS(B) at B = 1 + i */
  for (int k = 0; k < G; ++k) draft_temp[k] = sts_temp[k] = 1.0f;
  for (int r = 0; r < R; ++r) {
    x0[r] = (r * 37) % V;
    row_off[r] = r * (G + 1); /* padded target layout */
  }
  const uint64_t seed = 20261202ull;

  /* ---- device buffers ---- */
  float *dU = to_device(U, sizeof U), *dA = to_device(A, sizeof A), *dCt = to_device(Ct, sizeof Ct);
  float *dh = to_device(h, sizeof h), *dW1 = to_device(W1, sizeof W1), *dw = to_device(w, sizeof w);
  float *dtgt = to_device(tgt, sizeof tgt), *dsps = to_device(sps, sizeof sps);
  float *dT = to_device(draft_temp, sizeof draft_temp), *dST = to_device(sts_temp, sizeof sts_temp);
  int32_t *dx0 = to_device(x0, sizeof x0), *drow = to_device(row_off, sizeof row_off);
  int32_t *dx = to_device(NULL, sizeof(int32_t) * R * G);
  float *dq = to_device(NULL, sizeof(float) * R * G), *dl = to_device(NULL, sizeof(float) * R * G);
  float *dc = to_device(NULL, sizeof(float) * R * G), *da = to_device(NULL, sizeof(float) * R * G);
  int32_t *dell = to_device(NULL, sizeof(int32_t) * R), *dro = to_device(NULL, sizeof(int32_t) * (R + 1));
  double *dstats = to_device(NULL, 4 * sizeof(double));
  int32_t *dacc = to_device(NULL, sizeof(int32_t) * R), *dnout = to_device(NULL, sizeof(int32_t) * R);
  int32_t *dout = to_device(NULL, sizeof(int32_t) * R * (G + 1));
  uint32_t *dstatus = to_device(NULL, sizeof(uint32_t));
  size_t ws_d = spec_workspace_bytes(SPEC_STAGE_DRAFT, R, G, V, RANK);
  size_t ws_v = spec_workspace_bytes(SPEC_STAGE_VERIFY, R, G, V, RANK);
  void *dws_d = to_device(NULL, ws_d), *dws_v = to_device(NULL, ws_v);
  if (!dU || !dA || !dCt || !dh || !dW1 || !dw || !dtgt || !dsps || !dT || !dST || !dx0 || !drow ||
      !dx || !dq || !dl || !dc || !da || !dell || !dro || !dstats || !dacc || !dnout || !dout ||
      !dstatus || !dws_d || !dws_v) {
    fprintf(stderr, "device allocation or copy failed\n");
    return 1;
  }
  CHECK_CUDA(cudaMemset(dstatus, 0, sizeof(uint32_t)));

  /* ---- draft ---- */
  spec_draft_args d;
  memset(&d, 0, sizeof d); /* zeroed: the Markov head, no optional outputs */
  d.R = R, d.gamma = G, d.V = V, d.r = RANK, d.d = D, d.e = E;
  d.logit_dtype = d.fac_dtype = d.conf_dtype = SPEC_F32;
  d.U = dU, d.A = dA, d.Ct = dCt, d.x0 = dx0, d.draft_temp = dT;
  d.h = dh, d.W1 = dW1, d.w = dw, d.sts_temp = dST;
  d.x = dx, d.q_tok = dq, d.lse_q = dl, d.c = dc, d.a = da;
  d.workspace = dws_d, d.workspace_bytes = ws_d, d.status = dstatus;
  CHECK_SPEC(spec_draft_sample(&d, seed, NULL));

  /* ---- schedule ---- */
  spec_sched_args s;
  memset(&s, 0, sizeof s);
  s.R = R, s.gamma = G, s.a = da, s.sps = dsps, s.n_sps = NSPS, s.b_lo = 1.0, s.b_step = 1.0;
  s.K = R * G, s.mode = SPEC_SCHED_EARLY_STOP;
  s.ell = dell, s.row_off = dro, s.stats = dstats, s.status = dstatus;
  CHECK_SPEC(spec_schedule(&s, NULL));

  /* ---- verify ---- */
  spec_verify_args v;
  memset(&v, 0, sizeof v);
  v.mode = SPEC_VERIFY_SAMPLE, v.R = R, v.gamma = G, v.V = V, v.tgt_dtype = SPEC_F32;
  v.tgt = dtgt, v.tgt_row_off = drow, v.ell = dell, v.x = dx, v.q_tok = dq, v.lse_q = dl;
  v.target_temp = 1.0f, v.draft = &d;
  v.accept_len = dacc, v.out_tok = dout, v.n_out = dnout;
  v.workspace = dws_v, v.workspace_bytes = ws_v, v.status = dstatus;
  CHECK_SPEC(spec_verify(&v, seed, NULL));

  /* ---- results ---- */
  int32_t ell[R], acc[R], out[R * (G + 1)];
  uint32_t status = 0;
  double stats[4];
  CHECK_CUDA(cudaMemcpy(ell, dell, sizeof ell, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(acc, dacc, sizeof acc, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(stats, dstats, sizeof stats, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&status, dstatus, sizeof status, cudaMemcpyDeviceToHost));
  printf("status %u\n", status);
  printf("stats n=%d B=%d\n", (int)stats[0], (int)stats[1]);
  for (int r = 0; r < R; ++r) {
    printf("request %d ell %d accept %d tokens", r, ell[r], acc[r]);
    for (int j = 0; j <= acc[r]; ++j) printf(" %d", out[r * (G + 1) + j]);
    printf("\n");
  }
  return status == 0 ? 0 : 2;
}
