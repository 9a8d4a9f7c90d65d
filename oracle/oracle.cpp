// Oracle for the speculative-decoding round math: plain, slow, single-threaded
// C++17 in fp64.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
// benchmark's CPU-baseline leg call it; the product path never does.  It shares
// no code with the CUDA library (no headers, helpers, tables or generators).
//
// Sources (the three web pages this build follows):
//   [DSpark]  "DSpark: Confidence-Scheduled Speculative Decoding with
//             Semi-Autoregressive Generation" (summary, adg.csdn.net)
//   [History] speculative-decoding history article (wzjinhao.cn/news/15713)
//   [Philox]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
//             1, 2, 3", SC'11 -- the Philox-4x32 bijection with 10 rounds.
//
// Every floating-point step below runs in double precision on inputs that were
// converted exactly from fp32/bf16.  Nothing is blocked, fused or reordered:
// each function follows the definition it cites, step by step.
//
// Parity status: Philox, softmax, Gumbel-max sampling, the scheduler and the
// verifier are pinned by the tests under tests/ (curand host generator,
// closed forms, chi-square, brute force, hand-built fixtures).  The RNN head
// follows a reading of its own (the pages give no formula); it is pinned by a
// hand-computed case, its reduction to the Markov head and losslessness.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// ---------------------------------------------------------------- Philox ----
// [Philox] Philox-4x32: per round, two 32x32->64 products of words 0 and 2 with
// the multipliers M0, M1; the new words are (hi1 ^ w1 ^ k0, lo1, hi0 ^ w3 ^ k1,
// lo0).  Between rounds the key is bumped by the Weyl constants W0, W1.
const uint32_t kMulA = 0xD2511F53u;
const uint32_t kMulB = 0xCD9E8D57u;
const uint32_t kWeylA = 0x9E3779B9u;
const uint32_t kWeylB = 0xBB67AE85u;

void philox_block(const uint32_t counter[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t w[4] = {counter[0], counter[1], counter[2], counter[3]};
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kWeylA;
      k1 += kWeylB;
    }
    uint64_t prod0 = (uint64_t)kMulA * (uint64_t)w[0];
    uint64_t prod1 = (uint64_t)kMulB * (uint64_t)w[2];
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t next[4] = {hi1 ^ w[1] ^ k0, lo1, hi0 ^ w[3] ^ k1, lo0};
    w[0] = next[0];
    w[1] = next[1];
    w[2] = next[2];
    w[3] = next[3];
  }
  out[0] = w[0];
  out[1] = w[1];
  out[2] = w[2];
  out[3] = w[3];
}

// The random stream of this library: counter = (v / 4, position j, global
// request id, purpose), key = (seed low word, seed high word); vocabulary entry v
// takes word v % 4.  Word x maps to the open-interval uniform
// (2*(x & 0x7FFFFF)+1)*2^-24 (its low 23 bits),
// which is exact in fp32 and fp64 alike.
enum Purpose : uint32_t { kDraftGumbel = 0, kAcceptU = 1, kResidualGumbel = 2, kBonusGumbel = 3 };

double uniform_from_word(uint32_t x) { return (2.0 * (double)(x & 0x7fffffu) + 1.0) * 0x1p-24; }

struct Stream {
  uint32_t key[2];
  explicit Stream(uint64_t seed) {
    key[0] = (uint32_t)(seed & 0xffffffffu);
    key[1] = (uint32_t)(seed >> 32);
  }
  double uniform(uint32_t v, uint32_t j, uint32_t rid, uint32_t purpose) const {
    uint32_t counter[4] = {v / 4u, j, rid, purpose};
    uint32_t out[4];
    philox_block(counter, key, out);
    return uniform_from_word(out[v % 4u]);
  }
  // Standard Gumbel variate G = -ln(-ln u).
  double gumbel(uint32_t v, uint32_t j, uint32_t rid, uint32_t purpose) const {
    return -std::log(-std::log(uniform(v, j, rid, purpose)));
  }
};

const double kNegInf = -std::numeric_limits<double>::infinity();
const double kInf = std::numeric_limits<double>::infinity();

// log(sum_v exp(z_v)), written out with the usual max shift.
double log_sum_exp(const std::vector<double>& z) {
  double m = kNegInf;
  for (double zv : z) m = std::max(m, zv);
  double s = 0.0;
  for (double zv : z) s += std::exp(zv - m);
  return m + std::log(s);
}

// Gumbel-max: argmax_v (logw_v + G_v) over entries with logw_v > -inf.  Ties go
// to the lowest index.  *gap receives the top-1 minus top-2 score (inf if only
// one candidate).
int gumbel_argmax(const std::vector<double>& logw, const Stream& rng, uint32_t j, uint32_t rid,
                  uint32_t purpose, double* gap) {
  int best = -1;
  double s1 = kNegInf, s2 = kNegInf;
  for (size_t v = 0; v < logw.size(); ++v) {
    if (logw[v] == kNegInf) continue;
    double s = logw[v] + rng.gumbel((uint32_t)v, j, rid, purpose);
    if (s > s1) {
      s2 = s1;
      s1 = s;
      best = (int)v;
    } else if (s > s2) {
      s2 = s;
    }
  }
  if (gap) *gap = (s2 == kNegInf) ? kInf : s1 - s2;
  return best;
}

// [DSpark] "第二阶段：轻量顺序头" and [History] "杀招一": the Markov head draft
// logits at position k given the previous token x_prev:
//   z_v = (U_k[v] + B_k(x_prev)[v]) / T_k,   B_k(x)[v] = sum_i A_k[x, i] * C_k[i, v]
// with the low-rank factors stored A_k as [V, r] and C_k transposed as [V, r].
// The same with the bias taken from an explicit rank-r row: B_k[v] = row . C_k[:, v].
void draft_logits_row(int V, int r, const float* Uk, const double* row, const float* Ctk,
                      double temp, std::vector<double>& z) {
  z.assign((size_t)V, 0.0);
  for (int v = 0; v < V; ++v) {
    const float* crow = Ctk + (size_t)v * (size_t)r;
    double bias = 0.0;
    for (int i = 0; i < r; ++i) bias += row[i] * (double)crow[i];
    z[(size_t)v] = ((double)Uk[v] + bias) / temp;
  }
}

void draft_logits(int V, int r, const float* Uk, const float* Ak, const float* Ctk, int x_prev,
                  double temp, std::vector<double>& z) {
  const float* arow = Ak + (size_t)x_prev * (size_t)r;
  std::vector<double> row(arow, arow + r);
  draft_logits_row(V, r, Uk, row.data(), Ctk, temp, z);
}

// Draft logits of (req, j): the Markov row A_j[x_prev], or, when S is given
// (the RNN head), the stored state S[req, j-1, :].
void draft_logits_at(int V, int r, const float* Uk, const float* A, const float* Ct,
                     const float* S, int gamma, int req, int j, int x_prev, double temp,
                     std::vector<double>& z) {
  const float* Ctk = Ct + (size_t)(j - 1) * V * r;
  if (S) {
    const float* srow = S + ((size_t)req * gamma + (j - 1)) * r;
    std::vector<double> row(srow, srow + r);
    draft_logits_row(V, r, Uk, row.data(), Ctk, temp, z);
  } else {
    draft_logits(V, r, Uk, A + (size_t)(j - 1) * V * r, Ctk, x_prev, temp, z);
  }
}

// bf16 rounding (round to nearest, ties to even) of a value, as a double.
double round_bf16(double v) {
  const float f = (float)v;  // first to fp32, as a device stores its fp32 result
  uint32_t b;
  std::memcpy(&b, &f, 4);
  if ((b & 0x7f800000u) == 0x7f800000u) return (double)f;  // inf / nan
  const uint32_t lsb = (b >> 16) & 1u;
  b = (b + 0x7fffu + lsb) & 0xffff0000u;
  float o;
  std::memcpy(&o, &b, 4);
  return (double)o;
}

// SPS(B) from a table sampled at B_i = b_lo + i * b_step: linear interpolation
// between neighbours, clamped to the end values outside the grid.
double sps_lookup(const double* sps, int n_sps, double b_lo, double b_step, double B) {
  double t = (B - b_lo) / b_step;
  if (t <= 0.0) return sps[0];
  if (t >= (double)(n_sps - 1)) return sps[n_sps - 1];
  double fi = std::floor(t);
  int i = (int)fi;
  double f = t - fi;
  return (1.0 - f) * sps[i] + f * sps[i + 1];
}

}  // namespace

extern "C" {

// Raw Philox-4x32-10 block: out = Philox(counter, key).
void orc_philox4x32_10(const uint32_t* counter, const uint32_t* key, uint32_t* out) {
  philox_block(counter, key, out);
}

// Uniform in (0,1) for vocabulary entry v at (position j, request rid, purpose).
double orc_uniform(uint64_t seed, uint32_t v, uint32_t j, uint32_t rid, uint32_t purpose) {
  return Stream(seed).uniform(v, j, rid, purpose);
}

// Gumbel-max sample over V log-weights (entries equal to -inf are excluded).
int orc_gumbel_argmax(int V, const double* logw, uint64_t seed, uint32_t j, uint32_t rid,
                      uint32_t purpose, double* gap) {
  std::vector<double> lw(logw, logw + V);
  return gumbel_argmax(lw, Stream(seed), j, rid, purpose, gap);
}

// SPS table lookup (exported for tests).
double orc_sps_lookup(const double* sps, int n_sps, double b_lo, double b_step, double B) {
  return sps_lookup(sps, n_sps, b_lo, b_step, B);
}

// [DSpark] "2.1 置信度头": the acceptance probability of a token drawn from q
// and verified against p is c* = 1 - (1/2) ||p - q||_1 = sum_v min(p_v, q_v),
// with p = softmax(zt), q = softmax(zq).
double orc_accept_prob(int V, const double* zt, const double* zq) {
  std::vector<double> a(zt, zt + V), b(zq, zq + V);
  const double la = log_sum_exp(a), lb = log_sum_exp(b);
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += std::min(std::exp(a[(size_t)v] - la), std::exp(b[(size_t)v] - lb));
  return s;
}

// ------------------------------------------------------------------ draft ---
// [DSpark] "第二阶段：轻量顺序头"; [History] "杀招一".  For every request r and
// k = 1..gamma (sequential in k):
//   z = (U_{r,k} + A_k[x_{k-1}] C_k) / T_k,  P_k = softmax(z),
//   x_k = argmax_v (z_v + G_v)  with G from the stream (purpose 0, j = k),
//   q_tok = P_k[x_k],  lse = log sum exp z.
// U row of (r, k) starts at U + r*U_rstride + (k-1)*V.  x_cond (nullable,
// [R, gamma]) replaces the sampled x_k as the conditioning token of step k+1,
// which lets a test feed the same previous-stage tokens to both sides.
// P (nullable, [R, gamma, V]) receives the full draft distributions.
int orc_draft(int R, int gamma, int V, int r, const float* U, int64_t U_rstride, const float* A,
              const float* Ct, const int32_t* x0, const float* draft_temp, uint64_t seed,
              uint32_t rid_base, const int32_t* x_cond, int32_t* x, double* q_tok, double* lse,
              double* gap, double* P) {
  if (R < 0 || gamma <= 0 || V <= 0 || r <= 0) return -1;
  Stream rng(seed);
  std::vector<double> z;
  for (int req = 0; req < R; ++req) {
    uint32_t rid = rid_base + (uint32_t)req;
    int x_prev = x0[req];
    for (int k = 1; k <= gamma; ++k) {
      if (x_prev < 0 || x_prev >= V) return -2;
      const size_t kk = (size_t)(k - 1);
      const float* Uk = U + (size_t)req * (size_t)U_rstride + kk * (size_t)V;
      draft_logits(V, r, Uk, A + kk * (size_t)V * r, Ct + kk * (size_t)V * r, x_prev,
                   (double)draft_temp[kk], z);
      double l = log_sum_exp(z);
      double g;
      int xk = gumbel_argmax(z, rng, (uint32_t)k, rid, kDraftGumbel, &g);
      size_t o = (size_t)req * gamma + kk;
      x[o] = xk;
      q_tok[o] = std::exp(z[(size_t)xk] - l);
      lse[o] = l;
      if (gap) gap[o] = g;
      if (P) {
        double* Prow = P + o * (size_t)V;
        for (int v = 0; v < V; ++v) Prow[v] = std::exp(z[(size_t)v] - l);
      }
      x_prev = x_cond ? x_cond[o] : xk;
    }
  }
  return 0;
}

// ------------------------------------------------------------ RNN head ---
// [DSpark] "第二阶段：轻量顺序头": the sequential head comes in two forms, the
// Markov head (only the previous token, low-rank) and an RNN head that keeps a
// recurrent state for longer dependencies.  The pages give no formula for the
// latter; this library's reading is an Elman state in the same rank-r space:
//   s_0 = 0,  s_k = store(tanh(A_k[x_{k-1}] + s_{k-1} W_k)),  B_k = s_k C_k,
// with W_k [r, r] per position (row i maps s_{k-1}[i] to column j) and
// store() the state's storage precision (bf16 when `bf16_state`, else fp32).
// Everything else is the Markov draft: z = (U_k + B_k) / T_k, Gumbel-max with
// the purpose-0 stream.  S_out [R, gamma, r] receives the stored states.
// x_cond (nullable) replaces the sampled tokens as in orc_draft; s_cond
// (nullable, [R, gamma, r]) replaces the state carried to the next position
// and used for the bias, which lets a test feed the device's states.
int orc_draft_rnn(int R, int gamma, int V, int r, const float* U, int64_t U_rstride,
                  const float* A, const float* Ct, const float* W, const int32_t* x0,
                  const float* draft_temp, uint64_t seed, uint32_t rid_base, int bf16_state,
                  const int32_t* x_cond, const float* s_cond, int32_t* x, double* q_tok,
                  double* lse, double* gap, double* S_out, double* P) {
  if (R < 0 || gamma <= 0 || V <= 0 || r <= 0) return -1;
  Stream rng(seed);
  std::vector<double> z, st((size_t)r), prev((size_t)r);
  for (int req = 0; req < R; ++req) {
    const uint32_t rid = rid_base + (uint32_t)req;
    int x_prev = x0[req];
    std::fill(prev.begin(), prev.end(), 0.0);
    for (int k = 1; k <= gamma; ++k) {
      if (x_prev < 0 || x_prev >= V) return -2;
      const size_t kk = (size_t)(k - 1);
      const float* arow = A + kk * (size_t)V * r + (size_t)x_prev * r;
      const float* Wk = W + kk * (size_t)r * r;
      for (int j = 0; j < r; ++j) {
        double pre = (double)arow[j];
        for (int i = 0; i < r; ++i) pre += prev[(size_t)i] * (double)Wk[(size_t)i * r + j];
        const double t = std::tanh(pre);
        st[(size_t)j] = bf16_state ? round_bf16(t) : (double)(float)t;
      }
      const size_t o = (size_t)req * gamma + kk;
      for (int j = 0; j < r; ++j) S_out[o * r + j] = st[(size_t)j];
      const double* use = st.data();
      std::vector<double> cond;
      if (s_cond) {
        cond.assign(s_cond + o * r, s_cond + o * r + r);
        use = cond.data();
      }
      draft_logits_row(V, r, U + (size_t)req * U_rstride + kk * V, use, Ct + kk * (size_t)V * r,
                       (double)draft_temp[kk], z);
      const double l = log_sum_exp(z);
      double g;
      const int xk = gumbel_argmax(z, rng, (uint32_t)k, rid, kDraftGumbel, &g);
      x[o] = xk;
      q_tok[o] = std::exp(z[(size_t)xk] - l);
      lse[o] = l;
      if (gap) gap[o] = g;
      if (P)
        for (int v = 0; v < V; ++v) P[o * (size_t)V + (size_t)v] = std::exp(z[(size_t)v] - l);
      for (int j = 0; j < r; ++j) prev[(size_t)j] = use[j];
      x_prev = x_cond ? x_cond[o] : xk;
    }
  }
  return 0;
}


// ------------------------------------------------------------- confidence ---
// [DSpark] "2.1 置信度头": c_k = sigmoid(w . [h_k ; W1[x_{k-1}]]), with the
// sequential temperature of "后验温度缩放" applied as c_k = sigmoid(s_k / tau_k);
// [History] "杀招二": survival a_j = prod_{i<=j} c_i.
// h row of (r, k) starts at h + r*h_rstride + (k-1)*d.  The conditioning tokens
// are x0[r] for k = 1 and x[r, k-2] for k > 1.
int orc_confidence(int R, int gamma, int d, int e, int V, const float* h, int64_t h_rstride,
                   const float* W1, const float* w, const int32_t* x0, const int32_t* x,
                   const float* sts_temp, double* c, double* a) {
  if (R < 0 || gamma <= 0 || d < 0 || e < 0) return -1;
  for (int req = 0; req < R; ++req) {
    double surv = 1.0;
    for (int k = 1; k <= gamma; ++k) {
      int x_prev = (k == 1) ? x0[req] : x[(size_t)req * gamma + (k - 2)];
      if (x_prev < 0 || x_prev >= V) return -2;
      const float* hk = h + (size_t)req * (size_t)h_rstride + (size_t)(k - 1) * d;
      const float* emb = W1 + (size_t)x_prev * e;
      double s = 0.0;
      for (int i = 0; i < d; ++i) s += (double)w[i] * (double)hk[i];
      for (int i = 0; i < e; ++i) s += (double)w[d + i] * (double)emb[i];
      double ck = 1.0 / (1.0 + std::exp(-s / (double)sts_temp[k - 1]));
      surv *= ck;
      size_t o = (size_t)req * gamma + (k - 1);
      c[o] = ck;
      a[o] = surv;
    }
  }
  return 0;
}

// -------------------------------------------------------------- schedule ---
// [DSpark] "2.2 硬件感知前缀调度器": maximise Theta = tau * SPS(B) with
// B = sum_r (1 + l_r) and tau = sum_r sum_{j<=l_r} a_{r,j}; solved by sorting
// all candidates by survival (descending) and admitting them one by one while
// Theta rises ([History] "杀招三": keep a candidate only if the new throughput
// beats the best so far, stop at the first drop).  [DSpark] "挑战2" adds the
// top-K cap on the number admitted and the global search without early stop.
//   mode 0 = early stop, mode 1 = global argmax over all sorted prefixes.
//   mode 2 = static confidence threshold ([DSpark] comparison table: SpecDec++
//            schedules by a fixed confidence threshold; Figure 5 sweeps it):
//            every candidate whose survival a_{r,j} (the predicted probability
//            that the prefix up to j is accepted) is >= threshold, i.e. the
//            sorted prefix of those, still capped by K.  Theta is reported but
//            not used; the decisions are exact comparisons (margin +inf).
// Ties in the sort keep (request, position) order.  stats = {n, B, tau, Theta}.
// margin = smallest relative Theta difference among the comparisons made.
// order (nullable, [R*gamma]) receives the sorted candidate ids r*gamma + j-1;
// theta (nullable, [min(K,R*gamma)+1]) receives Theta_0..Theta_nmax.
int orc_schedule(int R, int gamma, const double* a, const double* sps, int n_sps, double b_lo,
                 double b_step, int K, int mode, double threshold, int32_t* ell,
                 int32_t* row_off, double* stats, double* margin, int32_t* order, double* theta) {
  if (R < 0 || gamma <= 0 || n_sps <= 0 || b_step <= 0.0 || K < 0 || mode < 0 || mode > 2)
    return -1;
  if (mode == 2 && std::isnan(threshold)) return -1;
  const int N = R * gamma;
  std::vector<int> ids((size_t)N);
  for (int i = 0; i < N; ++i) ids[(size_t)i] = i;
  std::stable_sort(ids.begin(), ids.end(), [&](int p, int q) { return a[p] > a[q]; });
  const int nmax = std::min(K, N);

  std::vector<double> tau((size_t)nmax + 1), th((size_t)nmax + 1);
  tau[0] = 0.0;
  th[0] = 0.0;
  for (int n = 1; n <= nmax; ++n) {
    tau[(size_t)n] = tau[(size_t)n - 1] + a[ids[(size_t)n - 1]];
    th[(size_t)n] = tau[(size_t)n] * sps_lookup(sps, n_sps, b_lo, b_step, (double)(R + n));
  }

  int nstar = 0;
  double mg = kInf;
  if (mode == 0) {
    while (nstar < nmax) {
      double cur = th[(size_t)nstar], nxt = th[(size_t)nstar + 1];
      double scale = std::max(std::fabs(cur), std::fabs(nxt));
      if (scale > 0.0) mg = std::min(mg, std::fabs(nxt - cur) / scale);
      if (nxt > cur)
        ++nstar;
      else
        break;
    }
  } else if (mode == 2) {
    while (nstar < nmax && a[ids[(size_t)nstar]] >= threshold) ++nstar;
  } else {
    for (int n = 1; n <= nmax; ++n)
      if (th[(size_t)n] > th[(size_t)nstar]) nstar = n;
    double best = th[(size_t)nstar];
    for (int n = 0; n <= nmax; ++n) {
      if (n == nstar || best <= 0.0) continue;
      mg = std::min(mg, (best - th[(size_t)n]) / best);
    }
  }

  for (int req = 0; req < R; ++req) ell[req] = 0;
  for (int n = 0; n < nstar; ++n) ell[ids[(size_t)n] / gamma] += 1;
  row_off[0] = 0;
  for (int req = 0; req < R; ++req) row_off[req + 1] = row_off[req] + 1 + ell[req];
  stats[0] = (double)nstar;
  stats[1] = (double)(R + nstar);
  stats[2] = tau[(size_t)nstar];
  stats[3] = th[(size_t)nstar];
  if (margin) *margin = mg;
  if (order)
    for (int i = 0; i < N; ++i) order[i] = ids[(size_t)i];
  if (theta)
    for (int n = 0; n <= nmax; ++n) theta[n] = th[(size_t)n];
  return 0;
}

// ---------------------------------------------------------------- verify ---
// [History] "1.1运行机制 / 拒绝采样": accept draft x_j if p(x_j) >= q(x_j), else
// accept with probability p/q; after the first rejection the rest of the draft
// is discarded.  [DSpark] Figure 1: the rejected position is regenerated by the
// target -- here from norm(max(0, p - q)), the residual that makes the round
// lossless ([History] "数学上的美感").  If every admitted position is accepted,
// one more token is sampled from the next target row (the "1 +" in B of [DSpark]
// "2.2").  Greedy mode accepts while x_j equals the target argmax (lowest index
// on ties) and emits the target argmax at the first mismatch or after the prefix.
//
// Target row of (r, j) is tgt + (row_off[r] + j - 1) * V, j = 1..l_r + 1, with
// p = softmax(L / target_temp).  The accept test at (r, j) is u < p(x_j)/q_tok
// with u from the stream (purpose 1, word 0 of block 0).  The residual needs the
// draft row at j*: z_q = (U_{r,j*} + A_{j*}[x_{j*-1}] C_{j*}) / T_{j*} and
// q = softmax(z_q).  Outputs: accept_len, out_tok[R, gamma+1] (-1 padded),
// n_out, margin (smallest decision margin: |u - p/q| of every accept test made
// and the Gumbel top-2 gap of the emitted sample; +inf in greedy mode, whose
// decisions are exact comparisons), jstar (first rejected position, 0 if none).
// margin_acc and margin_gap (nullable) split margin by kind: the smallest
// |u - p/q| of the accept tests, and the Gumbel gap of the emitted residual or
// bonus sample (+inf where the request made no such decision).
int orc_verify(int mode, int R, int gamma, int V, const float* tgt, const int32_t* row_off,
               const int32_t* ell, const int32_t* x, const double* q_tok, double target_temp,
               const float* U, int64_t U_rstride, const float* A, const float* Ct, int r,
               const int32_t* x0, const float* draft_temp, uint64_t seed, uint32_t rid_base,
               int32_t* accept_len, int32_t* out_tok, int32_t* n_out, double* margin,
               int32_t* jstar_out, const float* S, double* margin_acc, double* margin_gap) {
  if ((mode != 0 && mode != 1) || R < 0 || gamma <= 0 || V <= 0) return -1;
  Stream rng(seed);
  std::vector<double> zt, p, zq;
  for (int req = 0; req < R; ++req) {
    const uint32_t rid = rid_base + (uint32_t)req;
    const int l = ell[req];
    if (l < 0 || l > gamma) return -2;
    const int32_t* xr = x + (size_t)req * gamma;
    int32_t* out = out_tok + (size_t)req * (gamma + 1);
    for (int i = 0; i <= gamma; ++i) out[i] = -1;
    double mg = kInf, mg_acc = kInf, mg_gap = kInf;
    int jstar = 0;
    int y = -1;

    auto target_row = [&](int j) { return tgt + ((size_t)row_off[req] + (size_t)(j - 1)) * V; };

    if (mode == 1) {
      auto argmax_row = [&](int j) {
        const float* L = target_row(j);
        int best = 0;
        for (int v = 1; v < V; ++v)
          if ((double)L[v] > (double)L[best]) best = v;
        return best;
      };
      for (int j = 1; j <= l; ++j) {
        int t = argmax_row(j);
        if (xr[j - 1] != t) {
          jstar = j;
          y = t;
          break;
        }
      }
      if (jstar == 0) y = argmax_row(l + 1);
    } else {
      auto target_probs = [&](int j) {
        const float* L = target_row(j);
        zt.assign((size_t)V, 0.0);
        for (int v = 0; v < V; ++v) zt[(size_t)v] = (double)L[v] / target_temp;
        double l_t = log_sum_exp(zt);
        p.assign((size_t)V, 0.0);
        for (int v = 0; v < V; ++v) p[(size_t)v] = std::exp(zt[(size_t)v] - l_t);
      };
      for (int j = 1; j <= l; ++j) {
        target_probs(j);
        const int xj = xr[j - 1];
        if (xj < 0 || xj >= V) return -3;
        const double q = q_tok[(size_t)req * gamma + (j - 1)];
        const double u = rng.uniform(0u, (uint32_t)j, rid, kAcceptU);
        bool accept;
        if (q <= 0.0) {
          accept = true;
        } else {
          double ratio = p[(size_t)xj] / q;
          mg_acc = std::min(mg_acc, std::fabs(u - ratio));
          mg = std::min(mg, mg_acc);
          accept = u < ratio;
        }
        if (!accept) {
          jstar = j;
          break;
        }
      }
      double g;
      if (jstar > 0) {
        // Residual at j*: p is still the target distribution of row j*.
        const int kk = jstar - 1;
        const int x_prev = (jstar == 1) ? x0[req] : xr[jstar - 2];
        if (x_prev < 0 || x_prev >= V) return -3;
        draft_logits_at(V, r, U + (size_t)req * (size_t)U_rstride + (size_t)kk * V, A, Ct, S,
                        gamma, req, jstar, x_prev, (double)draft_temp[kk], zq);
        double l_q = log_sum_exp(zq);
        std::vector<double> logres((size_t)V, kNegInf);
        bool any = false;
        for (int v = 0; v < V; ++v) {
          double res = p[(size_t)v] - std::exp(zq[(size_t)v] - l_q);
          if (res > 0.0) {
            logres[(size_t)v] = std::log(res);
            any = true;
          }
        }
        if (!any) logres = zt;  // degenerate residual: sample from p itself
        y = gumbel_argmax(logres, rng, (uint32_t)jstar, rid, kResidualGumbel, &g);
      } else {
        target_probs(l + 1);
        y = gumbel_argmax(zt, rng, (uint32_t)(l + 1), rid, kBonusGumbel, &g);
      }
      mg_gap = g;
      mg = std::min(mg, g);
    }

    const int acc = (jstar > 0) ? jstar - 1 : l;
    for (int i = 0; i < acc; ++i) out[i] = xr[i];
    out[acc] = y;
    accept_len[req] = acc;
    n_out[req] = acc + 1;
    if (margin) margin[req] = mg;
    if (margin_acc) margin_acc[req] = mg_acc;
    if (margin_gap) margin_gap[req] = mg_gap;
    if (jstar_out) jstar_out[req] = jstar;
  }
  return 0;
}

// ------------------------------------------------- acceptance statistics ---
// LightSpec article, "无需额外训练，基于运行时统计的动态调度": acceptance rates
// are kept per batch-size class and per MTP length as exponential moving
// averages updated every round; a length with too few samples is estimated by
// interpolating the rates of the neighbouring lengths.
//
// One round's update of class `bucket` (rows of ema / count are classes, columns
// are the lengths L = 1..gamma):
//   n_L = number of requests with l_r = L, S_L = sum of their accept_len,
//   m_L = S_L / (L * n_L)  (the fraction of the L drafted tokens accepted);
//   for every L with n_L > 0: ema = m_L if no sample was seen before, else
//   ema = ema + beta * (m_L - ema) (as one fused multiply-add); count += n_L.
// Requests with l_r = 0 carry no draft and are skipped; an l_r outside
// [0, gamma] or an accept_len outside [0, l_r] is skipped and counted in *bad.
// estimate (nullable, [gamma]): for the updated class, the entry itself where
// count >= max(min_count, 1); otherwise linear interpolation in L between the
// nearest usable lengths below and above, the nearest one where only one side
// has a usable length, NaN where none has.
int orc_accept_stats(int R, int gamma, const int32_t* ell, const int32_t* accept_len, int bucket,
                     int n_buckets, double beta, int min_count, double* ema, int64_t* count,
                     double* estimate, int* bad) {
  if (R < 0 || gamma < 1 || n_buckets < 1 || bucket < 0 || bucket >= n_buckets ||
      !(beta > 0.0 && beta <= 1.0))
    return -1;
  std::vector<int64_t> n((size_t)gamma + 1, 0), S((size_t)gamma + 1, 0);
  int nbad = 0;
  for (int req = 0; req < R; ++req) {
    const int l = ell[req], acc = accept_len[req];
    if (l < 0 || l > gamma || acc < 0 || acc > l) {
      ++nbad;
      continue;
    }
    if (l == 0) continue;
    n[(size_t)l] += 1;
    S[(size_t)l] += acc;
  }
  double* e = ema + (size_t)bucket * gamma;
  int64_t* c = count + (size_t)bucket * gamma;
  for (int L = 1; L <= gamma; ++L) {
    if (n[(size_t)L] == 0) continue;
    const double m = (double)S[(size_t)L] / ((double)L * (double)n[(size_t)L]);
    if (c[L - 1] == 0)
      e[L - 1] = m;
    else
      e[L - 1] = std::fma(beta, m - e[L - 1], e[L - 1]);
    c[L - 1] += n[(size_t)L];
  }
  if (estimate) {
    const int64_t need = std::max(min_count, 1);
    for (int L = 1; L <= gamma; ++L) {
      if (c[L - 1] >= need) {
        estimate[L - 1] = e[L - 1];
        continue;
      }
      int lo = 0, hi = 0;
      for (int q = L - 1; q >= 1 && !lo; --q)
        if (c[q - 1] >= need) lo = q;
      for (int q = L + 1; q <= gamma && !hi; ++q)
        if (c[q - 1] >= need) hi = q;
      if (lo && hi) {
        const double w = (double)(L - lo) / (double)(hi - lo);
        estimate[L - 1] = std::fma(w, e[hi - 1] - e[lo - 1], e[lo - 1]);
      } else if (lo) {
        estimate[L - 1] = e[lo - 1];
      } else if (hi) {
        estimate[L - 1] = e[hi - 1];
      } else {
        estimate[L - 1] = std::numeric_limits<double>::quiet_NaN();
      }
    }
  }
  if (bad) *bad = nbad;
  return 0;
}

// ------------------------------------------------- calibration diagnostics ---
// [DSpark] "2.1 置信度头": the supervision target of the confidence head is the
// acceptance probability of the draft distribution against the target one,
// c* = 1 - (1/2) ||p - q||_1 = sum_v min(p_v, q_v).  For every verified draft
// row (r, j), j = 1..l_r: p = softmax(L / target_temp) of target row
// row_off[r] + j - 1 and q = softmax(z) of the draft logits of (r, j) given
// x_{j-1} (x_0 for j = 1).  c_star [R, gamma] receives it; positions past l_r
// get NaN (no target row exists for them).
int orc_cstar(int R, int gamma, int V, const float* tgt, const int32_t* row_off,
              const int32_t* ell, const int32_t* x, double target_temp, const float* U,
              int64_t U_rstride, const float* A, const float* Ct, int r, const int32_t* x0,
              const float* draft_temp, double* c_star, const float* S) {
  if (R < 0 || gamma <= 0 || V <= 0 || r <= 0 || !(target_temp > 0.0)) return -1;
  std::vector<double> zt((size_t)V), zq;
  for (int req = 0; req < R; ++req) {
    const int l = ell[req];
    if (l < 0 || l > gamma) return -2;
    for (int j = 1; j <= gamma; ++j) {
      double& out = c_star[(size_t)req * gamma + (j - 1)];
      if (j > l) {
        out = std::numeric_limits<double>::quiet_NaN();
        continue;
      }
      const float* row = tgt + (size_t)(row_off[req] + j - 1) * V;
      for (int v = 0; v < V; ++v) zt[(size_t)v] = (double)row[v] / target_temp;
      const int xp = (j == 1) ? x0[req] : x[(size_t)req * gamma + (j - 2)];
      draft_logits_at(V, r, U + (size_t)req * U_rstride + (size_t)(j - 1) * V, A, Ct, S, gamma,
                      req, j, xp, (double)draft_temp[j - 1], zq);
      out = orc_accept_prob(V, zt.data(), zq.data());
    }
  }
  return 0;
}

// [DSpark] Figure 6 and "2.1 置信度头" (sequential temperature scaling): the
// confidences are judged on a reliability diagram and by the expected
// calibration error against realised acceptance.  A round's tested positions
// are j = 1..min(l_r, accept_len_r + 1) of every request (the positions the
// verifier actually ruled on); position j counts as accepted iff
// j <= accept_len_r.  Each goes to bin b = min(floor(c_{r,j} * n_bins),
// n_bins - 1) of the equal-width diagram over [0, 1]: count_b += 1,
// sum_c_b += c, sum_acc_b += accepted.  The tables accumulate over calls.
// ECE = (1 / N) sum_b |sum_acc_b - sum_c_b| with N = sum_b count_b (NaN if 0),
// which is sum_b (n_b / N) |acc_b - conf_b| written without the divisions.
// Requests with l_r or accept_len_r out of range, and confidences outside
// [0, 1] or NaN, are skipped and counted in *bad.
int orc_calibration(int R, int gamma, const double* c, const int32_t* ell,
                    const int32_t* accept_len, int n_bins, int64_t* count, double* sum_c,
                    int64_t* sum_acc, double* ece, int* bad) {
  if (R < 0 || gamma <= 0 || n_bins <= 0) return -1;
  int nbad = 0;
  for (int req = 0; req < R; ++req) {
    const int l = ell[req], acc = accept_len[req];
    if (l < 0 || l > gamma || acc < 0 || acc > l) {
      ++nbad;
      continue;
    }
    const int tested = std::min(l, acc + 1);
    for (int j = 1; j <= tested; ++j) {
      const double cj = c[(size_t)req * gamma + (j - 1)];
      if (!(cj >= 0.0 && cj <= 1.0)) {
        ++nbad;
        continue;
      }
      const int b = std::min((int)std::floor(cj * (double)n_bins), n_bins - 1);
      count[b] += 1;
      sum_c[b] += cj;
      sum_acc[b] += (j <= acc) ? 1 : 0;
    }
  }
  if (ece) {
    int64_t N = 0;
    double dev = 0.0;
    for (int b = 0; b < n_bins; ++b) {
      N += count[b];
      dev += std::fabs((double)sum_acc[b] - sum_c[b]);
    }
    *ece = (N > 0) ? dev / (double)N : std::numeric_limits<double>::quiet_NaN();
  }
  if (bad) *bad = nbad;
  return 0;
}

}  // extern "C"


