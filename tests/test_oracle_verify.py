"""Pins for the oracle's verifier (CPU only).

* the lossless property of the history article's
  "数学上的美感": over 10^6 seeded rounds on a tiny vocabulary the emitted first
  token (gamma = 1) and the first two tokens (gamma = 2, completed by a second
  round when the first round emits one token) follow the target p, by
  chi-square; the acceptance frequency at j = 1 equals sum_v min(p_v, q_v), the
  closed form the DSpark summary ("2.1") gives as 1 - TV;
* the lossy reading (regenerate from p instead of the residual) must fail the
  same chi-square -- the test has the power to see the difference;
* greedy: accept length = longest prefix with
  x_j == argmax L_j (numpy argmax, lowest index on ties), brute force;
* DSpark Figure 1 as a scripted round (golden fixture).
"""
import json
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import expit, logit, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
N_TRIALS = 1_000_000


def _markov_draft_inputs(rng, V, gamma):
    """Full-table Markov draft: A_k = I, Ct_k = D_k^T, so q_k(.|x) = softmax(U_k + D_k[x])."""
    U = rng.normal(0, 1.0, size=(gamma, V)).astype(np.float32)
    D = rng.normal(0, 1.0, size=(gamma, V, V)).astype(np.float32)
    A = np.broadcast_to(np.eye(V, dtype=np.float32), (gamma, V, V)).copy()
    Ct = np.ascontiguousarray(np.transpose(D, (0, 2, 1)))
    return U, D, A, Ct


def _round(U_row, A, Ct, x0, tgt_fn, ell, seed, rid_base, mode=oracle.MODE_SAMPLE):
    R = x0.size
    gamma = U_row.shape[0]
    V = U_row.shape[1]
    U = np.broadcast_to(U_row, (R, gamma, V))
    d = oracle.draft(U, A, Ct, x0, np.ones(gamma), seed=seed, rid_base=rid_base)
    tgt = tgt_fn(d.x)                                  # [R, gamma + 1, V]
    row_off = (np.arange(R) * (gamma + 1)).astype(np.int32)
    v = oracle.verify(mode, tgt.reshape(-1, V), row_off, np.full(R, ell, np.int32), d.x, d.q_tok,
                      1.0, U, A, Ct, x0, np.ones(gamma), seed=seed, rid_base=rid_base)
    return d, v


def _chisq_p(counts, probs):
    probs = probs / probs.sum()
    return stats.chisquare(counts, probs * counts.sum()).pvalue


def test_lossless_first_token_gamma1():
    rng = np.random.default_rng(11)
    V = 12
    U, D, A, Ct = _markov_draft_inputs(rng, V, 1)
    t1 = rng.normal(0, 1.2, size=V).astype(np.float32)
    x0 = np.full(N_TRIALS, 2, np.int32)

    def tgt_fn(x):
        tgt = np.zeros((x.shape[0], 2, V), np.float32)
        tgt[:, 0] = t1
        return tgt

    d, v = _round(U, A, Ct, x0, tgt_fn, 1, seed=2024, rid_base=0)
    p = softmax(t1.astype(np.float64))
    q = softmax(U[0].astype(np.float64) + D[0, 2].astype(np.float64))
    first = v.out_tok[:, 0]
    assert _chisq_p(np.bincount(first, minlength=V), p) > 1e-3
    # acceptance frequency at j = 1 versus the closed form sum_v min(p_v, q_v)
    acc = (v.accept_len == 1).mean()
    cstar = np.minimum(p, q).sum()
    sigma = np.sqrt(cstar * (1 - cstar) / N_TRIALS)
    assert abs(acc - cstar) < 5 * sigma
    # the draft itself follows q
    assert _chisq_p(np.bincount(d.x[:, 0], minlength=V), q) > 1e-3
    # planted mistake, applied to a copy of the oracle's output on the CPU: the
    # lossy reading regenerates a rejected position from p instead of max(0,p-q)
    lossy = first.copy()
    rej = v.accept_len == 0
    lossy[rej] = np.random.default_rng(5).choice(V, size=rej.sum(), p=p)
    assert _chisq_p(np.bincount(lossy, minlength=V), p) < 1e-6


def test_lossless_first_two_tokens_gamma2():
    rng = np.random.default_rng(12)
    V = 6
    U, D, A, Ct = _markov_draft_inputs(rng, V, 2)
    t1 = rng.normal(0, 1.0, size=V).astype(np.float32)
    T2 = rng.normal(0, 1.0, size=(V, V)).astype(np.float32)    # target row 2 given token 1
    x0 = np.zeros(N_TRIALS, np.int32)

    def tgt_fn(x):
        tgt = np.zeros((x.shape[0], 3, V), np.float32)
        tgt[:, 0] = t1
        tgt[:, 1] = T2[x[:, 0]]
        return tgt

    d, v = _round(U, A, Ct, x0, tgt_fn, 2, seed=77, rid_base=0)
    first = v.out_tok[:, 0].copy()
    second = v.out_tok[:, 1].copy()
    need = v.n_out == 1
    # complete the pair with a second round (gamma = 1) that drafts from the
    # position-2 Markov head given the emitted token and verifies against T2[y]
    y = first[need]
    U2, A2, Ct2 = U[1:2], A[1:2], Ct[1:2]

    def tgt2_fn(x):
        tgt = np.zeros((x.shape[0], 2, V), np.float32)
        tgt[:, 0] = T2[y]
        return tgt

    _, v2 = _round(U2, A2, Ct2, y.astype(np.int32), tgt2_fn, 1, seed=78, rid_base=N_TRIALS)
    second[need] = v2.out_tok[:, 0]
    P = softmax(t1.astype(np.float64))[:, None] * softmax(T2.astype(np.float64), axis=1)
    counts = np.bincount(first * V + second, minlength=V * V)
    assert _chisq_p(counts, P.reshape(-1)) > 1e-3


def test_bonus_with_no_admitted_draft_is_plain_decoding():
    """l_r = 0: the round emits one token sampled from target row 1."""
    rng = np.random.default_rng(13)
    V = 10
    U, D, A, Ct = _markov_draft_inputs(rng, V, 3)
    t1 = rng.normal(0, 1.5, size=V).astype(np.float32)
    R = 200_000
    x0 = np.zeros(R, np.int32)

    def tgt_fn(x):
        tgt = np.zeros((x.shape[0], 4, V), np.float32)
        tgt[:, 0] = t1
        return tgt

    _, v = _round(U, A, Ct, x0, tgt_fn, 0, seed=9, rid_base=0)
    assert (v.n_out == 1).all() and (v.accept_len == 0).all() and (v.jstar == 0).all()
    assert _chisq_p(np.bincount(v.out_tok[:, 0], minlength=V), softmax(t1.astype(np.float64))) > 1e-3


def test_target_temperature():
    """p = softmax(L / T_t): at T_t = 2 the first token follows softmax(L/2)."""
    rng = np.random.default_rng(14)
    V = 8
    U, D, A, Ct = _markov_draft_inputs(rng, V, 1)
    t1 = rng.normal(0, 2.0, size=V).astype(np.float32)
    R = 300_000
    d = oracle.draft(np.broadcast_to(U, (R, 1, V)), A, Ct, np.zeros(R, np.int32), [1.0], seed=4)
    tgt = np.zeros((R, 2, V), np.float32)
    tgt[:, 0] = t1
    v = oracle.verify(oracle.MODE_SAMPLE, tgt.reshape(-1, V), np.arange(R, dtype=np.int32) * 2,
                      np.ones(R, np.int32), d.x, d.q_tok, 2.0, np.broadcast_to(U, (R, 1, V)), A, Ct,
                      np.zeros(R, np.int32), [1.0], seed=4)
    p = softmax(t1.astype(np.float64) / 2.0)
    assert _chisq_p(np.bincount(v.out_tok[:, 0], minlength=V), p) > 1e-3


def test_greedy_brute_force():
    """Greedy accept length: the longest prefix with x_j == argmax L_j."""
    rng = np.random.default_rng(15)
    R, gamma, V = 300, 6, 40
    # bf16-like coarse values so that exact ties occur
    tgt = np.round(rng.normal(0, 3, size=(R, gamma + 1, V)) * 2) / 2
    tgt = tgt.astype(np.float32)
    am = tgt.argmax(axis=2)                           # numpy: lowest index among maxima
    x = np.where(rng.uniform(size=(R, gamma)) < 0.7, am[:, :gamma],
                 rng.integers(0, V, (R, gamma))).astype(np.int32)
    ell = rng.integers(0, gamma + 1, R).astype(np.int32)
    row_off = (np.arange(R) * (gamma + 1)).astype(np.int32)
    v = oracle.verify(oracle.MODE_GREEDY, tgt.reshape(-1, V), row_off, ell, x,
                      np.ones((R, gamma)), 1.0, None, None, None, np.zeros(R, np.int32),
                      np.ones(gamma), seed=0)
    for r in range(R):
        n = 0
        while n < ell[r] and x[r, n] == am[r, n]:
            n += 1
        assert v.accept_len[r] == n
        assert list(v.out_tok[r, :n]) == list(x[r, :n])
        assert v.out_tok[r, n] == am[r, n]
        assert (v.out_tok[r, n + 1:] == -1).all() and v.n_out[r] == n + 1
    assert (tgt == tgt.max(axis=2, keepdims=True)).sum(axis=2).max() > 1  # ties were present


def test_figure1_round():
    with open(os.path.join(GOLDEN, "fig1_round.json")) as f:
        g = json.load(f)
    V, gamma, anchor = g["V"], g["gamma"], g["anchor"]
    draft_tok = np.array(g["draft"])
    U = np.zeros((1, gamma, V), np.float32)
    U[0, np.arange(gamma), draft_tok] = 50.0
    A = np.zeros((gamma, V, 1), np.float32)
    d = oracle.draft(U, A, A, np.array([anchor]), np.ones(gamma), seed=123)
    assert list(d.x[0]) == g["draft"]
    # confidences through w = e_0, h_{k,0} = logit(c_k)
    c_target = np.array(g["confidence"])
    h = np.zeros((1, gamma, 4))
    h[0, :, 0] = logit(c_target)
    w = np.zeros(4 + 2)
    w[0] = 1.0
    c, a = oracle.confidence(h, np.zeros((V, 2)), w, np.array([anchor]), d.x, np.ones(gamma))
    assert np.allclose(c[0], expit(h[0, :, 0].astype(np.float32).astype(np.float64)))
    s = oracle.schedule(a, g["sps"], g["b_lo"], g["b_step"], gamma, oracle.SCHED_EARLY_STOP)
    exp = g["expected"]
    assert s.ell[0] == exp["ell"] and s.B == exp["B"]
    tgt = np.zeros((1, gamma + 1, V), np.float32)
    tgt[0, 0, 4] = 50.0
    tgt[0, 1, 5] = 50.0
    tgt[0, 2, 6] = -50.0
    for seed in range(20):
        v = oracle.verify(oracle.MODE_SAMPLE, tgt.reshape(-1, V), np.array([0]), s.ell, d.x,
                          d.q_tok, 1.0, U, A, A, np.array([anchor]), np.ones(gamma), seed=seed)
        assert v.accept_len[0] == exp["accept_len"] and v.n_out[0] == exp["n_out"]
        assert list(v.out_tok[0, :2]) == exp["emitted_prefix"]
        assert v.out_tok[0, 2] != exp["rejected_token"] and v.jstar[0] == 3


def test_accept_prob_closed_form_matches_frequency():
    """orc_accept_prob is 1 - TV(p, q); pinned by the acceptance frequency of the
    oracle's own verifier over independent rounds and by the TV identity."""
    rng = np.random.default_rng(21)
    V = 9
    U, D, A, Ct = _markov_draft_inputs(rng, V, 1)
    t1 = rng.normal(0, 1.0, size=V).astype(np.float32)
    zq = U[0].astype(np.float64) + D[0, 0].astype(np.float64)
    cstar = oracle.accept_prob(t1.astype(np.float64), zq)
    p, q = softmax(t1.astype(np.float64)), softmax(zq)
    assert abs(cstar - (1 - 0.5 * np.abs(p - q).sum())) < 1e-14
    R = 400_000
    x0 = np.zeros(R, np.int32)

    def tgt_fn(x):
        tgt = np.zeros((x.shape[0], 2, V), np.float32)
        tgt[:, 0] = t1
        return tgt

    _, v = _round(U, A, Ct, x0, tgt_fn, 1, seed=31, rid_base=0)
    freq = (v.accept_len == 1).mean()
    assert abs(freq - cstar) < 5 * np.sqrt(cstar * (1 - cstar) / R)
