"""Pins for the oracle's RNN sequential head (CPU only).

DSpark summary, "第二阶段：轻量顺序头": besides the Markov head the sequential head
may keep a recurrent state.  The pages give no formula; the library reads it as
s_0 = 0, s_k = store(tanh(A_k[x_{k-1}] + s_{k-1} W_k)), B_k = s_k C_k.  The
pins: a hand-computed two-position case; with W = 0 the head is the Markov
head over the table store(tanh(A)) (the Markov draft is pinned by its own
tests), token for token on the same stream; the stored bf16 states equal
torch's bf16 rounding of the fp32 values; and verification of RNN drafts
against a target stays lossless by chi-square (the residual recomputes q from
the stored state, so a wrong state row would make it lossy).
"""
import math

import numpy as np
import pytest
import torch
from scipy import stats
from scipy.special import softmax

import oracle


def test_hand_computed_two_positions():
    # r = 1, V = 2, gamma = 2; tokens fixed through x_cond, fp32 states
    U = np.array([[[0.5, -0.25], [0.0, 1.0]]], np.float32)      # [R=1, gamma=2, V=2]
    A = np.array([[[0.3], [-0.6]], [[0.9], [0.2]]], np.float32)  # [gamma, V, r=1]
    Ct = np.array([[[2.0], [-1.0]], [[0.5], [1.5]]], np.float32)
    W = np.array([[[0.75]], [[-1.25]]], np.float32)
    x0 = np.array([1], np.int32)
    xc = np.array([[0, 1]], np.int32)
    out = oracle.draft_rnn(U, A, Ct, W, x0, np.ones(2, np.float32), seed=3, bf16_state=False,
                           x_cond=xc)
    s1 = float(np.float32(math.tanh(-0.6)))                     # A_1[x0 = 1], s_0 = 0
    s2 = float(np.float32(math.tanh(0.9 + s1 * -1.25)))          # A_2[x_1 = 0] + s_1 W_2
    assert out.S[0, 0, 0] == s1 and out.S[0, 1, 0] == s2
    z1 = np.array([0.5 + s1 * 2.0, -0.25 + s1 * -1.0])
    z2 = np.array([0.0 + s2 * 0.5, 1.0 + s2 * 1.5])
    lse = [math.log(np.exp(z1).sum()), math.log(np.exp(z2).sum())]
    assert out.lse[0] == pytest.approx(lse, rel=1e-12)
    q = [math.exp(z1[out.x[0, 0]] - lse[0]), math.exp(z2[out.x[0, 1]] - lse[1])]
    assert out.q_tok[0] == pytest.approx(q, rel=1e-12)


@pytest.mark.parametrize("bf16_state", [False, True])
def test_zero_recurrence_is_the_markov_head(bf16_state):
    rng = np.random.default_rng(4)
    R, gamma, V, r = 5, 4, 40, 6
    U = rng.normal(0, 2, (R, gamma, V)).astype(np.float32)
    A = rng.normal(0, 1, (gamma, V, r)).astype(np.float32)
    Ct = rng.normal(0, 0.5, (gamma, V, r)).astype(np.float32)
    W = np.zeros((gamma, r, r), np.float32)
    x0 = rng.integers(0, V, R).astype(np.int32)
    temps = np.ones(gamma, np.float32)
    rnn = oracle.draft_rnn(U, A, Ct, W, x0, temps, seed=9, bf16_state=bf16_state, want_P=True)
    tA = torch.tanh(torch.tensor(A, dtype=torch.float64)).float()
    table = (tA.to(torch.bfloat16).float() if bf16_state else tA).numpy()
    mk = oracle.draft(U, table, Ct, x0, temps, seed=9, want_P=True)
    assert np.array_equal(rnn.x, mk.x)
    assert np.allclose(rnn.q_tok, mk.q_tok, rtol=1e-12) and np.allclose(rnn.lse, mk.lse, rtol=1e-12)
    assert np.allclose(rnn.P, mk.P, rtol=1e-12, atol=0)


def test_bf16_states_match_torch_rounding():
    rng = np.random.default_rng(5)
    R, gamma, V, r = 3, 3, 20, 8
    U = rng.normal(0, 1, (R, gamma, V)).astype(np.float32)
    A = rng.normal(0, 1, (gamma, V, r)).astype(np.float32)
    Ct = rng.normal(0, 0.5, (gamma, V, r)).astype(np.float32)
    W = rng.normal(0, 0.4, (gamma, r, r)).astype(np.float32)
    x0 = rng.integers(0, V, R).astype(np.int32)
    out = oracle.draft_rnn(U, A, Ct, W, x0, np.ones(gamma, np.float32), seed=1, bf16_state=True)
    # recompute the recurrence with the oracle's own states and tokens, rounding with torch
    for req in range(R):
        prev = np.zeros(r)
        xp = x0[req]
        for k in range(gamma):
            pre = A[k, xp].astype(np.float64) + prev @ W[k].astype(np.float64)
            want = torch.tensor(np.tanh(pre), dtype=torch.float64).float().to(torch.bfloat16)
            assert np.array_equal(out.S[req, k], want.double().numpy())
            prev = out.S[req, k]
            xp = out.x[req, k]


def test_rnn_drafts_verify_losslessly():
    """Rejection sampling of RNN drafts (gamma = 1 after a fixed first state)
    emits the target distribution; the residual recomputes q from the state."""
    rng = np.random.default_rng(6)
    V, r, n = 8, 3, 200_000
    U1 = rng.normal(0, 1, (1, 1, V)).astype(np.float32)
    A = rng.normal(0, 1, (1, V, r)).astype(np.float32)
    Ct = rng.normal(0, 1, (1, V, r)).astype(np.float32)
    W = rng.normal(0, 0.5, (1, r, r)).astype(np.float32)
    x0 = np.full(n, 3, np.int32)
    U = np.broadcast_to(U1, (n, 1, V))
    d = oracle.draft_rnn(U, A, Ct, W, x0, np.ones(1, np.float32), seed=21, bf16_state=True)
    t1 = rng.normal(0, 1.2, V).astype(np.float32)
    tgt = np.zeros((n, 2, V), np.float32)
    tgt[:, 0] = t1
    row_off = (np.arange(n) * 2).astype(np.int32)
    v = oracle.verify(oracle.MODE_SAMPLE, tgt.reshape(-1, V), row_off, np.ones(n, np.int32), d.x,
                      d.q_tok, 1.0, U, A, Ct, x0, np.ones(1, np.float32), seed=21, S=d.S)
    p = softmax(t1.astype(np.float64))
    first = np.bincount(v.out_tok[:, 0], minlength=V)
    assert stats.chisquare(first, p * n).pvalue > 1e-3
    # c* of the first row against its measured acceptance
    cs = oracle.cstar(tgt[:1].reshape(-1, V), np.array([0], np.int32), np.ones(1, np.int32),
                      d.x[:1], 1.0, U[:1], A, Ct, x0[:1], np.ones(1, np.float32), S=d.S[:1])[0, 0]
    acc = (v.accept_len == 1).mean()
    assert abs(acc - cs) < 5 * math.sqrt(cs * (1 - cs) / n)
    # the wrong state (zeros) for the residual makes the round lossy
    vz = oracle.verify(oracle.MODE_SAMPLE, tgt.reshape(-1, V), row_off, np.ones(n, np.int32), d.x,
                       d.q_tok, 1.0, U, A, Ct, x0, np.ones(1, np.float32), seed=21,
                       S=np.zeros_like(d.S))
    bad = np.bincount(vz.out_tok[:, 0], minlength=V)
    assert stats.chisquare(bad, p * n).pvalue < 1e-6
