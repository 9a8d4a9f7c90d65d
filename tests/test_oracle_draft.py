"""Pins for the oracle's draft head and confidence head (CPU only).

The Markov bias is pinned by the full-table special case the history article
describes under "杀招一": with rank r = V and A_k = I the low-rank product
B_k(x) = A_k[x] C_k is just row x of a V x V transition table, so the draft
distribution must be softmax(U_k + T_k[x_{k-1}]) exactly (a table gather and a
library softmax).
"""
import numpy as np
import pytest
from scipy.special import expit, logsumexp, softmax

import oracle


def _table_case(R=3, gamma=4, V=9, seed=0, temps=None):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2, size=(R, gamma, V)).astype(np.float32)
    T = rng.normal(0, 1, size=(gamma, V, V)).astype(np.float32)    # T_k[x_prev, v]
    A = np.broadcast_to(np.eye(V, dtype=np.float32), (gamma, V, V)).copy()
    Ct = np.ascontiguousarray(np.transpose(T, (0, 2, 1)))           # Ct_k[v, i] = T_k[i, v]
    x0 = rng.integers(0, V, size=R).astype(np.int32)
    temps = np.ones(gamma, np.float32) if temps is None else np.asarray(temps, np.float32)
    return U, T, A, Ct, x0, temps


@pytest.mark.parametrize("temps", [None, [1.0, 2.0, 0.5, 1.5]])
def test_full_table_special_case(temps):
    U, T, A, Ct, x0, tt = _table_case(temps=temps)
    out = oracle.draft(U, A, Ct, x0, tt, seed=5, want_P=True)
    R, gamma, V = U.shape
    for r in range(R):
        prev = x0[r]
        for k in range(gamma):
            z = (U[r, k].astype(np.float64) + T[k, prev].astype(np.float64)) / float(tt[k])
            p = softmax(z)
            assert np.allclose(out.P[r, k], p, rtol=1e-12, atol=1e-15)
            assert abs(out.lse[r, k] - logsumexp(z)) < 1e-12
            assert abs(out.q_tok[r, k] - p[out.x[r, k]]) < 1e-14
            prev = out.x[r, k]


def test_sequential_dependency_on_previous_token():
    """Step k conditions on x_{k-1}: forcing a different x_{k-1} through x_cond
    changes the distribution of step k to the table row of the forced token."""
    U, T, A, Ct, x0, tt = _table_case(R=1, gamma=2, V=7, seed=3)
    forced = np.array([[4, 0]], np.int32)
    out = oracle.draft(U, A, Ct, x0, tt, seed=1, x_cond=forced, want_P=True)
    z = U[0, 1].astype(np.float64) + T[1, 4].astype(np.float64)
    assert np.allclose(out.P[0, 1], softmax(z), rtol=1e-12)


def test_rank_one_bias_is_outer_product():
    """A_k[x] = alpha_x (r = 1): bias_v = alpha_{x_prev} * Ct[v]; a scaled vector."""
    V, gamma = 6, 1
    alpha = np.arange(V, dtype=np.float32) - 2.0
    cvec = np.linspace(-1, 1, V).astype(np.float32)
    A = alpha.reshape(1, V, 1)
    Ct = cvec.reshape(1, V, 1)
    U = np.zeros((1, gamma, V), np.float32)
    out = oracle.draft(U, A, Ct, np.array([5], np.int32), [1.0], seed=0, want_P=True)
    assert np.allclose(out.P[0, 0], softmax(3.0 * cvec.astype(np.float64)), rtol=1e-12)


def test_draft_is_deterministic_and_keyed_by_request_id():
    U, T, A, Ct, x0, tt = _table_case(R=4, gamma=3, V=11, seed=9)
    a = oracle.draft(U, A, Ct, x0, tt, seed=3, rid_base=10)
    b = oracle.draft(U, A, Ct, x0, tt, seed=3, rid_base=10)
    assert (a.x == b.x).all()
    # request 2 of a batch with base 10 == request 0 of a batch with base 12
    c = oracle.draft(U[2:], A, Ct, x0[2:], tt, seed=3, rid_base=12)
    assert (c.x == a.x[2:]).all()


def test_confidence_closed_forms():
    R, gamma, d, e, V = 2, 4, 5, 3, 10
    x0 = np.array([1, 7], np.int32)
    x = np.array([[2, 3, 4, 5], [9, 8, 6, 0]], np.int32)
    # zero inputs: s = 0, c = 1/2 whatever the temperature, a = 2^-k
    c, a = oracle.confidence(np.zeros((R, gamma, d)), np.zeros((V, e)), np.zeros(d + e), x0, x,
                             [1, 2, 3, 4])
    assert np.all(c == 0.5) and np.allclose(a, 0.5 ** np.arange(1, gamma + 1))
    # w = e_0 reads h[..., 0]; STS divides by tau_k
    rng = np.random.default_rng(1)
    h = rng.normal(size=(R, gamma, d))
    w = np.zeros(d + e)
    w[0] = 1.0
    tau = np.array([1.0, 2.0, 1.5, 1.2])
    c, a = oracle.confidence(h, np.zeros((V, e)), w, x0, x, tau)
    h32 = h.astype(np.float32).astype(np.float64)
    assert np.allclose(c, expit(h32[:, :, 0] / tau), rtol=1e-13)
    assert np.allclose(a, np.cumprod(c, axis=1), rtol=1e-13)
    # w = e_{d+1} reads W1[x_{k-1}, 1]: x0 for k = 1, then the previous draft token
    W1 = rng.normal(size=(V, e))
    w = np.zeros(d + e)
    w[d + 1] = 1.0
    c, _ = oracle.confidence(np.zeros((R, gamma, d)), W1, w, x0, x, np.ones(gamma))
    prev = np.concatenate([x0[:, None], x[:, :-1]], axis=1)
    W132 = W1.astype(np.float32).astype(np.float64)
    assert np.allclose(c, expit(W132[prev, 1]), rtol=1e-13)


def test_survival_non_increasing():
    """Survival check: a_{r,j} = prod_{i<=j} c_{r,i} is non-increasing along j."""
    rng = np.random.default_rng(2)
    R, gamma, d, e, V = 8, 16, 32, 8, 50
    h = rng.normal(size=(R, gamma, d))
    W1 = rng.normal(size=(V, e))
    w = rng.normal(size=d + e)
    x0 = rng.integers(0, V, R)
    x = rng.integers(0, V, (R, gamma))
    _, a = oracle.confidence(h, W1, w, x0, x, 1 + np.arange(gamma) / 15)
    assert np.all(np.diff(a, axis=1) <= 0) and np.all(a > 0) and np.all(a <= 1)
