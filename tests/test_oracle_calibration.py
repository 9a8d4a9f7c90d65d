"""Pins for the oracle's calibration diagnostics (CPU only).

DSpark summary, "2.1 置信度头": the confidence head's target is the acceptance
probability c* = 1 - TV(p, q) = sum_v min(p_v, q_v); Figure 6 judges the
confidences by a reliability diagram and the expected calibration error (ECE)
against realised acceptance.  The pins: closed forms of c* (equal rows, two
tokens), the verifier's measured acceptance frequency at j = 1 against c*, a
hand-computed diagram, calibrated and over-confident synthetic streams against
their expected ECE, bin edges, and accumulation over calls.
"""
import numpy as np
import pytest

import oracle


def _round(rng, R, gamma, V, r, spread=1.0):
    U = rng.normal(0, spread, (R, gamma, V)).astype(np.float32)
    A = rng.normal(0, 0.3, (gamma, V, r)).astype(np.float32)
    Ct = rng.normal(0, 0.3, (gamma, V, r)).astype(np.float32)
    x0 = rng.integers(0, V, R).astype(np.int32)
    x = rng.integers(0, V, (R, gamma)).astype(np.int32)
    temps = np.ones(gamma, np.float32)
    return U, A, Ct, x0, x, temps


def test_cstar_is_one_for_equal_rows_and_nan_past_ell():
    rng = np.random.default_rng(1)
    R, gamma, V, r = 3, 3, 7, 2
    U, A, Ct, x0, x, temps = _round(rng, R, gamma, V, r)
    A[:] = 0.0  # no bias: q = softmax(U)
    ell = np.array([3, 1, 0], np.int32)
    row_off = np.arange(R, dtype=np.int32) * (gamma + 1)
    tgt = np.zeros((R * (gamma + 1), V), np.float32)
    for req in range(R):
        tgt[row_off[req]:row_off[req] + gamma] = U[req]
    cs = oracle.cstar(tgt, row_off, ell, x, 1.0, U, A, Ct, x0, temps)
    assert cs[0] == pytest.approx(1.0, abs=1e-14) and cs[1, 0] == pytest.approx(1.0, abs=1e-14)
    assert np.isnan(cs[1, 1:]).all() and np.isnan(cs[2]).all()


def test_cstar_two_tokens_closed_form():
    """V = 2: c* = 1 - |p_0 - q_0| with p_0 = sigmoid(L0 - L1), q_0 = sigmoid(z0 - z1)."""
    rng = np.random.default_rng(2)
    for _ in range(20):
        U, A, Ct, x0, x, temps = _round(rng, 1, 1, 2, 1)
        L = rng.normal(0, 2, (2, 2)).astype(np.float32)
        cs = oracle.cstar(L, np.array([0], np.int32), np.array([1], np.int32), x, 1.0, U, A, Ct,
                          x0, temps)
        bias = A[0, x0[0], 0] * Ct[0, :, 0].astype(np.float64)
        z = U[0, 0].astype(np.float64) + bias
        sig = lambda t: 1.0 / (1.0 + np.exp(-t))
        want = 1.0 - abs(sig(float(L[0, 0]) - float(L[0, 1])) - sig(z[0] - z[1]))
        assert cs[0, 0] == pytest.approx(want, abs=1e-12)


def test_cstar_matches_measured_acceptance_at_position_one():
    """The verifier accepts the first draft token with probability c* (history
    article, "1.1运行机制"): over 6000 independent requests with the same rows,
    the accepted fraction at j = 1 agrees with c* within 4 sigma."""
    rng = np.random.default_rng(3)
    V, r, n = 6, 2, 6000
    U1, A, Ct, x01, _, temps = _round(rng, 1, 1, V, r, spread=1.5)
    tgt1 = rng.normal(0, 1.5, (1, V)).astype(np.float32)
    cs = oracle.cstar(tgt1, np.array([0], np.int32), np.array([1], np.int32),
                      np.zeros((1, 1), np.int32), 1.0, U1, A, Ct, x01, temps)[0, 0]
    U = np.repeat(U1, n, axis=0)
    x0 = np.repeat(x01, n)
    d = oracle.draft(U, A, Ct, x0, temps, seed=11)
    tgt = np.repeat(np.concatenate([tgt1, tgt1]), n, axis=0).reshape(n * 2, V)
    row_off = (np.arange(n) * 2).astype(np.int32)
    ell = np.ones(n, np.int32)
    out = oracle.verify(oracle.MODE_SAMPLE, tgt, row_off, ell, d.x, d.q_tok, 1.0, U, A, Ct, x0,
                        temps, seed=12)
    freq = float((out.accept_len == 1).mean())
    sd = np.sqrt(cs * (1 - cs) / n)
    assert abs(freq - cs) < 4 * sd + 1e-9, (freq, cs)


def _tables(n_bins):
    return np.zeros(n_bins, np.int64), np.zeros(n_bins), np.zeros(n_bins, np.int64)


def test_hand_computed_diagram():
    c = np.array([[0.95, 0.55, 0.05], [0.35, 0.2, 0.1]])
    cnt, sc, sa = _tables(10)
    ece, bad = oracle.calibration(c, [3, 2], [1, 2], cnt, sc, sa)
    assert bad == 0
    assert list(np.flatnonzero(cnt)) == [2, 3, 5, 9] and cnt.sum() == 4
    assert list(sa[[2, 3, 5, 9]]) == [1, 1, 0, 1]
    assert ece == pytest.approx((0.05 + 0.55 + 0.65 + 0.8) / 4, rel=1e-14)


def test_bin_edges():
    c = np.array([[0.0, 0.25, 0.5, 1.0]])
    cnt, sc, sa = _tables(4)
    oracle.calibration(c, [4], [4], cnt, sc, sa)
    assert list(cnt) == [1, 1, 1, 1]  # 0 -> 0, 0.25 -> 1, 0.5 -> 2, 1.0 -> last


def _stream(rng, R, gamma, truth):
    """Requests with confidences c and positions accepted with probability
    truth(c) once the ones before were; every request admits all gamma."""
    c = rng.uniform(0.05, 1.0, (R, gamma))
    ok = rng.random((R, gamma)) < truth(c)
    first_fail = np.where(ok.all(axis=1), gamma, np.argmin(ok, axis=1))
    return c, np.full(R, gamma, np.int32), first_fail.astype(np.int32)


def test_calibrated_stream_has_small_ece():
    rng = np.random.default_rng(5)
    cnt, sc, sa = _tables(10)
    for _ in range(20):
        c, ell, acc = _stream(rng, 2000, 6, lambda c: c)
        ece, _ = oracle.calibration(c, ell, acc, cnt, sc, sa)
    assert ece < 0.01


def test_overconfident_stream_matches_expected_ece():
    """True acceptance c^2: ECE -> sum_b |sum c^2 - sum c| / N over the tested
    positions, i.e. the same diagram built from the expectations."""
    rng = np.random.default_rng(6)
    cnt, sc, sa = _tables(10)
    sq = np.zeros(10)
    for _ in range(20):
        c, ell, acc = _stream(rng, 2000, 6, lambda c: c * c)
        ece, _ = oracle.calibration(c, ell, acc, cnt, sc, sa)
        for req in range(c.shape[0]):
            for j in range(min(ell[req], acc[req] + 1)):
                b = min(int(c[req, j] * 10), 9)
                sq[b] += c[req, j] ** 2
    want = np.abs(sq - sc).sum() / cnt.sum()
    assert ece == pytest.approx(want, abs=0.01)
    assert ece > 0.1


def test_accumulation_equals_one_call_and_bad_entries():
    rng = np.random.default_rng(7)
    c1, l1, a1 = _stream(rng, 50, 4, lambda c: c)
    c2, l2, a2 = _stream(rng, 70, 4, lambda c: c)
    t1 = _tables(8)
    oracle.calibration(c1, l1, a1, *t1)
    e_two, _ = oracle.calibration(c2, l2, a2, *t1)
    t2 = _tables(8)
    e_one, _ = oracle.calibration(np.concatenate([c1, c2]), np.concatenate([l1, l2]),
                                  np.concatenate([a1, a2]), *t2)
    assert np.array_equal(t1[0], t2[0]) and np.array_equal(t1[2], t2[2])
    assert np.allclose(t1[1], t2[1], rtol=1e-14) and e_two == pytest.approx(e_one, rel=1e-13)
    cnt, sc, sa = _tables(4)
    c = np.array([[0.5, np.nan], [0.5, 0.5], [1.5, 0.5]])
    ece, bad = oracle.calibration(c, [2, 3, 1], [2, 0, 0], cnt, sc, sa)
    assert bad == 3 and cnt.sum() == 1  # NaN, l > gamma, c > 1
    empty = _tables(4)
    ece0, _ = oracle.calibration(np.zeros((0, 2)), [], [], *empty)
    assert np.isnan(ece0)
