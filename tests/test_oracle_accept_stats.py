"""Pins for the oracle's acceptance statistics (CPU only).

LightSpec article, "无需额外训练，基于运行时统计的动态调度": acceptance rates are
kept per batch-size class and per MTP length as exponential moving averages,
and lengths with too few samples are estimated by interpolating across
lengths.  The pins: a hand-computed round; the closed form of an EMA over a
sequence; fixed points; interpolation against straight lines; the verifier's
realised acceptance of i.i.d. positions against its closed form.
"""
import numpy as np
import pytest

import oracle


def _tables(n_buckets, gamma):
    return np.zeros((n_buckets, gamma)), np.zeros((n_buckets, gamma), np.int64)


def test_hand_computed_round():
    ema, cnt = _tables(2, 3)
    # l = 2, 2, 3, 0, 1 with 2, 1, 0, 0, 1 accepted
    est, bad = oracle.accept_stats([2, 2, 3, 0, 1], [2, 1, 0, 0, 1], ema, cnt, 1, 0.25)
    assert bad == 0
    assert list(ema[1]) == [1.0, 0.75, 0.0] and list(cnt[1]) == [1, 2, 1]
    assert not ema[0].any() and not cnt[0].any()  # other classes untouched
    assert list(est) == [1.0, 0.75, 0.0]


def test_ema_closed_form_over_a_sequence():
    """ema_n = (1-b)^(n-1) m_1 + sum_{i>=2} b (1-b)^(n-i) m_i for one length."""
    rng = np.random.default_rng(3)
    beta = 0.1
    ema, cnt = _tables(1, 4)
    ms = []
    for _ in range(40):
        acc = int(rng.integers(0, 5))
        oracle.accept_stats([4], [acc], ema, cnt, 0, beta)
        ms.append(acc / 4)
    n = len(ms)
    want = (1 - beta) ** (n - 1) * ms[0] + sum(beta * (1 - beta) ** (n - i) * ms[i - 1]
                                               for i in range(2, n + 1))
    assert ema[0, 3] == pytest.approx(want, rel=1e-12)
    assert cnt[0, 3] == n and cnt[0, :3].sum() == 0


def test_fixed_point_and_beta_one():
    ema, cnt = _tables(1, 2)
    for _ in range(25):
        oracle.accept_stats([2, 2], [1, 2], ema, cnt, 0, 0.3)
    assert ema[0, 1] == 0.75  # constant input stays exactly put
    oracle.accept_stats([2], [0], ema, cnt, 0, 1.0)
    assert ema[0, 1] == 0.0   # beta = 1 keeps only the newest round


def test_interpolation_across_lengths():
    ema, cnt = _tables(1, 6)
    oracle.accept_stats([1, 4], [1, 2], ema, cnt, 0, 0.5)   # rates 1.0 at L=1, 0.5 at L=4
    est, _ = oracle.accept_stats([], [], ema, cnt, 0, 0.5)
    assert est[0] == 1.0 and est[3] == 0.5
    assert est[1] == pytest.approx(1.0 - 0.5 / 3, rel=1e-15)
    assert est[2] == pytest.approx(1.0 - 1.0 / 3, rel=1e-15)
    assert est[4] == 0.5 and est[5] == 0.5                  # beyond the last: nearest
    # min_count: an entry with fewer samples is interpolated over as well
    est2, _ = oracle.accept_stats([], [], ema, cnt, 0, 0.5, min_count=2)
    assert np.isnan(est2).all()
    oracle.accept_stats([4], [2], ema, cnt, 0, 0.5)
    est3, _ = oracle.accept_stats([], [], ema, cnt, 0, 0.5, min_count=2)
    assert (est3 == 0.5).all()


def test_bad_entries_are_skipped_and_counted():
    ema, cnt = _tables(1, 3)
    est, bad = oracle.accept_stats([1, 4, -1, 2, 2], [0, 1, 0, 3, 2], ema, cnt, 0, 0.5)
    assert bad == 3
    assert list(cnt[0]) == [1, 1, 0] and list(ema[0, :2]) == [0.0, 1.0]


def test_invalid_arguments():
    ema, cnt = _tables(2, 3)
    for kw in [dict(bucket=2, beta=0.5), dict(bucket=-1, beta=0.5), dict(bucket=0, beta=0.0),
               dict(bucket=0, beta=1.5), dict(bucket=0, beta=float("nan"))]:
        with pytest.raises(ValueError):
            oracle.accept_stats([1], [1], ema, cnt, kw["bucket"], kw["beta"])


def test_tracks_the_verifier_acceptance_of_iid_positions():
    """Positions accepted independently with probability alpha until the first
    reject give E[accept_len] = sum_{k=1..L} alpha^k; the tracked rate of length
    L converges to that over L."""
    rng = np.random.default_rng(7)
    alpha, gamma, R = 0.8, 6, 512
    ema, cnt = _tables(1, gamma)
    for _ in range(60):
        ell = rng.integers(1, gamma + 1, R)
        ok = rng.random((R, gamma)) < alpha
        first_fail = np.where(ok.all(axis=1), gamma, np.argmin(ok, axis=1))
        oracle.accept_stats(ell, np.minimum(first_fail, ell), ema, cnt, 0, 0.2)
    for L in range(1, gamma + 1):
        want = sum(alpha ** k for k in range(1, L + 1)) / L
        assert ema[0, L - 1] == pytest.approx(want, abs=0.04)
