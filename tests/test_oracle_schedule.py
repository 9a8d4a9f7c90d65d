"""Pins for the oracle's prefix scheduler (CPU only).

* a hand-computed walk-through of the history article's "杀招三" (golden fixture);
* brute force over every l-vector (the benchmark spec check (d)): because a_{r,j} is
  non-increasing in j, the best admitted set of any size n is the top-n of the
  sorted list, so the global search must equal the brute-force optimum, and the
  early-stop result can only be lower (its ratio is reported);
* closed forms: a constant SPS admits every positive candidate up to the cap;
  a linear SPS table is reproduced exactly by the interpolating lookup.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _walkthrough():
    with open(os.path.join(GOLDEN, "scheduler_walkthrough.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case,mode", [("early_stop", oracle.SCHED_EARLY_STOP),
                                       ("global", oracle.SCHED_GLOBAL),
                                       ("global_K5", oracle.SCHED_GLOBAL)])
def test_walkthrough(case, mode):
    g = _walkthrough()
    exp = g[case]
    out = oracle.schedule(np.array(g["a"]), g["sps"], g["b_lo"], g["b_step"], exp["K"], mode)
    assert out.n == exp["n"] and out.B == exp["B"]
    assert list(out.ell) == exp["ell"] and list(out.row_off) == exp["row_off"]
    assert out.tau == pytest.approx(exp["tau"], rel=1e-12)
    assert out.theta == pytest.approx(exp["theta"], rel=1e-12)
    nmax = min(exp["K"], g["R"] * g["gamma"])
    assert np.allclose(out.theta_seq, g["theta_expected"][: nmax + 1], rtol=1e-12)


def _brute_force(a, sps_at, K):
    """max over all l in {0..gamma}^R with sum(l) <= K of tau(l) * SPS(R + sum l)."""
    R, gamma = a.shape
    best = 0.0
    for ell in itertools.product(range(gamma + 1), repeat=R):
        n = sum(ell)
        if n > K:
            continue
        tau = sum(a[r, :ell[r]].sum() for r in range(R))
        best = max(best, tau * sps_at(R + n))
    return best


def _random_instance(rng, R, gamma, kind):
    c = rng.uniform(0.05, 1.0, size=(R, gamma))
    a = np.cumprod(c, axis=1)
    nB = R * (gamma + 1) + 1
    if kind == "linear":
        sps = 100.0 - rng.uniform(0.5, 20.0) * np.arange(nB)
    elif kind == "sawtooth":
        sps = 100.0 / (1 + 0.3 * np.arange(nB)) * (1 + 0.5 * (np.arange(nB) % 3 == 0))
    else:
        sps = rng.uniform(1, 100, size=nB)
    return a, np.maximum(sps, 1e-3)


@pytest.mark.parametrize("R,gamma", [(1, 4), (2, 3), (3, 4), (3, 2)])
@pytest.mark.parametrize("kind", ["linear", "sawtooth", "random"])
def test_brute_force(R, gamma, kind):
    rng = np.random.default_rng(100 * R + gamma + len(kind))
    ratios = []
    for trial in range(6):
        a, sps = _random_instance(rng, R, gamma, kind)
        K = int(rng.integers(1, R * gamma + 2))
        sps_at = lambda B: sps[B]  # table at B = 0, 1, 2, ...: direct reads, no interpolation
        opt = _brute_force(a, sps_at, K)
        glob = oracle.schedule(a, sps, 0.0, 1.0, K, oracle.SCHED_GLOBAL)
        early = oracle.schedule(a, sps, 0.0, 1.0, K, oracle.SCHED_EARLY_STOP)
        assert glob.theta == pytest.approx(opt, rel=1e-12)
        assert early.theta <= opt * (1 + 1e-12)
        ratios.append(early.theta / opt if opt > 0 else 1.0)
        for out in (glob, early):
            assert out.ell.sum() == out.n <= K
            assert out.B == R + out.n == out.row_off[-1]
    assert min(ratios) > 0


def test_early_stop_equals_global_when_theta_unimodal():
    """A constant SPS makes Theta_n = tau_n * const increasing: admit all."""
    rng = np.random.default_rng(4)
    a = np.cumprod(rng.uniform(0.1, 1, (5, 6)), axis=1)
    for K in (0, 7, 30, 100):
        for mode in (oracle.SCHED_EARLY_STOP, oracle.SCHED_GLOBAL):
            out = oracle.schedule(a, [3.0], 1.0, 1.0, K, mode)
            assert out.n == min(K, 30)


def test_admission_is_prefix_closed_and_sorted():
    """The benchmark spec check (c): the admitted set is a prefix per request."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        R, gamma = int(rng.integers(1, 9)), int(rng.integers(1, 17))
        a = np.cumprod(rng.uniform(0.2, 1, (R, gamma)), axis=1)
        a = a.astype(np.float32).astype(np.float64)
        nB = R * (gamma + 1) + 1
        sps = np.maximum(100 - rng.uniform(0, 3) * np.arange(nB), 0.1)
        out = oracle.schedule(a, sps, 0.0, 1.0, int(rng.integers(0, R * gamma + 1)),
                              int(rng.integers(0, 2)))
        admitted = set(out.order[: out.n].tolist())
        for r in range(R):
            got = {i % gamma for i in admitted if i // gamma == r}
            assert got == set(range(out.ell[r]))
        keys = a.reshape(-1)[out.order]
        assert np.all(np.diff(keys) <= 0)


def test_ties_keep_request_then_position_order():
    a = np.array([[0.5, 0.5], [0.5, 0.25]])
    out = oracle.schedule(a, [1.0], 0.0, 1.0, 4, oracle.SCHED_GLOBAL)
    assert list(out.order) == [0, 1, 2, 3]


def test_sawtooth_trap_early_stop_below_global():
    """DSpark summary "挑战2": on a saw-tooth SPS early stop ends at a local optimum."""
    g = _walkthrough()
    e = oracle.schedule(np.array(g["a"]), g["sps"], 2, 1, 8, oracle.SCHED_EARLY_STOP)
    glob = oracle.schedule(np.array(g["a"]), g["sps"], 2, 1, 8, oracle.SCHED_GLOBAL)
    assert e.theta < glob.theta


def test_sps_lookup_linear_and_clamped():
    b_lo, b_step = 4.0, 2.5
    sps = 1000.0 - 7.0 * np.arange(16)        # value at B_i = b_lo + i*b_step
    lin = lambda B: 1000.0 - 7.0 * (B - b_lo) / b_step
    for B in np.linspace(b_lo, b_lo + 15 * b_step, 61):
        assert oracle.sps_lookup(sps, b_lo, b_step, B) == pytest.approx(lin(B), rel=1e-14)
    assert oracle.sps_lookup(sps, b_lo, b_step, 0.0) == sps[0]
    assert oracle.sps_lookup(sps, b_lo, b_step, 1e6) == sps[-1]


def test_zero_cap_admits_nothing():
    out = oracle.schedule(np.full((3, 2), 0.9), [1.0], 0, 1, 0, oracle.SCHED_EARLY_STOP)
    assert out.n == 0 and list(out.ell) == [0, 0, 0] and list(out.row_off) == [0, 1, 2, 3]
