"""Pins for the oracle's prefix scheduler (CPU only).

* a hand-computed walk-through of the history article's "杀招三" (golden fixture);
* brute force over every l-vector: because a_{r,j} is
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
    """Prefix closure: the admitted set is a prefix of each request."""
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


# ------------------------------------------------------- threshold admission --
# DSpark summary, comparison table (SpecDec++: a static confidence threshold) and
# Figure 5 (a threshold sweep): mode SCHED_THRESHOLD admits every candidate whose
# survival a_{r,j} reaches the threshold, capped by K.

def _non_increasing(rng, R, gamma):
    a = np.cumprod(rng.uniform(0.3, 1.0, (R, gamma)), axis=1)
    return a.astype(np.float32).astype(np.float64)


def test_threshold_admits_per_request_counts():
    """Without a binding cap, l_r is the number of positions of r with a >= theta
    (counted per request, not through the sorted list)."""
    rng = np.random.default_rng(11)
    for _ in range(30):
        R, gamma = int(rng.integers(1, 12)), int(rng.integers(1, 12))
        a = _non_increasing(rng, R, gamma)
        theta = float(rng.uniform(0.0, 1.0))
        out = oracle.schedule(a, [1.0], 0.0, 1.0, R * gamma, oracle.SCHED_THRESHOLD, theta)
        want = [int(sum(1 for j in range(gamma) if a[r, j] >= theta)) for r in range(R)]
        assert list(out.ell) == want
        assert out.n == sum(want) and out.B == R + sum(want)
        assert out.tau == pytest.approx(float(a[a >= theta].sum()), rel=1e-12, abs=0)
        assert out.margin == float("inf")


def test_threshold_cap_keeps_the_largest_survivals():
    rng = np.random.default_rng(12)
    for _ in range(30):
        R, gamma = int(rng.integers(1, 10)), int(rng.integers(1, 10))
        a = _non_increasing(rng, R, gamma)
        a[rng.random((R, gamma)) < 0.2] = 0.5  # planted ties
        a = np.minimum.accumulate(a, axis=1)
        theta = float(rng.uniform(0.0, 0.9))
        K = int(rng.integers(0, R * gamma + 1))
        out = oracle.schedule(a, [1.0], 0.0, 1.0, K, oracle.SCHED_THRESHOLD, theta)
        ids = [i for i in range(R * gamma) if a.reshape(-1)[i] >= theta]
        ids.sort(key=lambda i: (-a.reshape(-1)[i], i))
        chosen = ids[:K]
        want = np.zeros(R, int)
        for i in chosen:
            want[i // gamma] += 1
        assert list(out.ell) == list(want)


def test_threshold_ends():
    a = np.array([[0.9, 0.6, 0.2], [0.8, 0.8, 0.1]])
    everything = oracle.schedule(a, [1.0], 0.0, 1.0, 6, oracle.SCHED_THRESHOLD, 0.0)
    assert list(everything.ell) == [3, 3]
    nothing = oracle.schedule(a, [1.0], 0.0, 1.0, 6, oracle.SCHED_THRESHOLD, 0.95)
    assert nothing.n == 0 and list(nothing.row_off) == [0, 1, 2]
    equal = oracle.schedule(a, [1.0], 0.0, 1.0, 6, oracle.SCHED_THRESHOLD, 0.8)
    assert list(equal.ell) == [1, 2]  # a >= theta includes equality
    with pytest.raises(ValueError):
        oracle.schedule(a, [1.0], 0.0, 1.0, 6, oracle.SCHED_THRESHOLD, float("nan"))


def test_threshold_sweep_raises_acceptance_rate():
    """Figure 5: raising the threshold filters the likely rejections, so the
    accepted fraction of the admitted tokens rises.  With calibrated
    confidences (position j of r is accepted with probability c_{r,j} once the
    positions before it were), the expected accepted count of an admitted
    prefix is the sum of its survivals: the predicted rate tau / n must be
    non-decreasing in theta, and a simulation of the verifier agrees with it."""
    rng = np.random.default_rng(13)
    R, gamma = 256, 8
    c = rng.uniform(0.4, 1.0, (R, gamma))
    a = np.cumprod(c, axis=1)
    thresholds = [0.0, 0.2, 0.4, 0.6, 0.8]
    rates = []
    for th in thresholds:
        out = oracle.schedule(a, [1.0], 0.0, 1.0, R * gamma, oracle.SCHED_THRESHOLD, th)
        assert out.n > 0
        rates.append(out.tau / out.n)
        trials = 400
        acc = 0
        for _ in range(trials):
            ok = rng.random((R, gamma)) < c
            first_fail = np.where(ok.all(axis=1), gamma, np.argmin(ok, axis=1))
            acc += int(np.minimum(first_fail, out.ell).sum())
        sim = acc / (trials * out.n)
        assert sim == pytest.approx(out.tau / out.n, abs=0.01)
    assert all(x <= y for x, y in zip(rates, rates[1:]))
    assert rates[-1] > rates[0] + 0.1


@pytest.mark.parametrize("mode", [oracle.SCHED_EARLY_STOP, oracle.SCHED_THRESHOLD])
def test_cap_truncates_the_uncapped_decision(mode):
    """DSpark summary, "挑战2": the asynchronous cap only limits how many of
    the newest-ranked candidates are admitted.  For the rules that stop at the
    first failing candidate, the capped count is min(uncapped count, K) and
    the admitted set is the first n of the same sorted order -- what the
    device kernel uses to take both decisions from one scan."""
    rng = np.random.default_rng(11 + mode)
    R, gamma = 40, 6
    B = np.arange(1, R * (gamma + 1) + 1, dtype=np.float64)
    sps = 1.0 / (0.01 + 5e-4 * B)
    for trial in range(20):
        c = rng.uniform(0.05 * (trial % 10), 1.0, (R, gamma))
        a = np.cumprod(c, axis=1)
        free = oracle.schedule(a, sps, 1.0, 1.0, R * gamma, mode, 0.3)
        for K in (0, 1, free.n // 2, free.n, free.n + 3, R * gamma):
            got = oracle.schedule(a, sps, 1.0, 1.0, K, mode, 0.3)
            assert got.n == min(free.n, K)
            assert np.array_equal(got.order[:got.n], free.order[:got.n])


def test_global_cap_is_the_argmax_below_the_cap():
    """Global search under a cap: the smallest argmax of Theta over n <= K,
    which may differ from the uncapped argmax truncated to K."""
    rng = np.random.default_rng(5)
    R, gamma = 30, 5
    B = np.arange(1, R * (gamma + 1) + 1, dtype=np.float64)
    sps = (1.0 + 0.3 * ((B % 20) / 20.0)) / (0.01 + 5e-4 * B)  # sawtooth
    for _ in range(10):
        a = np.cumprod(rng.uniform(0.2, 1.0, (R, gamma)), axis=1)
        full = oracle.schedule(a, sps, 1.0, 1.0, R * gamma, oracle.SCHED_GLOBAL)
        th = full.theta_seq
        for K in (1, 7, full.n // 2, full.n, R * gamma):
            got = oracle.schedule(a, sps, 1.0, 1.0, K, oracle.SCHED_GLOBAL)
            want = int(np.argmax(th[: min(K, R * gamma) + 1]))
            assert got.n == want
