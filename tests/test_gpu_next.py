"""CUDA path versus the oracle for the scheduler's static-threshold mode and the
acceptance statistics, through the C ABI (needs a GB300).

* Threshold mode (DSpark summary, comparison table: SpecDec++; Figure 5): the
  admitted set, row offsets and n, B are bit-exact against the oracle at the
  sizes of the benchmark workloads and at the one-block maximum, with planted
  ties, survivals equal to the threshold, zeros, and caps that bind or not.
* Acceptance statistics (LightSpec article, runtime statistics): every entry
  of the EMA table, the counts and the interpolated estimates are bit-exact
  (every step is one correctly rounded fp64 operation on both sides) over a
  sequence of rounds in several classes, with bad entries flagged.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import verify_sampling_gb300 as vs
from parity import compare_schedule, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _survivals(rng, R, gamma):
    c = rng.uniform(0.3, 1.0, (R, gamma)).astype(np.float32)
    a = np.cumprod(c, axis=1, dtype=np.float32)
    # planted ties across requests, a survival equal to the threshold 0.5 and zeros
    a[rng.random((R, gamma)) < 0.05] = np.float32(0.5)
    a[rng.random(R) < 0.05, -1] = 0.0
    return np.minimum.accumulate(a, axis=1)


def _sps(R, gamma):
    B = np.arange(1, R * (gamma + 1) + 1, dtype=np.float64)
    return torch.tensor(1.0 / (0.01 + 2e-6 * B), dtype=torch.float32)


@pytest.mark.parametrize("R,gamma", [(512, 11), (256, 16), (744, 11), (3, 2), (1, 1)])
def test_schedule_threshold_parity(R, gamma):
    rng = np.random.default_rng(R * 100 + gamma)
    a_np = _survivals(rng, R, gamma)
    a = torch.tensor(a_np, device=DEV)
    inp = {"sps": _sps(R, gamma).to(DEV), "b_lo": 1.0, "b_step": 1.0}
    N = R * gamma
    checked = 0
    for theta in [0.0, 0.05, 0.3, 0.5, 0.99, 2.0]:
        for K in sorted({N, max(1, N // 3), 0}):
            s = vs.schedule(a, inp["sps"], 1.0, 1.0, K, vs.SCHED_THRESHOLD, threshold=theta,
                            want_order=True)
            torch.cuda.synchronize()
            rep = compare_schedule(inp, a, s, K, oracle.SCHED_THRESHOLD, threshold=theta)
            assert rep.near_ties == 0  # threshold decisions are exact comparisons
            n = int(to_np(s["stats"])[0])
            assert n == min(K, int((a_np >= theta).sum()))
            checked += 1
    assert checked == 6 * len({N, max(1, N // 3), 0})


def test_threshold_round_uses_the_schedule():
    """A full small round in threshold mode: the verifier reads the admitted rows."""
    wl = synth.WORKLOADS["c5"].scaled(R=8, gamma=6, V=12004, d=200, sched_mode=2,
                                      sched_threshold=0.3)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
         for k, v in synth.make_inputs(wl, "cpu").items()}
    din = synth.draft_inputs(g)
    out = vs.run_round(din, g["tgt"].view(-1, wl.V), g["tgt_row_off"], g["sps"], g["b_lo"],
                       g["b_step"], wl.K, 77, sched_mode=vs.SCHED_THRESHOLD,
                       sched_threshold=wl.sched_threshold)
    torch.cuda.synchronize()
    a = to_np(out["draft"]["a"])
    ell = to_np(out["sched"]["ell"])
    os_ = oracle.schedule(a.astype(np.float64), to_np(g["sps"]).astype(np.float64), g["b_lo"],
                          g["b_step"], wl.K, oracle.SCHED_THRESHOLD, wl.sched_threshold)
    assert (ell == os_.ell).all()
    acc = to_np(out["verify"]["accept_len"])
    assert ((acc >= 0) & (acc <= ell)).all()


def _round_inputs(rng, R, gamma):
    ell = rng.integers(0, gamma + 1, R).astype(np.int32)
    acc = np.array([rng.integers(0, l + 1) for l in ell], np.int32)
    return ell, acc


@pytest.mark.parametrize("R,gamma", [(512, 11), (256, 16), (5, 3), (0, 4), (3000, 64)])
def test_accept_stats_bit_exact(R, gamma):
    rng = np.random.default_rng(R + gamma)
    n_buckets = 3
    ema_o = np.zeros((n_buckets, gamma))
    cnt_o = np.zeros((n_buckets, gamma), np.int64)
    ema_g = torch.zeros((n_buckets, gamma), dtype=torch.float64, device=DEV)
    cnt_g = torch.zeros((n_buckets, gamma), dtype=torch.int64, device=DEV)
    est_g = torch.empty(gamma, dtype=torch.float64, device=DEV)
    for rnd in range(12):
        ell, acc = _round_inputs(rng, R, gamma)
        if R > 0 and rnd % 4 == 1:  # thin rounds leave lengths without samples
            thin = rng.random(R) < 0.9
            ell[thin] = 0
            acc[thin] = 0
        bucket = int(rng.integers(0, n_buckets))
        beta = float(rng.choice([0.05, 0.3, 1.0]))
        min_count = int(rng.integers(0, 40))
        est_o, bad = oracle.accept_stats(ell, acc, ema_o, cnt_o, bucket, beta, min_count)
        assert bad == 0
        vs.accept_stats(torch.tensor(ell, device=DEV), torch.tensor(acc, device=DEV), ema_g, cnt_g,
                        bucket, beta, min_count=min_count, estimate=est_g)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(cnt_g), cnt_o)
        assert np.array_equal(to_np(ema_g).view(np.uint64), ema_o.view(np.uint64))
        got = to_np(est_g)
        assert np.array_equal(np.isnan(got), np.isnan(est_o))
        fin = ~np.isnan(est_o)
        assert np.array_equal(got[fin].view(np.uint64), est_o[fin].view(np.uint64))


def test_accept_stats_bad_entries_set_status():
    ell = np.array([1, 4, -1, 2, 2, 3], np.int32)
    acc = np.array([0, 1, 0, 3, 2, 1], np.int32)
    ema_o, cnt_o = np.zeros((1, 3)), np.zeros((1, 3), np.int64)
    oracle.accept_stats(ell, acc, ema_o, cnt_o, 0, 0.5)
    ema_g = torch.zeros((1, 3), dtype=torch.float64, device=DEV)
    cnt_g = torch.zeros((1, 3), dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    vs.accept_stats(torch.tensor(ell, device=DEV), torch.tensor(acc, device=DEV), ema_g, cnt_g, 0,
                    0.5, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & vs.STATUS_BAD_ELL
    assert np.array_equal(to_np(cnt_g), cnt_o)
    assert np.array_equal(to_np(ema_g), ema_o)
