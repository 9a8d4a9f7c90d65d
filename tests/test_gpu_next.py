"""CUDA path versus the oracle for the scheduler's static-threshold mode, the
acceptance statistics and the calibration diagnostics, through the C ABI
(needs a GB300).

* Threshold mode (DSpark summary, comparison table: SpecDec++; Figure 5): the
  admitted set, row offsets and n, B are bit-exact against the oracle at the
  sizes of the benchmark workloads and at the one-block maximum, with planted
  ties, survivals equal to the threshold, zeros, and caps that bind or not.
* Acceptance statistics (LightSpec article, runtime statistics): every entry
  of the EMA table, the counts and the interpolated estimates are bit-exact
  (every step is one correctly rounded fp64 operation on both sides) over a
  sequence of rounds in several classes, with bad entries flagged.
* Calibration (DSpark summary, "2.1 置信度头" and Figure 6): c* = sum min(p, q)
  of every verified row within the probability tolerance, on the generic and
  the tensor-core passes, small and at full size; the reliability diagram's
  counts exactly and its sums and ECE to fp64 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import verify_sampling_gb300 as vs
from parity import compare_schedule, record, to_np

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
            record(f"schedule_threshold_R{R}_g{gamma}", rep)
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


# ------------------------------------------------------- calibration (c*) ----
from parity import PROB_TOL  # noqa: E402

CSTAR_CASES = {
    "tiny": synth.WORKLOADS["tiny"],                                          # generic, fp32 factors
    "c3_small": synth.WORKLOADS["c3"].scaled(R=12, gamma=8, V=8195, d=128),  # generic, ragged V
    "tc_c5_small": synth.WORKLOADS["c5"].scaled(R=8, gamma=6, V=12004, d=200),
    "tc_c3_R130": synth.WORKLOADS["c3"].scaled(R=130, gamma=3, V=4136, d=64),  # two row tiles
}


def _cstar_oracle(inp, reqs, x, ell, draft_temp):
    """The oracle's c* of the sampled requests, fed the GPU's tokens and l_r
    (tensors are indexed where they live, then copied)."""
    V = inp["U"].shape[-1]
    G = x.shape[1]
    reqs = list(reqs)
    idx = torch.tensor(reqs, device=inp["U"].device)
    tgt = inp["tgt"].view(-1, V)
    off = to_np(inp["tgt_row_off"])
    rows = torch.stack([tgt[int(off[r]) + j] for r in reqs for j in range(G + 1)])
    sub_off = (np.arange(len(reqs)) * (G + 1)).astype(np.int32)
    return oracle.cstar(to_np(rows), sub_off, ell[reqs], x[reqs], 1.0, to_np(inp["U"][idx]),
                        to_np(inp["A"]), to_np(inp["Ct"]), to_np(inp["x0"][idx]), draft_temp)


def _cstar_run(g, wl, seed, K):
    din = synth.draft_inputs(g)
    d = vs.draft_sample(din, seed)
    s = vs.schedule(d["a"], g["sps"], g["b_lo"], g["b_step"], K, vs.SCHED_THRESHOLD, threshold=0.0)
    v = vs.verify(vs.VERIFY_SAMPLE, g["tgt"].view(-1, wl.V), g["tgt_row_off"], s["ell"], d["x"],
                  seed, q_tok=d["q_tok"], lse_q=d["lse_q"], draft=din, want_cstar=True)
    torch.cuda.synchronize()
    return d, s, v


def _check_cstar(got, want):
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert fin.any()
    err = np.abs(got[fin] - want[fin]).max()
    assert err < PROB_TOL, err
    assert (got[fin] > 0).all() and (got[fin] <= 1 + 1e-5).all()


@pytest.mark.parametrize("name", list(CSTAR_CASES))
def test_cstar_parity_small(name):
    wl = CSTAR_CASES[name]
    inp = synth.make_inputs(wl, "cpu")
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    K = max(1, (wl.R * wl.gamma * 2) // 3)  # a cap that binds: some rows past l_r
    d, s, v = _cstar_run(g, wl, 31, K)
    ell, x = to_np(s["ell"]), to_np(d["x"])
    assert ell.sum() == min(K, wl.R * wl.gamma)
    want = _cstar_oracle(inp, range(wl.R), x, ell, to_np(inp["draft_temp"]))
    _check_cstar(to_np(v["c_star"]), want)


def test_cstar_full_size_c5_sampled():
    wl = synth.WORKLOADS["c5"]
    g = synth.make_inputs(wl, DEV, seed=wl.seed)
    d, s, v = _cstar_run(g, wl, 4243, wl.K)
    ell, x = to_np(s["ell"]), to_np(d["x"])
    # 32 requests spread over l_r (every verified row of each is compared)
    order = np.argsort(ell, kind="stable")
    reqs = sorted({int(order[i]) for i in np.linspace(0, wl.R - 1, 32).round().astype(int)}
                  | {0, wl.R - 1})
    assert len(reqs) >= 32 and len({int(ell[r]) for r in reqs}) >= 4
    want = _cstar_oracle(g, reqs, x, ell, to_np(g["draft_temp"]))
    _check_cstar(to_np(v["c_star"])[reqs], want)
    assert np.isnan(to_np(v["c_star"])[ell == 0]).all()


def test_calibration_parity_and_accumulation():
    rng = np.random.default_rng(21)
    n_bins = 10
    cnt_o, sc_o, sa_o = np.zeros(n_bins, np.int64), np.zeros(n_bins), np.zeros(n_bins, np.int64)
    tab = vs.calibration_tables(n_bins, DEV)
    for rnd in range(6):
        R, G = 512, 11
        c = rng.uniform(0, 1, (R, G)).astype(np.float32)
        c[0, 0], c[1, 0], c[2, 0] = 0.0, 1.0, 0.5  # bin edges
        ell, acc = _round_inputs(rng, R, G)
        ece_o, bad = oracle.calibration(c.astype(np.float64), ell, acc, cnt_o, sc_o, sa_o)
        assert bad == 0
        vs.calibration(torch.tensor(c, device=DEV), torch.tensor(ell, device=DEV),
                       torch.tensor(acc, device=DEV), tab)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(tab["count"]), cnt_o)
        assert np.array_equal(to_np(tab["sum_acc"]), sa_o)
        assert np.allclose(to_np(tab["sum_c"]), sc_o, rtol=1e-12, atol=0)
        assert abs(float(tab["ece"].item()) - ece_o) <= 1e-12 * max(1.0, ece_o)


def test_calibration_bad_entries_and_empty():
    tab = vs.calibration_tables(4, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    c = torch.tensor([[0.5, float("nan")], [0.5, 0.5], [1.5, 0.5]], device=DEV)
    ell = torch.tensor([2, 3, 1], dtype=torch.int32, device=DEV)
    acc = torch.tensor([2, 0, 0], dtype=torch.int32, device=DEV)
    vs.calibration(c, ell, acc, tab, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & vs.STATUS_BAD_ELL and st & vs.STATUS_BAD_SURVIVAL
    assert int(tab["count"].sum()) == 1
    empty = vs.calibration_tables(4, DEV)
    vs.calibration(torch.zeros((0, 2), device=DEV), torch.zeros(0, dtype=torch.int32, device=DEV),
                   torch.zeros(0, dtype=torch.int32, device=DEV), empty)
    torch.cuda.synchronize()
    assert np.isnan(float(empty["ece"].item()))


def _level_survivals(rng, R, gamma, lo):
    c = rng.uniform(lo, 1.0, (R, gamma)).astype(np.float32)
    return np.cumprod(c, axis=1, dtype=np.float32)


@pytest.mark.parametrize("mode", [oracle.SCHED_EARLY_STOP, oracle.SCHED_GLOBAL,
                                  oracle.SCHED_THRESHOLD])
def test_async_cap_chain(mode):
    """DSpark summary, "挑战2": round t is capped by the uncapped count of
    round t - 2, through one device word per parity of t (read, then written,
    by the same launch).  Every round's decision and its uncapped count equal
    the oracle's, run with the cap the oracle's own chain gives."""
    R, gamma, K = 512, 11, 2048
    N = R * gamma
    rng = np.random.default_rng(90 + mode)
    # confidence levels that make the two-rounds-back cap bind (a low round
    # followed, two rounds later, by a high one)
    levels = [0.05, 0.1, 0.9, 0.95, 0.2, 0.6]
    sps = _sps(R, gamma).to(DEV)
    sps_np = to_np(sps).astype(np.float64)
    thr = 0.3
    cap = torch.full((2,), K, dtype=torch.int32, device=DEV)
    free_seen, bound = [], 0
    for t, lo in enumerate(levels):
        a_np = _level_survivals(rng, R, gamma, lo)
        a = torch.tensor(a_np, device=DEV)
        word = cap[t % 2: t % 2 + 1]
        s = vs.schedule(a, sps, 1.0, 1.0, K, mode, threshold=thr, K_dev=word, n_free=word)
        torch.cuda.synchronize()
        k_t = K if t < 2 else min(K, free_seen[t - 2])
        inp = {"sps": sps, "b_lo": 1.0, "b_step": 1.0}
        rep = compare_schedule(inp, a, s, k_t, mode, threshold=thr)
        record(f"async_cap_mode{mode}", rep)
        of = oracle.schedule(a_np.astype(np.float64), sps_np, 1.0, 1.0, N, mode, thr)
        if of.margin >= 1e-6 and rep.near_ties == 0:
            assert int(word.item()) == of.n, (t, int(word.item()), of.n)
        free_seen.append(int(word.item()))
        bound += int(int(to_np(s["stats"])[0]) < min(K, of.n))
    assert bound >= 1  # the lagged cap took effect at least once


@pytest.mark.parametrize("R,gamma", [(512, 11), (128, 64), (3, 7), (1, 40)])
def test_schedule_unordered_survivals(R, gamma):
    """Survivals that rise along j (not products of confidences): the sort
    orders every run itself before merging.  Order, l_r and stats equal the
    oracle's in all three modes."""
    rng = np.random.default_rng(R + gamma)
    a_np = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
    a_np[rng.random((R, gamma)) < 0.05] = np.float32(0.5)  # ties across requests
    a = torch.tensor(a_np, device=DEV)
    inp = {"sps": _sps(R, gamma).to(DEV), "b_lo": 1.0, "b_step": 1.0}
    for mode in (oracle.SCHED_EARLY_STOP, oracle.SCHED_GLOBAL, oracle.SCHED_THRESHOLD):
        K = max(1, (R * gamma) // 2)
        s = vs.schedule(a, inp["sps"], 1.0, 1.0, K, mode, threshold=0.4, want_order=True)
        torch.cuda.synchronize()
        rep = compare_schedule(inp, a, s, K, mode, threshold=0.4)
        assert rep.checked + rep.near_ties == 1
        record(f"schedule_unordered_R{R}_g{gamma}", rep)
