"""RNN sequential head: CUDA path versus the oracle, through the C ABI (needs a
GB300).

DSpark summary, "第二阶段：轻量顺序头": the head may carry a recurrent state
instead of the previous token alone.  The library reads it as
s_k = store(tanh(A_k[x_{k-1}] + s_{k-1} W_k)), B_k = s_k C_k (the oracle's
reading, pinned there by reduction to the Markov head and by losslessness).
Each case runs a whole round -- draft with the state kernel between positions,
schedule, verify with the residual and c* recomputed from the stored states --
on the generic kernels (fp32 factors; bf16 rows that are not 16-byte
multiples) and on the tensor-core kernels (one and two 128-request tiles, r 64,
128 and 256), with W_k staged in shared memory or read from global memory, then
at the benchmark's full size on sampled requests.  Stages are
isolated as in the Markov parity tests: the oracle takes the CUDA path's
tokens and states as its conditioning.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import verify_sampling_gb300 as vs
from parity import (PROB_TOL, compare_draft_rnn, compare_verify, pick_full_size_requests, record,
                    to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "c3_small": synth.WORKLOADS["c3"].scaled(R=12, gamma=8, V=8195, d=128),
    "tc_c5_small": synth.WORKLOADS["c5"].scaled(R=8, gamma=6, V=12004, d=200),
    "tc_c3_small_R130": synth.WORKLOADS["c3"].scaled(R=130, gamma=3, V=4136, d=64),
    "tc_c5_r64": synth.WORKLOADS["c5"].scaled(R=5, gamma=4, V=3000, d=16, r=64),
    # W_k too large to stage in shared memory (read from global memory instead)
    "tc_c5_r256": synth.WORKLOADS["c5"].scaled(R=6, gamma=3, V=2048, d=16, r=256),
    "fp32_r160": synth.WORKLOADS["tiny"].scaled(R=5, gamma=3, V=777, r=160),
    # degenerate sizes: one token, one position, one request
    "v1": synth.WORKLOADS["tiny"].scaled(R=2, gamma=1, V=1, r=1, d=3, e=1),
    "r1_gamma1": synth.WORKLOADS["c2"].scaled(R=1, gamma=1, V=4097, d=64, e=16, r=16),
    "tc_gamma1": synth.WORKLOADS["c5"].scaled(R=3, gamma=1, V=2048, d=16, r=64),
}
SAMPLED = {"tc_c3_small_R130": [0, 1, 2, 64, 127, 128, 129]}


def _round(g, wl, W, seed, want_P):
    S = torch.full((wl.R, wl.gamma, wl.r), float("nan"), dtype=wl.fac_dtype, device=DEV)
    din = synth.draft_inputs(g)
    din.Wrnn, din.S = W, S
    d = vs.draft_sample(din, seed, want_P=want_P)
    s = vs.schedule(d["a"], g["sps"], g["b_lo"], g["b_step"], g["K"], wl.sched_mode,
                    threshold=wl.sched_threshold)
    v = vs.verify(vs.VERIFY_SAMPLE, g["tgt"].view(-1, wl.V), g["tgt_row_off"], s["ell"], d["x"],
                  seed, q_tok=d["q_tok"], lse_q=d["lse_q"], draft=din, want_p=True, want_cstar=True)
    torch.cuda.synchronize()
    return S, d, s, v


def _cstar_oracle(g, reqs, x, ell, S):
    V = g["U"].shape[-1]
    G = x.shape[1]
    idx = torch.tensor(reqs, device=g["U"].device)
    tgt = g["tgt"].view(-1, V)
    off = to_np(g["tgt_row_off"])
    rows = torch.stack([tgt[int(off[r]) + j] for r in reqs for j in range(G + 1)])
    sub_off = (np.arange(len(reqs)) * (G + 1)).astype(np.int32)
    return oracle.cstar(to_np(rows), sub_off, ell[reqs], x[reqs], 1.0, to_np(g["U"][idx]),
                        to_np(g["A"]), to_np(g["Ct"]), to_np(g["x0"][idx]), to_np(g["draft_temp"]),
                        S=to_np(S[idx]))


def _check(g, wl, W, seed, S, d, s, v, reqs, config):
    rep = compare_draft_rnn(g, W, S, d, seed, reqs)
    assert rep.near_ties <= max(1, len(reqs) * wl.gamma // 100)
    record(config, rep)
    rep = compare_verify(g, d, s["ell"], v, seed, oracle.MODE_SAMPLE, reqs, S=S)
    assert rep.checked >= len(reqs) - max(1, len(reqs) // 20)
    record(config, rep)
    ell, x = to_np(s["ell"]), to_np(d["x"])
    want = _cstar_oracle(g, list(reqs), x, ell, S)
    got = to_np(v["c_star"])[list(reqs)]
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    if fin.any():
        assert np.abs(got[fin] - want[fin]).max() < PROB_TOL


@pytest.mark.parametrize("name", list(CASES))
def test_rnn_round_parity_small(name):
    wl = CASES[name]
    g = {k: (t.to(DEV) if isinstance(t, torch.Tensor) else t)
         for k, t in synth.make_inputs(wl, "cpu").items()}
    W = synth.rnn_weights(wl, DEV)
    seed = 1234
    S, d, s, v = _round(g, wl, W, seed, want_P=wl.V <= 20000)
    assert not torch.isnan(S.float()).any()
    reqs = SAMPLED.get(name, range(wl.R))
    _check(g, wl, W, seed, S, d, s, v, list(reqs), "rnn_" + name)


def test_rnn_differs_from_markov_and_reruns_identically():
    wl = CASES["tc_c5_small"]
    g = {k: (t.to(DEV) if isinstance(t, torch.Tensor) else t)
         for k, t in synth.make_inputs(wl, "cpu").items()}
    W = synth.rnn_weights(wl, DEV)
    S1, d1, _, v1 = _round(g, wl, W, 77, want_P=False)
    S2, d2, _, v2 = _round(g, wl, W, 77, want_P=False)
    assert torch.equal(S1, S2) and torch.equal(d1["x"], d2["x"])
    assert torch.equal(v1["out_tok"], v2["out_tok"])
    mk = vs.draft_sample(synth.draft_inputs(g), 77)
    torch.cuda.synchronize()
    # the first position's bias rows differ (tanh of A_1[x0] against A_1[x0]),
    # so the distributions must too
    assert not torch.equal(mk["lse_q"], d1["lse_q"])


def test_rnn_full_size_c5_sampled():
    wl = synth.WORKLOADS["c5"]
    g = synth.make_inputs(wl, DEV, seed=wl.seed)
    W = synth.rnn_weights(wl, DEV)
    seed = 4243
    S, d, s, v = _round(g, wl, W, seed, want_P=False)
    assert not torch.isnan(S.float()).any()
    reqs, rejected, bonus = pick_full_size_requests(to_np(s["ell"]), to_np(v["accept_len"]), wl.R)
    assert len(rejected) >= 8 and len(bonus) >= 8 and len(reqs) >= 32
    _check(g, wl, W, seed, S, d, s, v, reqs, "rnn_c5")


def test_rnn_request_sharding_is_invariant():
    """The state is per request and the stream is keyed by the global request
    id: drafting the last requests alone, with request_id_base = their first
    global id, gives the same tokens and states (one and two request tiles)."""
    wl = CASES["tc_c3_small_R130"]
    g = {k: (t.to(DEV) if isinstance(t, torch.Tensor) else t)
         for k, t in synth.make_inputs(wl, "cpu").items()}
    W = synth.rnn_weights(wl, DEV)
    S_all, d_all, _, _ = _round(g, wl, W, 5, want_P=False)
    lo = 70
    half = {k: (v[lo:] if isinstance(v, torch.Tensor) and k in ("U", "x0", "h") else v)
            for k, v in g.items()}
    din = synth.draft_inputs(half, request_id_base=lo)
    din.Wrnn = W
    din.S = torch.zeros(wl.R - lo, wl.gamma, wl.r, dtype=wl.fac_dtype, device=DEV)
    d_half = vs.draft_sample(din, 5)
    torch.cuda.synchronize()
    assert torch.equal(d_half["x"], d_all["x"][lo:])
    assert torch.equal(din.S, S_all[lo:])
