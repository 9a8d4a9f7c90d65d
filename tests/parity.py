"""Comparison of the CUDA path with the oracle, stage by stage.

Rules (from the method's statement of correctness):
  * token ids, accept lengths, l_r: bit-exact, except decisions whose oracle
    margin (Gumbel top-2 score gap, |u - p/q|, relative Theta gap) is below
    NEAR_TIE; those are counted and the request is excluded downstream;
  * probabilities and confidences: within PROB_TOL absolute (fp32 path; the
    arithmetic is fp32 on exactly upcast bf16 inputs, so one tolerance serves
    both input dtypes); log-sum-exp values within PROB_TOL relative.
Stage isolation: every oracle stage is fed the CUDA path's outputs of the
previous stage (draft tokens, survivals, l_r), so each stage is compared on its
own decisions.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import near_ties
import oracle

NEAR_TIE = 1e-6
PROB_TOL = 1e-5


@dataclass
class Report:
    """checked: decisions compared bit-exactly; near_ties: exempted decisions
    (oracle margin below NEAR_TIE) on which the two sides disagreed; kinds:
    per decision kind, [checked, near, differ] (see near_ties.py)."""
    checked: int = 0
    near_ties: int = 0
    notes: list = field(default_factory=list)
    kinds: dict = field(default_factory=dict)

    def count(self, kind: str, checked: int = 0, near: int = 0, differ: int = 0) -> None:
        row = self.kinds.setdefault(kind, [0, 0, 0])
        row[0] += int(checked)
        row[1] += int(near)
        row[2] += int(differ)


def record(config: str, rep: Report) -> Report:
    """Add a report's per-kind counts to the session's near-tie record."""
    for kind, (checked, near, differ) in rep.kinds.items():
        near_ties.add(config, kind, checked, near, differ)
    return rep


def pick_full_size_requests(ell, accept_len, R: int, n_rejected: int = 32, n_bonus: int = 12,
                            always=(0, 1)):
    """Requests to compare at full size: every request the GPU rejected, up
    to n_rejected of them, taken round-robin over the rejected position j* (so
    the residual pass's per-position tiles are all reached); n_bonus of the
    requests that accepted every admitted position (their bonus row is
    sampled), spread over l_r; plus `always`, the middle and the last request.
    Returns (sorted requests, rejected among them, bonus among them)."""
    ell, acc = np.asarray(ell), np.asarray(accept_len)
    rej = np.flatnonzero(acc < ell)
    by_pos = {}
    for r in rej:
        by_pos.setdefault(int(acc[r]) + 1, []).append(int(r))
    picked_rej = []
    while len(picked_rej) < min(n_rejected, len(rej)):
        for j in sorted(by_pos):
            if by_pos[j] and len(picked_rej) < n_rejected:
                picked_rej.append(by_pos[j].pop(0))
    bon = np.flatnonzero(acc == ell)
    order = bon[np.argsort(ell[bon], kind="stable")]
    picked_bon = [int(order[i]) for i in np.linspace(0, len(order) - 1, min(n_bonus, len(order))
                                                    ).round().astype(int)] if len(order) else []
    reqs = sorted(set(picked_rej) | set(picked_bon) | {int(a) for a in always} | {R // 2, R - 1})
    return reqs, [r for r in reqs if acc[r] < ell[r]], [r for r in reqs if acc[r] == ell[r]]


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def compare_draft(inp: dict, out: dict, seed: int, reqs, rid_base: int = 0, rep=None) -> Report:
    rep = rep or Report()
    A, Ct = to_np(inp["A"]), to_np(inp["Ct"])
    x_gpu = to_np(out["x"])
    for r in reqs:
        od = oracle.draft(to_np(inp["U"][r:r + 1]), A, Ct, to_np(inp["x0"][r:r + 1]),
                          to_np(inp["draft_temp"]), seed, rid_base=rid_base + r,
                          x_cond=x_gpu[r:r + 1], want_P="P" in out)
        same = od.x[0] == x_gpu[r]
        tie = od.gap[0] < NEAR_TIE
        assert np.all(same | tie), (r, od.x[0], x_gpu[r], od.gap[0])
        rep.near_ties += int(np.sum(~same & tie))
        rep.checked += len(same)
        rep.count("draft_gap", len(same), np.sum(tie), np.sum(~same & tie))
        q = to_np(out["q_tok"][r])
        lse = to_np(out["lse_q"][r])
        ok = same  # values of a near-tie row refer to different tokens
        assert np.all(np.abs(q - od.q_tok[0])[ok] < PROB_TOL), (r, q, od.q_tok[0])
        assert np.all((np.abs(lse - od.lse[0]) / np.maximum(1, np.abs(od.lse[0])))[ok] < PROB_TOL)
        if "P" in out:
            assert np.abs(to_np(out["P"][r]) - od.P[0]).max() < PROB_TOL
    return rep


def compare_confidence(inp: dict, out: dict, reqs) -> None:
    sl = list(reqs)
    c, a = oracle.confidence(to_np(inp["h"][sl]), to_np(inp["W1"]), to_np(inp["w"]),
                             to_np(inp["x0"][sl]), to_np(out["x"][sl]), to_np(inp["sts_temp"]))
    assert np.abs(c - to_np(out["c"][sl])).max() < PROB_TOL
    assert np.abs(a - to_np(out["a"][sl])).max() < PROB_TOL


def compare_schedule(inp: dict, a_gpu: torch.Tensor, sched: dict, K: int, mode: int,
                     rep=None, threshold: float = 0.0) -> Report:
    rep = rep or Report()
    os_ = oracle.schedule(to_np(a_gpu).astype(np.float64), to_np(inp["sps"]).astype(np.float64),
                          inp["b_lo"], inp["b_step"], K, mode, threshold)
    stats = to_np(sched["stats"])
    if os_.margin < NEAR_TIE:
        # exempt: the decision is compared with a relative Theta step below the
        # margin, so record whether the two sides agreed but do not assert it
        same = (to_np(sched["ell"]) == os_.ell).all()
        rep.near_ties += 0 if same else 1
        rep.count("theta_step", 1, 1, 0 if same else 1)
        rep.notes.append(f"schedule near-tie margin {os_.margin:.3g} (agree: {same})")
        if not same:
            return rep
    else:
        rep.count("theta_step", 1)
    assert (to_np(sched["ell"]) == os_.ell).all()
    assert (to_np(sched["row_off"]) == os_.row_off).all()
    assert int(stats[0]) == os_.n and int(stats[1]) == os_.B
    assert abs(stats[2] - os_.tau) <= 1e-9 * max(1.0, abs(os_.tau))
    assert abs(stats[3] - os_.theta) <= 1e-9 * max(1.0, abs(os_.theta))
    if "order" in sched:
        assert (to_np(sched["order"]) == os_.order).all()
    rep.checked += 1
    return rep


def compare_draft_rnn(inp: dict, W: torch.Tensor, S: torch.Tensor, out: dict, seed: int, reqs,
                      rid_base: int = 0, rep=None) -> Report:
    """RNN head, stage-isolated per position: the oracle recomputes each state
    from the CUDA path's previous state and token, and draws each token from
    the CUDA path's state.  States: bf16 within one unit in the last place of
    the stored value (the pre-activation is summed in fp32 on the device and
    in fp64 by the oracle, so a value near a rounding boundary may round the
    other way), with at most 1% of them off; fp32 within 1e-5."""
    rep = rep or Report()
    A, Ct, Wn = to_np(inp["A"]), to_np(inp["Ct"]), to_np(W)
    bf16 = S.dtype == torch.bfloat16
    x_gpu, S_gpu = to_np(out["x"]), to_np(S)
    off = total = 0
    for r in reqs:
        od = oracle.draft_rnn(to_np(inp["U"][r:r + 1]), A, Ct, Wn, to_np(inp["x0"][r:r + 1]),
                              to_np(inp["draft_temp"]), seed, rid_base=rid_base + r, bf16_state=bf16,
                              x_cond=x_gpu[r:r + 1], s_cond=S_gpu[r:r + 1], want_P="P" in out)
        diff = np.abs(od.S[0] - S_gpu[r])
        if bf16:
            ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(od.S[0]), 1e-30))[1] - 8)
            assert np.all(diff <= ulp * 1.0000001), (r, diff.max())
            off += int(np.count_nonzero(diff))
        else:
            assert diff.max() < 1e-5, (r, diff.max())
        total += diff.size
        same = od.x[0] == x_gpu[r]
        tie = od.gap[0] < NEAR_TIE
        assert np.all(same | tie), (r, od.x[0], x_gpu[r], od.gap[0])
        rep.near_ties += int(np.sum(~same & tie))
        rep.checked += len(same)
        rep.count("draft_gap", len(same), np.sum(tie), np.sum(~same & tie))
        q, lse = to_np(out["q_tok"][r]), to_np(out["lse_q"][r])
        assert np.all(np.abs(q - od.q_tok[0])[same] < PROB_TOL), (r, q, od.q_tok[0])
        assert np.all((np.abs(lse - od.lse[0]) / np.maximum(1, np.abs(od.lse[0])))[same] < PROB_TOL)
        if "P" in out:
            assert np.abs(to_np(out["P"][r]) - od.P[0]).max() < PROB_TOL
    assert off <= 0.01 * total, (off, total)
    rep.notes.append(f"rnn states one ulp off: {off} of {total}")
    return rep


def compare_verify(inp: dict, d_out: dict, ell: torch.Tensor, v_out: dict, seed: int, mode: int,
                   reqs, target_temp: float = 1.0, rid_base: int = 0, rep=None,
                   S: torch.Tensor | None = None) -> Report:
    rep = rep or Report()
    tgt_all = inp["tgt"]
    V = tgt_all.shape[-1]
    G = (d_out["x"] if d_out is not None else inp["x"]).shape[1]
    row_off = to_np(inp["tgt_row_off"])
    ellv = to_np(ell)
    if mode != oracle.MODE_GREEDY:
        A, Ct, temps = to_np(inp["A"]), to_np(inp["Ct"]), to_np(inp["draft_temp"])
    for r in reqs:
        rows = to_np(tgt_all.reshape(-1, V)[row_off[r]: row_off[r] + ellv[r] + 1])
        x = to_np((d_out["x"] if d_out is not None else inp["x"])[r:r + 1])
        if mode == oracle.MODE_GREEDY:
            ov = oracle.verify(mode, rows, np.array([0]), ellv[r:r + 1], x, np.ones((1, G)), 1.0,
                               None, None, None, np.zeros(1, np.int32), np.ones(G), seed,
                               rid_base=rid_base + r)
        else:
            ov = oracle.verify(mode, rows, np.array([0]), ellv[r:r + 1], x,
                               to_np(d_out["q_tok"][r:r + 1]).astype(np.float64), target_temp,
                               to_np(inp["U"][r:r + 1]), A, Ct,
                               to_np(inp["x0"][r:r + 1]), temps, seed,
                               rid_base=rid_base + r,
                               S=None if S is None else to_np(S[r:r + 1]))
        got = to_np(v_out["out_tok"][r])
        if mode == oracle.MODE_GREEDY:
            rep.count("greedy_argmax", 1)
        differ = not (got == ov.out_tok[0]).all()
        near_acc, near_gap = ov.margin_acc[0] < NEAR_TIE, ov.margin_gap[0] < NEAR_TIE
        rep.count("accept_margin", np.isfinite(ov.margin_acc[0]), near_acc, differ and near_acc)
        rep.count("sample_gap", np.isfinite(ov.margin_gap[0]), near_gap,
                  differ and near_gap and not near_acc)
        if ov.margin[0] < NEAR_TIE and differ:
            rep.near_ties += 1
            rep.notes.append(f"verify near-tie r={r} margin={ov.margin[0]:.3g}")
            continue
        assert (got == ov.out_tok[0]).all(), (r, got, ov.out_tok[0], ov.margin[0])
        assert int(v_out["accept_len"][r]) == ov.accept_len[0]
        assert int(v_out["n_out"][r]) == ov.n_out[0]
        rep.checked += 1
        if "p_tok" in v_out and mode == oracle.MODE_SAMPLE:
            z = rows.astype(np.float64) / target_temp
            m = z.max(axis=1, keepdims=True)
            lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
            lse_gpu = to_np(v_out["lse_t"][r])[: ellv[r] + 1]
            assert np.all(np.abs(lse_gpu - lse) / np.maximum(1, np.abs(lse)) < PROB_TOL)
            for j in range(1, ellv[r] + 1):
                p = np.exp(z[j - 1, x[0, j - 1]] - lse[j - 1])
                assert abs(float(v_out["p_tok"][r, j - 1]) - p) < PROB_TOL
    return rep
