"""Seeded synthetic workloads for the speculative-decoding round.

This module only draws inputs: random logits, factors, hidden states, tables and
planted structure.  It holds none of the method's arithmetic (no softmax, no
sampling, no schedule, no verification), so the CUDA library and the oracle
can both consume what it produces.  The pages measure on models and datasets
(Qwen3, DeepSeek-V4, ShareGPT, HumanEval, GSM8K, Alpaca) that are not
available here; these workloads stand in for them with the shapes named below.

Workloads (R requests, gamma draft positions, V vocabulary, r bias rank,
d hidden size, e Markov-embedding size):

  tiny     R=4   gamma=4  V=1000    r=8   fp32 logits and factors
  c2       R=64  gamma=8  V=151936  r=64  bf16, planted +8 peak, target noise
                                          tuned to ~70% acceptance at j=1
  c3       R=256 gamma=16 V=151936  r=64  bf16, acceptance ~0.8*0.95^(k-1),
                                          saw-tooth SPS, STS temps 1..2
  greedy   R=256 gamma=11 V=129280        bf16 target N(0,3) (ties at the row
                                          maximum arise from the rounding); drafts
                                          equal the lowest-index argmax w.p. 0.9^k
  c5       R=512 gamma=11 V=129280 r=128  fp32 logits N(0,4), Zipf(1.1) target
                                          over U's rank, top-K cap 2048
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
CALIBRATION = os.path.join(_HERE, "calibration.json")


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    r: int
    d: int
    e: int
    logit_dtype: torch.dtype
    fac_dtype: torch.dtype
    conf_dtype: torch.dtype
    mode: str            # "sample" (full round) or "greedy" (verify only)
    K: int
    sched_mode: int      # 0 early stop, 1 global, 2 static threshold
    target: str          # "noise", "zipf" or "planted_argmax"
    sps_kind: str        # "linear16", "linear", "sawtooth"
    u_std: float
    peak: float
    seed: int
    sts_ramp: bool = False
    sched_threshold: float = 0.0  # read by the static-threshold mode only
    head: str = "markov"          # sequential head: "markov" or "rnn" (rnn_weights)
    async_cap: bool = False       # cap round t by the uncapped count of round t - 2

    def scaled(self, **kw) -> "Workload":
        """Same recipe at other sizes (for parity cases the oracle finishes quickly).
        Unless given, K keeps its share of the R * gamma candidates."""
        w = replace(self, **kw)
        if "K" not in kw:
            share = self.K / (self.R * self.gamma)
            w = replace(w, K=max(1, min(w.R * w.gamma, round(share * w.R * w.gamma))))
        return w


WORKLOADS = {
    "tiny": Workload("tiny", 4, 4, 1000, 8, 64, 8, torch.float32, torch.float32, torch.float32,
                     "sample", 16, 0, "noise", "linear16", 2.0, 0.0, 0),
    "c2": Workload("c2", 64, 8, 151936, 64, 2048, 64, torch.bfloat16, torch.bfloat16,
                   torch.bfloat16, "sample", 512, 0, "noise", "linear", 3.0, 8.0, 2),
    "c3": Workload("c3", 256, 16, 151936, 64, 2048, 64, torch.bfloat16, torch.bfloat16,
                   torch.bfloat16, "sample", 4096, 0, "noise", "sawtooth", 3.0, 8.0, 3,
                   sts_ramp=True),
    "greedy": Workload("greedy", 256, 11, 129280, 1, 0, 0, torch.bfloat16, torch.bfloat16,
                       torch.bfloat16, "greedy", 2816, 0, "planted_argmax", "linear", 3.0, 0.0, 4),
    "c5": Workload("c5", 512, 11, 129280, 128, 2048, 128, torch.float32, torch.bfloat16,
                   torch.bfloat16, "sample", 2048, 0, "zipf", "sawtooth", 4.0, 0.0, 5),
}
# Profiling case: the c5 per-launch shape (R=512, V=129280, r=128, fp32) with two
# draft positions, small enough for a multi-pass profiler capture (~1.3 GB).
WORKLOADS["c5p"] = WORKLOADS["c5"].scaled(name="c5p", gamma=2)


def _calibration() -> dict:
    if os.path.exists(CALIBRATION):
        with open(CALIBRATION) as f:
            return json.load(f)
    return {}


def target_noise_std(wl: Workload) -> list[float]:
    """Per-position std of the target noise (from calibration.json, else a default)."""
    cal = _calibration().get(wl.name)
    if cal is not None:
        return [float(s) for s in cal["sigma_t"]]
    return [0.5] * (wl.gamma + 1)


def sps_table(wl: Workload):
    """SPS lookup table (float32 values at B_i = b_lo + i * b_step)."""
    R, g = wl.R, wl.gamma
    if wl.sps_kind == "linear16":
        i = np.arange(16, dtype=np.float64)
        return (1000.0 * (1.0 - 0.04 * i)).astype(np.float32), float(R), 1.0
    if wl.sps_kind == "linear":
        n = R * g + 1
        i = np.arange(n, dtype=np.float64)
        return (1000.0 * (1.0 - 0.5 * i / max(1, R * g))).astype(np.float32), float(R), 1.0
    # saw-tooth: steps/s of a 10 ms + 2 us/row forward, +20% ramp inside every 256-row window
    B = np.arange(1, R * (g + 1) + 1, dtype=np.float64)
    sps = 1.0 / (0.010 + 2e-6 * B) * (1.0 + 0.2 * ((B % 256) / 256.0))
    return sps.astype(np.float32), 1.0, 1.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std)


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input of one round.  Returns a dict of tensors on `device`:
    U, A, Ct, x0, draft_temp, h, W1, w, sts_temp (draft), tgt [R, gamma+1, V] with
    tgt_row_off (padded layout), sps/b_lo/b_step/K, and for the greedy workload
    the planted drafts x and l_r = gamma."""
    seed = wl.seed if seed is None else seed
    g = _gen(seed, device)
    R, G, V, r, d, e = wl.R, wl.gamma, wl.V, wl.r, wl.d, wl.e
    out: dict = {"workload": wl}
    sps, b_lo, b_step = sps_table(wl)
    out.update(sps=torch.from_numpy(sps).to(device), b_lo=b_lo, b_step=b_step, K=wl.K)
    out["tgt_row_off"] = (torch.arange(R, dtype=torch.int32, device=device) * (G + 1))

    if wl.mode == "greedy":
        # Target rows N(0,3) in the logit dtype, nothing clipped or planted: at
        # bf16 resolution about one row in ten has its maximum at more than one
        # token.  To plant the drafts, the generator finds each row's maximum
        # at the lowest index (a torch reduction; the verifier and the oracle
        # each find it on their own).  The draft keeps that token w.p. 0.9^k
        # and otherwise takes a uniformly drawn different token, which may be
        # another index of a tied maximum.
        tgt = _randn((R, G + 1, V), g, device, wl.u_std).to(wl.logit_dtype)
        top = torch.empty((R, G), dtype=torch.int64, device=device)
        idx = torch.arange(V, device=device, dtype=torch.int32)
        for r0 in range(0, R, 16):
            t = tgt[r0:r0 + 16, :G].float()
            at_max = t == t.amax(dim=2, keepdim=True)
            top[r0:r0 + 16] = torch.where(at_max, idx, V).amin(dim=2)
        keep = torch.rand((R, G), generator=g, device=device) < \
            (0.9 ** torch.arange(1, G + 1, device=device, dtype=torch.float32))
        other = (top + torch.randint(1, V, (R, G), generator=g, device=device)) % V
        x = torch.where(keep, top, other).to(torch.int32)
        out.update(tgt=tgt, x=x, ell=torch.full((R,), G, dtype=torch.int32, device=device))
        return out

    # draft head inputs
    U = _randn((R, G, V), g, device, wl.u_std)
    if wl.peak:
        pk = torch.randint(0, V, (R, G), generator=g, device=device)
        U.scatter_add_(2, pk.unsqueeze(-1), torch.full((R, G, 1), wl.peak, device=device))
    A = _randn((G, V, r), g, device, 1.0 / math.sqrt(r))
    Ct = _randn((G, V, r), g, device, 0.5)
    x0 = torch.randint(0, V, (R,), generator=g, device=device, dtype=torch.int32)
    # confidence head: h ~ N(0,1) with h[...,0] = 2 - 0.25 (k-1); w_0 = 1,
    # other w ~ N(0, 1/(d+e)); W1 ~ N(0,1)
    h = _randn((R, G, d), g, device)
    if d > 0:
        h[:, :, 0] = 2.0 - 0.25 * torch.arange(G, device=device, dtype=torch.float32)
    W1 = _randn((V, e), g, device)
    w = _randn((d + e,), g, device, 1.0 / math.sqrt(max(1, d + e)))
    if d + e > 0:
        w[0] = 1.0
    sts = (1.0 + torch.arange(G, device=device, dtype=torch.float32) / max(1, G - 1)) \
        if wl.sts_ramp else torch.ones(G, device=device)
    Ub = U.to(wl.logit_dtype)
    out.update(U=Ub, A=A.to(wl.fac_dtype), Ct=Ct.to(wl.fac_dtype), x0=x0,
               draft_temp=torch.ones(G, device=device), h=h.to(wl.conf_dtype),
               W1=W1.to(wl.conf_dtype), w=w.to(wl.conf_dtype), sts_temp=sts)

    # target rows 1..gamma+1 (row gamma+1 is a fresh backbone-like row)
    extra = _randn((R, 1, V), g, device, wl.u_std)
    base = torch.cat([Ub.float(), extra], dim=1)
    if wl.target == "zipf":
        # L_t[v] = -1.1 ln rank(v), rank 1 = largest backbone logit of the row
        order = torch.argsort(base, dim=2, descending=True)
        ranks = torch.empty_like(order)
        ranks.scatter_(2, order, torch.arange(1, V + 1, device=device).expand(R, G + 1, V))
        tgt = -1.1 * torch.log(ranks.to(torch.float32))
    else:
        sig = torch.tensor(target_noise_std(wl)[: G + 1], device=device, dtype=torch.float32)
        tgt = base + _randn((R, G + 1, V), g, device) * sig.view(1, G + 1, 1)
    out["tgt"] = tgt.to(wl.logit_dtype)
    return out


def rnn_weights(wl: Workload, device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    """Recurrence matrices W_k of the RNN sequential head: [gamma, r, r], entries
    N(0, 1/r) (unit gain on a random state), in the workload's factor dtype.
    Drawn from their own stream (seed + 1), so the round's other inputs are the
    same as for the Markov head."""
    seed = wl.seed if seed is None else seed
    g = _gen(seed + 1, device)
    return _randn((wl.gamma, wl.r, wl.r), g, device, 1.0 / math.sqrt(wl.r)).to(wl.fac_dtype)


def draft_inputs(inp: dict, request_id_base: int = 0):
    """The library's DraftInputs view of a make_inputs() dict (device tensors)."""
    from verify_sampling_gb300 import DraftInputs
    return DraftInputs(U=inp["U"], A=inp["A"], Ct=inp["Ct"], x0=inp["x0"],
                       draft_temp=inp["draft_temp"], h=inp["h"], W1=inp["W1"], w=inp["w"],
                       sts_temp=inp["sts_temp"], request_id_base=request_id_base)
