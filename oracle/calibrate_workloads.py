"""Calibrate the target-noise levels of the synthetic workloads with the oracle.

Writes synth/calibration.json: for each noise-target workload the per-position
standard deviation sigma_t of the noise added to the backbone logits so that the
acceptance probability of one draft token, sum_v min(p_v, q_v) (the oracle's
accept_prob), averaged over a few requests, hits the workload's target:
  c2  ~0.70 at every position (tuned at position 1)
  c3  0.8 * 0.95^(k-1) at position k
The draft distributions q come from the oracle's draft head on the same
synthetic inputs; only the oracle computes anything here.

Usage: python oracle/calibrate_workloads.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

TARGETS = {
    "c2": lambda k: 0.70,
    "c3": lambda k: 0.8 * 0.95 ** (k - 1),
}


def _bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def calibrate(name: str, n_req: int = 4, seed: int = 1) -> dict:
    wl = synth.WORKLOADS[name].scaled(R=n_req)
    inp = synth.make_inputs(wl, "cpu", seed=seed)
    U = inp["U"].float().numpy()
    d = oracle.draft(U, inp["A"].float().numpy(), inp["Ct"].float().numpy(), inp["x0"].numpy(),
                     inp["draft_temp"].numpy(), seed=seed, want_P=True)
    rng = np.random.default_rng(seed)
    sig, acc = [], []
    for k in range(1, wl.gamma + 1):
        target = TARGETS[name](k)
        noise = rng.standard_normal((n_req, wl.V))
        logq = np.log(np.maximum(d.P[:, k - 1], 1e-300))

        def mean_acc(s):
            return float(np.mean([oracle.accept_prob(_bf16(U[r, k - 1] + s * noise[r]), logq[r])
                                  for r in range(n_req)]))

        lo, hi = 0.0, 8.0
        for _ in range(30):
            mid = 0.5 * (lo + hi)
            if mean_acc(mid) > target:
                lo = mid
            else:
                hi = mid
        s = 0.5 * (lo + hi)
        sig.append(round(s, 5))
        acc.append(round(mean_acc(s), 4))
        print(f"{name} k={k}: sigma_t={s:.4f} acceptance={acc[-1]:.4f} (target {target:.4f})",
              flush=True)
        if name == "c2":  # one level for every position
            sig = [sig[0]] * wl.gamma
            acc = [acc[0]] * wl.gamma
            break
    sig.append(sig[-1])  # bonus row gamma + 1
    return {"sigma_t": sig, "acceptance": acc, "requests": n_req, "seed": seed}


def main():
    out = {}
    if os.path.exists(synth.CALIBRATION):
        with open(synth.CALIBRATION) as f:
            out = json.load(f)
    for name in (sys.argv[1:] or list(TARGETS)):
        out[name] = calibrate(name)
    with open(synth.CALIBRATION, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", synth.CALIBRATION)


if __name__ == "__main__":
    main()
