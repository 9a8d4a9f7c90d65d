"""Benchmark of one speculative-decoding round on GB300.

A step is one full round over one batch: draft (gamma sampling steps of the
Markov head, or of the RNN head with --head rnn, + confidence head), prefix
schedule, verification (rejection sampling, residual, bonus).  Default
workload: R=512 requests, gamma=11, V=129280, r=128, fp32 logits, bf16
factors, top-K cap 2048 (the largest configuration).
Inputs are synthetic and seeded (synth/), resident in HBM, larger than L2.

Metric: draft+verified positions per second = (R * gamma + B) / step time,
B = sum_r (1 + l_r) verify rows, summed over ranks (one replica per GPU).
Also reported: logit bytes per second of the dominant kernel against the
measured HBM copy bandwidth, the oracle on the host cores, an end-to-end
figure through host buffers, and SM clocks sampled during the timed region.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config c5]
Under torchrun every rank runs its own replica (weak scaling, no collective on
the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="c5", choices=["tiny", "c2", "c3", "c5", "c5p", "greedy"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--sched-mode", default="workload",
                   choices=["workload", "early_stop", "global", "threshold"],
                   help="scheduler admission rule (default: the workload's own)")
    p.add_argument("--sched-threshold", type=float, default=0.3,
                   help="survival threshold of --sched-mode threshold")
    p.add_argument("--accept-stats", action="store_true",
                   help="fold every round into the per-length acceptance EMA table")
    p.add_argument("--head", default="markov", choices=["markov", "rnn"],
                   help="sequential draft head: the Markov head, or the RNN head with a "
                        "recurrent state (synthetic recurrence W_k ~ N(0, 1/r))")
    p.add_argument("--async-cap", action="store_true",
                   help="cap each round's admissions by the uncapped count of the round two "
                        "earlier, kept on the device (the first two rounds use K); the c5 "
                        "workload's own cap, so its default")
    p.add_argument("--static-cap", action="store_true",
                   help="cap every round by the fixed K only (also for c5)")
    p.add_argument("--calibration", action="store_true",
                   help="also compute c* = sum min(p, q) of every verified row and fold the "
                        "round into the reliability diagram (ECE)")
    return p.parse_args()


def _workload(args):
    import dataclasses
    import synth
    wl = synth.WORKLOADS[args.config]
    if args.sched_mode != "workload":
        mode = {"early_stop": 0, "global": 1, "threshold": 2}[args.sched_mode]
        wl = dataclasses.replace(wl, sched_mode=mode, sched_threshold=args.sched_threshold)
    if args.head != "markov":
        if wl.mode == "greedy":
            raise SystemExit("--head applies to workloads with a draft stage")
        wl = dataclasses.replace(wl, head=args.head)
    static = getattr(args, "static_cap", False)
    if args.async_cap and static:
        raise SystemExit("--async-cap and --static-cap exclude each other")
    if args.async_cap:
        if wl.mode == "greedy":
            raise SystemExit("--async-cap applies to workloads with a schedule")
        wl = dataclasses.replace(wl, async_cap=True)
    elif not static and wl.name in ASYNC_CAP_WORKLOADS:
        # the workload's stated cap: top-K from the confidences of two rounds back
        wl = dataclasses.replace(wl, async_cap=True)
    return wl


# Workloads whose stated top-K cap is the asynchronous one (K_t from round t-2).
ASYNC_CAP_WORKLOADS = ("c5", "c5p")


# DRAM bytes (read + write) of one launch of the dominant kernel, taken with
# ncu on the same per-launch shape (R=512, V=129280, r=128, fp32 logits, one
# draft position; the committed draft-kernel profile gives the command),
# keyed by a hash of the kernel's sources: a changed kernel reports null until
# it is profiled again.
DRAFT_TC_SOURCES = ["draft_tc.cu", "draft_tc.cuh", "fused_tc.cuh", "tc.cuh", "common.cuh"]
MEASURED_TRAFFIC = {("c5", "2b875fbd8ee25322"): 298082560 + 4012800}
# Tensor-pipe utilisation (%, sm__pipe_tensor_cycles_active) of the same
# capture: the bias GEMM A_k[x] C_k on tcgen05, keyed the same way.
MEASURED_TENSOR_PIPE = {("c5", "2b875fbd8ee25322"): 8.44}


def _source_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "verify_sampling_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling SM clocks and throttle reasons every 10 ms.  It is
    started before the warm-up steps (so that it is running when the timed
    region starts) and keeps only the samples whose timestamps fall inside the
    timed region's wall-clock window."""

    INTERVAL_MS = 10

    def __init__(self, gpu_index: int):
        self.proc = None
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_bench_", suffix=".csv")
        self.f = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_QUERY}", "--format=csv",
                 "-lms", str(self.INTERVAL_MS)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            self.f.close()
            os.remove(self.path)

    def stop(self, t_start, t_end):
        """Samples taken between the datetimes t_start and t_end (local time,
        as nvidia-smi stamps them); the first one after t_start if the window
        holds none."""
        if self.proc is None:
            return None
        time.sleep(2.5 * self.INTERVAL_MS / 1000.0)  # let the sample after t_end arrive
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        import datetime
        rows = []
        with open(self.path) as f:
            lines = f.read().strip().splitlines()[1:]
        try:
            os.remove(self.path)
        except OSError:
            pass
        for ln in lines:
            c = [x.strip() for x in ln.split(",")]
            if len(c) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(c[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(c[2].split()[0]), float(c[3].split()[0]), c))
            except ValueError:
                continue
        inside = [r for r in rows if t_start <= r[0] <= t_end]
        if not inside:
            inside = [r for r in rows if r[0] >= t_start][:1]
        if not inside:
            return None
        sm = [r[1] for r in inside]
        mx = [r[2] for r in inside]
        reasons = set()
        for r in inside:
            c = r[3]
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if c[col].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "interval_ms": self.INTERVAL_MS,
                "window_ms": round((t_end - t_start).total_seconds() * 1000.0, 1),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------- reference ----
def _oracle_round(wl, inp_cpu, seed: int, n_req: int, chain=None) -> tuple[int, float]:
    """The oracle as it stands on a sub-batch of n_req requests of the workload:
    draft, confidence, schedule over the sub-batch, verify.  Returns
    (positions, seconds).  With the asynchronous cap, `chain` (a list kept by
    the caller) holds the uncapped counts of the earlier rounds."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    f = lambda t: t.float().numpy()
    G = wl.gamma
    if wl.mode == "greedy":  # verify only: every row of the sub-batch
        rows = f(inp_cpu["tgt"][:n_req]).reshape(-1, wl.V)
        x = inp_cpu["x"][:n_req].numpy()
        oracle.verify(oracle.MODE_GREEDY, rows, (np.arange(n_req) * (G + 1)).astype(np.int32),
                      inp_cpu["ell"][:n_req].numpy(), x, np.ones(x.shape), 1.0, None, None, None,
                      np.zeros(n_req, np.int32), np.ones(G), 0)
        return n_req * (G + 1), time.perf_counter() - t0
    U = f(inp_cpu["U"][:n_req])
    A, Ct = inp_cpu["A_np"], inp_cpu["Ct_np"]
    x0 = inp_cpu["x0"][:n_req].numpy()
    temps = inp_cpu["draft_temp"].numpy()
    S = None
    if wl.head == "rnn":
        d = oracle.draft_rnn(U, A, Ct, inp_cpu["Wrnn_np"], x0, temps, seed,
                             bf16_state=inp_cpu["A"].dtype == torch_bf16())
        S = d.S
    else:
        d = oracle.draft(U, A, Ct, x0, temps, seed)
    _, a = oracle.confidence(f(inp_cpu["h"][:n_req]), inp_cpu["W1_np"], inp_cpu["w_np"], x0, d.x,
                             inp_cpu["sts_temp"].numpy())
    K = max(1, round(wl.K * n_req / wl.R))
    if wl.async_cap and chain is not None:
        if len(chain) >= 2:
            K = min(K, chain[-2])
        chain.append(oracle.schedule(a, inp_cpu["sps"].numpy(), inp_cpu["b_lo"], inp_cpu["b_step"],
                                     n_req * G, wl.sched_mode, wl.sched_threshold).n)
    s = oracle.schedule(a, inp_cpu["sps"].numpy(), inp_cpu["b_lo"], inp_cpu["b_step"], K,
                        wl.sched_mode, wl.sched_threshold)
    rows = f(inp_cpu["tgt"][:n_req]).reshape(-1, wl.V)
    oracle.verify(oracle.MODE_SAMPLE, rows, (np.arange(n_req) * (G + 1)).astype(np.int32), s.ell,
                  d.x, d.q_tok, 1.0, U, A, Ct, x0, temps, seed, S=S)
    return n_req * G + s.B, time.perf_counter() - t0


def torch_bf16():
    import torch
    return torch.bfloat16


def _cpu_inputs(wl):
    import synth
    small = wl.scaled(R=min(wl.R, 8), K=max(1, round(wl.K * min(wl.R, 8) / wl.R)))
    inp = synth.make_inputs(small, "cpu", seed=wl.seed)
    if wl.mode != "greedy":  # the greedy workload has no draft stage
        inp["A_np"] = inp["A"].float().numpy()
        inp["Ct_np"] = inp["Ct"].float().numpy()
        inp["W1_np"] = inp["W1"].float().numpy()
        inp["w_np"] = inp["w"].float().numpy()
        if wl.head == "rnn":
            inp["Wrnn_np"] = synth.rnn_weights(small, "cpu").float().numpy()
    return inp


def _stages(wl, n: int) -> str:
    if wl.mode == "greedy":
        return "greedy verify of every row"
    return f"draft, confidence, schedule over the {n}, verify"


def cpu_baseline(wl, budget_s: float = 15.0) -> dict:
    """The oracle on sub-batches of 8 requests, fresh seeds, until ~budget_s."""
    inp = _cpu_inputs(wl)
    n = min(wl.R, 8)
    pos_tot, sec_tot, rounds = 0, 0.0, 0
    chain = []
    while sec_tot < budget_s and rounds < 1000:
        pos, sec = _oracle_round(wl, inp, 100 + rounds, n, chain)
        pos_tot, sec_tot, rounds = pos_tot + pos, sec_tot + sec, rounds + 1
    return {"value": pos_tot / sec_tot, "unit": "positions/s", "cores": 1, "kind": "oracle",
            "sample": f"{rounds} rounds of {n} of the {wl.R} requests of the same workload "
                      f"({_stages(wl, n)}), single-threaded fp64",
            "seconds": round(sec_tot, 3)}


def _cpu_worker(args):
    """One process of the all-cores oracle run: its own sub-batch inputs, then
    rounds with its own seeds until the budget is spent."""
    wl, wid, budget_s = args
    inp = _cpu_inputs(wl)
    n = min(wl.R, 8)
    pos_tot, sec_tot, rounds = 0, 0.0, 0
    chain = []
    while sec_tot < budget_s and rounds < 1000:
        pos, sec = _oracle_round(wl, inp, 100000 * (wid + 1) + rounds, n, chain)
        pos_tot, sec_tot, rounds = pos_tot + pos, sec_tot + sec, rounds + 1
    return pos_tot, sec_tot, rounds


def cpu_baseline_all_cores(wl, budget_s: float = 10.0) -> dict:
    """The same oracle rounds on every host core at once (one process per core,
    started with spawn): requests are independent, so sub-batches run side by
    side.  Throughput = all positions / the longest worker's time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_cpu_worker, [(wl, i, budget_s) for i in range(cores)])
    pos = sum(r[0] for r in res)
    sec = max(r[1] for r in res)
    return {"value": pos / sec, "unit": "positions/s", "cores": cores, "kind": "oracle",
            "sample": f"{sum(r[2] for r in res)} rounds of {min(wl.R, 8)} requests over {cores} "
                      "processes, single-threaded fp64 each",
            "seconds": round(sec, 3)}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = _cpu_inputs(wl)
    n = 2
    for i in range(args.warmup):
        _oracle_round(wl, inp, 100 + i, 1)
    tot_pos, tot_sec = 0, 0.0
    chain = []
    for i in range(args.steps):
        p, s = _oracle_round(wl, inp, 1000 + i, n, chain)
        tot_pos += p
        tot_sec += s
    value = tot_pos / tot_sec
    line = {"metric": "draft+verified positions/s", "value": value, "unit": "positions/s",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * tot_sec / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "positions/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} of {wl.R} requests per step ({_stages(wl, n)}); "
                                       f"the schedule runs over those {n} with K scaled to "
                                       f"them, so l_r (and B) come from a {n}-request "
                                       "schedule"},
            "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ replicas ----
def replica_layout(rank: int, wl) -> tuple[int, int]:
    """Rank `rank` runs its own batch of wl.R requests: input seed and global
    request id of its first request (Philox is keyed by global request ids, so
    the ranks' random streams never overlap)."""
    return wl.seed + rank, rank * wl.R


def combine_over_ranks(ms: float, positions: float, device, world: int) -> tuple[float, float]:
    """Whole-job figures of a replica run: the slowest rank's time and the
    positions of all ranks (all_reduce MAX and SUM; no-op for one rank)."""
    if world == 1:
        return ms, positions
    import torch
    import torch.distributed as dist
    tm = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tm, op=dist.ReduceOp.MAX)
    tp = torch.tensor([positions], dtype=torch.float64, device=device)
    dist.all_reduce(tp, op=dist.ReduceOp.SUM)
    return float(tm.item()), float(tp.item())


def _config(wl, world: int) -> dict:
    """The workload as reported in the JSON line (both arms)."""
    import torch
    return {"workload": wl.name, "R": wl.R, "gamma": wl.gamma, "V": wl.V, "r": wl.r, "K": wl.K,
            "logits": str(wl.logit_dtype).replace("torch.", ""),
            "factors": str(wl.fac_dtype).replace("torch.", ""),
            "l2": (f"inputs per step {_step_input_bytes(wl) / 1e6:.0f} MB, larger than L2 "
                   "(no flush)") if _step_input_bytes(wl) >= 2 * L2_BYTES else
                  "L2 flushed between timed steps (256 MB written)",
            "parallelism": f"replicas x{world}",
            **_sched_config(wl), **({"head": "rnn"} if wl.head == "rnn" else {})}


def _step_input_bytes(wl) -> int:
    """Logit and factor bytes one step reads: the padded target rows, and for
    workloads with a draft stage the backbone logits and C."""
    import torch
    es = lambda dt: 2 if dt == torch.bfloat16 else 4
    n = wl.R * (wl.gamma + 1) * wl.V * es(wl.logit_dtype)
    if wl.mode != "greedy":
        n += wl.R * wl.gamma * wl.V * es(wl.logit_dtype) + wl.gamma * wl.V * wl.r * es(wl.fac_dtype)
    return n


def _sched_config(wl) -> dict:
    names = {0: "early_stop", 1: "global", 2: "threshold"}
    out = {"sched_mode": names[wl.sched_mode]}
    if wl.sched_mode == 2:
        out["sched_threshold"] = wl.sched_threshold
    if wl.async_cap:
        out["async_cap"] = "K_t = uncapped n of round t-2"
    return out


# ------------------------------------------------------------------ ours ----
def main():
    args = _args()
    import synth
    wl = _workload(args)
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import torch.distributed as dist
    import verify_sampling_gb300 as vs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    seed_in, rid_base = replica_layout(rank, wl)
    g = synth.make_inputs(wl, dev, seed=seed_in)
    greedy = wl.mode == "greedy"
    din = None if greedy else synth.draft_inputs(g, request_id_base=rid_base)
    R, G, V = wl.R, wl.gamma, wl.V
    rnn = wl.head == "rnn"
    if rnn:  # the recurrence is a weight (resident); S is written by the draft, read by verify
        din.Wrnn = synth.rnn_weights(wl, dev, seed=seed_in)
        din.S = torch.empty(R, G, wl.r, dtype=wl.fac_dtype, device=dev)
    stats_hist = torch.zeros(max(1, args.steps), 4, dtype=torch.float64, device=dev)
    # per timed step: l_r and accept_len (residual rows = requests rejected at j <= l_r)
    acc_hist = torch.zeros(max(1, args.steps), 2, R, dtype=torch.int32, device=dev)
    # inputs read per step; below twice the L2 size the L2 is flushed between
    # timed steps (outside their events)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) \
        if _step_input_bytes(wl) < 2 * L2_BYTES else None

    bufs = {}
    if not greedy:
        bufs["draft"] = vs.draft_outputs(R, G, V, dev)
        bufs["ws_draft"] = torch.empty(vs.workspace_bytes(vs.STAGE_DRAFT, R, G, V, wl.r),
                                       dtype=torch.uint8, device=dev)
    bufs["ws_verify"] = torch.empty(vs.workspace_bytes(vs.STAGE_VERIFY, R, G, V), dtype=torch.uint8,
                                    device=dev)
    acc_tab = None
    if args.accept_stats and not greedy:
        acc_tab = {"ema": torch.zeros(1, G, dtype=torch.float64, device=dev),
                   "count": torch.zeros(1, G, dtype=torch.int64, device=dev),
                   "estimate": torch.zeros(G, dtype=torch.float64, device=dev)}
    calib = vs.calibration_tables(10, dev) if args.calibration and not greedy else None
    # asynchronous cap: word t % 2 holds the uncapped count of round t - 2
    cap_words = torch.full((2,), wl.K, dtype=torch.int32, device=dev) if wl.async_cap else None
    stream = torch.cuda.current_stream()
    nev = max(1, args.steps)
    ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
          for k in ("d0", "d1", "s1", "v1")}

    def step(i: int, timed: bool):
        seed = 7000 + i
        if greedy:
            if timed:
                ev["d0"][i].record(stream)
            bufs["verify"] = vs.verify(vs.VERIFY_GREEDY, g["tgt"].view(-1, V), g["tgt_row_off"],
                                       g["ell"], g["x"], seed, out=bufs.get("verify"),
                                       workspace=bufs["ws_verify"])
            if timed:
                ev["v1"][i].record(stream)
                acc_hist[i, 0].copy_(g["ell"], non_blocking=True)
                acc_hist[i, 1].copy_(bufs["verify"]["accept_len"], non_blocking=True)
            return
        if timed:
            ev["d0"][i].record(stream)
        d = vs.draft_sample(din, seed, out=bufs["draft"], workspace=bufs["ws_draft"])
        if timed:
            ev["d1"][i].record(stream)
        word = cap_words[i % 2: i % 2 + 1] if cap_words is not None else None
        s = vs.schedule(d["a"], g["sps"], g["b_lo"], g["b_step"], wl.K, wl.sched_mode,
                        threshold=wl.sched_threshold, K_dev=word, n_free=word,
                        out=bufs.get("sched"))
        bufs["sched"] = s
        if timed:
            ev["s1"][i].record(stream)
        v = vs.verify(vs.VERIFY_SAMPLE, g["tgt"].view(-1, V), g["tgt_row_off"], s["ell"], d["x"],
                      seed, q_tok=d["q_tok"], lse_q=d["lse_q"], draft=din,
                      request_id_base=rid_base, want_cstar=calib is not None,
                      out=bufs.get("verify"), workspace=bufs["ws_verify"])
        bufs["verify"] = v
        if acc_tab is not None:
            vs.accept_stats(s["ell"], v["accept_len"], acc_tab["ema"], acc_tab["count"], 0, 0.1,
                            estimate=acc_tab["estimate"])
        if calib is not None:
            vs.calibration(d["c"], s["ell"], v["accept_len"], calib)
        if timed:
            ev["v1"][i].record(stream)
            stats_hist[i].copy_(s["stats"], non_blocking=True)
            acc_hist[i, 0].copy_(s["ell"], non_blocking=True)
            acc_hist[i, 1].copy_(v["accept_len"], non_blocking=True)

    import datetime
    clocks = ClockSampler(local) if rank == 0 else None
    try:
        for i in range(args.warmup):
            step(-1 - i, False)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        wall0 = datetime.datetime.now()
        t0.record(stream)
        for i in range(args.steps):
            if flush is not None:  # evict the previous step's inputs (not timed)
                flush.zero_()
            step(i, True)
        t1.record(stream)
        torch.cuda.synchronize()
        wall1 = datetime.datetime.now()
    except BaseException:
        if clocks is not None and clocks.proc is not None:
            clocks.proc.kill()
        raise
    if world > 1:
        dist.barrier()
    clk = clocks.stop(wall0, wall1) if clocks else None
    stage_ms = {"draft": 0.0, "schedule": 0.0, "verify": 0.0}
    step_ms = 0.0
    for i in range(args.steps):
        step_ms += ev["d0"][i].elapsed_time(ev["v1"][i])
        if not greedy:
            stage_ms["draft"] += ev["d0"][i].elapsed_time(ev["d1"][i])
            stage_ms["schedule"] += ev["d1"][i].elapsed_time(ev["s1"][i])
            stage_ms["verify"] += ev["s1"][i].elapsed_time(ev["v1"][i])
        else:
            stage_ms["verify"] += ev["d0"][i].elapsed_time(ev["v1"][i])
    # with inputs larger than L2 the whole region is timed; with the flush,
    # the steps' own events (the flushes between them are left out)
    ms = t0.elapsed_time(t1) if flush is None else step_ms
    if greedy:
        B_sum = float(args.steps * R * (G + 1))
        positions = B_sum
    else:
        B_sum = float(stats_hist[:, 1].sum())
        positions = args.steps * R * G + B_sum
    ms_max, pos_all = combine_over_ranks(ms, positions, dev, world)
    value = pos_all / (ms_max / 1000.0)

    # ------------------------------------------------ roofline (rank 0) ----
    hbm, peak_kind = _peaks()
    es_u = 4 if wl.logit_dtype == torch.float32 else 2
    es_f = 4 if wl.fac_dtype == torch.float32 else 2
    stage_bytes = _round_bytes(wl, to_cpu(acc_hist), args.steps)
    if greedy:
        # the rows up to each request's first mismatch (or row l_r + 1)
        per_launch = int(stage_bytes["verify"])
        dur_ms = ms / args.steps
        kernel = "verify_rows (greedy argmax; rows past a request's first mismatch skipped)"
        launches = 2  # row plan, row pass
    else:
        # dominant kernel: the draft step, gamma launches per round; one launch
        # streams the R backbone rows of position k and the factor C_k.
        per_launch = R * V * es_u + V * wl.r * es_f
        dur_ms = stage_ms["draft"] / (args.steps * G)
        kernel = "draft_step (one launch per position k)"
        # per round: gamma draft steps, confidence, schedule, verify row plan,
        # verify rows, fused residual, residual fallback (gated, exits at once
        # when unused); the EMA update; the c* plan, c* pass and diagram
        launches = G + 6 + (1 if acc_tab is not None else 0) + (3 if calib is not None else 0)
        if rnn:  # the state kernel before every draft step
            launches += G
            kernel = "draft_step (one launch per position k; RNN head, state rows gathered)"
    achieved = per_launch / (dur_ms / 1000.0) / 1e9
    # measured on the Markov head's launch (the RNN head's gathers other rows)
    src = _source_hash(DRAFT_TC_SOURCES)
    traffic = None if greedy or rnn else MEASURED_TRAFFIC.get((wl.name, src))
    tensor_pipe = None if greedy or rnn else MEASURED_TENSOR_PIPE.get((wl.name, src))
    roofline = {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": hbm,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "frac_of_8tbs": round(achieved / 8000.0, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": per_launch,
                # DRAM bytes the profiler counted per launch over the same
                # event-timed duration (null with traffic)
                "achieved_dram": None if traffic is None else round(traffic / (dur_ms / 1000.0) / 1e9, 1),
                # tcgen05 pipe utilisation of the bias GEMM in the same capture
                "tensor_pipe_pct": tensor_pipe}

    # ---------------------------------------- round-level algorithmic bytes ----
    round_bytes = sum(stage_bytes.values())
    stages = {}
    for k in ("draft", "schedule", "verify"):
        ms_k = stage_ms[k] / args.steps
        st = {"ms": round(ms_k, 4)}
        if stage_bytes.get(k):
            st["algorithmic_bytes"] = int(stage_bytes[k])
            st["gbs"] = round(stage_bytes[k] / (ms_k / 1000.0) / 1e9, 1)
            st["frac"] = round(st["gbs"] / hbm, 4)
        stages[k] = st
    round_gbs = round_bytes / (ms_max / args.steps / 1000.0) / 1e9
    round_logit = {"algorithmic_bytes_per_step": int(round_bytes), "gbs": round(round_gbs, 1),
                   "frac": round(round_gbs / hbm, 4), "frac_of_8tbs": round(round_gbs / 8000.0, 4),
                   "floor_ms": round(round_bytes / (hbm * 1e9) * 1000.0, 4)}

    line = {"metric": "draft+verified positions/s", "value": value, "unit": "positions/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if es_u == 4 else "bf16", "data": "synthetic",
            "config": {**_config(wl, world),
                       **({"accept_stats": True} if acc_tab is not None else {}),
                       **({"calibration": True} if calib is not None else {})},
            "stage_ms_per_step": {k: round(v / args.steps, 4) for k, v in stage_ms.items()},
            "stages": stages, "round_logit_gbs": round_logit,
            "mean_verify_rows": B_sum / args.steps,
            "roofline": roofline, "gpu_launches": launches * args.steps, "clocks": clk}
    if calib is not None:
        line["ece"] = float(calib["ece"].item())

    # ----------------------------------------------------- e2e (rank 0) ----
    if rank == 0 and not args.no_e2e and not greedy:
        # one round at a time, and two in flight on two streams: which is faster
        # depends on how the host link serves copy-engine transfers and the
        # gather's loads at once (it differed between machines); both are
        # measured and reported, the faster one as the value
        runs = [_e2e(wl, g, din, vs, torch, dev, bufs, rid_base, steps=min(args.steps, 8),
                     cap_words=cap_words, in_flight=n) for n in (1, 2)]
        best = min(runs, key=lambda e: e["ms_per_step"])
        best["ms_per_step_by_rounds_in_flight"] = {str(e["rounds_in_flight"]): e["ms_per_step"]
                                                   for e in runs}
        line["e2e"] = best
    if rank == 0 and not args.no_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


L2_BYTES = 129 * 2 ** 20


def to_cpu(t):
    return t.cpu().numpy()


def _round_bytes(wl, acc_hist, steps: int) -> dict:
    """Algorithmic bytes of one round, per stage, averaged over the timed steps.
    draft: gamma launches of the R backbone rows and C_k, plus the confidence
    head's hidden states and W1 rows; verify: the target rows a verifier must
    read -- each request's rows up to its end, accept_len + 1 of them (its
    first rejection or mismatch, or row l_r + 1) -- and, for every request
    rejected at j*, its backbone row at j* plus C_{j*} once per position that
    has a rejection (the residual pass)."""
    import numpy as np
    import torch
    es = lambda dt: 2 if dt == torch.bfloat16 else 4
    R, G, V, r = wl.R, wl.gamma, wl.V, wl.r
    e_u, e_f, e_c = es(wl.logit_dtype), es(wl.fac_dtype), es(wl.conf_dtype)
    rows = resid = 0.0
    for i in range(steps):
        ell, acc = acc_hist[i, 0], acc_hist[i, 1]
        rows += float((acc + 1).sum())
        if wl.mode != "greedy":
            rej = acc < ell
            resid += int(rej.sum()) * V * e_u + len(np.unique(acc[rej] + 1)) * V * r * e_f
    verify = (rows * V * e_u + resid) / steps
    if wl.mode == "greedy":
        return {"verify": verify}
    draft = G * (R * V * e_u + V * r * e_f) + R * G * (wl.d + wl.e) * e_c
    return {"draft": draft, "verify": verify}


def _link_gbs(torch, src, dev) -> float:
    """Host-to-device bandwidth of one copy of `src` (pinned) into the device."""
    dst = torch.empty(src.shape, dtype=src.dtype, device=dev)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    e0.record(s)
    dst.copy_(src, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize()
    return src.numel() * src.element_size() / (e0.elapsed_time(e1) / 1000.0) / 1e9


def _e2e(wl, g, din, vs, torch, dev, bufs, rid_base, steps: int, cap_words=None,
         in_flight: int = 2) -> dict:
    """Same round through the public API (one spec_round_host call per step)
    with the per-step inputs taken from pinned host memory and the results
    (tokens, lengths, stats) copied back; the model weights (A, Ct, W1, w) stay
    resident.  U, h and x0 are copied whole.  Of the target logits, held on the
    host for every candidate row [R, gamma + 1, V], only the B rows the
    schedule admits are read -- the rows a target model computes for the
    round -- by the library's gather from the mapped host buffer.

    `in_flight` rounds are in flight, on as many streams with their own device
    buffers: while one round computes, the next one's inputs cross the link.
    Step i's results are read on the host before step i + in_flight reuses
    its buffers."""
    names = ["U", "h", "x0", "tgt"]
    host = {n: g[n].cpu().pin_memory() for n in names}
    whole = sum(host[n].numel() * host[n].element_size() for n in ("U", "h", "x0"))
    row_bytes = wl.V * host["tgt"].element_size()
    R, G, V = wl.R, wl.gamma, wl.V
    streams = [torch.cuda.Stream(device=dev) for _ in range(in_flight)]
    sets = []
    for _ in range(in_flight):
        devb = {n: torch.empty_like(g[n]) for n in names}
        outs = {"out_tok": torch.empty(R, G + 1, dtype=torch.int32).pin_memory(),
                "accept_len": torch.empty(R, dtype=torch.int32).pin_memory(),
                "n_out": torch.empty(R, dtype=torch.int32).pin_memory(),
                "stats": torch.empty(4, dtype=torch.float64).pin_memory()}
        d_in = vs.DraftInputs(U=devb["U"], A=g["A"], Ct=g["Ct"], x0=devb["x0"],
                              draft_temp=g["draft_temp"], h=devb["h"], W1=g["W1"], w=g["w"],
                              sts_temp=g["sts_temp"], request_id_base=rid_base, Wrnn=din.Wrnn,
                              S=None if din.S is None else torch.empty_like(din.S))
        b = {"draft": vs.draft_outputs(R, G, V, dev),
             "ws_draft": torch.empty_like(bufs["ws_draft"]),
             "ws_verify": torch.empty_like(bufs["ws_verify"]),
             "sched": {"ell": torch.empty(R, dtype=torch.int32, device=dev),
                       "row_off": torch.empty(R + 1, dtype=torch.int32, device=dev),
                       "stats": torch.empty(4, dtype=torch.float64, device=dev)},
             "verify": {"accept_len": torch.empty(R, dtype=torch.int32, device=dev),
                        "out_tok": torch.empty(R, G + 1, dtype=torch.int32, device=dev),
                        "n_out": torch.empty(R, dtype=torch.int32, device=dev)}}
        sets.append((devb, outs, d_in, b))
    d2h = sum(t.numel() * t.element_size() for t in sets[0][1].values())
    torch.cuda.synchronize()

    def issue(i):
        # one C-ABI call: host inputs in, host results out (asynchronous)
        devb, outs, d_in, b = sets[i % in_flight]
        vs.run_round_host(d_in, devb["tgt"].view(-1, V), g["tgt_row_off"], g["sps"], g["b_lo"],
                          g["b_step"], wl.K, 9000 + i, host_in=host, host_out=outs,
                          sched_mode=wl.sched_mode, sched_threshold=wl.sched_threshold,
                          tgt_scheduled_only=True,
                          K_dev=None if cap_words is None else cap_words[i % 2: i % 2 + 1],
                          n_free=None if cap_words is None else cap_words[i % 2: i % 2 + 1],
                          bufs=b, stream=streams[i % in_flight])

    def collect(i):
        streams[i % in_flight].synchronize()
        B = float(sets[i % in_flight][1]["stats"][1])
        return R * G + B, B

    for i in range(in_flight):  # warm-up
        issue(i)
    for i in range(in_flight):
        collect(i)
    t0 = time.perf_counter()
    res = []
    for i in range(steps):
        if i >= in_flight:
            res.append(collect(i - in_flight))
        issue(i)
    for i in range(max(0, steps - in_flight), steps):
        res.append(collect(i))
    sec = time.perf_counter() - t0
    pos = sum(p for p, _ in res)
    B_mean = sum(b for _, b in res) / steps
    h2d = int(whole + B_mean * row_bytes)
    link = _link_gbs(torch, host["U"], dev)
    return {"value": pos / sec, "unit": "positions/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "rounds_in_flight": in_flight, "ms_per_step": round(1000.0 * sec / steps, 3),
            # one pinned copy of U's size, timed right after: the link's own rate,
            # and the step time that rate alone would give for the step's bytes
            "link_gbs": round(link, 1), "link_floor_ms": round(h2d / (link * 1e9) * 1000.0, 3),
            "target_rows": "the B scheduled rows of each step (mean %.1f), read from the "
                           "pinned [R, gamma+1, V] host array" % B_mean}


if __name__ == "__main__":
    main()
