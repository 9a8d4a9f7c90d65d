"""Multi-process host logic, on CPU with the gloo backend (world size 2).

The benchmark runs one replica per GPU: each rank drafts, schedules and
verifies its own batch of requests, keyed by global request ids, and rank 0
reports the slowest rank's time and the positions of all ranks.  These tests
cover that logic without a GPU:

  * replica_layout gives every rank a disjoint range of global request ids;
  * combine_over_ranks takes the MAX of the step times and the SUM of the
    positions;
  * a batch split over two ranks by request (each rank runs the oracle on its
    shard with request_id_base = its first global id, the survivals are
    all-gathered so that every rank runs the same schedule, and each rank
    verifies its own shard) gives exactly the tokens, lengths and schedule of
    the whole batch in one process -- the property that makes request
    sharding free of any collective other than that one all-gather.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank: int, port: int):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)


def _round(inp, wl, lo, hi, rid_base, seed, a_all=None, W=None):
    """Oracle draft + confidence on requests [lo, hi); schedule over a_all (or
    the shard's own survivals); verify the shard.  W: the RNN head's
    recurrence (None: the Markov head)."""
    f = lambda t: t.float().numpy()
    U = f(inp["U"][lo:hi])
    A, Ct = f(inp["A"]), f(inp["Ct"])
    x0 = inp["x0"][lo:hi].numpy()
    temps = inp["draft_temp"].numpy()
    S = None
    if W is None:
        d = oracle.draft(U, A, Ct, x0, temps, seed, rid_base=rid_base)
    else:
        d = oracle.draft_rnn(U, A, Ct, W, x0, temps, seed, rid_base=rid_base, bf16_state=False)
        S = d.S
    _, a = oracle.confidence(f(inp["h"][lo:hi]), f(inp["W1"]), f(inp["w"]), x0, d.x,
                             inp["sts_temp"].numpy())
    s = oracle.schedule(a if a_all is None else a_all, inp["sps"].numpy(), inp["b_lo"],
                        inp["b_step"], wl.K, wl.sched_mode)
    G, V = wl.gamma, wl.V
    ell = s.ell[lo:hi] if a_all is not None else s.ell
    rows = f(inp["tgt"][lo:hi]).reshape(-1, V)
    v = oracle.verify(oracle.MODE_SAMPLE, rows, (np.arange(hi - lo) * (G + 1)).astype(np.int32),
                      ell, d.x, d.q_tok, 1.0, U, A, Ct, x0, temps, seed, rid_base=rid_base, S=S)
    return d, a, s, v


def _worker_combine(rank, port, q):
    _init(rank, port)
    try:
        ms, pos = [3.0, 5.0][rank], [100.0, 250.0][rank]
        q.put((rank, bench.combine_over_ranks(ms, pos, "cpu", WORLD)))
    finally:
        dist.destroy_process_group()


def _shard_inputs(rnn: bool):
    wl = synth.WORKLOADS["tiny"].scaled(R=6, V=300)
    inp = synth.make_inputs(wl, "cpu")
    W = synth.rnn_weights(wl, "cpu").numpy() if rnn else None
    return wl, inp, W


def _worker_shard(rank, port, q, rnn=False):
    _init(rank, port)
    try:
        wl, inp, W = _shard_inputs(rnn)
        per = wl.R // WORLD
        lo, hi = rank * per, (rank + 1) * per
        seed = 77
        # stage 1: draft + confidence on the shard, all-gather the survivals
        d, a, _, _ = _round(inp, wl, lo, hi, lo, seed, W=W)
        parts = [torch.zeros(per, wl.gamma, dtype=torch.float64) for _ in range(WORLD)]
        dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(a)))
        a_all = torch.cat(parts).numpy()
        # stage 2: identical schedule on every rank, verify the shard
        _, _, s, v = _round(inp, wl, lo, hi, lo, seed, a_all=a_all, W=W)
        got = {k: torch.from_numpy(np.ascontiguousarray(t)) for k, t in
               (("x", d.x), ("acc", v.accept_len), ("out", v.out_tok), ("n", v.n_out))}
        gathered = {}
        for k, t in got.items():
            bufs = [torch.zeros_like(t) for _ in range(WORLD)]
            dist.all_gather(bufs, t)
            gathered[k] = torch.cat(bufs).numpy()
        q.put((rank, gathered, s.ell.copy(), s.B))
    finally:
        dist.destroy_process_group()


def _worker_shard_rnn(rank, port, q):
    _worker_shard(rank, port, q, rnn=True)


def _spawn(fn):
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    codes = [p.exitcode for p in procs]
    assert codes == [0] * WORLD, codes
    return [q.get() for _ in range(WORLD)]


def test_replica_layout_disjoint_request_ids():
    wl = synth.WORKLOADS["c5"]
    spans = [bench.replica_layout(r, wl) for r in range(8)]
    seeds = {s for s, _ in spans}
    bases = [b for _, b in spans]
    assert len(seeds) == 8
    for r in range(7):
        assert bases[r] + wl.R == bases[r + 1]


def test_combine_over_ranks_gloo():
    res = dict(_spawn(_worker_combine))
    for rank in range(WORLD):
        assert res[rank] == (5.0, 350.0)
    assert bench.combine_over_ranks(3.0, 100.0, "cpu", 1) == (3.0, 100.0)


@pytest.mark.parametrize("rnn", [False, True])
def test_request_sharded_round_equals_whole_batch_gloo(rnn):
    """Markov head, and the RNN head (its state is per request, so the shards
    carry no state of one another)."""
    out = _spawn(_worker_shard_rnn if rnn else _worker_shard)
    wl, inp, W = _shard_inputs(rnn)
    d, _, s, v = _round(inp, wl, 0, wl.R, 0, 77, W=W)
    for _, g, ell, B in out:
        np.testing.assert_array_equal(g["x"], d.x)
        np.testing.assert_array_equal(ell, s.ell)
        assert B == s.B
        np.testing.assert_array_equal(g["acc"], v.accept_len)
        np.testing.assert_array_equal(g["out"], v.out_tok)
        np.testing.assert_array_equal(g["n"], v.n_out)
