"""Oracle for the speculative-decoding round math -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded fp64 C++ implementation (``oracle.cpp``) of the
draft / confidence / schedule / verify definitions, wrapped here with ctypes
and numpy.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  It shares no code with the CUDA
library in ``verify_sampling_gb300``.

Each wrapper cites the passage of the pages it follows (see ``oracle.cpp``):
  * draft      -- DSpark summary, "第二阶段：轻量顺序头"; history article "杀招一"
  * confidence -- DSpark summary, "2.1 置信度头" (+ sequential temperature scaling)
  * schedule   -- DSpark summary, "2.2 硬件感知前缀调度器" and "挑战2"; history "杀招三"
  * verify     -- history article, "1.1运行机制" (rejection sampling); DSpark Figure 1
  * schedule, threshold mode -- DSpark summary, comparison table (SpecDec++) and Figure 5
  * accept_stats -- LightSpec article, "无需额外训练，基于运行时统计的动态调度"
  * cstar, calibration -- DSpark summary, "2.1 置信度头" and Figure 6
  * draft_rnn  -- DSpark summary, "第二阶段：轻量顺序头" (the RNN head; no formula is
                  given there: s_k = store(tanh(A_k[x_{k-1}] + s_{k-1} W_k)) is this
                  library's reading, pinned by its reduction to the Markov head)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

DRAFT_GUMBEL, ACCEPT_U, RESIDUAL_GUMBEL, BONUS_GUMBEL = 0, 1, 2, 3
MODE_SAMPLE, MODE_GREEDY = 0, 1
SCHED_EARLY_STOP, SCHED_GLOBAL, SCHED_THRESHOLD = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (fp contraction off, so x86 and Arm agree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, u32, u64, f64 = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                                   ctypes.c_uint64, ctypes.c_double)
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_philox4x32_10.restype = None
        L.orc_uniform.argtypes = [u64, u32, u32, u32, u32]
        L.orc_uniform.restype = f64
        L.orc_gumbel_argmax.argtypes = [i32, P, u64, u32, u32, u32, P]
        L.orc_gumbel_argmax.restype = i32
        L.orc_sps_lookup.argtypes = [P, i32, f64, f64, f64]
        L.orc_sps_lookup.restype = f64
        L.orc_accept_prob.argtypes = [i32, P, P]
        L.orc_accept_prob.restype = f64
        L.orc_draft.argtypes = [i32, i32, i32, i32, P, i64, P, P, P, P, u64, u32, P, P, P, P, P, P]
        L.orc_draft.restype = i32
        L.orc_confidence.argtypes = [i32, i32, i32, i32, i32, P, i64, P, P, P, P, P, P, P]
        L.orc_confidence.restype = i32
        L.orc_schedule.argtypes = [i32, i32, P, P, i32, f64, f64, i32, i32, f64, P, P, P, P, P, P]
        L.orc_schedule.restype = i32
        L.orc_verify.argtypes = [i32, i32, i32, i32, P, P, P, P, P, f64, P, i64, P, P, i32, P, P,
                                 u64, u32, P, P, P, P, P, P, P, P]
        L.orc_verify.restype = i32
        L.orc_accept_stats.argtypes = [i32, i32, P, P, i32, i32, f64, i32, P, P, P, P]
        L.orc_accept_stats.restype = i32
        L.orc_cstar.argtypes = [i32, i32, i32, P, P, P, P, f64, P, i64, P, P, i32, P, P, P, P]
        L.orc_draft_rnn.argtypes = [i32, i32, i32, i32, P, i64, P, P, P, P, P, u64, u32, i32, P, P,
                                    P, P, P, P, P, P]
        L.orc_draft_rnn.restype = i32
        L.orc_cstar.restype = i32
        L.orc_calibration.argtypes = [i32, i32, P, P, P, i32, P, P, P, P, P]
        L.orc_calibration.restype = i32
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# ---------------------------------------------------------------- random ----
def philox4x32_10(counter, key) -> np.ndarray:
    c = np.asarray(counter, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, v: int, j: int, rid: int, purpose: int) -> float:
    return lib().orc_uniform(seed, v, j, rid, purpose)


def gumbel_argmax(logw, seed: int, j: int, rid: int, purpose: int):
    lw = _f64(logw)
    gap = ctypes.c_double()
    idx = lib().orc_gumbel_argmax(lw.size, _ptr(lw), seed, j, rid, purpose, ctypes.byref(gap))
    return idx, gap.value


def sps_lookup(sps, b_lo: float, b_step: float, B: float) -> float:
    s = _f64(sps)
    return lib().orc_sps_lookup(_ptr(s), s.size, b_lo, b_step, B)


def accept_prob(zt, zq) -> float:
    """sum_v min(softmax(zt)_v, softmax(zq)_v): acceptance probability of one draft token."""
    a, b = _f64(zt), _f64(zq)
    assert a.size == b.size
    return lib().orc_accept_prob(a.size, _ptr(a), _ptr(b))


# ----------------------------------------------------------------- draft ----
@dataclass
class DraftOut:
    x: np.ndarray       # [R, gamma] int32
    q_tok: np.ndarray   # [R, gamma] f64
    lse: np.ndarray     # [R, gamma] f64
    gap: np.ndarray     # [R, gamma] f64 Gumbel top-2 score gap
    P: np.ndarray | None


def draft(U, A, Ct, x0, draft_temp, seed: int, rid_base: int = 0, x_cond=None,
          want_P: bool = False) -> DraftOut:
    """U [R, gamma, V]; A, Ct [gamma, V, r]; x0 [R]; draft_temp [gamma]."""
    U = _f32(U)
    R, gamma, V = U.shape
    A, Ct = _f32(A), _f32(Ct)
    r = A.shape[2]
    assert A.shape == (gamma, V, r) and Ct.shape == (gamma, V, r)
    x0, temp = _i32(x0), _f32(draft_temp)
    xc = None if x_cond is None else _i32(x_cond)
    x = np.zeros((R, gamma), np.int32)
    q, l, g = (np.zeros((R, gamma)) for _ in range(3))
    P = np.zeros((R, gamma, V)) if want_P else None
    rc = lib().orc_draft(R, gamma, V, r, _ptr(U), gamma * V, _ptr(A), _ptr(Ct), _ptr(x0),
                         _ptr(temp), seed, rid_base, _ptr(xc), _ptr(x), _ptr(q), _ptr(l),
                         _ptr(g), _ptr(P))
    if rc != 0:
        raise ValueError(f"orc_draft failed ({rc})")
    return DraftOut(x, q, l, g, P)


# ------------------------------------------------------------ confidence ----
def confidence(h, W1, w, x0, x, sts_temp):
    """h [R, gamma, d]; W1 [V, e]; w [d + e]; x0 [R]; x [R, gamma] -> (c, a) f64."""
    h = _f32(h)
    R, gamma, d = h.shape
    W1, w = _f32(W1), _f32(w)
    V, e = W1.shape
    assert w.size == d + e
    x0, x, t = _i32(x0), _i32(x), _f32(sts_temp)
    c = np.zeros((R, gamma))
    a = np.zeros((R, gamma))
    rc = lib().orc_confidence(R, gamma, d, e, V, _ptr(h), gamma * d, _ptr(W1), _ptr(w), _ptr(x0),
                              _ptr(x), _ptr(t), _ptr(c), _ptr(a))
    if rc != 0:
        raise ValueError(f"orc_confidence failed ({rc})")
    return c, a


# -------------------------------------------------------------- schedule ----
@dataclass
class ScheduleOut:
    ell: np.ndarray
    row_off: np.ndarray
    n: int
    B: int
    tau: float
    theta: float
    margin: float
    order: np.ndarray
    theta_seq: np.ndarray


def schedule(a, sps, b_lo: float, b_step: float, K: int, mode: int = SCHED_EARLY_STOP,
             threshold: float = 0.0) -> ScheduleOut:
    """a [R, gamma] survival probabilities; sps table at B_i = b_lo + i*b_step.
    ``threshold`` is used by SCHED_THRESHOLD only (admit a >= threshold)."""
    a = _f64(a)
    R, gamma = a.shape
    s = _f64(sps)
    ell = np.zeros(R, np.int32)
    row_off = np.zeros(R + 1, np.int32)
    stats = np.zeros(4)
    mg = ctypes.c_double()
    order = np.zeros(R * gamma, np.int32)
    nmax = min(K, R * gamma)
    th = np.zeros(nmax + 1)
    rc = lib().orc_schedule(R, gamma, _ptr(a), _ptr(s), s.size, b_lo, b_step, K, mode,
                            float(threshold), _ptr(ell),
                            _ptr(row_off), _ptr(stats), ctypes.byref(mg), _ptr(order), _ptr(th))
    if rc != 0:
        raise ValueError(f"orc_schedule failed ({rc})")
    return ScheduleOut(ell, row_off, int(stats[0]), int(stats[1]), float(stats[2]),
                       float(stats[3]), mg.value, order, th)


# ---------------------------------------------------------------- verify ----
@dataclass
class VerifyOut:
    accept_len: np.ndarray
    out_tok: np.ndarray
    n_out: np.ndarray
    margin: np.ndarray
    jstar: np.ndarray
    margin_acc: np.ndarray  # smallest |u - p/q| of the accept tests (+inf: none made)
    margin_gap: np.ndarray  # Gumbel top-2 gap of the emitted sample (+inf in greedy mode)


def verify(mode: int, tgt, row_off, ell, x, q_tok, target_temp: float, U, A, Ct, x0, draft_temp,
           seed: int, rid_base: int = 0, S=None) -> VerifyOut:
    """tgt [rows, V]; row (r, j) = row_off[r] + j - 1.  U [R, gamma, V]; A, Ct [gamma, V, r]."""
    tgt = _f32(tgt)
    V = tgt.shape[-1]
    tgt = tgt.reshape(-1, V)
    x = _i32(x)
    R, gamma = x.shape
    row_off, ell, x0 = _i32(row_off), _i32(ell), _i32(x0)
    q = _f64(q_tok)
    temp = _f32(draft_temp)
    if U is None:  # greedy mode never reads the draft rows
        assert mode == MODE_GREEDY
        A = Ct = None
        r = 0
    else:
        U, A, Ct = _f32(U), _f32(A), _f32(Ct)
        r = A.shape[2]
    acc = np.zeros(R, np.int32)
    out = np.zeros((R, gamma + 1), np.int32)
    n_out = np.zeros(R, np.int32)
    mg = np.zeros(R)
    mg_acc = np.zeros(R)
    mg_gap = np.zeros(R)
    js = np.zeros(R, np.int32)
    rc = lib().orc_verify(mode, R, gamma, V, _ptr(tgt), _ptr(row_off), _ptr(ell), _ptr(x), _ptr(q),
                          target_temp, _ptr(U), gamma * V, _ptr(A), _ptr(Ct), r, _ptr(x0),
                          _ptr(temp), seed, rid_base, _ptr(acc), _ptr(out), _ptr(n_out), _ptr(mg),
                          _ptr(js), _ptr(None if S is None else _f32(S)), _ptr(mg_acc), _ptr(mg_gap))
    if rc != 0:
        raise ValueError(f"orc_verify failed ({rc})")
    return VerifyOut(acc, out, n_out, mg, js, mg_acc, mg_gap)


# ----------------------------------------------------- acceptance statistics --
def accept_stats(ell, accept_len, ema, count, bucket: int, beta: float, min_count: int = 1):
    """One round's EMA update of acceptance rates per MTP length (LightSpec
    runtime statistics).  ``ema`` [n_buckets, gamma] f64 and ``count``
    [n_buckets, gamma] int64 are updated IN PLACE; returns (estimate [gamma],
    bad) with the interpolated rates of ``bucket`` after the update."""
    ell, acc = _i32(ell), _i32(accept_len)
    assert ema.dtype == np.float64 and count.dtype == np.int64
    assert ema.flags.c_contiguous and count.flags.c_contiguous and ema.shape == count.shape
    n_buckets, gamma = ema.shape
    est = np.zeros(gamma)
    bad = ctypes.c_int()
    rc = lib().orc_accept_stats(ell.size, gamma, _ptr(ell), _ptr(acc), bucket, n_buckets,
                                float(beta), int(min_count), _ptr(ema), _ptr(count), _ptr(est),
                                ctypes.byref(bad))
    if rc != 0:
        raise ValueError(f"orc_accept_stats failed ({rc})")
    return est, bad.value


# --------------------------------------------------- calibration diagnostics --
def cstar(tgt, row_off, ell, x, target_temp: float, U, A, Ct, x0, draft_temp, S=None) -> np.ndarray:
    """c* = sum_v min(p_v, q_v) for every verified draft row (r, j <= l_r);
    NaN past l_r.  Layouts as in ``verify``."""
    tgt = _f32(tgt)
    V = tgt.shape[-1]
    tgt = tgt.reshape(-1, V)
    x = _i32(x)
    R, gamma = x.shape
    U, A, Ct = _f32(U), _f32(A), _f32(Ct)
    out = np.zeros((R, gamma))
    rc = lib().orc_cstar(R, gamma, V, _ptr(tgt), _ptr(_i32(row_off)), _ptr(_i32(ell)), _ptr(x),
                         float(target_temp), _ptr(U), gamma * V, _ptr(A), _ptr(Ct), A.shape[2],
                         _ptr(_i32(x0)), _ptr(_f32(draft_temp)), _ptr(out),
                         _ptr(None if S is None else _f32(S)))
    if rc != 0:
        raise ValueError(f"orc_cstar failed ({rc})")
    return out


def calibration(c, ell, accept_len, count, sum_c, sum_acc):
    """Fold one round's tested positions into the reliability diagram (tables
    updated IN PLACE: count int64, sum_c f64, sum_acc int64, [n_bins] each);
    returns (ece, bad)."""
    c = _f64(c)
    R, gamma = c.shape
    assert count.dtype == np.int64 and sum_acc.dtype == np.int64 and sum_c.dtype == np.float64
    ece = ctypes.c_double()
    bad = ctypes.c_int()
    rc = lib().orc_calibration(R, gamma, _ptr(c), _ptr(_i32(ell)), _ptr(_i32(accept_len)),
                               count.size, _ptr(count), _ptr(sum_c), _ptr(sum_acc),
                               ctypes.byref(ece), ctypes.byref(bad))
    if rc != 0:
        raise ValueError(f"orc_calibration failed ({rc})")
    return ece.value, bad.value


# ------------------------------------------------------------------ RNN head --
@dataclass
class DraftRnnOut:
    x: np.ndarray       # [R, gamma] int32
    q_tok: np.ndarray   # [R, gamma] f64
    lse: np.ndarray     # [R, gamma] f64
    gap: np.ndarray     # [R, gamma] f64
    S: np.ndarray       # [R, gamma, r] f64 stored states
    P: np.ndarray | None = None  # [R, gamma, V] draft distributions (want_P)


def draft_rnn(U, A, Ct, W, x0, draft_temp, seed: int, rid_base: int = 0, bf16_state: bool = True,
              x_cond=None, s_cond=None, want_P: bool = False) -> DraftRnnOut:
    """RNN sequential head: s_k = store(tanh(A_k[x_{k-1}] + s_{k-1} W_k)),
    B_k = s_k C_k.  U [R, gamma, V]; A, Ct [gamma, V, r]; W [gamma, r, r]."""
    U = _f32(U)
    R, gamma, V = U.shape
    A, Ct, W = _f32(A), _f32(Ct), _f32(W)
    r = A.shape[2]
    assert W.shape == (gamma, r, r)
    x = np.zeros((R, gamma), np.int32)
    q, l, g = (np.zeros((R, gamma)) for _ in range(3))
    S = np.zeros((R, gamma, r))
    xc = None if x_cond is None else _i32(x_cond)
    sc = None if s_cond is None else _f32(s_cond)
    P = np.zeros((R, gamma, V)) if want_P else None
    rc = lib().orc_draft_rnn(R, gamma, V, r, _ptr(U), gamma * V, _ptr(A), _ptr(Ct), _ptr(W),
                             _ptr(_i32(x0)), _ptr(_f32(draft_temp)), seed, rid_base, int(bf16_state),
                             _ptr(xc), _ptr(sc), _ptr(x), _ptr(q), _ptr(l), _ptr(g), _ptr(S), _ptr(P))
    if rc != 0:
        raise ValueError(f"orc_draft_rnn failed ({rc})")
    return DraftRnnOut(x, q, l, g, S, P)
