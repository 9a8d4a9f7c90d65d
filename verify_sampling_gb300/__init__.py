"""verify_sampling_gb300 -- Python binding of libspec, the sm_103a CUDA library
for the batched speculative-decoding round (draft / schedule / verify).

The binding only marshals arguments: it checks tensor shapes and dtypes,
allocates output and workspace tensors with torch (device memory and streams
are all torch is used for), fills the C argument structs of ``include/spec.h``
and calls the library.  Every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if ``libspec.so`` is missing, every
call raises.

Entry points mirror the C ABI: :func:`draft_sample`, :func:`schedule`,
:func:`verify`, plus :func:`run_round` that chains the three on one stream
without a host synchronisation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspec.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_ALIGNMENT, SPEC_ERR_WORKSPACE, \
    SPEC_ERR_CUDA = range(6)
SPEC_F32, SPEC_BF16 = 0, 1
VERIFY_SAMPLE, VERIFY_GREEDY = 0, 1
SCHED_EARLY_STOP, SCHED_GLOBAL, SCHED_THRESHOLD = 0, 1, 2
STAGE_DRAFT, STAGE_SCHEDULE, STAGE_VERIFY = 0, 1, 2
HEAD_MARKOV, HEAD_RNN = 0, 1
STATUS_BAD_TOKEN, STATUS_BAD_ELL, STATUS_BAD_SURVIVAL, STATUS_BAD_ROW = 0x1, 0x2, 0x4, 0x8
STATUS_TIMEOUT = 0x10

_P = ctypes.c_void_p


class DraftArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("gamma", ctypes.c_int), ("V", ctypes.c_int), ("r", ctypes.c_int),
                ("d", ctypes.c_int), ("e", ctypes.c_int), ("logit_dtype", ctypes.c_int),
                ("fac_dtype", ctypes.c_int), ("conf_dtype", ctypes.c_int),
                ("request_id_base", ctypes.c_uint32),
                ("U", _P), ("A", _P), ("Ct", _P), ("x0", _P), ("draft_temp", _P), ("h", _P),
                ("W1", _P), ("w", _P), ("sts_temp", _P), ("x", _P), ("q_tok", _P), ("lse_q", _P),
                ("c", _P), ("a", _P), ("P_out", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t), ("status", _P),
                ("head", ctypes.c_int), ("Wrnn", _P), ("S", _P)]


class SchedArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("gamma", ctypes.c_int), ("a", _P), ("sps", _P),
                ("n_sps", ctypes.c_int), ("b_lo", ctypes.c_double), ("b_step", ctypes.c_double),
                ("K", ctypes.c_int), ("mode", ctypes.c_int), ("ell", _P), ("row_off", _P),
                ("stats", _P), ("order", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t), ("status", _P),
                ("threshold", ctypes.c_double), ("K_dev", _P), ("n_free", _P)]


class AcceptStatsArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("gamma", ctypes.c_int), ("ell", _P), ("accept_len", _P),
                ("bucket", ctypes.c_int), ("n_buckets", ctypes.c_int), ("beta", ctypes.c_double),
                ("min_count", ctypes.c_int), ("ema", _P), ("count", _P), ("estimate", _P),
                ("status", _P)]


class CalibrationArgs(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("gamma", ctypes.c_int), ("c", _P), ("ell", _P),
                ("accept_len", _P), ("n_bins", ctypes.c_int), ("count", _P), ("sum_c", _P),
                ("sum_acc", _P), ("ece", _P), ("status", _P)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("R", ctypes.c_int), ("gamma", ctypes.c_int),
                ("V", ctypes.c_int), ("tgt_dtype", ctypes.c_int),
                ("request_id_base", ctypes.c_uint32), ("tgt", _P), ("tgt_row_off", _P),
                ("ell", _P), ("x", _P), ("q_tok", _P), ("lse_q", _P),
                ("target_temp", ctypes.c_float), ("draft", ctypes.POINTER(DraftArgs)),
                ("accept_len", _P), ("out_tok", _P), ("n_out", _P), ("p_tok", _P), ("lse_t", _P),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("status", _P),
                ("c_star", _P)]


class RoundHostArgs(ctypes.Structure):
    _fields_ = [("draft", ctypes.POINTER(DraftArgs)), ("sched", ctypes.POINTER(SchedArgs)),
                ("verify", ctypes.POINTER(VerifyArgs)), ("U_host", _P), ("h_host", _P),
                ("x0_host", _P), ("tgt_host", _P), ("tgt_rows", ctypes.c_size_t),
                ("out_tok_host", _P), ("accept_len_host", _P), ("n_out_host", _P),
                ("stats_host", _P), ("tgt_scheduled_only", ctypes.c_int)]


class SpecError(RuntimeError):
    pass


_lib = None


def lib() -> ctypes.CDLL:
    """Load libspec.so (built in-tree by ``build.py``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise SpecError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                            "g.build()'` (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        L.spec_draft_sample.argtypes = [ctypes.POINTER(DraftArgs), ctypes.c_uint64, _P]
        L.spec_schedule.argtypes = [ctypes.POINTER(SchedArgs), _P]
        L.spec_verify.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.c_uint64, _P]
        L.spec_accept_stats.argtypes = [ctypes.POINTER(AcceptStatsArgs), _P]
        L.spec_calibration.argtypes = [ctypes.POINTER(CalibrationArgs), _P]
        L.spec_round_host.argtypes = [ctypes.POINTER(RoundHostArgs), ctypes.c_uint64, _P]
        for f in (L.spec_draft_sample, L.spec_schedule, L.spec_verify, L.spec_accept_stats,
                  L.spec_calibration, L.spec_round_host):
            f.restype = ctypes.c_int
        L.spec_workspace_bytes.argtypes = [ctypes.c_int] * 5
        L.spec_workspace_bytes.restype = ctypes.c_size_t
        L.spec_error_string.argtypes = [ctypes.c_int]
        L.spec_error_string.restype = ctypes.c_char_p
        L.spec_version.restype = ctypes.c_int
        L.spec_wait_selftest.argtypes = [ctypes.c_uint64, _P, _P]
        L.spec_wait_selftest.restype = ctypes.c_int
        L.spec_stream_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                           ctypes.c_uint32, ctypes.c_int, _P, _P, _P]
        L.spec_stream_uniforms.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != SPEC_OK:
        raise SpecError(f"{what}: {lib().spec_error_string(rc).decode()} (code {rc})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(stage: int, R: int, gamma: int, V: int, r: int = 1) -> int:
    return int(lib().spec_workspace_bytes(stage, R, gamma, V, r))


def _workspace(nbytes: int, device, given: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    if given is not None:
        if given.numel() * given.element_size() < nbytes:
            raise ValueError("workspace too small")
        return given
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def stream_uniforms(seed: int, j: int, rid: int, purpose: int, V: int, device="cuda",
                    stream=None):
    """spec_stream_uniforms: (u, -ln u) of vocabulary entries 0..V-1 for one draw site."""
    u = torch.empty(V, dtype=torch.float32, device=device)
    e = torch.empty(V, dtype=torch.float32, device=device)
    _check(lib().spec_stream_uniforms(seed & 0xFFFFFFFFFFFFFFFF, j, rid, purpose, V, _ptr(u),
                                      _ptr(e), _stream_handle(stream)), "spec_stream_uniforms")
    return u, e


def wait_selftest(limit_ns: int, status: torch.Tensor, stream=None) -> None:
    """spec_wait_selftest: a bounded wait that nothing completes gives up after
    limit_ns and sets STATUS_TIMEOUT in ``status`` (int32 device word)."""
    status = _dev(status, "status")
    _check(lib().spec_wait_selftest(int(limit_ns), _ptr(status), _stream_handle(stream)),
           "spec_wait_selftest")


# -------------------------------------------------------------------- draft --
@dataclass
class DraftInputs:
    """Inputs of the draft stage (device tensors; see include/spec.h for layouts)."""
    U: torch.Tensor            # [R, gamma, V]
    A: torch.Tensor            # [gamma, V, r]
    Ct: torch.Tensor           # [gamma, V, r]  C_k transposed (vocabulary-major)
    x0: torch.Tensor           # [R] int32
    draft_temp: torch.Tensor   # [gamma] f32
    h: torch.Tensor            # [R, gamma, d]
    W1: torch.Tensor           # [V, e]
    w: torch.Tensor            # [d + e]
    sts_temp: torch.Tensor     # [gamma] f32
    request_id_base: int = 0
    # RNN sequential head (both or neither; factor dtype): the recurrence W_k and
    # the state array the draft writes and the verifier reads back
    Wrnn: Optional[torch.Tensor] = None   # [gamma, r, r]
    S: Optional[torch.Tensor] = None      # [R, gamma, r]


def _draft_struct(inp: DraftInputs, outs: dict, ws: Optional[torch.Tensor], status) -> DraftArgs:
    U, A, Ct = (_dev(inp.U, "U"), _dev(inp.A, "A"), _dev(inp.Ct, "Ct"))
    R, gamma, V = U.shape
    r = A.shape[2]
    if A.shape != (gamma, V, r) or Ct.shape != (gamma, V, r) or A.dtype != Ct.dtype:
        raise ValueError("A and Ct must both be [gamma, V, r] of one dtype")
    h, W1, w = _dev(inp.h, "h"), _dev(inp.W1, "W1"), _dev(inp.w, "w")
    d, e = h.shape[2], W1.shape[1]
    if h.shape[:2] != (R, gamma) or W1.shape[0] != V or w.numel() != d + e:
        raise ValueError("confidence-head shapes do not match")
    if not (h.dtype == W1.dtype == w.dtype):
        raise ValueError("h, W1 and w must share one dtype")
    for name, t, dt in (("x0", inp.x0, torch.int32), ("draft_temp", inp.draft_temp, torch.float32),
                        ("sts_temp", inp.sts_temp, torch.float32)):
        if _dev(t, name).dtype != dt:
            raise TypeError(f"{name} must be {dt}")
    a = DraftArgs()
    a.R, a.gamma, a.V, a.r, a.d, a.e = R, gamma, V, r, d, e
    a.logit_dtype, a.fac_dtype, a.conf_dtype = _dtype_code(U), _dtype_code(A), _dtype_code(h)
    a.request_id_base = inp.request_id_base
    a.U, a.A, a.Ct, a.x0, a.draft_temp = _ptr(U), _ptr(A), _ptr(Ct), _ptr(inp.x0), _ptr(inp.draft_temp)
    a.h, a.W1, a.w, a.sts_temp = _ptr(h), _ptr(W1), _ptr(w), _ptr(inp.sts_temp)
    if (inp.Wrnn is None) != (inp.S is None):
        raise ValueError("the RNN head needs both Wrnn and S")
    if inp.Wrnn is not None:
        Wr, S = _dev(inp.Wrnn, "Wrnn"), _dev(inp.S, "S")
        if Wr.shape != (gamma, r, r) or S.shape != (R, gamma, r) or not (Wr.dtype == S.dtype == A.dtype):
            raise ValueError("Wrnn must be [gamma, r, r] and S [R, gamma, r], in the dtype of A")
        a.head, a.Wrnn, a.S = HEAD_RNN, _ptr(Wr), _ptr(S)
    if outs:
        a.x, a.q_tok, a.lse_q = _ptr(outs["x"]), _ptr(outs["q_tok"]), _ptr(outs["lse_q"])
        a.c, a.a, a.P_out = _ptr(outs["c"]), _ptr(outs["a"]), _ptr(outs.get("P"))
    a.workspace = _ptr(ws)
    a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    a.status = _ptr(status)
    return a


def draft_outputs(R: int, gamma: int, V: int, device, want_P: bool = False) -> dict:
    f = dict(dtype=torch.float32, device=device)
    outs = {"x": torch.empty(R, gamma, dtype=torch.int32, device=device),
            "q_tok": torch.empty(R, gamma, **f), "lse_q": torch.empty(R, gamma, **f),
            "c": torch.empty(R, gamma, **f), "a": torch.empty(R, gamma, **f)}
    if want_P:
        outs["P"] = torch.empty(R, gamma, V, **f)
    return outs


def draft_sample(inp: DraftInputs, seed: int, *, want_P: bool = False, out: Optional[dict] = None,
                 workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 stream=None) -> dict:
    """spec_draft_sample: sample x_1..x_gamma, q(x_k), lse_k, confidences and survivals."""
    R, gamma, V = inp.U.shape
    r = inp.A.shape[2]
    outs = out if out is not None else draft_outputs(R, gamma, V, inp.U.device, want_P)
    ws = _workspace(workspace_bytes(STAGE_DRAFT, R, gamma, V, r), inp.U.device, workspace)
    a = _draft_struct(inp, outs, ws, status)
    _check(lib().spec_draft_sample(ctypes.byref(a), seed & 0xFFFFFFFFFFFFFFFF, _stream_handle(stream)),
           "spec_draft_sample")
    return outs


# ----------------------------------------------------------------- schedule --
def _sched_struct(a, sps, b_lo, b_step, K, mode, threshold, outs, status, K_dev=None,
                  n_free=None) -> SchedArgs:
    R, gamma = a.shape
    s = SchedArgs()
    s.R, s.gamma = R, gamma
    s.a, s.sps, s.n_sps = _ptr(a), _ptr(sps), sps.numel()
    s.b_lo, s.b_step, s.K, s.mode = float(b_lo), float(b_step), int(K), int(mode)
    s.threshold = float(threshold)
    s.ell, s.row_off, s.stats = _ptr(outs["ell"]), _ptr(outs["row_off"]), _ptr(outs["stats"])
    s.order = _ptr(outs.get("order"))
    s.status = _ptr(status)
    for name, t in (("K_dev", K_dev), ("n_free", n_free)):
        if t is not None and (_dev(t, name).dtype != torch.int32 or t.numel() < 1):
            raise TypeError(f"{name} must be an int32 device tensor")
    s.K_dev, s.n_free = _ptr(K_dev), _ptr(n_free)
    return s


def schedule(a: torch.Tensor, sps: torch.Tensor, b_lo: float, b_step: float, K: int,
             mode: int = SCHED_EARLY_STOP, *, threshold: float = 0.0, want_order: bool = False,
             K_dev: Optional[torch.Tensor] = None, n_free: Optional[torch.Tensor] = None,
             out: Optional[dict] = None, status: Optional[torch.Tensor] = None,
             stream=None) -> dict:
    """spec_schedule: l_r, packed row offsets and {n, B, tau, Theta} on the device.
    ``threshold`` is read by SCHED_THRESHOLD only (admit survivals >= threshold).
    Asynchronous cap: ``K_dev`` (int32 device word, may alias ``n_free``) lowers
    the cap to min(K, K_dev[0]); ``n_free`` receives the uncapped n."""
    a = _dev(a, "a")
    sps = _dev(sps, "sps")
    if a.dtype != torch.float32 or sps.dtype != torch.float32:
        raise TypeError("a and sps must be float32")
    R, gamma = a.shape
    dev = a.device
    outs = out if out is not None else {
        "ell": torch.empty(R, dtype=torch.int32, device=dev),
        "row_off": torch.empty(R + 1, dtype=torch.int32, device=dev),
        "stats": torch.empty(4, dtype=torch.float64, device=dev)}
    if want_order and "order" not in outs:
        outs["order"] = torch.empty(R * gamma, dtype=torch.int32, device=dev)
    s = _sched_struct(a, sps, b_lo, b_step, K, mode, threshold, outs, status, K_dev, n_free)
    _check(lib().spec_schedule(ctypes.byref(s), _stream_handle(stream)), "spec_schedule")
    return outs


# ------------------------------------------------------------------- verify --
def _verify_struct(mode, tgt, tgt_row_off, ell, x, q_tok, lse_q, target_temp, draft,
                   request_id_base, outs, ws, status):
    """VerifyArgs plus the DraftArgs it points to (keep it alive for the call)."""
    R, gamma = x.shape
    V = tgt.shape[-1]
    v = VerifyArgs()
    v.mode, v.R, v.gamma, v.V, v.tgt_dtype = int(mode), R, gamma, V, _dtype_code(tgt)
    v.request_id_base = request_id_base
    v.tgt, v.tgt_row_off, v.ell, v.x = _ptr(tgt), _ptr(_dev(tgt_row_off, "tgt_row_off")), \
        _ptr(_dev(ell, "ell")), _ptr(x)
    v.q_tok, v.lse_q = _ptr(q_tok), _ptr(lse_q)
    v.target_temp = float(target_temp)
    keep = None
    if draft is not None:
        keep = _draft_struct(draft, {}, None, None)
        v.draft = ctypes.pointer(keep)
    v.accept_len, v.out_tok, v.n_out = _ptr(outs["accept_len"]), _ptr(outs["out_tok"]), \
        _ptr(outs["n_out"])
    v.p_tok, v.lse_t = _ptr(outs.get("p_tok")), _ptr(outs.get("lse_t"))
    v.c_star = _ptr(outs.get("c_star"))
    v.workspace = _ptr(ws)
    v.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    v.status = _ptr(status)
    return v, keep


def verify(mode: int, tgt: torch.Tensor, tgt_row_off: torch.Tensor, ell: torch.Tensor,
           x: torch.Tensor, seed: int, *, q_tok: Optional[torch.Tensor] = None,
           lse_q: Optional[torch.Tensor] = None, target_temp: float = 1.0,
           draft: Optional[DraftInputs] = None, request_id_base: int = 0, want_p: bool = False,
           want_cstar: bool = False,
           out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
           status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """spec_verify: accept lengths and emitted tokens (sample or greedy mode)."""
    tgt = _dev(tgt, "tgt")
    x = _dev(x, "x")
    R, gamma = x.shape
    V = tgt.shape[-1]
    dev = tgt.device
    outs = out if out is not None else {
        "accept_len": torch.empty(R, dtype=torch.int32, device=dev),
        "out_tok": torch.empty(R, gamma + 1, dtype=torch.int32, device=dev),
        "n_out": torch.empty(R, dtype=torch.int32, device=dev)}
    if want_cstar and "c_star" not in outs:
        outs["c_star"] = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    if want_p and "p_tok" not in outs:
        outs["p_tok"] = torch.empty(R, gamma, dtype=torch.float32, device=dev)
        outs["lse_t"] = torch.empty(R, gamma + 1, dtype=torch.float32, device=dev)
    ws = _workspace(workspace_bytes(STAGE_VERIFY, R, gamma, V), dev, workspace)
    v, keep = _verify_struct(mode, tgt, tgt_row_off, ell, x, q_tok, lse_q, target_temp, draft,
                             request_id_base, outs, ws, status)
    _check(lib().spec_verify(ctypes.byref(v), seed & 0xFFFFFFFFFFFFFFFF, _stream_handle(stream)),
           "spec_verify")
    del keep
    return outs


# ---------------------------------------------------------- acceptance stats --
def accept_stats(ell: torch.Tensor, accept_len: torch.Tensor, ema: torch.Tensor,
                 count: torch.Tensor, bucket: int, beta: float, *, min_count: int = 1,
                 estimate: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 stream=None) -> Optional[torch.Tensor]:
    """spec_accept_stats: fold one verified round into the per-length EMA table
    ``ema`` [n_buckets, gamma] f64 / ``count`` [n_buckets, gamma] int64 (both
    updated in place on the device); returns ``estimate`` [gamma] f64 if given."""
    ell, accept_len = _dev(ell, "ell"), _dev(accept_len, "accept_len")
    ema, count = _dev(ema, "ema"), _dev(count, "count")
    if ell.dtype != torch.int32 or accept_len.dtype != torch.int32:
        raise TypeError("ell and accept_len must be int32")
    if ema.dtype != torch.float64 or count.dtype != torch.int64 or ema.shape != count.shape \
            or ema.dim() != 2:
        raise TypeError("ema must be float64 and count int64, both [n_buckets, gamma]")
    a = AcceptStatsArgs()
    a.R, (a.n_buckets, a.gamma) = ell.numel(), ema.shape
    a.ell, a.accept_len = _ptr(ell), _ptr(accept_len)
    a.bucket, a.beta, a.min_count = int(bucket), float(beta), int(min_count)
    a.ema, a.count = _ptr(ema), _ptr(count)
    if estimate is not None:
        estimate = _dev(estimate, "estimate")
        if estimate.dtype != torch.float64 or estimate.numel() < a.gamma:
            raise TypeError("estimate must be float64 with gamma entries")
    a.estimate = _ptr(estimate)
    a.status = _ptr(status)
    _check(lib().spec_accept_stats(ctypes.byref(a), _stream_handle(stream)), "spec_accept_stats")
    return estimate


def calibration(c: torch.Tensor, ell: torch.Tensor, accept_len: torch.Tensor,
                tables: dict, *, status: Optional[torch.Tensor] = None, stream=None) -> dict:
    """spec_calibration: fold one verified round into the reliability diagram
    ``tables`` = {"count": int64 [n_bins], "sum_c": float64 [n_bins],
    "sum_acc": int64 [n_bins], "ece": float64 [1] (optional)}, updated in place
    on the device (see ``calibration_tables``)."""
    c, ell, accept_len = _dev(c, "c"), _dev(ell, "ell"), _dev(accept_len, "accept_len")
    if c.dtype != torch.float32 or c.dim() != 2:
        raise TypeError("c must be float32 [R, gamma]")
    if ell.dtype != torch.int32 or accept_len.dtype != torch.int32:
        raise TypeError("ell and accept_len must be int32")
    cnt, sc, sa = (_dev(tables[k], k) for k in ("count", "sum_c", "sum_acc"))
    if cnt.dtype != torch.int64 or sa.dtype != torch.int64 or sc.dtype != torch.float64 or \
            not (cnt.numel() == sc.numel() == sa.numel()):
        raise TypeError("count / sum_acc int64 and sum_c float64, all [n_bins]")
    a = CalibrationArgs()
    a.R, a.gamma = c.shape
    a.c, a.ell, a.accept_len = _ptr(c), _ptr(ell), _ptr(accept_len)
    a.n_bins = cnt.numel()
    a.count, a.sum_c, a.sum_acc = _ptr(cnt), _ptr(sc), _ptr(sa)
    a.ece = _ptr(tables.get("ece"))
    a.status = _ptr(status)
    _check(lib().spec_calibration(ctypes.byref(a), _stream_handle(stream)), "spec_calibration")
    return tables


def calibration_tables(n_bins: int, device) -> dict:
    """Zeroed device tables for ``calibration``."""
    return {"count": torch.zeros(n_bins, dtype=torch.int64, device=device),
            "sum_c": torch.zeros(n_bins, dtype=torch.float64, device=device),
            "sum_acc": torch.zeros(n_bins, dtype=torch.int64, device=device),
            "ece": torch.zeros(1, dtype=torch.float64, device=device)}


# -------------------------------------------------------------------- round --
def run_round(draft_in: DraftInputs, tgt: torch.Tensor, tgt_row_off: torch.Tensor,
              sps: torch.Tensor, b_lo: float, b_step: float, K: int, seed: int, *,
              sched_mode: int = SCHED_EARLY_STOP, sched_threshold: float = 0.0,
              target_temp: float = 1.0, bufs: Optional[dict] = None, stream=None) -> dict:
    """One full round -- draft, schedule, verify -- on one stream, no host sync."""
    bufs = {} if bufs is None else bufs
    d = draft_sample(draft_in, seed, out=bufs.get("draft"), workspace=bufs.get("ws_draft"),
                     status=bufs.get("status"), stream=stream)
    s = schedule(d["a"], sps, b_lo, b_step, K, sched_mode, threshold=sched_threshold,
                 out=bufs.get("sched"), status=bufs.get("status"), stream=stream)
    v = verify(VERIFY_SAMPLE, tgt, tgt_row_off, s["ell"], d["x"], seed, q_tok=d["q_tok"],
               lse_q=d["lse_q"], target_temp=target_temp, draft=draft_in,
               request_id_base=draft_in.request_id_base, out=bufs.get("verify"),
               workspace=bufs.get("ws_verify"), status=bufs.get("status"), stream=stream)
    return {"draft": d, "sched": s, "verify": v}


def _host(t: Optional[torch.Tensor], like: torch.Tensor, name: str):
    """Pointer of a host tensor that mirrors the device tensor ``like``."""
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous host tensor")
    if t.dtype != like.dtype or t.numel() != like.numel():
        raise ValueError(f"{name} must match its device buffer ({like.dtype}, {like.numel()} elements)")
    return ctypes.c_void_p(t.data_ptr())


def run_round_host(draft_in: DraftInputs, tgt: torch.Tensor, tgt_row_off: torch.Tensor,
                   sps: torch.Tensor, b_lo: float, b_step: float, K: int, seed: int, *,
                   host_in: dict, host_out: dict, sched_mode: int = SCHED_EARLY_STOP,
                   sched_threshold: float = 0.0, target_temp: float = 1.0,
                   tgt_scheduled_only: bool = False, K_dev: Optional[torch.Tensor] = None,
                   n_free: Optional[torch.Tensor] = None,
                   bufs: Optional[dict] = None, stream=None) -> dict:
    """spec_round_host: one round whose per-round inputs come from host tensors
    ``host_in`` {"U", "h", "x0", "tgt"} (copied into draft_in.U / .h / .x0 and
    ``tgt``) and whose results go to host tensors ``host_out`` {"out_tok",
    "accept_len", "n_out", "stats"}; every key is optional.  Page-locked host
    tensors keep the call asynchronous (synchronise before reading host_out).
    ``tgt_scheduled_only``: host_in["tgt"] is the padded [R, gamma + 1, V]
    page-locked array and only the scheduled rows are read from it, into
    ``tgt`` (room for R * (gamma + 1) rows) in the schedule's packed layout;
    ``tgt_row_off`` is then ignored.  ``K_dev`` / ``n_free``: the scheduler's
    asynchronous cap words, as for schedule()."""
    bufs = {} if bufs is None else bufs
    U = _dev(draft_in.U, "U")
    R, gamma, V = U.shape
    dev = U.device
    d_outs = bufs.get("draft") or draft_outputs(R, gamma, V, dev)
    ws_d = _workspace(workspace_bytes(STAGE_DRAFT, R, gamma, V, draft_in.A.shape[2]), dev,
                      bufs.get("ws_draft"))
    da = _draft_struct(draft_in, d_outs, ws_d, bufs.get("status"))
    s_outs = bufs.get("sched") or {
        "ell": torch.empty(R, dtype=torch.int32, device=dev),
        "row_off": torch.empty(R + 1, dtype=torch.int32, device=dev),
        "stats": torch.empty(4, dtype=torch.float64, device=dev)}
    sa = _sched_struct(d_outs["a"], _dev(sps, "sps"), b_lo, b_step, K, sched_mode,
                       sched_threshold, s_outs, bufs.get("status"), K_dev, n_free)
    tgt = _dev(tgt, "tgt")
    if tgt_scheduled_only:
        ht = host_in.get("tgt")
        if ht is None or not ht.is_pinned() or ht.numel() != R * (gamma + 1) * V:
            raise ValueError("tgt_scheduled_only needs a pinned host tgt of R*(gamma+1)*V entries")
        if tgt.numel() < R * (gamma + 1) * V:
            raise ValueError("tgt must hold R*(gamma+1) rows")
        tgt_row_off = s_outs["row_off"]
    v_outs = bufs.get("verify") or {
        "accept_len": torch.empty(R, dtype=torch.int32, device=dev),
        "out_tok": torch.empty(R, gamma + 1, dtype=torch.int32, device=dev),
        "n_out": torch.empty(R, dtype=torch.int32, device=dev)}
    ws_v = _workspace(workspace_bytes(STAGE_VERIFY, R, gamma, V), dev, bufs.get("ws_verify"))
    va, keep = _verify_struct(VERIFY_SAMPLE, tgt, tgt_row_off, s_outs["ell"], d_outs["x"],
                              d_outs["q_tok"], d_outs["lse_q"], target_temp, draft_in,
                              draft_in.request_id_base, v_outs, ws_v, bufs.get("status"))
    h = RoundHostArgs()
    h.draft, h.sched, h.verify = ctypes.pointer(da), ctypes.pointer(sa), ctypes.pointer(va)
    h.U_host = _host(host_in.get("U"), U, "host U")
    h.h_host = _host(host_in.get("h"), draft_in.h, "host h")
    h.x0_host = _host(host_in.get("x0"), draft_in.x0, "host x0")
    h.tgt_host = _host(host_in.get("tgt"), tgt, "host tgt")
    h.tgt_rows = tgt.numel() // V
    h.out_tok_host = _host(host_out.get("out_tok"), v_outs["out_tok"], "host out_tok")
    h.accept_len_host = _host(host_out.get("accept_len"), v_outs["accept_len"], "host accept_len")
    h.n_out_host = _host(host_out.get("n_out"), v_outs["n_out"], "host n_out")
    h.stats_host = _host(host_out.get("stats"), s_outs["stats"], "host stats")
    h.tgt_scheduled_only = int(bool(tgt_scheduled_only))
    _check(lib().spec_round_host(ctypes.byref(h), seed & 0xFFFFFFFFFFFFFFFF, _stream_handle(stream)),
           "spec_round_host")
    del keep
    return {"draft": d_outs, "sched": s_outs, "verify": v_outs}
