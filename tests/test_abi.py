"""The C ABI library loads and exports every symbol include/spec.h declares; the
ctypes mirrors of the argument structs match the C layout; host-side argument
checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec.h")


@pytest.fixture(scope="module")
def spec():
    import verify_sampling_gb300 as vs
    if not os.path.exists(vs.LIB_PATH):
        from verify_sampling_gb300 import build
        build.build()
    return vs


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(spec):
    names = _declared_functions()
    assert {"spec_draft_sample", "spec_schedule", "spec_verify", "spec_workspace_bytes",
            "spec_error_string", "spec_stream_uniforms", "spec_version",
            "spec_accept_stats", "spec_calibration", "spec_round_host"} <= set(names)
    lib = spec.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", spec.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (spec_\w+)", out))
    assert set(names) == exported


def test_struct_layout_matches_c(spec, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "spec.h"\n'
        "#define P(T, f) printf(#T \".\" #f \" %zu\\n\", offsetof(T, f));\n"
        "int main(void){\n"
        'printf("spec_draft_args %zu\\n", sizeof(spec_draft_args));\n'
        'printf("spec_sched_args %zu\\n", sizeof(spec_sched_args));\n'
        'printf("spec_verify_args %zu\\n", sizeof(spec_verify_args));\n'
        'printf("spec_accept_stats_args %zu\\n", sizeof(spec_accept_stats_args));\n'
        'printf("spec_calibration_args %zu\\n", sizeof(spec_calibration_args));\n'
        'printf("spec_round_host_args %zu\\n", sizeof(spec_round_host_args));\n'
        "P(spec_draft_args, status) P(spec_draft_args, workspace_bytes) P(spec_draft_args, U)\n"
        "P(spec_draft_args, head) P(spec_draft_args, Wrnn) P(spec_draft_args, S)\n"
        "P(spec_sched_args, b_lo) P(spec_sched_args, stats) P(spec_sched_args, status)\n"
        "P(spec_sched_args, threshold) P(spec_sched_args, K_dev) P(spec_sched_args, n_free)\n"
        "P(spec_accept_stats_args, beta)\n"
        "P(spec_accept_stats_args, ema) P(spec_accept_stats_args, status)\n"
        "P(spec_verify_args, c_star) P(spec_calibration_args, n_bins)\n"
        "P(spec_calibration_args, ece) P(spec_calibration_args, status)\n"
        "P(spec_round_host_args, tgt_rows) P(spec_round_host_args, stats_host)\n"
        "P(spec_round_host_args, tgt_scheduled_only)\n"
        "P(spec_verify_args, target_temp) P(spec_verify_args, draft) P(spec_verify_args, status)\n"
        "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                         text=True).stdout.splitlines())
    assert int(got["spec_draft_args"]) == ctypes.sizeof(spec.DraftArgs)
    assert int(got["spec_sched_args"]) == ctypes.sizeof(spec.SchedArgs)
    assert int(got["spec_verify_args"]) == ctypes.sizeof(spec.VerifyArgs)
    assert int(got["spec_accept_stats_args"]) == ctypes.sizeof(spec.AcceptStatsArgs)
    assert int(got["spec_calibration_args"]) == ctypes.sizeof(spec.CalibrationArgs)
    assert int(got["spec_round_host_args"]) == ctypes.sizeof(spec.RoundHostArgs)
    for key, (cls, field) in {"spec_draft_args.status": (spec.DraftArgs, "status"),
                              "spec_draft_args.workspace_bytes": (spec.DraftArgs, "workspace_bytes"),
                              "spec_draft_args.U": (spec.DraftArgs, "U"),
                              "spec_draft_args.head": (spec.DraftArgs, "head"),
                              "spec_draft_args.Wrnn": (spec.DraftArgs, "Wrnn"),
                              "spec_draft_args.S": (spec.DraftArgs, "S"),
                              "spec_sched_args.b_lo": (spec.SchedArgs, "b_lo"),
                              "spec_sched_args.stats": (spec.SchedArgs, "stats"),
                              "spec_sched_args.status": (spec.SchedArgs, "status"),
                              "spec_sched_args.threshold": (spec.SchedArgs, "threshold"),
                              "spec_sched_args.K_dev": (spec.SchedArgs, "K_dev"),
                              "spec_sched_args.n_free": (spec.SchedArgs, "n_free"),
                              "spec_accept_stats_args.beta": (spec.AcceptStatsArgs, "beta"),
                              "spec_accept_stats_args.ema": (spec.AcceptStatsArgs, "ema"),
                              "spec_accept_stats_args.status": (spec.AcceptStatsArgs, "status"),
                              "spec_verify_args.c_star": (spec.VerifyArgs, "c_star"),
                              "spec_calibration_args.n_bins": (spec.CalibrationArgs, "n_bins"),
                              "spec_calibration_args.ece": (spec.CalibrationArgs, "ece"),
                              "spec_calibration_args.status": (spec.CalibrationArgs, "status"),
                              "spec_round_host_args.tgt_rows": (spec.RoundHostArgs, "tgt_rows"),
                              "spec_round_host_args.stats_host": (spec.RoundHostArgs, "stats_host"),
                              "spec_round_host_args.tgt_scheduled_only":
                                  (spec.RoundHostArgs, "tgt_scheduled_only"),
                              "spec_verify_args.target_temp": (spec.VerifyArgs, "target_temp"),
                              "spec_verify_args.draft": (spec.VerifyArgs, "draft"),
                              "spec_verify_args.status": (spec.VerifyArgs, "status")}.items():
        assert int(got[key]) == getattr(cls, field).offset, key


def test_error_strings_and_version(spec):
    lib = spec.lib()
    assert lib.spec_version() >= 10000
    for code in range(6):
        assert lib.spec_error_string(code)
    assert b"unknown" in lib.spec_error_string(99)


def test_workspace_sizes(spec):
    assert spec.workspace_bytes(spec.STAGE_SCHEDULE, 64, 8, 1000) == 0
    d = spec.workspace_bytes(spec.STAGE_DRAFT, 512, 11, 129280, 128)
    v = spec.workspace_bytes(spec.STAGE_VERIFY, 512, 11, 129280)
    assert d > 0 and d % 256 == 0 and v > 0 and v % 256 == 0
    assert spec.workspace_bytes(spec.STAGE_DRAFT, 0, 11, 129280, 128) == 0
    assert spec.workspace_bytes(spec.STAGE_DRAFT, 4, 11, 100, 257) == 0   # rank > 256
    assert spec.workspace_bytes(7, 4, 4, 100, 8) == 0


def test_host_side_rejections_launch_nothing(spec):
    lib = spec.lib()
    assert lib.spec_draft_sample(None, 0, None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_schedule(None, None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify(None, 0, None) == spec.SPEC_ERR_INVALID_ARG
    a = spec.DraftArgs()
    a.R, a.gamma, a.V, a.r = 4, 4, 100, 8
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG  # nulls
    a.gamma = 65
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG
    # the sequential head: valid pointers reach the workspace check; a bad head
    # value, a missing RNN buffer or a misaligned state array is refused first
    a.gamma, a.fac_dtype = 4, spec.SPEC_BF16
    for f in ("U", "A", "Ct", "x0", "draft_temp", "sts_temp", "x", "q_tok", "lse_q", "c", "a"):
        setattr(a, f, ctypes.c_void_p(256))
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_WORKSPACE
    a.head = 2
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_draft_sample_static(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG
    a.head, a.Wrnn = spec.HEAD_RNN, ctypes.c_void_p(256)
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG  # no S
    assert lib.spec_draft_sample_static(ctypes.byref(a), 0, None) == spec.SPEC_ERR_INVALID_ARG
    a.S = ctypes.c_void_p(257)
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_ALIGNMENT
    assert lib.spec_draft_sample_static(ctypes.byref(a), 0, None) == spec.SPEC_ERR_ALIGNMENT
    a.S = ctypes.c_void_p(256)
    assert lib.spec_draft_sample(ctypes.byref(a), 0, None) == spec.SPEC_ERR_WORKSPACE
    s = spec.SchedArgs()
    s.R, s.gamma, s.n_sps, s.b_step, s.K = 100, 100, 1, 1.0, 5
    s.a = s.sps = s.ell = s.row_off = s.stats = ctypes.c_void_p(256)
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_UNSUPPORTED  # 10^4 > 8192
    s.gamma, s.b_step = 2, 0.0
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_INVALID_ARG
    s.b_step = 1.0
    s.stats = ctypes.c_void_p(260)  # not 8-byte aligned
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_ALIGNMENT
    s.stats = ctypes.c_void_p(256)
    s.n_free = ctypes.c_void_p(258)  # not 4-byte aligned
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_ALIGNMENT
    s.n_free, s.K_dev = None, ctypes.c_void_p(257)
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_ALIGNMENT
    s.K_dev = None
    s.mode, s.threshold = spec.SCHED_THRESHOLD, float("nan")
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_INVALID_ARG
    s.mode = 3
    assert lib.spec_schedule(ctypes.byref(s), None) == spec.SPEC_ERR_INVALID_ARG
    st = spec.AcceptStatsArgs()
    assert lib.spec_accept_stats(None, None) == spec.SPEC_ERR_INVALID_ARG
    st.R, st.gamma, st.n_buckets, st.bucket, st.beta = 4, 4, 2, 0, 0.5
    st.ell = st.accept_len = st.ema = st.count = ctypes.c_void_p(256)
    st.bucket = 2
    assert lib.spec_accept_stats(ctypes.byref(st), None) == spec.SPEC_ERR_INVALID_ARG
    st.bucket, st.beta = 1, 0.0
    assert lib.spec_accept_stats(ctypes.byref(st), None) == spec.SPEC_ERR_INVALID_ARG
    st.beta, st.gamma = 0.5, 2000
    assert lib.spec_accept_stats(ctypes.byref(st), None) == spec.SPEC_ERR_UNSUPPORTED
    st.gamma, st.ema = 4, ctypes.c_void_p(260)
    assert lib.spec_accept_stats(ctypes.byref(st), None) == spec.SPEC_ERR_ALIGNMENT
    ca = spec.CalibrationArgs()
    assert lib.spec_calibration(None, None) == spec.SPEC_ERR_INVALID_ARG
    ca.R, ca.gamma, ca.n_bins = 4, 4, 0
    ca.c = ca.ell = ca.accept_len = ca.count = ca.sum_c = ca.sum_acc = ctypes.c_void_p(256)
    assert lib.spec_calibration(ctypes.byref(ca), None) == spec.SPEC_ERR_INVALID_ARG
    ca.n_bins = 2000
    assert lib.spec_calibration(ctypes.byref(ca), None) == spec.SPEC_ERR_UNSUPPORTED
    ca.n_bins, ca.sum_c = 10, ctypes.c_void_p(260)
    assert lib.spec_calibration(ctypes.byref(ca), None) == spec.SPEC_ERR_ALIGNMENT
    # a host round whose stages are not chained through the same buffers
    assert lib.spec_round_host(None, 0, None) == spec.SPEC_ERR_INVALID_ARG
    da, sa, va = spec.DraftArgs(), spec.SchedArgs(), spec.VerifyArgs()
    da.R = sa.R = va.R = 4
    da.gamma = sa.gamma = va.gamma = 2
    da.V = va.V = 100
    da.a, sa.a = ctypes.c_void_p(256), ctypes.c_void_p(512)  # schedule reads another buffer
    rh = spec.RoundHostArgs()
    rh.draft, rh.sched, rh.verify = ctypes.pointer(da), ctypes.pointer(sa), ctypes.pointer(va)
    assert lib.spec_round_host(ctypes.byref(rh), 0, None) == spec.SPEC_ERR_INVALID_ARG
    # the scheduled-rows mode: a verify that does not read the schedule's row
    # offsets is refused, and so is host memory the device cannot address
    # (checked before anything is copied or launched)
    sa.a = da.a
    va.ell = sa.ell = ctypes.c_void_p(1024)
    va.x, va.q_tok, va.lse_q = (ctypes.c_void_p(2048), ctypes.c_void_p(3072), ctypes.c_void_p(4096))
    da.x, da.q_tok, da.lse_q = va.x, va.q_tok, va.lse_q
    da.U = da.A = da.Ct = da.x0 = ctypes.c_void_p(8192)
    va.draft = ctypes.pointer(da)
    va.tgt = ctypes.c_void_p(16384)
    da.logit_dtype = da.conf_dtype = va.tgt_dtype = spec.SPEC_F32
    host_tgt = (ctypes.c_float * 16)()
    rh.tgt_host, rh.tgt_scheduled_only = ctypes.cast(host_tgt, ctypes.c_void_p), 1
    sa.row_off, va.tgt_row_off = ctypes.c_void_p(5120), ctypes.c_void_p(6144)
    assert lib.spec_round_host(ctypes.byref(rh), 0, None) == spec.SPEC_ERR_INVALID_ARG
    va.tgt_row_off = sa.row_off
    assert lib.spec_round_host(ctypes.byref(rh), 0, None) == spec.SPEC_ERR_UNSUPPORTED
    v = spec.VerifyArgs()
    v.mode, v.R, v.gamma, v.V = 0, 2, 2, 10
    v.tgt = v.tgt_row_off = v.ell = v.x = v.accept_len = v.out_tok = v.n_out = ctypes.c_void_p(256)
    v.target_temp = 1.0
    assert lib.spec_verify(ctypes.byref(v), 0, None) == spec.SPEC_ERR_INVALID_ARG  # no draft
    v.mode = 7
    assert lib.spec_verify(ctypes.byref(v), 0, None) == spec.SPEC_ERR_INVALID_ARG
    v.mode, v.c_star = 1, ctypes.c_void_p(256)  # c* needs sample mode
    assert lib.spec_verify(ctypes.byref(v), 0, None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_stream_uniforms(0, 1, 0, 0, 0, None, None, None) == spec.SPEC_ERR_INVALID_ARG
    # the wait self-test: limits outside [1 ns, 2 s], no status word, a misaligned one
    assert lib.spec_wait_selftest(0, ctypes.c_void_p(256), None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_wait_selftest(3_000_000_000, ctypes.c_void_p(256), None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_wait_selftest(1000, None, None) == spec.SPEC_ERR_INVALID_ARG
    assert lib.spec_wait_selftest(1000, ctypes.c_void_p(258), None) == spec.SPEC_ERR_ALIGNMENT


def test_missing_library_fails_loudly(spec, monkeypatch):
    monkeypatch.setattr(spec, "_lib", None)
    monkeypatch.setattr(spec, "LIB_PATH", "/nonexistent/libspec.so")
    with pytest.raises(spec.SpecError):
        spec.lib()
