"""spec_draft_sample_static: the draft stage with library-owned scratch memory,
for callers that cannot allocate device memory themselves.  Through the C ABI,
its outputs must equal those of spec_draft_sample (caller workspace) on the
same inputs, on two calls in a row (the shared scratch keeps the last call's
contents, so the second call checks that everything that must start at zero
is cleared)."""
import ctypes

import pytest
import torch

import synth
import verify_sampling_gb300 as vs

pytestmark = pytest.mark.gpu

CASES = {
    "fused_fp32": synth.WORKLOADS["c5"].scaled(R=130, gamma=3, V=4100, d=64),
    "fused_bf16": synth.WORKLOADS["c2"].scaled(R=7, gamma=4, V=8192, d=64),
    "generic_fp32": synth.WORKLOADS["tiny"],
}


def _static_call(din, outs, seed):
    a = vs._draft_struct(din, outs, None, None)
    lib = vs.lib()
    lib.spec_draft_sample_static.argtypes = [ctypes.POINTER(vs.DraftArgs), ctypes.c_uint64,
                                            ctypes.c_void_p]
    lib.spec_draft_sample_static.restype = ctypes.c_int
    rc = lib.spec_draft_sample_static(ctypes.byref(a), seed, vs._stream_handle(None))
    assert rc == vs.SPEC_OK, lib.spec_error_string(rc)


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_entry_point(name):
    wl = CASES[name]
    g = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v)
         for k, v in synth.make_inputs(wl, "cpu").items()}
    din = synth.draft_inputs(g)
    for seed in (11, 12):  # two calls in a row
        ref = vs.draft_sample(din, seed)
        got = vs.draft_outputs(wl.R, wl.gamma, wl.V, "cuda")
        _static_call(din, got, seed)
        torch.cuda.synchronize()
        assert torch.equal(got["x"], ref["x"])
        for key in ("q_tok", "lse_q", "c", "a"):
            assert torch.allclose(got[key], ref[key], rtol=0, atol=1e-5), key


def test_static_scratch_allocates_no_device_memory():
    """The defining property: after a first call (which resolves the scratch
    array's address and loads the kernels), further calls leave the device's
    free memory unchanged (cudaMemGetInfo)."""
    wl = CASES["fused_fp32"]
    g = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v)
         for k, v in synth.make_inputs(wl, "cpu").items()}
    din = synth.draft_inputs(g)
    got = vs.draft_outputs(wl.R, wl.gamma, wl.V, "cuda")
    _static_call(din, got, 3)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for seed in (4, 5, 6):
        _static_call(din, got, seed)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_scratch_rejects_oversized_batches():
    wl = synth.WORKLOADS["tiny"].scaled(R=60000, gamma=20, V=8)
    din = vs.DraftInputs(U=torch.zeros(wl.R, wl.gamma, wl.V, device="cuda"),
                         A=torch.zeros(wl.gamma, wl.V, 8, device="cuda"),
                         Ct=torch.zeros(wl.gamma, wl.V, 8, device="cuda"),
                         x0=torch.zeros(wl.R, dtype=torch.int32, device="cuda"),
                         draft_temp=torch.ones(wl.gamma, device="cuda"),
                         h=torch.zeros(wl.R, wl.gamma, 0, device="cuda"),
                         W1=torch.zeros(wl.V, 0, device="cuda"), w=torch.zeros(0, device="cuda"),
                         sts_temp=torch.ones(wl.gamma, device="cuda"))
    outs = vs.draft_outputs(wl.R, wl.gamma, wl.V, "cuda")
    a = vs._draft_struct(din, outs, None, None)
    lib = vs.lib()
    lib.spec_draft_sample_static.argtypes = [ctypes.POINTER(vs.DraftArgs), ctypes.c_uint64,
                                            ctypes.c_void_p]
    lib.spec_draft_sample_static.restype = ctypes.c_int
    assert lib.spec_draft_sample_static(ctypes.byref(a), 1, None) == vs.SPEC_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["fused_fp32", "generic_fp32"])
def test_static_scratch_rnn_head(name):
    """The RNN head through the static entry point: same tokens and states."""
    wl = CASES[name]
    g = {k: (v.to("cuda") if isinstance(v, torch.Tensor) else v)
         for k, v in synth.make_inputs(wl, "cpu").items()}
    din = synth.draft_inputs(g)
    din.Wrnn = synth.rnn_weights(wl, "cuda")
    din.S = torch.zeros(wl.R, wl.gamma, wl.r, dtype=wl.fac_dtype, device="cuda")
    ref = vs.draft_sample(din, 5)
    torch.cuda.synchronize()
    S_ref = din.S.clone()
    din.S.fill_(float("nan"))
    got = vs.draft_outputs(wl.R, wl.gamma, wl.V, "cuda")
    _static_call(din, got, 5)
    torch.cuda.synchronize()
    assert torch.equal(got["x"], ref["x"])
    assert torch.equal(din.S, S_ref)
    for key in ("q_tok", "lse_q"):
        assert torch.allclose(got[key], ref[key], rtol=0, atol=1e-5), key
