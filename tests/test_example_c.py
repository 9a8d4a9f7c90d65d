"""The standalone C example (examples/round.c): it builds against include/spec.h
and libspec.so alone (CPU), and on a GPU its round equals the Python binding's
on the same inputs (a port of the example's LCG), token for token."""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
R, G, V, RANK, D, E = 4, 3, 1000, 8, 16, 8
SEED = 20261202


def _build(tmp_path) -> str:
    from verify_sampling_gb300 import build as spec_build
    libdir = os.path.dirname(spec_build.build())
    cudalib = next((os.path.join(CUDA, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib",
                                                    "targets/x86_64-linux/lib")
                    if os.path.exists(os.path.join(CUDA, d, "libcudart.so"))), None)
    if shutil.which("gcc") is None or cudalib is None:
        pytest.skip("gcc or libcudart not available")
    exe = str(tmp_path / "round")
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "examples", "round.c"),
           "-L", libdir, f"-Wl,-rpath,{libdir}", "-lspec", "-L", cudalib, f"-Wl,-rpath,{cudalib}",
           "-lcudart", "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_example_builds_against_the_c_abi(tmp_path):
    assert os.access(_build(tmp_path), os.X_OK)


def _lcg(n, state):
    out = np.empty(n, np.float32)
    for i in range(n):
        state = (state * 6364136223846793005 + 1442695040888963407) & 0xFFFFFFFFFFFFFFFF
        out[i] = np.float32((state >> 11) * (1.0 / 9007199254740992.0) * 2.0 - 1.0)
    return out, state


def _inputs():
    st = 0x2545F4914F6CDD1D
    parts = {}
    for name, n, scale in (("U", R * G * V, 2.0), ("A", G * V * RANK, 0.3), ("Ct", G * V * RANK, 0.5),
                           ("h", R * G * D, 1.0), ("W1", V * E, 1.0), ("w", D + E, 0.2)):
        x, st = _lcg(n, st)
        parts[name] = np.float32(scale) * x
    noise, st = _lcg(R * (G + 1) * V, st)
    U = parts["U"].reshape(R, G, V)
    tgt = np.empty((R, G + 1, V), np.float32)
    for r in range(R):
        for j in range(G + 1):
            tgt[r, j] = U[r, min(j, G - 1)] + np.float32(0.5) * noise[(r * (G + 1) + j) * V:
                                                                      (r * (G + 1) + j + 1) * V]
    return parts, tgt


@pytest.mark.gpu
def test_example_round_equals_the_binding(tmp_path):
    import torch

    import verify_sampling_gb300 as vs
    exe = _build(tmp_path)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    lines = [l for l in res.stdout.splitlines() if l.startswith("request")]
    got = {}
    for l in lines:
        m = re.match(r"request (\d+) ell (\d+) accept (\d+) tokens(( -?\d+)*)", l)
        got[int(m.group(1))] = (int(m.group(2)), int(m.group(3)), [int(t) for t in m.group(4).split()])

    parts, tgt = _inputs()
    dev = "cuda"
    t = lambda a, shape: torch.tensor(a.reshape(shape), device=dev)
    din = vs.DraftInputs(U=t(parts["U"], (R, G, V)), A=t(parts["A"], (G, V, RANK)),
                         Ct=t(parts["Ct"], (G, V, RANK)),
                         x0=torch.tensor([(r * 37) % V for r in range(R)], dtype=torch.int32, device=dev),
                         draft_temp=torch.ones(G, device=dev), h=t(parts["h"], (R, G, D)),
                         W1=t(parts["W1"], (V, E)), w=t(parts["w"], (D + E,)),
                         sts_temp=torch.ones(G, device=dev))
    d = vs.draft_sample(din, SEED)
    sps = torch.tensor([1000.0 - 10.0 * i for i in range(R * (G + 1) + 1)], dtype=torch.float32,
                       device=dev)
    s = vs.schedule(d["a"], sps, 1.0, 1.0, R * G, vs.SCHED_EARLY_STOP)
    row_off = torch.arange(R, dtype=torch.int32, device=dev) * (G + 1)
    v = vs.verify(vs.VERIFY_SAMPLE, torch.tensor(tgt.reshape(-1, V), device=dev), row_off, s["ell"],
                  d["x"], SEED, q_tok=d["q_tok"], lse_q=d["lse_q"], draft=din)
    torch.cuda.synchronize()
    ell, acc, out = s["ell"].cpu().tolist(), v["accept_len"].cpu().tolist(), v["out_tok"].cpu().tolist()
    for r in range(R):
        assert got[r] == (ell[r], acc[r], out[r][: acc[r] + 1]), (r, got[r], ell[r], acc[r], out[r])
