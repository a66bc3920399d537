"""The single-token AWQ kernel's index arithmetic, run on the CPU.

tests/host_awq_m1.cu runs the kernel's steps on the host through the
kernel's own lane functions (csrc/decode_awq_m1.cuh), with mma.sync emulated
from the PTX fragment layouts.  Its output is compared with the oracle on
seeded inputs: the item split across CTAs and warps, the piece numbering,
the staged operand orders, the scale / zero addressing and the fold all have
to be right for it to match.  The GPU parity tests check the kernel itself.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from top_moe_expert_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_awq_m1.cu")
HDR = os.path.join(ROOT, "top_moe_expert_gb300", "csrc", "decode_awq_m1.cuh")
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_awq_m1.so")
REL_TOL = 2e-3          # the layer tolerance: max|err| <= 2e-3 max|ref|


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def emu():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    t = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < t:
        os.makedirs(os.path.dirname(OUT), exist_ok=True)
        subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                        "-I", os.path.dirname(HDR), SRC, "-o", OUT], check=True, capture_output=True)
    return ctypes.CDLL(OUT)


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _run(emu, d, I, E, k, seed, xdt, G, ids=None, wts=None, xscale=1.0):
    wl = inputs.Workload("awq_m1_host", M=1, d=d, I=I, E=E, k=k, fmt="awq4", seed=seed)
    x = (inputs.activations(wl, dtype=torch.float32) * xscale).to(xdt)
    if ids is None:
        ids, wts = oracle.topk_softmax(inputs.router_logits(wl, 0), k)
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(1, k)
    wts = np.ascontiguousarray(wts, dtype=np.float32).reshape(1, k)
    q13, s13, z13 = inputs.awq_weights(wl, "w13")
    q2, s2, z2 = inputs.awq_weights(wl, "w2")
    xb = inputs.bits16(x)
    gp = np.full(k * (2 * I // 8) * 4 * 8, np.nan, dtype=np.float32)   # a piece read before written is NaN
    y = np.full(d, np.nan, dtype=np.float32)
    st = np.zeros(2, dtype=np.int32)
    smem = emu.awq_m1_emulate(_p(xb), ctypes.c_int(int(xdt == torch.bfloat16)), _p(ids), _p(wts), _p(q13), _p(s13),
                              _p(z13), _p(q2), _p(s2), _p(z2), _p(gp), _p(y), k, d, I, E, G, _p(st))
    assert smem > 0, (smem, st)
    ref = oracle.moe_layer(x.to(torch.float64).numpy(), ids, wts.astype(np.float64), E,
                           {"fmt": "awq4", "q": q13, "s": s13, "z": z13},
                           {"fmt": "awq4", "q": q2, "s": s2, "z": z2})["y"][0]
    assert np.all(np.isfinite(y))
    invalid = int(np.sum((ids < 0) | (ids >= E)))
    assert st[0] == invalid
    scale = np.abs(ref).max()
    err = np.abs(y.astype(np.float64) - ref).max()
    assert err <= REL_TOL * scale, (err, scale)
    return smem


@pytest.mark.parametrize("d,I,E,k,G", [(1024, 256, 16, 4, 152), (1024, 256, 16, 4, 37), (2048, 768, 8, 8, 152),
                                       (2048, 768, 8, 8, 148), (1024, 512, 12, 3, 152)])
@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
def test_host_emulation_matches_oracle(emu, d, I, E, k, G, xdt):
    smem = _run(emu, d, I, E, k, 7, xdt, G)
    assert smem <= 220 * 1024


def test_host_emulation_activation_scales(emu):
    # the power-of-two staging of x keeps tiny and large activations exact
    _run(emu, 2048, 768, 8, 8, 3, torch.float16, 152, xscale=1e-3)
    _run(emu, 2048, 768, 8, 8, 3, torch.bfloat16, 152, xscale=3e3)


def test_host_emulation_duplicate_and_invalid_routes(emu):
    _run(emu, 1024, 512, 16, 6, 5, torch.float16, 152, ids=[3, 3, -1, 16, 0, 15],
         wts=[0.3, 0.2, 0.1, 0.1, 0.2, 0.1])
    _run(emu, 1024, 256, 16, 1, 5, torch.float16, 152, ids=[4], wts=[1.0])


def test_host_emulation_no_valid_route_gives_zero(emu):
    d, I, E, k = 1024, 128, 4, 2
    wl = inputs.Workload("awq_m1_host", M=1, d=d, I=I, E=E, k=k, fmt="awq4", seed=5)
    q13, s13, z13 = inputs.awq_weights(wl, "w13")
    q2, s2, z2 = inputs.awq_weights(wl, "w2")
    xb = inputs.bits16(inputs.activations(wl, dtype=torch.float16))
    ids = np.array([-1, 99], dtype=np.int32)
    wts = np.array([0.5, 0.5], dtype=np.float32)
    gp = np.zeros(k * (2 * I // 8) * 4 * 8, dtype=np.float32)
    y = np.full(d, np.nan, dtype=np.float32)
    st = np.zeros(2, dtype=np.int32)
    assert emu.awq_m1_emulate(_p(xb), 0, _p(ids), _p(wts), _p(q13), _p(s13), _p(z13), _p(q2), _p(s2), _p(z2),
                              _p(gp), _p(y), k, d, I, E, 152, _p(st)) > 0
    assert st[0] == 2
    assert np.all(y == 0)
