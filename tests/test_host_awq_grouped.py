"""The small-block grouped AWQ kernel's index arithmetic, run on the CPU.

tests/host_awq_grouped.cu runs the kernel's two phases and the combine on the
host through the kernel's own lane functions (csrc/grouped_awq_mma.cuh), with
mma.sync emulated from the PTX fragment layouts, on the oracle's alignment of
seeded routes.  The result is compared with the exact oracle; the unit split,
the staged operands, the per-block completion counts and the piece of Yr each
route owns all have to be right for it to match.  The GPU parity tests check
the kernel itself.
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
SRC = os.path.join(ROOT, "tests", "host_awq_grouped.cu")
CSRC = os.path.join(ROOT, "top_moe_expert_gb300", "csrc")
DEPS = [SRC, os.path.join(CSRC, "grouped_awq_mma.cuh"), os.path.join(CSRC, "decode_awq_m1.cuh")]
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_awq_grouped.so")
REL_TOL = 2e-3          # the layer tolerance: max|err| <= 2e-3 max|ref|


@pytest.fixture(scope="module")
def emu():
    nvcc = next((c for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc")
                 if c and os.path.exists(c)), None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    t = max(os.path.getmtime(p) for p in DEPS)
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < t:
        os.makedirs(os.path.dirname(OUT), exist_ok=True)
        subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC, SRC, "-o", OUT],
                       check=True, capture_output=True)
    return ctypes.CDLL(OUT)


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _run(emu, wl, b, xdt, G, ids=None, w=None, layer=None):
    x = inputs.activations(wl, dtype=xdt)
    if ids is None:
        ids, w = oracle.topk_softmax(inputs.router_logits(wl, 0), wl.k)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    q13, s13, z13, q2, s2, z2 = layer if layer is not None else (*inputs.awq_weights(wl, "w13"),
                                                                  *inputs.awq_weights(wl, "w2"))
    srt, ex, npp, _ = oracle.align(ids, wl.E, b)
    M, k, d, I = wl.M, wl.k, wl.d, wl.I
    gu = np.full(M * k * 2 * I, np.nan, dtype=np.float32)
    yr = np.full(M * k * d, np.nan, dtype=np.float32)       # entries never written stay NaN
    y = np.full(M * d, np.nan, dtype=np.float32)
    xb = inputs.bits16(x)
    rc = emu.awq_grouped_emulate(_p(xb), int(xdt == torch.bfloat16), _p(ids), _p(w), _p(srt), _p(ex), npp, _p(q13),
                                 _p(s13), _p(z13), _p(q2), _p(s2), _p(z2), _p(gu), _p(yr), _p(y), M, k, d, I, wl.E,
                                 b, G)
    assert rc > 0, rc
    assert rc <= 220 * 1024
    y = y.reshape(M, d)
    ref = oracle.moe_layer(x.to(torch.float64).numpy(), ids, w.astype(np.float64), wl.E,
                           {"fmt": "awq4", "q": q13, "s": s13, "z": z13},
                           {"fmt": "awq4", "q": q2, "s": s2, "z": z2})["y"]
    assert np.all(np.isfinite(y))
    scale = np.abs(ref).max()
    err = np.abs(y.astype(np.float64) - ref).max()
    assert err <= REL_TOL * scale, (err, scale)
    return y


SMALL = inputs.Workload("awq_grouped_host", M=40, d=1024, I=256, E=16, k=4, fmt="awq4", seed=8)


@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
def test_block_sizes_agree_and_match_oracle(emu, xdt):
    layer = (*inputs.awq_weights(SMALL, "w13"), *inputs.awq_weights(SMALL, "w2"))
    y8 = _run(emu, SMALL, 8, xdt, 152, layer=layer)
    y16 = _run(emu, SMALL, 16, xdt, 152, layer=layer)
    y16b = _run(emu, SMALL, 16, xdt, 37, layer=layer)
    # a route's rows do not depend on its block's other rows or on the grid
    assert np.array_equal(y8, y16) and np.array_equal(y16, y16b)


def test_shapes_not_multiple_of_256(emu):
    wl = inputs.Workload("awq_grouped_host_1152", M=9, d=1152, I=384, E=8, k=3, fmt="awq4", seed=4)
    _run(emu, wl, 16, torch.float16, 152)


def test_duplicate_and_invalid_routes(emu):
    wl = inputs.Workload("awq_grouped_host_dup", M=6, d=1024, I=256, E=8, k=3, fmt="awq4", seed=6)
    ids = np.array([[1, 1, 7], [2, -1, 9], [0, 3, 3], [5, 5, 5], [8, 2, 4], [6, 0, 1]], dtype=np.int32)
    w = np.random.default_rng(2).uniform(0.1, 1.0, size=(6, 3)).astype(np.float32)
    _run(emu, wl, 8, torch.bfloat16, 152, ids=ids, w=w)


def test_many_routes_per_expert(emu):
    # experts with more than 16 routes span several blocks
    wl = inputs.Workload("awq_grouped_host_many", M=64, d=1024, I=256, E=4, k=2, fmt="awq4", seed=5)
    _run(emu, wl, 16, torch.float16, 152)
