"""The single-token MXFP8 kernel's index arithmetic, run on the CPU.

tests/host_mx_m1.cu runs the kernel's steps on the host through the kernel's
own lane functions (csrc/decode_mx_m1.cuh), with mma.sync emulated from the
PTX fragment layouts, and its output is compared with the exact oracle on
seeded inputs (weights quantized by the oracle's MXFP8 quantizer, which the
GPU quantizer matches bit for bit).  The GPU parity tests check the kernel
itself.
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
SRC = os.path.join(ROOT, "tests", "host_mx_m1.cu")
CSRC = os.path.join(ROOT, "top_moe_expert_gb300", "csrc")
DEPS = [SRC, os.path.join(CSRC, "decode_mx_m1.cuh"), os.path.join(CSRC, "decode_awq_m1.cuh")]
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_mx_m1.so")
REL_TOL = 2e-3


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


def _weights(wl):
    f13 = inputs.weights_fp32(wl, "w13").astype(np.float64)
    f2 = inputs.weights_fp32(wl, "w2").astype(np.float64)
    q13, s13 = oracle.mxfp8_quantize_3d(f13)
    q2, s2 = oracle.mxfp8_quantize_3d(f2)
    return [np.ascontiguousarray(a) for a in (q13, s13, q2, s2)]


def _run(emu, wl, G, ids=None, w=None, weights=None, xscale=1.0, stage=1):
    x = (inputs.activations(wl, dtype=torch.float32) * xscale).to(torch.bfloat16)[:1]
    if ids is None:
        ids, w = oracle.topk_softmax(inputs.router_logits(wl, 0), wl.k)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(1, wl.k))
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float32).reshape(1, wl.k))
    q13, s13, q2, s2 = weights if weights is not None else _weights(wl)
    gp = np.full(wl.k * (2 * wl.I // 8) * 4 * 8, np.nan, dtype=np.float32)
    y = np.full(wl.d, np.nan, dtype=np.float32)
    st = np.zeros(2, dtype=np.int32)
    xb = inputs.bits16(x)
    rc = emu.mx_m1_emulate(_p(xb), _p(ids), _p(w), _p(q13), _p(s13), _p(q2), _p(s2), _p(gp), _p(y), wl.k, wl.d,
                           wl.I, wl.E, G, stage, _p(st))
    assert rc > 0, (rc, st)
    assert rc <= 220 * 1024
    ref = oracle.moe_layer(x.to(torch.float64).numpy(), ids, w.astype(np.float64), wl.E,
                           {"fmt": "mxfp8", "q": q13, "s": s13}, {"fmt": "mxfp8", "q": q2, "s": s2})["y"][0]
    assert np.all(np.isfinite(y))
    assert st[0] == int(np.sum((ids < 0) | (ids >= wl.E)))
    scale = np.abs(ref).max()
    err = np.abs(y.astype(np.float64) - ref).max()
    assert err <= REL_TOL * max(scale, 1e-30), (err, scale)
    return y


DECODE8 = inputs.Workload("mx_m1_host", M=1, d=2048, I=768, E=8, k=8, seed=3)


def test_decode_shape_matches_oracle_and_grid_independent(emu):
    weights = _weights(DECODE8)
    y152 = _run(emu, DECODE8, 152, weights=weights)
    y148 = _run(emu, DECODE8, 148, weights=weights)
    assert np.allclose(y152, y148, rtol=1e-5, atol=1e-7 * np.abs(y152).max())
    # W2 read from global memory (the form used when its rows do not fit in
    # shared memory) gives the same bits
    assert np.array_equal(_run(emu, DECODE8, 152, weights=weights, stage=0), y152)


def test_small_shapes_scales_and_routes(emu):
    wl = inputs.Workload("mx_m1_host_small", M=1, d=1024, I=256, E=16, k=4, seed=7)
    weights = _weights(wl)
    _run(emu, wl, 152, weights=weights)
    _run(emu, wl, 37, weights=weights, xscale=1e-3)
    _run(emu, wl, 152, weights=weights, xscale=3e3)
    _run(emu, wl, 152, ids=[3, 3, -1, 16], w=[0.4, 0.3, 0.2, 0.1], weights=weights)


def test_large_expert_shape_reads_w2_from_global(emu):
    # d = 7168, I = 2048: the CTA's W2 rows do not fit in shared memory
    wl = inputs.Workload("mx_m1_host_large", M=1, d=7168, I=2048, E=8, k=8, seed=4)
    _run(emu, wl, 152, stage=0)
