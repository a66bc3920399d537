"""The small-batch MXFP8 kernel's index arithmetic, run on the CPU.

tests/host_mx_grouped.cu runs the kernel's two phases and the combine on the
host through the kernel's own lane functions (csrc/grouped_mx_mma.cuh and
csrc/decode_mx_m1.cuh), with mma.sync emulated from the PTX fragment
layouts, on the oracle's alignment of seeded routes into blocks of 16 rows.
The result is compared with the exact oracle, and a token's rows are checked
to be independent of the rest of the batch bit for bit.
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
SRC = os.path.join(ROOT, "tests", "host_mx_grouped.cu")
CSRC = os.path.join(ROOT, "top_moe_expert_gb300", "csrc")
DEPS = [SRC, os.path.join(CSRC, "grouped_mx_mma.cuh"), os.path.join(CSRC, "decode_mx_m1.cuh"),
        os.path.join(CSRC, "decode_awq_m1.cuh")]
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_mx_grouped.so")
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


def _emulate(emu, wl, x, ids, w, weights, G):
    q13, s13, q2, s2 = weights
    M, k, d, I = x.shape[0], ids.shape[1], wl.d, wl.I
    srt, ex, npp, _ = oracle.align(ids, wl.E, 16)
    gu = np.full(M * k * 2 * I, np.nan, dtype=np.float32)
    yr = np.full(M * k * d, np.nan, dtype=np.float32)
    y = np.full(M * d, np.nan, dtype=np.float32)
    xb = inputs.bits16(x)
    rc = emu.mx_grouped_emulate(_p(xb), _p(ids), _p(w), _p(srt), _p(ex), npp, _p(q13), _p(s13), _p(q2), _p(s2),
                                _p(gu), _p(yr), _p(y), M, k, d, I, wl.E, G)
    assert rc > 0, rc
    assert rc <= 220 * 1024
    return y.reshape(M, d)


def _check(wl, x, ids, w, weights, y):
    q13, s13, q2, s2 = weights
    ref = oracle.moe_layer(x.to(torch.float64).numpy(), ids, w.astype(np.float64), wl.E,
                           {"fmt": "mxfp8", "q": q13, "s": s13}, {"fmt": "mxfp8", "q": q2, "s": s2})["y"]
    assert np.all(np.isfinite(y))
    scale = np.abs(ref).max()
    err = np.abs(y.astype(np.float64) - ref).max()
    assert err <= REL_TOL * scale, (err, scale)


def test_matches_oracle_and_rows_independent_of_batch(emu):
    wl = inputs.Workload("mx_small_host", M=12, d=1024, I=256, E=16, k=4, seed=8)
    weights = _weights(wl)
    x = inputs.activations(wl)
    ids, w = oracle.topk_softmax(inputs.router_logits(wl, 0), wl.k)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = _emulate(emu, wl, x, ids, w, weights, 152)
    _check(wl, x, ids, w, weights, y)
    # two tokens alone, another grid: the same bits as inside the batch
    y2 = _emulate(emu, wl, x[3:5], ids[3:5].copy(), w[3:5].copy(), weights, 37)
    assert np.array_equal(y2, y[3:5])


def test_decode_shape_and_invalid_routes(emu):
    wl = inputs.Workload("mx_small_host_2048", M=4, d=2048, I=768, E=12, k=8, seed=5)
    weights = _weights(wl)
    x = inputs.activations(wl)
    ids, w = oracle.topk_softmax(inputs.router_logits(wl, 0), wl.k)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    ids[1, 2] = -1
    ids[2, 0] = wl.E
    _check(wl, x, ids, w, weights, _emulate(emu, wl, x, ids, w, weights, 152))


def test_many_routes_per_expert(emu):
    wl = inputs.Workload("mx_small_host_many", M=40, d=1024, I=256, E=3, k=2, seed=6)
    weights = _weights(wl)
    x = inputs.activations(wl)
    ids, w = oracle.topk_softmax(inputs.router_logits(wl, 0), wl.k)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    _check(wl, x, ids, w, weights, _emulate(emu, wl, x, ids, w, weights, 152))
