"""The NVFP4S decode kernels' chunk decoding, run on the CPU.

tests/host_nvfp4s.cu forms each row's dot product with x through the
kernels' own chunk function (csrc/nvfp4s.cuh), reading every chunk's bytes at
the kernels' offsets; the result is compared with the oracle's dequantized
row (paired 4:8 sparse NVFP4, "Hardware-Native Joint Sparse-Quantization ...",
App. A) dotted with x in binary64.  The GPU parity test checks the kernels.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_nvfp4s.cu")
CSRC = os.path.join(ROOT, "top_moe_expert_gb300", "csrc")
DEPS = [SRC, os.path.join(CSRC, "nvfp4s.cuh")]
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_nvfp4s.so")


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
    L = ctypes.CDLL(OUT)
    L.nv4_rows_dot.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_void_p, ctypes.c_void_p]
    return L


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


@pytest.mark.parametrize("N,K,seed", [(16, 64, 0), (24, 512, 1), (8, 2048, 2)])
def test_chunk_decoding_matches_the_oracle(emu, N, K, seed):
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((N, K)) * np.exp(rng.uniform(-2, 2, (N, 1))) * 0.02
    p = oracle.nvfp4s_quantize(W)
    x = rng.standard_normal(K).astype(np.float32)
    out = np.empty(N, dtype=np.float64)
    emu.nv4_rows_dot(_p(p["v"]), _p(p["m"]), _p(p["s"]), float(p["alpha"]), N, K, _p(x), _p(out))
    w = {"fmt": "nvfp4s", "v": p["v"][None], "m": p["m"][None], "s": p["s"][None],
         "alpha": np.array([p["alpha"]], dtype=np.float32)}
    ref = np.array([oracle.dequant_row(w, 1, 0, n) @ x.astype(np.float64) for n in range(N)])
    # FP32 sums within each 64-weight chunk: a few ulps of the chunk's magnitude
    scale = np.array([np.abs(oracle.dequant_row(w, 1, 0, n)) @ np.abs(x.astype(np.float64)) for n in range(N)])
    assert (np.abs(out - ref) <= 1e-6 * scale).all()


def test_every_pattern_and_code(emu):
    """All six patterns and all sixteen E2M1 codes, against x = distinct powers
    of two, so that each kept position shows up exactly in the sum."""
    K = 64
    patterns = [a | (b << 2) for a in range(4) for b in range(a + 1, 4)]
    v = np.zeros((1, K // 4), dtype=np.uint8)
    m = np.zeros((1, K // 16), dtype=np.uint8)
    s = np.array([[0x38, 0x40]], dtype=np.uint8)                    # UE4M3 1.0 and 2.0
    for g in range(8):
        nib = patterns[g % 6]
        m[0, g // 2] |= nib << (4 * (g % 2))
        codes = [(4 * g + i) % 16 for i in range(4)]
        v[0, 2 * g] = codes[0] | (codes[1] << 4)
        v[0, 2 * g + 1] = codes[2] | (codes[3] << 4)
    w = {"fmt": "nvfp4s", "v": v[None], "m": m[None], "s": s[None], "alpha": np.array([0.5], dtype=np.float32)}
    dense = oracle.dequant_row(w, 1, 0, 0)
    for pos in range(K):
        x = np.zeros(K, dtype=np.float32)
        x[pos] = 1.0
        out = np.empty(1, dtype=np.float64)
        emu.nv4_rows_dot(_p(v), _p(m), _p(s), 0.5, 1, K, _p(x), _p(out))
        assert out[0] == dense[pos], pos
