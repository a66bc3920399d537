"""The single-token kernels' CTA split, run on the CPU.

tests/host_split.cu calls the kernels' own split (32-bit arithmetic) for
every CTA; each CTA's share is checked against the even split written out
in 64-bit integers: the (route, neuron) pairs q = r * I + n in
[nv * I * c / G, nv * I * (c + 1) / G) and the output rows in
[d * c / G, d * (c + 1) / G), so that the CTAs' shares tile both spaces
exactly once, with the stage counts that follow from them.  The shapes are
every (d, I) the single-token kernels are built for, every route count up
to 32, and grids from 1 CTA to more SMs than this GPU has.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_split.cu")
CSRC = os.path.join(ROOT, "top_moe_expert_gb300", "csrc")
DEPS = [SRC, os.path.join(CSRC, "pipe_common.cuh")]
OUT = os.path.join(ROOT, "top_moe_expert_gb300", "_build", "host_split.so")

SHAPES = [(512, 256), (1024, 256), (1024, 512), (2048, 512), (2048, 768), (2048, 1024)]
GRIDS = [1, 7, 132, 148, 152, 160, 264]


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
    L.split_all.argtypes = [ctypes.c_int] * 6 + [ctypes.c_void_p]
    return L


def _reference(nv, I, d, G, RPS, PS):
    c = np.arange(G, dtype=np.int64)
    q_lo = nv * I * c // G
    P = nv * I * (c + 1) // G - q_lo
    o0 = d * c // G
    nrows = d * (c + 1) // G - o0
    S = (P + PS - 1) // PS
    SW = np.where(nrows > 0, (nv + RPS - 1) // RPS, 0)
    return np.stack([q_lo, P, S, o0, nrows, SW], axis=1)


@pytest.mark.parametrize("d,I", SHAPES)
def test_split_matches_the_even_split(emu, d, I):
    for G in GRIDS:
        for nv in range(1, 33):
            for RPS, PS in ((1, 4), (2, 8), (3, 4)):
                out = np.zeros((G, 6), dtype=np.int32)
                emu.split_all(nv, I, d, G, RPS, PS, out.ctypes.data)
                ref = _reference(nv, I, d, G, RPS, PS)
                np.testing.assert_array_equal(out, ref, err_msg=f"nv={nv} I={I} d={d} G={G}")
                # the shares tile both spaces exactly once
                assert out[0, 0] == 0 and out[0, 3] == 0
                assert (out[1:, 0] == out[:-1, 0] + out[:-1, 1]).all()
                assert (out[1:, 3] == out[:-1, 3] + out[:-1, 4]).all()
                assert out[-1, 0] + out[-1, 1] == nv * I and out[-1, 3] + out[-1, 4] == d
