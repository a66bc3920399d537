"""The C-ABI library builds, loads and exports what include/*.h declares.

CPU only: no call here launches a kernel.  Host-side entry points (status
names, capacities, workspace sizes) are exercised, and argument validation is
checked to reject bad calls before anything would reach the GPU.
"""
import ctypes
import glob
import os
import re

import pytest

import top_moe_expert_gb300 as moe
from top_moe_expert_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "moe_ffn_decode" in names and "moe_align_block_size" in names
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding knows every declared entry point
    assert set(names) <= set(moe._PROTOS), set(names) - set(moe._PROTOS)


def test_exchange_stall_hook_validates_its_argument(L):
    # host only: sets a process-wide flag read at the next launch
    assert L.moe_debug_exchange_stall(2) == 1 and L.moe_debug_exchange_stall(-1) == 1
    assert L.moe_debug_exchange_stall(1) == 0 and L.moe_debug_exchange_stall(0) == 0


def test_status_names_and_version(L):
    for code, name in moe.STATUS_NAMES.items():
        assert L.moe_status_string(code).decode() == name
    assert L.moe_abi_version() == 3


def test_align_capacity_bound():
    # the packed-AWQ study's shape: 168 routes, worst case every route alone
    cr, cb = moe.moe_align_capacity(21, 8, 128, 8)
    assert cr == 168 + 128 * 7 and cb == cr // 8
    cr, cb = moe.moe_align_capacity(1, 8, 128, 8)
    assert cr == 8 * 8 and cb == 8
    assert moe.moe_align_workspace_size(21, 8, 128, 8) == 0
    assert moe.moe_align_workspace_size(16384, 8, 128, 16) == 64 * 128 * 4


def test_decode_workspace_size():
    _r256 = lambda n: (n + 255) // 256 * 256
    # 256 + 80 KiB reserved for the single-token kernel (its CTA count and its
    # h exchange words), then h [M*k][I] f32 of every other decode path
    R = 256 + 80 * 1024
    assert moe.moe_ffn_decode_workspace_size(65, 8, 512, 768) == R + 65 * 8 * 768 * 4
    assert moe.moe_ffn_decode_workspace_size(1, 8, 512, 768) == R + 8 * 768 * 4
    assert moe.moe_ffn_decode_workspace_size(3, 8, 512, 100) % 256 == 0
    for M, k, d, I in ((2, 8, 512, 768), (64, 8, 512, 768), (1, 8, 2048, 768)):
        assert moe.moe_ffn_decode_workspace_size(M, k, d, I) == R + _r256(M * k * I * 4)


def _r256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("M,k,d,I,b", [(21, 8, 2048, 768, 8), (64, 8, 2048, 768, 16), (512, 8, 2048, 768, 64),
                                       (8, 8, 7168, 2048, 16), (3, 4, 1024, 256, 136)])
def test_grouped_workspace_size_matches_documented_layout(M, k, d, I, b):
    """moe_ffn_grouped_workspace_size is the larger of the documented
    layouts: MXFP8 [Xq | Xs | Hq | Hs | Yr | D] and AWQ [Xg | Hg | Yr | D],
    each part rounded up to 256 bytes."""
    cap_rows = moe.moe_align_capacity(M, k, 128, b)[0]
    cap_blocks = cap_rows // b
    n_mma = (b + 15) // 16 * 16
    nsf = (n_mma + 127) // 128
    mx = (_r256(cap_rows * d) + _r256(cap_blocks * (d // 128) * nsf * 512) + _r256(cap_rows * I)
          + _r256(cap_blocks * (I // 128) * nsf * 512) + _r256(M * k * d * 4) + _r256(cap_blocks * 4))
    awq = _r256(cap_rows * d * 2) + _r256(cap_rows * I * 2) + _r256(M * k * d * 4) + _r256(cap_blocks * 4)
    assert moe.moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows) == max(mx, awq)


def test_host_validation_rejects_before_launch(L):
    # invalid shapes / null pointers return synchronously, nothing launched
    assert L.moe_topk_softmax(None, 4, 128, 0, None, None, None) == 1
    assert L.moe_topk_softmax(None, 4, 8, 9, None, None, None) == 1
    assert L.moe_align_block_size(None, 1, 8, 2048, 8, None, None, None, 64, 8, None, 0, None, None) == 2
    assert L.moe_align_block_size(16, 21, 8, 128, 8, 16, 16, 16, 100, 100, None, 0, None, None) == 3
    assert L.moe_mxfp8_quantize(None, 2, 4, 33, None, None, None) == 1
    assert L.moe_mxfp8_quantize(None, 1, 4, 32, None, None, None) == 2
    w = moe.moe_weights_t(0, 4, 64, 512, 16, 16, None)
    w2 = moe.moe_weights_t(0, 4, 512, 32, 16, 16, None)
    # W2 K (=I) must match W13 N/2
    bad = moe.moe_weights_t(0, 4, 512, 64, 16, 16, None)
    assert L.moe_ffn_decode(16, 0, 1, 512, 16, 16, 8, ctypes.byref(w), ctypes.byref(bad), 16, 0,
                            None, 0, None, None) == 1
    # workspace missing
    assert L.moe_ffn_decode(16, 0, 1, 512, 16, 16, 8, ctypes.byref(w), ctypes.byref(w2), 16, 0,
                            None, 0, None, None) == 4
    # unsupported output dtype
    assert L.moe_ffn_decode(16, 0, 1, 512, 16, 16, 8, ctypes.byref(w), ctypes.byref(w2), 16, 1,
                            None, 0, None, None) == 2
    # d not a multiple of 512
    w3 = moe.moe_weights_t(0, 4, 64, 256, 16, 16, None)
    w4 = moe.moe_weights_t(0, 4, 256, 32, 16, 16, None)
    assert L.moe_ffn_decode(16, 0, 1, 256, 16, 16, 8, ctypes.byref(w3), ctypes.byref(w4), 16, 0,
                            None, 0, None, None) == 2
    # M == 0 is a no-op that succeeds without touching the GPU
    assert L.moe_topk_softmax(None, 0, 128, 8, None, None, None) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        moe.lib()


def test_python_layout_helper_matches_library():
    """grouped_workspace_layout (used by the tests to find Xq/Hq/Hs) totals the
    MXFP8 layout the library sizes, where that layout is the larger one."""
    for M, k, d, I, b in ((64, 8, 2048, 768, 16), (512, 8, 2048, 768, 64)):
        cap_rows = moe.moe_align_capacity(M, k, 128, b)[0]
        L = moe.grouped_workspace_layout(M, k, d, I, b, cap_rows)
        assert moe.moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows) >= L["total"]
        awq = _r256(cap_rows * d * 2) + _r256(cap_rows * I * 2) + _r256(M * k * d * 4) + _r256(cap_rows // b * 4)
        assert moe.moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows) == max(L["total"], awq)


def test_select_path_at_the_measured_crossover(L):
    """Path choice (host only): one token takes the output-centric path
    where its single-kernel form is built for the format (MXFP8 or 4-bit
    AWQ), and the grouped path otherwise.  The block size is twice
    the expected rows per expert rounded up to a power of two within the
    format's range."""
    D, G = moe.MOE_PATH_DECODE, moe.MOE_PATH_GROUPED
    mx, awq = moe.MOE_W_MXFP8, moe.MOE_W_AWQ4
    sel = lambda M, fmt=mx, k=8, E=128, d=2048, I=768: moe.moe_ffn_select_path(M, k, E, d, I, fmt)
    assert sel(1) == (D, 0)
    # 2*M*k/E rows per expert: 0.25 .. 64 -> 16 up to 64; 128 caps
    assert [sel(M) for M in (2, 3, 4, 64, 256, 512, 16384)] == [(G, 16), (G, 16), (G, 16), (G, 16), (G, 32), (G, 64),
                                                                 (G, 128)]
    assert sel(0) == (D, 0)                                  # an empty batch: the cheap path
    # AWQ: grouped at every M; fixture A (M=21, k=8, E=128) gets b = 8
    assert sel(1, awq) == (D, 0) and sel(21, awq) == (G, 8) and sel(512, awq) == (G, 64)
    assert sel(1, awq, d=3072, I=256) == (G, 8)              # no single-kernel AWQ form at this shape
    # shapes one path does not take go to the other
    assert sel(1, d=1152, I=384) == (G, 16)                  # decode needs d % 512 == 0
    # one token takes the decode path only where its single-kernel form is
    # built (the large-expert shape and k beyond its shared-memory plan go
    # to the grouped path, which is faster there than the two-kernel decode)
    assert sel(1, d=7168, I=2048, E=384) == (G, 16)
    # (every CTA's gate/up stages within one lap of the ring: k <= 8 here)
    assert sel(1, k=8) == (D, 0) and sel(1, k=9) == (G, 16)
    assert sel(1, d=2048, I=1024, k=6) == (D, 0) and sel(1, d=2048, I=1024, k=7) == (G, 16)
    assert sel(64, d=1536, I=96) == (D, 0)                   # grouped needs I % 128 == 0
    assert sel(21, awq, d=9216, I=256) == (D, 0)             # AWQ grouped: d / 128 <= 64
    assert sel(21, awq, d=3072, I=256) == (G, 8)
    with pytest.raises(moe.MoeError) as err:
        sel(4, d=1152, I=96)                                 # neither path
    assert err.value.status == 2
    with pytest.raises(moe.MoeError):
        sel(21, awq, d=1152, I=256)                          # AWQ: neither (d % 256, d % 1024)
    with pytest.raises(moe.MoeError):
        moe.moe_ffn_select_path(4, 8, 128, 2048, 768, 2)       # the retired K-outer MXFP8 layout
    # paired 4:8 sparse NVFP4: one token on its single-kernel form, the W4A4
    # grouped path from two tokens (blocks from 8, as AWQ)
    nv4 = moe.MOE_W_NVFP4S
    assert sel(1, nv4) == (D, 0) and sel(2, nv4) == (G, 8) and sel(512, nv4) == (G, 64)
    assert sel(1, nv4, k=13) == (D, 0) and sel(1, nv4, k=14) == (G, 8)    # the exchange's tag words
    assert sel(1, nv4, d=3072, I=256) == (G, 8)              # no single-kernel NVFP4S form at this shape
    assert sel(4, nv4, d=1152, I=256) == (D, 0)              # grouped needs d % 256 == 0
