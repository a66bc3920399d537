"""The Python binding's argument checks, on CPU.

Every pointer the binding passes to the library is checked first (device,
contiguity, dtype, shape, output capacity), so that a wrong argument raises
ValueError on the host instead of reaching a kernel.  Here the entry points
that launch work are replaced by a recorder: the tests show that valid
arguments reach the C entry point once, and that each kind of wrong argument
is refused before it.  The library's host-only size and capacity functions
are the real ones.
"""
import ctypes
import dataclasses

import pytest
import torch

import top_moe_expert_gb300 as moe

_LAUNCHING = {"moe_topk_softmax", "moe_align_block_size", "moe_mxfp8_quantize",
              "moe_ffn_decode", "moe_ffn_decode_logits", "moe_ffn_decode_noalloc", "moe_grouped_prepare",
              "moe_ffn_grouped", "moe_grouped_prepare_nvfp4s"}


class _Recorder:
    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if name in _LAUNCHING:
            def record(*args):
                self.calls.append((name, args))
                return 0
            return record
        return getattr(self.real, name)


@pytest.fixture
def rec(monkeypatch):
    """CPU tensors stand in for device tensors; launches are recorded."""
    r = _Recorder(moe.lib())
    monkeypatch.setattr(moe, "lib", lambda: r)
    monkeypatch.setattr(moe, "_is_gpu", lambda t: True)
    monkeypatch.setattr(moe, "_stream", lambda stream=None, device=None: ctypes.c_void_p(0))
    return r


def _mx(E, N, K):
    return moe.Weights(moe.MOE_W_MXFP8, torch.zeros((E, N, K), dtype=torch.uint8),
                       torch.zeros((E, N, K // 32), dtype=torch.uint8))


def _awq(E, N, K):
    return moe.Weights(moe.MOE_W_AWQ4, torch.zeros((E, N, K // 8), dtype=torch.int32),
                       torch.zeros((E, N, K // 128), dtype=torch.float16),
                       torch.zeros((E, N // 8, K // 128), dtype=torch.int32))


def _route(M, k):
    return torch.zeros((M, k), dtype=torch.int32), torch.zeros((M, k), dtype=torch.float32)


def test_host_tensors_are_refused_without_the_stand_in():
    # no monkeypatching: a CPU tensor never reaches the library
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        moe.moe_topk_softmax(torch.zeros((4, 16)), 2)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        moe.moe_mxfp8_quantize(torch.zeros((4, 64)))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _mx(4, 256, 256)


def test_valid_calls_reach_the_library_once(rec):
    M, k, d, I, E = 3, 2, 256, 128, 4
    ids, w = _route(M, k)
    x = torch.zeros((M, d), dtype=torch.bfloat16)
    w13, w2 = _mx(E, 2 * I, d), _mx(E, d, I)
    moe.moe_topk_softmax(torch.zeros((M, E)), k)
    aligned = moe.moe_align_block_size(ids, E, 8)
    moe.moe_mxfp8_quantize(torch.zeros((5, 64)))
    y = moe.moe_ffn_decode(x, ids, w, w13, w2, out_dtype=torch.float32)
    moe.moe_ffn_decode_logits(torch.zeros((M, E)), x, k, w13, w2)
    moe.moe_ffn_decode_noalloc(x, ids, w, w13, w2)
    sfa13, sfa2 = moe.moe_grouped_prepare(w13, w2)
    moe.moe_ffn_grouped(x, ids, w, w13, w2, sfa13, sfa2, aligned, 8)
    a13, a2 = _awq(E, 2 * I, d), _awq(E, d, I)
    moe.moe_ffn_decode(x.half(), ids, w, a13, a2)
    moe.moe_ffn_grouped(x.half(), ids, w, a13, a2, None, None, aligned, 8)
    names = [c[0] for c in rec.calls]
    assert names == ["moe_topk_softmax", "moe_align_block_size", "moe_mxfp8_quantize",
                     "moe_ffn_decode", "moe_ffn_decode_logits", "moe_ffn_decode_noalloc", "moe_grouped_prepare",
                     "moe_ffn_grouped", "moe_ffn_decode", "moe_ffn_grouped"]
    assert y.shape == (M, d) and y.dtype == torch.float32
    # the decode call passes M, d, k and the workspace size in bytes
    args = rec.calls[3][1]
    assert (args[2], args[3], args[6]) == (M, d, k)
    assert args[12] == moe.moe_ffn_decode_workspace_size(M, k, d, I)


def _decode_case(bad):
    M, k, d, I, E = 3, 2, 256, 128, 4
    ids, w = _route(M, k)
    x = torch.zeros((M, d), dtype=torch.bfloat16)
    q13, s13 = torch.zeros((E, 2 * I, d), dtype=torch.uint8), torch.zeros((E, 2 * I, d // 32), dtype=torch.uint8)
    kw = {}
    if bad == "ids_dtype":
        ids = ids.long()
    elif bad == "w_shape":
        w = torch.zeros((M, k + 1))
    elif bad == "x_dtype":
        x = x.to(torch.int16)
    elif bad == "x_strided":
        x = torch.zeros((d, M), dtype=torch.bfloat16).t()
    elif bad == "y_shape":
        kw["y"] = torch.zeros((M, d - 1), dtype=torch.float32)
    elif bad == "y_dtype":
        kw["y"] = torch.zeros((M, d), dtype=torch.float16)
    elif bad == "status_short":
        kw["dev_status"] = torch.zeros(1, dtype=torch.int32)
    elif bad == "w13_dtype":
        q13 = q13.to(torch.int8)
    elif bad == "w13_scale_shape":
        s13 = s13[:, :, :-1].contiguous()
    elif bad == "ws_strided":
        kw["ws"] = torch.zeros((64, 2), dtype=torch.uint8).t()
    w13 = moe.Weights(moe.MOE_W_MXFP8, q13, s13)
    if bad == "w2_K":
        w2 = moe.Weights(moe.MOE_W_MXFP8, torch.zeros((E, d, 100), dtype=torch.uint8),
                         torch.zeros((E, d, 3), dtype=torch.uint8))
    else:
        w2 = _mx(E, d, I)
    moe.moe_ffn_decode(x, ids, w, w13, w2, **kw)


@pytest.mark.parametrize("bad", ["ids_dtype", "w_shape", "x_dtype", "x_strided", "y_shape", "y_dtype",
                                 "status_short", "w13_dtype", "w13_scale_shape", "w2_K", "ws_strided"])
def test_decode_arguments_refused(rec, bad):
    with pytest.raises(ValueError):
        _decode_case(bad)
    assert rec.calls == []


def _awq_case(bad):
    M, k, d, I, E = 3, 2, 256, 128, 4
    ids, w = _route(M, k)
    x = torch.zeros((M, d), dtype=torch.float16)
    q = torch.zeros((E, 2 * I, d // 8), dtype=torch.int32)
    sc = torch.zeros((E, 2 * I, d // 128), dtype=torch.float16)
    z = torch.zeros((E, 2 * I // 8, d // 128), dtype=torch.int32)
    if bad == "scale_dtype":
        sc = sc.float()
    elif bad == "zero_missing":
        z = None
    elif bad == "zero_shape":
        z = z[:, :-1].contiguous()
    elif bad == "q_dtype":
        q = q.to(torch.uint8)
    a13 = moe.Weights(moe.MOE_W_AWQ4, q, sc, z)
    if bad == "N_not_8":
        a2 = moe.Weights(moe.MOE_W_AWQ4, torch.zeros((E, 12, I // 8), dtype=torch.int32),
                         torch.zeros((E, 12, 1), dtype=torch.float16), torch.zeros((E, 1, 1), dtype=torch.int32))
    else:
        a2 = _awq(E, d, I)
    moe.moe_ffn_decode(x, ids, w, a13, a2)


@pytest.mark.parametrize("bad", ["scale_dtype", "zero_missing", "zero_shape", "q_dtype", "N_not_8"])
def test_awq_weights_refused(rec, bad):
    with pytest.raises(ValueError):
        _awq_case(bad)
    assert rec.calls == []


def test_weights_are_immutable_and_device_checked(rec):
    w = _mx(2, 64, 64)
    with pytest.raises(dataclasses.FrozenInstanceError):
        w.q = torch.zeros((2, 64, 64), dtype=torch.uint8)
    with pytest.raises(ValueError, match="is on"):
        w.on("w13", torch.device("cuda", 1))
    w.on("w13", torch.device("cpu"))


def test_output_buffers_must_hold_the_result(rec):
    M, k, E = 5, 2, 8
    with pytest.raises(ValueError):        # topk outputs of the wrong shape
        moe.moe_topk_softmax(torch.zeros((M, E)), k, torch.zeros((M, k + 1), dtype=torch.int32),
                             torch.zeros((M, k)))
    with pytest.raises(ValueError):        # logits must be fp32
        moe.moe_topk_softmax(torch.zeros((M, E), dtype=torch.float16), k)
    with pytest.raises(ValueError):        # quantize outputs too short
        moe.moe_mxfp8_quantize(torch.zeros((4, 64)), torch.zeros(100, dtype=torch.uint8))
    with pytest.raises(ValueError):        # a row length that is not whole scale blocks
        moe.moe_mxfp8_quantize(torch.zeros((4, 40)))
    ids = torch.zeros((M, k), dtype=torch.int32)
    with pytest.raises(ValueError):        # alignment ids must be int32
        moe.moe_align_block_size(ids.long(), E, 4)
    with pytest.raises(ValueError):        # a capacity above the given buffer
        moe.moe_align_block_size(ids, E, 4, cap_rows=64,
                                 out=(torch.zeros(32, dtype=torch.int32), torch.zeros(16, dtype=torch.int32),
                                      torch.zeros(1, dtype=torch.int32)))
    assert rec.calls == []
    # capacities default to the given buffers' lengths
    out = (torch.zeros(48, dtype=torch.int32), torch.zeros(12, dtype=torch.int32), torch.zeros(1, dtype=torch.int32))
    moe.moe_align_block_size(ids, E, 4, out=out)
    args = rec.calls[-1][1]
    assert (args[8], args[9]) == (48, 12)


def test_grouped_needs_the_scale_atoms_for_mxfp8(rec):
    M, k, d, I, E = 3, 2, 256, 128, 4
    ids, w = _route(M, k)
    x = torch.zeros((M, d), dtype=torch.bfloat16)
    w13, w2 = _mx(E, 2 * I, d), _mx(E, d, I)
    aligned = moe.moe_align_block_size(ids, E, 8)
    with pytest.raises(ValueError):
        moe.moe_ffn_grouped(x, ids, w, w13, w2, None, None, aligned, 8)
    sfa13, sfa2 = moe.moe_grouped_prepare(w13, w2)
    with pytest.raises(ValueError):
        moe.moe_ffn_grouped(x, ids, w, w13, w2, sfa13[:-1], sfa2, aligned, 8)
    with pytest.raises(ValueError):        # expert_ids shorter than the block count of the rows
        moe.moe_ffn_grouped(x, ids, w, w13, w2, sfa13, sfa2, (aligned[0], aligned[1][:1], aligned[2]), 8)
    assert [c[0] for c in rec.calls] == ["moe_align_block_size", "moe_grouped_prepare"]


def _nv4(E, N, K):
    return moe.Weights(moe.MOE_W_NVFP4S, torch.zeros((E, N, K // 4), dtype=torch.uint8),
                       torch.zeros((E, N, K // 32), dtype=torch.uint8), torch.zeros((E, N, K // 16), dtype=torch.uint8),
                       torch.ones(E, dtype=torch.float32))


def test_grouped_nvfp4s_needs_its_prepared_buffers(rec):
    M, k, d, I, E = 3, 2, 256, 128, 4
    ids, w = _route(M, k)
    x = torch.zeros((M, d), dtype=torch.bfloat16)
    w13, w2 = _nv4(E, 2 * I, d), _nv4(E, d, I)
    aligned = moe.moe_align_block_size(ids, E, 8)
    with pytest.raises(ValueError):                       # the activation scales must be finite and > 0
        moe.moe_grouped_prepare_nvfp4s(w13, w2, 0.0, 0.1)
    with pytest.raises(ValueError):
        moe.moe_grouped_prepare_nvfp4s(w13, w2, 0.1, float("inf"))
    with pytest.raises(ValueError):                       # MXFP8 weights have no NVFP4S preparation
        moe.moe_grouped_prepare_nvfp4s(_mx(E, 2 * I, d), _mx(E, d, I), 0.1, 0.1)
    p13, p2 = moe.moe_grouped_prepare_nvfp4s(w13, w2, 0.01, 0.02)
    # head + per-expert factors + one 16-byte side record per row and k-step of 128
    assert p13.numel() == 256 + 256 + E * 2 * I * (d // 128) * 16
    assert p2.numel() == 256 + 256 + E * d * (I // 128) * 16
    with pytest.raises(ValueError):
        moe.moe_ffn_grouped(x, ids, w, w13, w2, None, None, aligned, 8)
    with pytest.raises(ValueError):
        moe.moe_ffn_grouped(x, ids, w, w13, w2, p13, p2[:-1], aligned, 8)
    moe.moe_ffn_grouped(x, ids, w, w13, w2, p13, p2, aligned, 8)
    names = [c[0] for c in rec.calls]
    assert names == ["moe_align_block_size", "moe_grouped_prepare_nvfp4s", "moe_ffn_grouped"]
    args = rec.calls[1][1]
    assert abs(args[2] - 0.01) < 1e-9 and abs(args[3] - 0.02) < 1e-9
