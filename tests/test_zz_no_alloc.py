"""The allocation-free decode entry point against the regular one and the
oracle.

moe_ffn_decode_noalloc serves callers that cannot hand the library device
memory (strict graph capture, pre-planned serving memory, operator plugins);
its intermediate lives in a fixed array inside the library.  This file runs
last so that a stop-at-first-failure run has already run every other test,
and it builds all of its own inputs, so it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import top_moe_expert_gb300 as moe
from top_moe_expert_gb300 import inputs

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3      # the layer tolerance used by the other decode tests


def _layer():
    wl = inputs.TINY                      # M=21, d=512, I=256, E=128, k=8
    dev = "cuda"
    f13 = torch.from_numpy(inputs.weights_fp32(wl, "w13")).to(dev)
    f2 = torch.from_numpy(inputs.weights_fp32(wl, "w2")).to(dev)
    q13, s13 = moe.moe_mxfp8_quantize(f13)
    q2, s2 = moe.moe_mxfp8_quantize(f2)
    ids, w = oracle.topk_softmax(inputs.router_logits(wl), wl.k)
    x = inputs.activations(wl).to(dev)
    return (wl, x, torch.from_numpy(ids).to(dev), torch.from_numpy(w.astype(np.float32)).to(dev),
            moe.Weights(moe.MOE_W_MXFP8, q13, s13), moe.Weights(moe.MOE_W_MXFP8, q2, s2))


def _oracle_y(wl, x, ids, w):
    """The oracle's exact-mode layer on its own MXFP8 codes of the same fp32
    draws (checked equal to the device codes by the other GPU tests)."""
    oq13, os13 = oracle.mxfp8_quantize_3d(inputs.weights_fp32(wl, "w13").astype(np.float64))
    oq2, os2 = oracle.mxfp8_quantize_3d(inputs.weights_fp32(wl, "w2").astype(np.float64))
    return oracle.moe_layer(x.cpu().to(torch.float64).numpy(), ids.cpu().numpy(),
                            w.cpu().numpy().astype(np.float64), wl.E, {"fmt": "mxfp8", "q": oq13, "s": os13},
                            {"fmt": "mxfp8", "q": oq2, "s": os2})["y"]


def _call_c_abi(x, ids, w, w13, w2, y, status):
    """Straight through the C ABI (ctypes), no Python wrapper logic."""
    L = moe.lib()
    a, b = w13.c_struct(), w2.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.moe_ffn_decode_noalloc(ctypes.c_void_p(x.data_ptr()), moe.MOE_BF16, x.shape[0], x.shape[1],
                                    ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()), ids.shape[1],
                                    ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(y.data_ptr()),
                                    moe.MOE_FP32, ctypes.c_void_p(status.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_on_two_calls():
    assert torch.cuda.is_available()
    wl, x, ids, w, w13, w2 = _layer()
    ref = moe.moe_ffn_decode(x, ids, w, w13, w2, out_dtype=torch.float32)
    scale = float(ref.abs().max())
    exact = _oracle_y(wl, x, ids, w)
    escale = float(np.abs(exact).max())
    for call in range(2):                  # the shared array is reused by the second call
        y = torch.full_like(ref, float("nan"))
        status = torch.zeros(2, dtype=torch.int32, device="cuda")
        assert _call_c_abi(x, ids, w, w13, w2, y, status) == moe.MOE_OK
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        err = float((y - ref).abs().max())
        assert err <= REL_TOL * scale, (call, err, scale)
        # the same kernels with the same summation order: the same bits
        assert torch.equal(y, ref), call
        eerr = float(np.abs(y.cpu().double().numpy() - exact).max())
        assert eerr <= REL_TOL * escale, (call, eerr, escale)
    # a second, different batch through the same array
    x2 = inputs.activations(wl, step=1).to("cuda")
    ref2 = moe.moe_ffn_decode(x2, ids, w, w13, w2, out_dtype=torch.float32)
    y2 = moe.moe_ffn_decode_noalloc(x2, ids, w, w13, w2, out_dtype=torch.float32)
    assert float((y2 - ref2).abs().max()) <= REL_TOL * float(ref2.abs().max())


def test_noalloc_rejects_oversized_intermediate():
    # M*k*I*4 = 64 * 8 * 2304 * 4 bytes = 4.5 MiB > the fixed 4 MiB: refused
    # with MOE_ERR_CAPACITY before anything is launched (weights unread)
    M, k, d, I, E = 64, 8, 512, 2304, 4
    w13 = moe.Weights(moe.MOE_W_MXFP8, torch.zeros((E, 2 * I, d), dtype=torch.uint8, device="cuda"),
                      torch.zeros((E, 2 * I, d // 32), dtype=torch.uint8, device="cuda"))
    w2 = moe.Weights(moe.MOE_W_MXFP8, torch.zeros((E, d, I), dtype=torch.uint8, device="cuda"),
                     torch.zeros((E, d, I // 32), dtype=torch.uint8, device="cuda"))
    x = torch.zeros((M, d), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    y = torch.empty((M, d), dtype=torch.float32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert _call_c_abi(x, ids, w, w13, w2, y, status) == 3      # MOE_ERR_CAPACITY
