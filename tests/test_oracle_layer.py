"""Pins for the oracle's routed expert-FFN layer and top-k routing.

Independent checks (none re-types the oracle's loops):
  * a dense "run every expert on every token, then mask and weight" recompute
    with numpy/PyTorch float64 matmuls over weights decoded by PyTorch's
    float8 casts;
  * k=1, w=1 reduces to one SwiGLU FFN: torch.nn.functional.silu and matmul;
  * a closed-form layer computed by hand (tests/golden/closed_form_layer.json);
  * exact invariants: power-of-two scale linearity, zero up-rows give y=0,
    slot permutation, duplicate experts merge their weights, invalid routes
    contribute nothing;
  * the block-scaled mode against the library quantizer of tests/refdecode.py;
  * top-k routing against torch.topk / torch.softmax.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests import refdecode as rd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_layer(seed, M=5, d=64, I=32, E=6, k=3, fmt="mxfp8"):
    g = np.random.Generator(np.random.PCG64(seed))
    x = torch.from_numpy(g.standard_normal((M, d)).astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    ids = np.stack([g.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    w = g.uniform(0.1, 1.0, size=(M, k))
    w /= w.sum(1, keepdims=True)
    if fmt == "mxfp8":
        q13, s13 = oracle.mxfp8_quantize_3d(g.standard_normal((E, 2 * I, d)) * 0.02)
        q2, s2 = oracle.mxfp8_quantize_3d(g.standard_normal((E, d, I)) * 0.02)
        w13 = {"fmt": "mxfp8", "q": q13, "s": s13}
        w2 = {"fmt": "mxfp8", "q": q2, "s": s2}
        W13 = rd.dequant_mxfp8(q13, s13)
        W2 = rd.dequant_mxfp8(q2, s2)
    else:
        def awq(N, K):
            qv = g.integers(0, 16, size=(E, N, K))
            zv = g.integers(0, 16, size=(E, N, K // 128))
            s = torch.from_numpy(g.uniform(0.005, 0.02, size=(E, N, K // 128)).astype(np.float32)).to(torch.float16)
            q, z = rd.pack_awq(qv, zv)
            sb = s.view(torch.int16).numpy().view(np.uint16)
            return {"fmt": "awq4", "q": q, "s": sb, "z": z}, rd.dequant_awq(q, sb, z)
        w13, W13 = awq(2 * I, d)
        w2, W2 = awq(d, I)
    return x, ids, w, w13, w2, W13, W2


def _dense(x, ids, w, W13, W2, hround=None, xround=None):
    """Every expert on every token with float64 matmuls, then mask and weight."""
    E, twoI, d = W13.shape
    I = twoI // 2
    xt = torch.from_numpy(xround(x) if xround else x)
    y = torch.zeros(x.shape, dtype=torch.float64)
    for e in range(E):
        gu = xt @ torch.from_numpy(W13[e]).T
        h = torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]
        if hround is not None:
            h = torch.from_numpy(hround(h.numpy()))
        ye = h @ torch.from_numpy(W2[e]).T
        coef = torch.from_numpy(((ids == e) * w).sum(1))
        y += coef[:, None] * ye
    return y.numpy()


@pytest.mark.parametrize("fmt", ["mxfp8", "awq4"])
def test_layer_matches_dense_masked_formulation(fmt):
    d = 256 if fmt == "awq4" else 64
    I = 128 if fmt == "awq4" else 32
    x, ids, w, w13, w2, W13, W2 = _random_layer(1, d=d, I=I, fmt=fmt)
    y = oracle.moe_layer(x, ids, w, 6, w13, w2)["y"]
    ref = _dense(x, ids, w, W13, W2)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_k1_w1_is_a_single_swiglu_ffn():
    x, ids, w, w13, w2, W13, W2 = _random_layer(2, k=1)
    w[:] = 1.0
    y = oracle.moe_layer(x, ids, w, 6, w13, w2)["y"]
    for t in range(x.shape[0]):
        e = ids[t, 0]
        xt = torch.from_numpy(x[t])
        g = torch.from_numpy(W13[e, :32]) @ xt
        u = torch.from_numpy(W13[e, 32:]) @ xt
        ffn = torch.from_numpy(W2[e]) @ (torch.nn.functional.silu(g) * u)
        np.testing.assert_allclose(y[t], ffn.numpy(), rtol=1e-12, atol=1e-14)


def test_closed_form_layer():
    """One-hot input and constant rows: h_n = SiLU(a)*b for every n, so
    y_o = w * I * c * SiLU(a) * b (values in tests/golden/closed_form_layer.json,
    computed with math.exp)."""
    g = json.load(open(os.path.join(GOLDEN, "closed_form_layer.json")))
    d, I, E = g["d"], g["I"], g["E"]
    code = {v: c for c, v in enumerate(rd.e4m3_table()) if not math.isnan(v) and c < 128}
    q13 = np.zeros((E, 2 * I, d), dtype=np.uint8)
    q13[:, :I, 0] = code[g["a"]]
    q13[:, I:, 0] = code[g["b"]]
    s13 = np.full((E, 2 * I, d // 32), 127, dtype=np.uint8)
    q2 = np.full((E, d, I), code[g["c"]], dtype=np.uint8)
    s2 = np.full((E, d, I // 32), 127, dtype=np.uint8)
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    ids = np.array([[1]], dtype=np.int32)
    w = np.array([[g["w"]]])
    y = oracle.moe_layer(x, ids, w, E, {"fmt": "mxfp8", "q": q13, "s": s13},
                         {"fmt": "mxfp8", "q": q2, "s": s2})["y"]
    np.testing.assert_allclose(y[0], g["y"], rtol=1e-14)


def test_power_of_two_scale_linearity_and_zero_rows():
    x, ids, w, w13, w2, W13, W2 = _random_layer(3)
    y = oracle.moe_layer(x, ids, w, 6, w13, w2)["y"]
    w2b = dict(w2, s=w2["s"] + 1)                       # every down scale x2
    assert np.array_equal(oracle.moe_layer(x, ids, w, 6, w13, w2b)["y"], 2 * y)
    s13 = w13["s"].copy()
    s13[:, 32:] += 1                                    # every up-row scale x2
    assert np.array_equal(oracle.moe_layer(x, ids, w, 6, dict(w13, s=s13), w2)["y"], 2 * y)
    q13 = w13["q"].copy()
    q13[:, 32:] = 0                                     # up rows all zero
    assert np.all(oracle.moe_layer(x, ids, w, 6, dict(w13, q=q13), w2)["y"] == 0)


def test_slot_permutation_duplicates_and_invalid_routes():
    x, ids, w, w13, w2, W13, W2 = _random_layer(4)
    y = oracle.moe_layer(x, ids, w, 6, w13, w2)["y"]
    perm = [2, 0, 1]
    yp = oracle.moe_layer(x, ids[:, perm], w[:, perm], 6, w13, w2)["y"]
    np.testing.assert_allclose(yp, y, rtol=1e-13, atol=1e-15)
    # duplicate expert: (e, e) with (w1, w2) equals (e) with w1 + w2
    ids_d = ids.copy()
    ids_d[:, 1] = ids_d[:, 0]
    yd = oracle.moe_layer(x, ids_d, w, 6, w13, w2)["y"]
    ids_m = ids_d.copy()
    ids_m[:, 1] = -1
    wm = w.copy()
    wm[:, 0] += wm[:, 1]
    ym = oracle.moe_layer(x, ids_m, wm, 6, w13, w2)["y"]
    np.testing.assert_allclose(yd, ym, rtol=1e-13, atol=1e-15)
    # invalid ids (negative, >= E) contribute nothing
    ids_i = ids.copy()
    ids_i[:, 2] = 6
    w_i = w.copy()
    yi = oracle.moe_layer(x, ids_i, w_i, 6, w13, w2)["y"]
    w_z = w.copy()
    w_z[:, 2] = 0.0
    np.testing.assert_allclose(yi, oracle.moe_layer(x, ids, w_z, 6, w13, w2)["y"], rtol=1e-13, atol=1e-15)


def _mx_rt(v):
    q, s = rd.mx_quantize_lib(np.ascontiguousarray(v.reshape(-1, v.shape[-1])))
    return rd.dequant_mxfp8(q, s).reshape(v.shape)


def test_block_scaled_mode_matches_library_quantizer():
    x, ids, w, w13, w2, W13, W2 = _random_layer(5)
    out = oracle.moe_layer(x, ids, w, 6, w13, w2, mode=oracle.MODE_MX, want_hq=True, want_h=True)
    ref = _dense(x, ids, w, W13, W2, hround=_mx_rt, xround=_mx_rt)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # stage-wise entry: feeding the oracle's own quantized h back changes nothing
    again = oracle.moe_layer(x, ids, w, 6, w13, w2, mode=oracle.MODE_MX,
                             hq_in=out["hq"], hs_in=out["hs"])
    assert np.array_equal(again["y"], out["y"])
    # quantized h codes agree with the library quantizer applied to h
    q, s = rd.mx_quantize_lib(out["h"])
    assert np.array_equal(q, out["hq"]) and np.array_equal(s, out["hs"])


def test_fp16_intermediate_mode_matches_numpy_rounding():
    x, ids, w, w13, w2, W13, W2 = _random_layer(6, d=256, I=128, fmt="awq4")
    y = oracle.moe_layer(x, ids, w, 6, w13, w2, mode=oracle.MODE_H16)["y"]
    ref = _dense(x, ids, w, W13, W2,
                 hround=lambda h: h.astype(np.float16).astype(np.float64))  # numpy rounds f64->f16 directly; torch goes through f32 (double rounding)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_topk_softmax_matches_torch():
    g = np.random.Generator(np.random.PCG64(7))
    logits = g.standard_normal((40, 128)).astype(np.float32)
    ids, w = oracle.topk_softmax(logits, 8)
    lt = torch.from_numpy(logits)
    val, idx = torch.topk(lt, 8, dim=1, sorted=True)
    assert np.array_equal(ids, idx.numpy().astype(np.int32))
    p = torch.softmax(lt.to(torch.float64), dim=1)
    sel = torch.gather(p, 1, idx)
    np.testing.assert_allclose(w, (sel / sel.sum(1, keepdim=True)).numpy(), rtol=1e-14)


def test_topk_ties_go_to_lower_expert_id():
    logits = np.zeros((2, 8), dtype=np.float32)
    logits[0, [6, 2, 4]] = 1.0                           # three-way tie on top
    logits[1, :] = [0.5, 0.25, 0.5, 0.25, 0.0, 0.5, 0.0, 0.0]
    ids, w = oracle.topk_softmax(logits, 4)
    assert ids[0].tolist() == [2, 4, 6, 0]
    assert ids[1].tolist() == [0, 2, 5, 1]
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)
    e = math.exp(1.0)
    np.testing.assert_allclose(w[0], [e / (3 * e + 1)] * 3 + [1 / (3 * e + 1)], rtol=1e-14)
