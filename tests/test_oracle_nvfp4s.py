"""Pins of the oracle's paired 4:8 sparse NVFP4 weight format (CPU).

"Hardware-Native Joint Sparse-Quantization for Trillion-Scale
Mixture-of-Experts", App. A (feasible set Eq. 6, Figure 3, storage Eq. 7) and
Sec. 3.4 (block scales, Eq. 5).  Each check ties the oracle to something other
than itself: the values the page prints (tests/golden/nvfp4_paired_sparse.json),
a library decoding (torch float8), brute force over the six patterns and the
eight E2M1 magnitudes, Eq. 5's closed form, and a dense numpy recomputation
of the layer from the dequantized weights.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_paired_sparse.json")))
GRID = np.array(GOLDEN["e2m1_magnitudes"], dtype=np.float64)


def _dense(p, K):
    """All rows of one packed matrix, dequantized by the oracle."""
    w = {"fmt": "nvfp4s", "v": p["v"][None], "m": p["m"][None], "s": p["s"][None],
         "alpha": np.array([p["alpha"]], dtype=np.float32)}
    return np.stack([oracle.dequant_row(w, 1, 0, n) for n in range(p["v"].shape[0])])


def _kept(p, n, g):
    nib = (p["m"][n, g // 2] >> (4 * (g % 2))) & 0xF
    return oracle.pair_pattern(int(nib))


def test_e2m1_codes_are_the_printed_grid():
    v = oracle.e2m1_value(np.arange(16))
    np.testing.assert_array_equal(v[:8], GRID)                       # sign bit clear: the grid, in order
    np.testing.assert_array_equal(v[8:], -GRID)                      # sign bit set: its negatives
    assert np.signbit(v[8]) and not np.signbit(v[0])
    assert v.max() == GOLDEN["e2m1_max"]


def test_ue4m3_against_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes[:0x7F].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.ue4m3_value(codes[:0x7F]), ref)
    assert oracle.ue4m3_value(0x7E) == GOLDEN["e4m3_max"]
    assert np.isnan(oracle.ue4m3_value(codes[0x7F:])).all()         # 0x7F and every signed code


def test_six_paired_patterns():
    pats = [oracle.pair_pattern(n) for n in range(16)]
    kept = [p for p in pats if p is not None]
    assert len(kept) == GOLDEN["patterns"]
    assert sorted(kept) == list(itertools.combinations(range(4), 2))
    for p0, p1 in kept:                                              # two adjacent pairs: 4 of 8 positions
        pos = {2 * p0, 2 * p0 + 1, 2 * p1, 2 * p1 + 1}
        assert len(pos) == GOLDEN["group_size"] // 2


def test_storage_is_eq7_bits_per_weight():
    N, K = 24, 256
    p = oracle.nvfp4s_quantize(np.random.default_rng(1).standard_normal((N, K)))
    bits = 8 * (p["v"].nbytes + p["m"].nbytes + p["s"].nbytes)
    assert bits / (N * K) == GOLDEN["bits_per_weight"]


def test_eq5_largest_block_scale_is_448_and_alpha():
    W = np.random.default_rng(2).standard_normal((16, 128)) * 0.02
    p = oracle.nvfp4s_quantize(W)
    assert p["s"].max() == 0x7E and (p["s"] <= 0x7E).all()
    # alpha = 1 / gamma, gamma = 448 / (max |kept weight| / 6), in binary32
    Wd = _dense(p, 128)
    kept_max = max(abs(W[n, 8 * g + 2 * pj + c]) for n in range(16) for g in range(16)
                   for pj in _kept(p, n, g) for c in range(2))
    assert p["alpha"] == np.float32(kept_max / 6.0 / 448.0)
    assert np.abs(Wd).max() <= 6 * 448 * float(p["alpha"])


def test_dequantized_weights_lie_in_the_feasible_set():
    """Eq. 6: every group of 8 is zero outside one of the six patterns, and
    every block of 32 is a UE4M3 scale (times the per-matrix constant) times
    E2M1 grid values."""
    W = np.random.default_rng(3).standard_normal((8, 256))
    p = oracle.nvfp4s_quantize(W)
    Wd = _dense(p, 256)
    alpha = float(p["alpha"])
    for n in range(8):
        for g in range(32):
            p0, p1 = _kept(p, n, g)
            mask = np.zeros(8, dtype=bool)
            mask[[2 * p0, 2 * p0 + 1, 2 * p1, 2 * p1 + 1]] = True
            assert (Wd[n, 8 * g:8 * g + 8][~mask] == 0).all()
        for b in range(8):
            s = alpha * oracle.ue4m3_value(p["s"][n, b])
            assert np.isin(np.abs(Wd[n, 32 * b:32 * b + 32]) / s, GRID).all()


def test_patterns_keep_the_most_energy():
    """Brute force over the six patterns: the kept pairs carry the most
    energy (random data has no ties)."""
    W = np.random.default_rng(4).standard_normal((6, 128))
    p = oracle.nvfp4s_quantize(W)
    for n in range(6):
        for g in range(16):
            w = W[n, 8 * g:8 * g + 8]
            en = lambda pp: sum(w[2 * j] ** 2 + w[2 * j + 1] ** 2 for j in pp)
            best = max(itertools.combinations(range(4), 2), key=en)
            assert _kept(p, n, g) == best


def test_equal_pairs_keep_the_lowest_indices():
    W = np.ones((1, 32))
    p = oracle.nvfp4s_quantize(W)
    assert all(_kept(p, 0, g) == (0, 1) for g in range(4))


def test_value_codes_are_the_nearest_grid_point_ties_to_even():
    """Brute force: each kept weight's code is the E2M1 magnitude nearest to
    |w| / (alpha * scale), an exact tie going to the even code, saturating
    at 6; the sign bit is the weight's sign."""
    rng = np.random.default_rng(5)
    W = rng.standard_normal((8, 128)) * np.exp(rng.uniform(-3, 3, (8, 1)))
    p = oracle.nvfp4s_quantize(W)
    Wd = _dense(p, 128)
    alpha = float(p["alpha"])
    for n in range(8):
        for g in range(16):
            s = alpha * oracle.ue4m3_value(p["s"][n, (8 * g) // 32])
            for i, (pj, c) in enumerate((pj, c) for pj in _kept(p, n, g) for c in range(2)):
                w = W[n, 8 * g + 2 * pj + c]
                code = (p["v"][n, 2 * g + i // 2] >> (4 * (i % 2))) & 0xF
                a = abs(w) / s
                dist = np.abs(GRID - min(a, 6.0))
                near = np.flatnonzero(dist == dist.min())
                want = near[0] if len(near) == 1 else near[near % 2 == 0][0]
                assert code & 0x7 == want and bool(code & 0x8) == (w < 0)
                # and the dequantized weight sits at that weight's own position
                assert Wd[n, 8 * g + 2 * pj + c] == np.copysign(GRID[want] * s, w)


def test_ties_round_to_even_codes():
    # the largest weight 6 * 0.875 = 5.25 gives gamma = 448 / (5.25 / 6) =
    # 512, so alpha = 1/512 exactly, the block's scale code RNE(448) = 0x7E
    # and its scale 448/512 = 0.875: each w / 0.875 is an exact midpoint
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    W = np.zeros((1, 64))
    W[0, 0:2], W[0, 8:10], W[0, 16:18], W[0, 24:26] = 0.875 * mids[0:2], 0.875 * mids[2:4], 0.875 * mids[4:6], \
        0.875 * mids[6:8]
    p = oracle.nvfp4s_quantize(W)
    assert float(p["alpha"]) == 1 / 512 and p["s"][0, 0] == 0x7E
    codes = [(p["v"][0, 2 * g + i // 2] >> (4 * (i % 2))) & 0xF for g in range(4) for i in range(2)]
    # 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0, 6 -> 6
    assert oracle.e2m1_value(np.array(codes)).tolist() == [0, 1, 1, 2, 2, 4, 4, 6]


def _layer(M=5, k=2, E=4, d=64, I=32, seed=6):
    rng = np.random.default_rng(seed)
    W13 = rng.standard_normal((E, 2 * I, d)) * 0.05
    W2 = rng.standard_normal((E, d, I)) * 0.05
    x = rng.standard_normal((M, d))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (M, k))
    return x, ids, w, oracle.nvfp4s_quantize_3d(W13), oracle.nvfp4s_quantize_3d(W2)


def _dense_3d(w, E):
    return np.stack([np.stack([oracle.dequant_row(w, E, e, n) for n in range(w["v"].shape[1])])
                     for e in range(E)])


def test_layer_equals_dense_recomputation():
    """The oracle layer on packed weights equals SwiGLU experts evaluated with
    numpy on the dequantized dense matrices (an independent formulation)."""
    M, k, E, d, I = 5, 2, 4, 64, 32
    x, ids, w, w13, w2 = _layer(M, k, E, d, I)
    y = oracle.moe_layer(x, ids, w, E, w13, w2)["y"]
    D13, D2 = _dense_3d(w13, E), _dense_3d(w2, E)
    ref = np.zeros((M, d))
    for t in range(M):
        for j in range(k):
            e = ids[t, j]
            g, u = D13[e, :I] @ x[t], D13[e, I:] @ x[t]
            ref[t] += w[t, j] * (D2[e] @ (g / (1 + np.exp(-g)) * u))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_invalid_metadata_is_refused():
    x, ids, w, w13, w2 = _layer()
    w13["m"] = w13["m"].copy()
    w13["m"][0, 0, 0] = 0x00                                         # pair indices (0, 0): not a pattern
    with pytest.raises(ValueError):
        oracle.moe_layer(x, ids, w, 4, w13, w2)
