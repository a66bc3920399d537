"""Pins of the oracle's run-time activation quantizer Q_a and of its W4A4
layer mode (CPU).

"Hardware-Native Joint Sparse-Quantization for Trillion-Scale
Mixture-of-Experts", Sec. 3.4 and App. D.1: expert activations are quantized
at run time into 32-element blocks with one UE4M3 scale each (the block
scale of Eq. 5), before the first GEMM and again after SwiGLU; the
tensor-wide scales of both operands fold into one factor per expert.  The
checks tie the oracle to values worked by hand below, to brute force over
the eight E2M1 magnitudes, to closed-form invariances (a power-of-two change
of the tensor-wide scale changes no code), and to the exact layer.
"""
import numpy as np

import oracle

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _block(vals):
    v = np.zeros((1, 32), dtype=np.float32)
    v[0, :len(vals)] = vals
    return v


def _q(vals, alpha):
    c, s = oracle.nvfp4_act_quantize(_block(vals), alpha)
    return c[0, :len(vals)].tolist(), int(s[0, 0])


def test_worked_block():
    # alpha = 0.5: r6 = binary32(1/3); amax 6 gives t = binary32(2.00000006) = 2,
    # S = 2, q = 1 / (0.5 * 2) = 1, so each code is the grid point nearest v
    codes, s = _q([6, 3, 1, 0.5, -2, 0, 0.2], 0.5)
    assert oracle.ue4m3_value(s) == 2.0
    assert codes == [7, 5, 2, 1, 8 | 4, 0, 0]
    c, sc = oracle.nvfp4_act_quantize(_block([6, 3, 1, 0.5, -2, 0, 0.2]), 0.5)
    np.testing.assert_array_equal(0.5 * oracle.nvfp4_act_values(c, sc)[0, :7], [6, 3, 1, 0.5, -2, 0, 0])


def test_ties_go_to_the_even_code():
    # as above (S = 2, q = 1): the midpoints between grid points
    codes, _ = _q([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5], 0.5)
    assert GRID[codes[1:]].tolist() == [0, 1, 1, 2, 2, 4, 4]


def test_element_saturates_at_six():
    # amax 6.2: t = 2.0667 rounds to S = 2 (2.25 is farther), so 6.2 * q = 6.2 > 6
    codes, s = _q([6.2, -6.2, 1.0], 0.5)
    assert oracle.ue4m3_value(s) == 2.0 and codes == [7, 15, 2]


def test_scale_saturates_at_448():
    # t = 10000 / 3 is far above 448: S = 448, q = 1/224, 10000/224 > 6
    codes, s = _q([10000.0, -1.0], 0.5)
    assert s == 0x7E and codes[0] == 7
    c, sc = oracle.nvfp4_act_quantize(_block([10000.0]), 0.5)
    assert 0.5 * oracle.nvfp4_act_values(c, sc)[0, 0] == 0.5 * 448 * 6


def test_subnormal_scale():
    # amax 0.01: t = 0.00333 = 1.71 * 2^-9 rounds to the subnormal 2 * 2^-9;
    # q = 1 / (0.5 * 2^-8) = 512 and 0.01 * 512 = 5.12 rounds to 6
    codes, s = _q([0.01], 0.5)
    assert s == 0x02 and oracle.ue4m3_value(s) == 2.0 ** -8 and codes == [7]


def test_scale_underflow_gives_zero_codes_with_signs():
    # t = 3.3e-7 is below half the smallest UE4M3 step (2^-10): S = 0
    codes, s = _q([1e-6, -1e-6, 0.0], 0.5)
    assert s == 0 and codes == [0, 8, 0]


def test_codes_are_nearest_grid_points():
    """Brute force: every magnitude code is a grid point nearest |v * q|, the
    lower-mantissa one on a tie, and the scale is the UE4M3 value nearest
    amax / (6 alpha) (checked against all 127 codes)."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((64, 128)) * rng.uniform(0.01, 20, (64, 1))).astype(np.float32)
    alpha = 0.37
    codes, scales = oracle.nvfp4_act_quantize(v, alpha)
    ue = oracle.ue4m3_value(np.arange(0x7F))
    r6 = np.float32(1.0 / (6.0 * np.float64(np.float32(alpha))))
    for r in range(v.shape[0]):
        for b in range(v.shape[1] // 32):
            blk = v[r, 32 * b:32 * b + 32]
            t = np.float32(np.abs(blk).max() * r6)
            dist = np.abs(ue - np.float64(t))
            best = np.flatnonzero(dist == dist.min())
            s = scales[r, b]
            assert s in best and (len(best) == 1 or s % 2 == 0)
            S = np.float32(ue[s])
            q = np.float32(1) / np.float32(np.float32(alpha) * S)
            for i in range(32):
                u = abs(float(np.float32(blk[i] * q)))
                dg = np.abs(GRID - min(u, 6.0))
                cand = np.flatnonzero(dg == dg.min())
                m = codes[r, 32 * b + i] & 7
                assert m in cand and (len(cand) == 1 or m % 2 == 0)
                assert (codes[r, 32 * b + i] >> 3) == int(np.signbit(blk[i]))


def test_power_of_two_change_of_alpha_changes_no_code():
    """Q_a(2^j v; 2^j alpha) has the same codes and scales (Eq. 5 depends on v
    only through v / alpha; every step scales exactly by 2^j)."""
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((16, 64)) * 3).astype(np.float32)
    c0, s0 = oracle.nvfp4_act_quantize(v, 0.05)
    for j in (-3, -1, 1, 4):
        c, s = oracle.nvfp4_act_quantize(v * np.float32(2.0 ** j), 0.05 * 2.0 ** j)
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(s, s0)


def test_roundtrip_error_bound():
    """|v - alpha S E2M1| is at most half a grid step of |v q| (a quarter of
    |v q| above 1, 0.25 below), plus the binary32 rounding of v q."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((32, 256)) * 2).astype(np.float32)
    alpha = 0.02
    c, s = oracle.nvfp4_act_quantize(v, alpha)
    deq = alpha * oracle.nvfp4_act_values(c, s)
    S = np.repeat(oracle.ue4m3_value(s), 32, axis=1)
    u = np.abs(v) / (alpha * S)
    bound = alpha * S * np.where(u <= 6.0, np.maximum(0.25, u / 4), u - 6.0 + 1.0) * (1 + 1e-6)
    assert (np.abs(v - deq) <= bound).all()


# ------------------------------------------------------------------ the layer

def _layer(M=4, k=2, E=4, d=64, I=64, seed=8):
    rng = np.random.default_rng(seed)
    W13 = rng.standard_normal((E, 2 * I, d)) * 0.05
    W2 = rng.standard_normal((E, d, I)) * 0.05
    x = rng.standard_normal((M, d)).astype(np.float32).astype(np.float64)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (M, k))
    return x, ids, w, oracle.nvfp4s_quantize_3d(W13), oracle.nvfp4s_quantize_3d(W2)


def test_layer_on_grid_x_matches_exact_h():
    """When every block of x is already on the NVFP4 grid (its maximum
    6 alpha S, the rest alpha S E2M1), Q_a(x) = x, so h equals the exact
    layer's h bit for bit."""
    M, k, E, d, I = 3, 2, 4, 64, 64
    _, ids, w, w13, w2 = _layer(M, k, E, d, I)
    rng = np.random.default_rng(9)
    alpha = 0.25
    S = np.array([0.5, 1.0, 1.125, 2.0, 3.5])[rng.integers(0, 5, (M, d // 32))]
    vals = GRID[rng.integers(0, 8, (M, d))] * np.where(rng.random((M, d)) < 0.5, -1, 1)
    vals[:, ::32] = 6.0
    x = alpha * np.repeat(S, 32, axis=1) * vals
    a4 = oracle.moe_layer_a4(x, ids, w, E, w13, w2, alpha, 0.1, want_xv=True, want_h=True)
    ex = oracle.moe_layer(x, ids, w, E, w13, w2, want_h=True)
    np.testing.assert_array_equal(alpha * a4["xv"], x)
    np.testing.assert_array_equal(a4["h"], ex["h"])


def test_layer_alpha_power_of_two_invariance():
    """y does not change when alpha_x or alpha_h doubles: the codes stay and
    the dequantized activations are the same numbers."""
    x, ids, w, w13, w2 = _layer()
    y0 = oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 0.02, 0.01)["y"]
    np.testing.assert_array_equal(oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 0.04, 0.01)["y"], y0)
    np.testing.assert_array_equal(oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 0.02, 0.005)["y"], y0)


def test_layer_stages_compose():
    """hv is Q_a of h rounded to binary32, and feeding it back reproduces y."""
    x, ids, w, w13, w2 = _layer()
    r = oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 0.02, 0.01, want_h=True, want_hv=True)
    c, s = oracle.nvfp4_act_quantize(r["h"].astype(np.float32), 0.01)
    np.testing.assert_array_equal(oracle.nvfp4_act_values(c, s), r["hv"])
    y2 = oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 0.02, 0.01, hv_in=r["hv"])["y"]
    np.testing.assert_array_equal(y2, r["y"])


def test_layer_close_to_exact_and_invalid_routes_skip():
    x, ids, w, w13, w2 = _layer(M=6)
    a4 = oracle.moe_layer_a4(x, ids, w, 4, w13, w2, 4.0 / (6 * 448), 0.002)["y"]
    ex = oracle.moe_layer(x, ids, w, 4, w13, w2)["y"]
    rel = np.sqrt(np.mean((a4 - ex) ** 2)) / np.sqrt(np.mean(ex ** 2))
    assert 1e-3 < rel < 0.25                      # 4-bit activations: a visible but bounded error
    ids2 = ids.copy()
    ids2[:, 1] = -1
    w2_ = w.copy()
    w2_[:, 1] = 0.0
    y_inv = oracle.moe_layer_a4(x, ids2, w, 4, w13, w2, 0.02, 0.01)["y"]
    y_zero = oracle.moe_layer_a4(x, ids, w2_, 4, w13, w2, 0.02, 0.01)["y"]
    np.testing.assert_array_equal(y_inv, y_zero)
