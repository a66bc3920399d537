"""Pins for the oracle's number formats: every code against library casts."""
import numpy as np
import pytest
import torch

import oracle
from tests import refdecode as rd


def _same(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_e4m3_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    assert _same(oracle.e4m3_value(codes), rd.e4m3_table())
    # the two NaN codes and the extremes of the format
    v = oracle.e4m3_value(codes)
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6


def test_e8m0_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    assert _same(oracle.e8m0_value(codes), rd.e8m0_table())
    assert oracle.e8m0_value(np.uint8(127)) == 1.0


def test_bf16_and_fp16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert _same(oracle.bf16_value(bits), rd.bf16_from_bits(bits))
    assert _same(oracle.fp16_value(bits), rd.fp16_from_bits(bits))


@pytest.mark.parametrize("scale", [1.0, 0.02, 1e-30, 3e30, 7.0])
def test_mxfp8_quantizer_matches_library_quantizer(scale):
    g = np.random.Generator(np.random.PCG64(11))
    v = g.standard_normal((64, 256)) * scale
    v[3, :32] = 0.0                        # an all-zero block
    v[5, 40] = -1e-300 * scale             # a tiny value that rounds to -0
    q, s = oracle.mxfp8_quantize(v)
    q2, s2 = rd.mx_quantize_lib(v)
    assert np.array_equal(s, s2)
    assert np.array_equal(q, q2)


def test_mxfp8_quantizer_scale_rule_and_saturation():
    g = np.random.Generator(np.random.PCG64(12))
    v = g.standard_normal((32, 128)) * 3.0
    q, s = oracle.mxfp8_quantize(v)
    X = s.astype(np.int64) - 127
    amax = np.abs(v.reshape(32, 4, 32)).max(-1)
    ratio = amax / np.ldexp(1.0, X)
    assert np.all((ratio >= 256) & (ratio < 512))        # floor(log2 amax) - 8
    # values between 448 and 512 times the scale saturate to the 448 code
    assert np.all((q & 0x7F) <= 0x7E)
    big = np.abs(v.reshape(32, 4, 32)) / np.ldexp(1.0, X)[..., None] >= 464
    assert np.all((q.reshape(32, 4, 32)[big] & 0x7F) == 0x7E)


def test_mxfp8_zero_block_and_sign_of_zero():
    v = np.zeros((1, 64))
    v[0, 33] = -2.0 ** -200
    v[0, 34] = 1.0
    q, s = oracle.mxfp8_quantize(v)
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    assert q[0, 33] == 0x80                              # -0 keeps its sign
    assert oracle.e4m3_value(q[0, 34]) * oracle.e8m0_value(s[0, 1]) == 1.0


def test_mxfp8_roundtrip_of_representable_values():
    g = np.random.Generator(np.random.PCG64(13))
    codes = g.integers(0, 256, size=(16, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E
    codes[:, 0] = 0x7E                   # each block's amax is 448 * 2^X, so the
    codes[:, 32] = 0xFE                  # OCP rule gives back exactly that X
    X = g.integers(-20, 20, size=(16, 2))
    v = rd.e4m3_table()[codes] * np.repeat(np.ldexp(1.0, X), 32, axis=1)
    q, s = oracle.mxfp8_quantize(v)
    back = rd.dequant_mxfp8(q, s)
    assert np.array_equal(back, v)


def test_awq_dequant_row_matches_packed_integers():
    g = np.random.Generator(np.random.PCG64(14))
    S, N, K = 2, 16, 256
    qv = g.integers(0, 16, size=(S, N, K))
    zv = g.integers(0, 16, size=(S, N, K // 128))
    sv = torch.from_numpy(g.uniform(0.005, 0.02, size=(S, N, K // 128)).astype(np.float32)).to(torch.float16)
    q, z = rd.pack_awq(qv, zv)
    s_bits = sv.view(torch.int16).numpy().view(np.uint16)
    w = {"fmt": "awq4", "q": q, "s": s_bits, "z": z}
    want = (qv - np.repeat(zv, 128, axis=-1)) * np.repeat(sv.to(torch.float64).numpy(), 128, axis=-1)
    for e in range(S):
        for n in range(N):
            assert np.array_equal(oracle.dequant_row(w, S, e, n), want[e, n])
    assert np.array_equal(rd.dequant_awq(q, s_bits, z), want)
