"""The algorithmic bytes behind every roofline fraction, pinned to the data.

bench.py's per-expert and per-step byte counts are compared with the sizes of
the arrays the kernels actually read, built by the formats' own producers:
the oracle's MXFP8 quantizer, the AWQ and NVFP4S generators of inputs.py, the
library's prepared NVFP4S side records (its size query, host only), and the
step's x, router logits and bf16 y.  A wrong term in a byte formula (a
missing scale array, a 4-bit field counted as a byte, one constant of two)
changes these sums.
"""
import ctypes

import numpy as np

import bench
import oracle
import top_moe_expert_gb300 as moe
from top_moe_expert_gb300 import inputs

D, I = 2048, 768


def _wl(fmt, routing="uniform"):
    return inputs.Workload(f"bytes_{fmt}", M=1, d=D, I=I, E=128, k=8, fmt=fmt, routing=routing, seed=5)


def _mxfp8_expert_arrays(wl):
    out = []
    for which in ("w13", "w2"):
        W = inputs.weights_fp32(wl, which, experts=[0])[0]
        q, s = oracle.mxfp8_quantize(W)
        out += [q, s]
    return out


def test_mxfp8_expert_bytes_are_the_quantizer_arrays():
    wl = _wl("mxfp8")
    arrays = _mxfp8_expert_arrays(wl)
    assert bench.expert_bytes(wl, "decode") == bench.expert_bytes(wl, "grouped") == sum(a.nbytes for a in arrays)


def test_awq_expert_bytes_are_the_packed_arrays():
    wl = _wl("awq4")
    n = sum(a.nbytes for which in ("w13", "w2") for a in inputs.awq_weights(wl, which, experts=[0]))
    assert bench.expert_bytes(wl, "decode") == bench.expert_bytes(wl, "grouped") == n


def test_nvfp4s_expert_bytes_are_the_packed_fields_and_prepared_records():
    wl = _wl("nvfp4s")
    fields = {which: inputs.nvfp4s_weights(wl, which, experts=[0]) for which in ("w13", "w2")}
    # decode: kept codes, patterns, scales and the expert's constant of each matrix
    assert bench.expert_bytes(wl, "decode") == sum(a.nbytes for f in fields.values() for a in f)

    # grouped: kept codes plus the library's prepared side records and factors,
    # per expert (the prepared buffers' growth over 64 experts: the factor
    # arrays are padded to 256 bytes, 64 experts' worth of fp32)
    def prepared(E):
        a = moe.moe_weights_t(moe.MOE_W_NVFP4S, E, 2 * I, D, None, None, None, None)
        b = moe.moe_weights_t(moe.MOE_W_NVFP4S, E, D, I, None, None, None, None)
        n13, n2 = ctypes.c_size_t(), ctypes.c_size_t()
        assert moe.lib().moe_grouped_prepare_size(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n13),
                                                  ctypes.byref(n2)) == 0
        return n13.value + n2.value

    codes = fields["w13"][0].nbytes + fields["w2"][0].nbytes
    grown = prepared(65) - prepared(1)
    assert grown % 64 == 0
    assert bench.expert_bytes(wl, "grouped") == codes + grown // 64


def test_decode_step_bytes_at_the_benchmark_shape():
    """decode_m1: 8 distinct experts' MXFP8 arrays, x (bf16), the router
    logits (fp32) and y (bf16); the layer call's bytes are the same here."""
    wl = bench.workload_from_name("decode_m1")
    ids = np.arange(8, dtype=np.int32).reshape(1, 8) * 3
    expert = sum(a.nbytes for a in _mxfp8_expert_arrays(wl))
    x = inputs.activations(wl)
    logits = inputs.router_logits(wl)
    y_bytes = x.numel() * 2
    want = 8 * expert + x.numel() * x.element_size() + logits.nbytes + y_bytes
    assert bench.step_bytes(wl, ids, "decode") == want == 38_937_088


def test_repeated_and_invalid_experts_count_once_or_not_at_all():
    wl = bench.workload_from_name("decode_m1")
    base = bench.step_bytes(wl, np.arange(8, dtype=np.int32).reshape(1, 8), "decode")
    dup = np.array([[0, 0, 1, 2, 3, 4, 5, 6]], dtype=np.int32)
    inv = np.array([[-1, 1, 2, 3, 4, 5, 6, 7]], dtype=np.int32)
    e = bench.expert_bytes(wl, "decode")
    assert bench.step_bytes(wl, dup, "decode") == base - e
    assert bench.step_bytes(wl, inv, "decode") == base - e
