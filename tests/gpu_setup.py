"""Test-side setup shared by the GPU parity tests.

Builds each workload twice from the same seeded draws (top_moe_expert_gb300.
inputs): once on the device through the library (its MXFP8 quantize kernel),
once on the host for the oracle (its own quantizer).  The two code sets are
compared bit for bit before either is used, so a layer comparison never feeds
the oracle anything computed by the CUDA path.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import top_moe_expert_gb300 as moe
from top_moe_expert_gb300 import inputs

# Layer tolerance stated for the path: max |err| <= 2e-3 * max |ref| (FP32
# accumulation); bf16 outputs additionally get half a bf16 ulp of the value.
REL_TOL = 2e-3
MIN_COSINE = 0.999996


def need_gpu():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU test run without a CUDA device")
    moe.lib()


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 2.0 ** -134)


def assert_layer_close(y_gpu: torch.Tensor, y_ref: np.ndarray, rel_tol: float = REL_TOL,
                       min_cos: float = MIN_COSINE):
    y = y_gpu.detach().double().cpu().numpy()
    assert y.shape == y_ref.shape
    assert np.all(np.isfinite(y))
    scale = np.abs(y_ref).max()
    tol = rel_tol * scale
    if y_gpu.dtype == torch.bfloat16:
        tol = tol + bf16_half_ulp(y_ref)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {err.size} outside tolerance; "
                           f"max |err| / max|ref| = {err.max() / scale:.3e}")
    cos = float((y * y_ref).sum() / math.sqrt((y * y).sum() * (y_ref * y_ref).sum()))
    assert cos >= min_cos, f"cosine {cos}"
    return err.max() / scale, cos


def x_exact(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.float64).numpy()


class MxLayer:
    """MXFP8 weights of one workload on the device, plus host access to the
    fp32 draws of any expert for the oracle."""

    def __init__(self, wl: inputs.Workload, device="cuda", host_draw: bool | None = None,
                 experts=None):
        self.wl = wl
        self.device = device
        E, d, I = wl.E, wl.d, wl.I
        # host draws are cheap for the small layers; big ones draw per expert
        # on the device
        self.host_draw = (E * 3 * I * d <= 64 * 2 ** 20) if host_draw is None else host_draw
        self.q13 = torch.zeros((E, 2 * I, d), dtype=torch.uint8, device=device)
        self.s13 = torch.zeros((E, 2 * I, d // 32), dtype=torch.uint8, device=device)
        self.q2 = torch.zeros((E, d, I), dtype=torch.uint8, device=device)
        self.s2 = torch.zeros((E, d, I // 32), dtype=torch.uint8, device=device)
        fill = range(E) if experts is None else sorted(set(int(e) for e in experts))
        if self.host_draw:
            f13 = torch.from_numpy(inputs.weights_fp32(wl, "w13")).to(device)
            f2 = torch.from_numpy(inputs.weights_fp32(wl, "w2")).to(device)
            moe.moe_mxfp8_quantize(f13, self.q13, self.s13)
            moe.moe_mxfp8_quantize(f2, self.q2, self.s2)
            del f13, f2
        else:
            for e in fill:
                moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w13", e, device), self.q13[e], self.s13[e])
                moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w2", e, device), self.q2[e], self.s2[e])
        torch.cuda.synchronize()
        self.w13 = moe.Weights(moe.MOE_W_MXFP8, self.q13, self.s13)
        self.w2 = moe.Weights(moe.MOE_W_MXFP8, self.q2, self.s2)

    def fp32_host(self, which: str, experts) -> np.ndarray:
        if self.host_draw:
            return inputs.weights_fp32(self.wl, which, experts)
        return np.stack([inputs.weights_fp32_device(self.wl, which, e, self.device).cpu().numpy()
                         for e in experts])

    def oracle_weights(self, experts, check_codes: bool = True):
        """Oracle-side MXFP8 weights of `experts` (quantized by the oracle from
        the fp32 draws), with a slot map; optionally checks that the device
        codes of those experts are bit-identical."""
        experts = sorted(set(int(e) for e in experts if 0 <= e < self.wl.E))
        slot = np.full(self.wl.E, -1, dtype=np.int32)
        slot[experts] = np.arange(len(experts), dtype=np.int32)
        out = {}
        for which, (qd, sd) in (("w13", (self.q13, self.s13)), ("w2", (self.q2, self.s2))):
            qs, ss = [], []
            for e in experts:                  # one expert at a time: bounded host memory
                f = self.fp32_host(which, [e])[0].astype(np.float64)
                q, s = oracle.mxfp8_quantize(f)
                if check_codes:
                    assert np.array_equal(qd[e].cpu().numpy(), q), f"{which} codes of expert {e} differ"
                    assert np.array_equal(sd[e].cpu().numpy(), s), f"{which} scales of expert {e} differ"
                qs.append(q)
                ss.append(s)
            out[which] = {"fmt": "mxfp8", "q": np.stack(qs), "s": np.stack(ss), "slot": slot}
        return out["w13"], out["w2"]


class AwqLayer:
    """4-bit AWQ weights (drawn directly as packed integers) on both sides."""

    def __init__(self, wl: inputs.Workload, device="cuda"):
        self.wl = wl
        q13, s13, z13 = inputs.awq_weights(wl, "w13")
        q2, s2, z2 = inputs.awq_weights(wl, "w2")
        self.host13 = {"fmt": "awq4", "q": q13, "s": s13, "z": z13}
        self.host2 = {"fmt": "awq4", "q": q2, "s": s2, "z": z2}
        t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
        self.w13 = moe.Weights(moe.MOE_W_AWQ4, t(q13), t(s13).view(torch.float16), t(z13))
        self.w2 = moe.Weights(moe.MOE_W_AWQ4, t(q2), t(s2).view(torch.float16), t(z2))


def routing(wl: inputs.Workload, step: int = 0):
    """(ids int32 [M,k], w float32 [M,k]) from the oracle's top-k of the seeded
    logits (host), or the closed-form fixture."""
    if wl.routing == "fixture_a":
        return inputs.fixture_a_ids(wl.M, wl.k, wl.E), inputs.fixture_a_weights(wl.M, wl.k, wl.seed)
    ids, w = oracle.topk_softmax(inputs.router_logits(wl, step), wl.k)
    return ids, w.astype(np.float32)
