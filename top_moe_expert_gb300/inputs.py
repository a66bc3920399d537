"""Seeded synthetic workloads for the routed MoE expert-FFN layer.

This module only draws random numbers (and the closed-form routing fixture);
it holds none of the layer's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.  Quantization of the drawn fp32 weights to MXFP8 is
done separately by each side (the library's quantize kernel, the oracle's own
quantizer) and compared bit for bit.

Workload shapes follow the pages' layers: d=2048 / I=768 / E=128 / top-8
(the 30B-A3B-class shape of the packed-AWQ study and of the grouped-GEMM
benchmark table) and d=7168 / I=2048 / E=384 (the trillion-scale shape).  The
pages measure on real checkpoints, which are not available here; seeded
N(0, 0.02) weights, N(0, 1) activations and N(0, 1) router logits stand in.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    d: int
    I: int
    E: int
    k: int
    b: int = 8
    fmt: str = "mxfp8"          # "mxfp8", "awq4" or "nvfp4s"
    routing: str = "uniform"    # "uniform", "zipf", "fixture_a"
    seed: int = 0

    @property
    def mk(self) -> int:
        return self.M * self.k


# The configurations the layer is specified on.
TINY = Workload("tiny_m21_d512_i256_e128_k8", M=21, d=512, I=256, E=128, k=8, seed=0)
DECODE = Workload("decode_m1_d2048_i768_e128_k8", M=1, d=2048, I=768, E=128, k=8, seed=1)
AWQ_FIXTURE = Workload("awq_fixtureA_m21_d2048_i768_e128_k8", M=21, d=2048, I=768, E=128, k=8,
                       fmt="awq4", routing="fixture_a", seed=3)
LARGE_M1 = Workload("large_m1_d7168_i2048_e384_k8", M=1, d=7168, I=2048, E=384, k=8, seed=4)
LARGE_M8 = Workload("large_m8_d7168_i2048_e384_k8", M=8, d=7168, I=2048, E=384, k=8, seed=4)
SWEEP_M = (1, 4, 8, 16, 32, 64, 512)


def sweep(M: int, routing: str = "uniform") -> Workload:
    return Workload(f"sweep_m{M}_{routing}_d2048_i768_e128_k8", M=M, d=2048, I=768, E=128, k=8,
                    routing=routing, seed=2)


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(BASE_SEED + 1000 * seed + stream))


# ---------------------------------------------------------------- activations

def activations(wl: Workload, step: int = 0, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """x [M, d] ~ N(0, 1), rounded to bf16 (or fp16 for the AWQ layer)."""
    g = rng(wl.seed, 10 + 7919 * step)
    x = g.standard_normal((wl.M, wl.d), dtype=np.float32)
    return torch.from_numpy(x).to(dtype)


def router_logits(wl: Workload, step: int = 0) -> np.ndarray:
    """Router logits [M, E] fp32 ~ N(0, 1); the Zipf(s=1.1) variant adds
    ln p_e with p_e proportional to (1 + rank_e)^-1.1, ranks from a seeded
    permutation of the experts."""
    g = rng(wl.seed, 20 + 7919 * step)
    logits = g.standard_normal((wl.M, wl.E), dtype=np.float32)
    if wl.routing == "zipf":
        rank = rng(wl.seed, 21).permutation(wl.E)
        p = (1.0 + rank.astype(np.float64)) ** -1.1
        p /= p.sum()
        logits = (logits.astype(np.float64) + np.log(p)[None, :]).astype(np.float32)
    return logits


def fixture_a_ids(M: int = 21, k: int = 8, E: int = 128) -> np.ndarray:
    """Closed-form routing with the packed-AWQ study's counts: token t, slot j
    goes to expert (5 * ((8t + j) mod 50)) mod 128.  At M=21, k=8 this gives
    168 valid routes over 50 distinct experts (18 with 4 routes, 32 with 3),
    i.e. 400 aligned rows in 50 blocks at b=8."""
    t = np.arange(M)[:, None]
    j = np.arange(k)[None, :]
    return ((5 * ((8 * t + j) % 50)) % E).astype(np.int32)


def fixture_a_weights(M: int = 21, k: int = 8, seed: int = 3) -> np.ndarray:
    """Positive routing weights for the fixture, drawn as a softmax over k
    N(0,1) draws per token (so each row sums to 1)."""
    z = rng(seed, 30).standard_normal((M, k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def imbalanced_counts(N: int, G: int) -> np.ndarray:
    """Per-expert token counts of the grouped-GEMM benchmark ("Hardware-Native
    Joint Sparse-Quantization ...", App. D.2): the pattern {N, 3N/4, N/2, N/4}
    repeated over the G experts (rounded down, at least 1)."""
    pat = np.array([N, 3 * N // 4, N // 2, N // 4], dtype=np.int64)
    return np.maximum(pat[np.arange(G) % 4], 1)


def imbalanced_routing(N: int, G: int, seed: int = 6) -> np.ndarray:
    """ids [sum of the counts, 1]: one route per token, expert g taking
    imbalanced_counts(N, G)[g] tokens; the tokens' order is a seeded
    permutation (the page fixes only the counts)."""
    ids = np.repeat(np.arange(G, dtype=np.int32), imbalanced_counts(N, G))
    return rng(seed, 40 + N + 7 * G).permutation(ids).reshape(-1, 1).astype(np.int32)


# ---------------------------------------------------------------- weights

def weights_fp32(wl: Workload, which: str, experts=None) -> np.ndarray:
    """fp32 expert weights ~ N(0, 0.02) on the host: which = "w13" ([E,2I,d])
    or "w2" ([E,d,I]).  One generator per (expert, matrix), so any expert can
    be drawn alone; `experts` restricts the draw to a list of expert ids."""
    N, K = (2 * wl.I, wl.d) if which == "w13" else (wl.d, wl.I)
    experts = range(wl.E) if experts is None else experts
    out = np.empty((len(experts), N, K), dtype=np.float32)
    mat = 0 if which == "w13" else 1
    for i, e in enumerate(experts):
        g = rng(wl.seed, 100000 + 2 * int(e) + mat)
        out[i] = g.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    return out


def weights_fp32_device(wl: Workload, which: str, e: int, device) -> torch.Tensor:
    """fp32 weights ~ N(0, 0.02) of one expert, drawn on the device with a
    per-(expert, matrix) torch generator (used for the full-size layers whose
    weights are too large to draw on the host).  The same call reproduces the
    same values, so a test can re-draw any expert and move it to the host."""
    N, K = (2 * wl.I, wl.d) if which == "w13" else (wl.d, wl.I)
    mat = 0 if which == "w13" else 1
    g = torch.Generator(device=device)
    g.manual_seed(BASE_SEED + 1000 * wl.seed + 2 * int(e) + mat)
    return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * 0.02


def awq_weights(wl: Workload, which: str, experts=None):
    """4-bit AWQ weights (group 128 along K): q int32 [E,N,K/8] of uniform
    random nibbles, s fp16 [E,N,K/128] ~ U(0.005, 0.02) (returned as raw
    uint16 bits), z int32 [E,N/8,K/128] of uniform random nibbles."""
    N, K = (2 * wl.I, wl.d) if which == "w13" else (wl.d, wl.I)
    experts = range(wl.E) if experts is None else experts
    mat = 0 if which == "w13" else 1
    n = len(experts)
    q = np.empty((n, N, K // 8), dtype=np.int32)
    s = np.empty((n, N, K // 128), dtype=np.uint16)
    z = np.empty((n, N // 8, K // 128), dtype=np.int32)
    for i, e in enumerate(experts):
        g = rng(wl.seed, 200000 + 2 * int(e) + mat)
        q[i] = g.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
        z[i] = g.integers(0, 2 ** 32, size=(N // 8, K // 128), dtype=np.uint64).astype(np.uint32).view(np.int32)
        sv = g.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float32)
        s[i] = torch.from_numpy(sv).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    return q, s, z


# the six paired 4:8 patterns as nibbles p0 | p1 << 2 (p0 < p1, kept pair indices)
NV4_PATTERNS = np.array([a | (b << 2) for a in range(4) for b in range(a + 1, 4)], dtype=np.uint8)


def nvfp4s_weights(wl: Workload, which: str, experts=None):
    """Random admissible paired 4:8 sparse NVFP4 weights (no quantizer: the
    packed fields are drawn directly): v uint8 [E,N,K/4] of uniform random
    E2M1 codes, m uint8 [E,N,K/16] of patterns drawn uniformly from the six,
    s uint8 [E,N,K/32] UE4M3 codes uniform in [0x30, 0x40] (0.5 .. 2), and
    alpha float32 [E] = 0.01 (kept weights of RMS about 0.03, the draws'
    N(0, 0.02) with half the pairs pruned)."""
    N, K = (2 * wl.I, wl.d) if which == "w13" else (wl.d, wl.I)
    experts = range(wl.E) if experts is None else experts
    mat = 0 if which == "w13" else 1
    n = len(experts)
    v = np.empty((n, N, K // 4), dtype=np.uint8)
    m = np.empty((n, N, K // 16), dtype=np.uint8)
    sc = np.empty((n, N, K // 32), dtype=np.uint8)
    for i, e in enumerate(experts):
        g = rng(wl.seed, 300000 + 2 * int(e) + mat)
        v[i] = g.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
        pat = NV4_PATTERNS[g.integers(0, 6, size=(N, K // 8))]
        m[i] = pat[:, 0::2] | (pat[:, 1::2] << 4)
        sc[i] = g.integers(0x30, 0x41, size=(N, K // 32), dtype=np.uint8)
    return v, m, sc, np.full(n, 0.01, dtype=np.float32)


def nvfp4s_weights_device(wl: Workload, which: str, device):
    """nvfp4s_weights' distribution drawn on the device (for large grids), one
    seeded generator per matrix, expert by expert: kept codes, patterns,
    scale codes, alpha, as torch tensors."""
    N, K = (2 * wl.I, wl.d) if which == "w13" else (wl.d, wl.I)
    g = torch.Generator(device=device)
    g.manual_seed(BASE_SEED + 1000 * wl.seed + (400000 if which == "w13" else 400001))
    E = wl.E
    v = torch.empty((E, N, K // 4), dtype=torch.uint8, device=device)
    m = torch.empty((E, N, K // 16), dtype=torch.uint8, device=device)
    sc = torch.empty((E, N, K // 32), dtype=torch.uint8, device=device)
    pats = torch.from_numpy(NV4_PATTERNS).to(device)
    for e in range(E):
        v[e] = torch.randint(0, 256, (N, K // 4), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
        pat = pats[torch.randint(0, 6, (N, K // 8), generator=g, device=device)]
        m[e] = pat[:, 0::2] | (pat[:, 1::2] << 4)
        sc[e] = torch.randint(0x30, 0x41, (N, K // 32), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    return v, m, sc, torch.full((E,), 0.01, dtype=torch.float32, device=device)


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16/fp16 tensor, as numpy uint16."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
