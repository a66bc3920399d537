"""Independent decoders used to pin the oracle (test side only).

These reach the same quantities as the oracle through library routines --
PyTorch's float8 / bf16 / fp16 casts and numpy's frexp / ldexp -- so that a
mistake in the oracle's own hand-written format code fails a comparison.
"""
from __future__ import annotations

import numpy as np
import torch


def e4m3_table() -> np.ndarray:
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e8m0_table() -> np.ndarray:
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return c.view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def dequant_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """q [..., K] codes, s [..., K/32] scale bytes -> float64 values."""
    vals = e4m3_table()[q]
    scl = e8m0_table()[s]
    return vals * np.repeat(scl, 32, axis=-1)


def dequant_awq(q: np.ndarray, s_bits: np.ndarray, z: np.ndarray) -> np.ndarray:
    """q int32 [S,N,K/8], s fp16 bits [S,N,K/128], z int32 [S,N/8,K/128]."""
    S, N, K8 = q.shape
    K = K8 * 8
    qu = q.view(np.uint32)
    nib = np.stack([(qu >> np.uint32(4 * i)) & np.uint32(15) for i in range(8)], axis=-1)
    qv = nib.reshape(S, N, K).astype(np.float64)
    zu = z.view(np.uint32)
    znib = np.stack([(zu >> np.uint32(4 * i)) & np.uint32(15) for i in range(8)], axis=2)
    zv = znib.reshape(S, N, K // 128).astype(np.float64)     # row 8a+i <- nibble i of word a
    sv = torch.from_numpy(s_bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    return (qv - np.repeat(zv, 128, axis=-1)) * np.repeat(sv, 128, axis=-1)


def pack_awq(qv: np.ndarray, zv: np.ndarray):
    """Inverse of dequant_awq's unpacking: qv ints [S,N,K], zv ints [S,N,K/128]."""
    S, N, K = qv.shape
    q = np.zeros((S, N, K // 8), dtype=np.uint32)
    for i in range(8):
        q |= (qv[:, :, i::8].astype(np.uint32) & 15) << np.uint32(4 * i)
    z = np.zeros((S, N // 8, K // 128), dtype=np.uint32)
    for i in range(8):
        z |= (zv[:, i::8, :].astype(np.uint32) & 15) << np.uint32(4 * i)
    return q.view(np.int32), z.view(np.int32)


def mx_quantize_lib(v: np.ndarray):
    """MXFP8 quantization through library routines: the shared exponent from
    numpy.frexp, the element rounding from PyTorch's RNE float8_e4m3fn cast
    (which turns |u| >= 464 into NaN instead of saturating, so those are
    clamped to 448 first: saturating conversion).  Inputs with more than 24
    significant bits may be double-rounded by the cast; the pins feed it
    bf16/fp32-derived values or compare codes away from ties."""
    rows, K = v.shape
    blocks = v.reshape(rows, K // 32, 32)
    amax = np.abs(blocks).max(axis=-1)
    _, e2 = np.frexp(amax)
    X = np.where(amax == 0, -127, np.clip(e2 - 1 - 8, -127, 127)).astype(np.int64)
    u = np.ldexp(blocks, -X[..., None])
    u = np.clip(u, -448.0, 448.0)
    q = torch.from_numpy(np.ascontiguousarray(u)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q.reshape(rows, K), (X + 127).astype(np.uint8)


def bf16_from_bits(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def fp16_from_bits(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
