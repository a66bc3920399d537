"""CPU oracle for the routed MoE expert-FFN layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``top_moe_expert_gb300``) never imports, links or falls back to it, and the
two share no code: the arithmetic lives in ``moe_oracle.c`` (binary64, plain
loops, each routine citing the passage it follows), this module only marshals
numpy arrays through ctypes, plus two small pure-Python host checks
(block-membership identity and the split-K schedule derivation).

Pages cited:
  [RB] "Route-Block Membership Selects Packed-AWQ Arithmetic" (arXiv 2607.26316)
  [SQ] "Hardware-Native Joint Sparse-Quantization for Trillion-Scale
       Mixture-of-Experts" (arXiv 2610.02241)
  [WD] "Warp decode" (cursor.com blog)

Parity unpinned: bit equality with the pages' own kernels (warp decode, the
Marlin AWQ path, the sparse grouped GEMM) -- no code or checkpoint for them
exists here, so nothing is claimed against them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_EXACT = 0  # x, h exact: the output-centric decode path [WD]
MODE_MX = 1     # x, h MXFP8-quantized: block-scaled grouped path [SQ]
MODE_H16 = 2    # h rounded to fp16: fp16 tensor-core AWQ grouped path


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc into liboracle.so (OpenMP, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Weights(ctypes.Structure):
    _fields_ = [
        ("fmt", ctypes.c_int32), ("E", ctypes.c_int32),
        ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("q8", ctypes.c_void_p), ("s8", ctypes.c_void_p),
        ("q4", ctypes.c_void_p), ("s16", ctypes.c_void_p), ("z4", ctypes.c_void_p),
        ("slot", ctypes.c_void_p),
        ("v4", ctypes.c_void_p), ("m4", ctypes.c_void_p), ("sc8", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_e8m0_value.restype = ctypes.c_double
            lib.orc_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.orc_fp16_value.restype = ctypes.c_double
            lib.orc_fp16_value.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_value.restype = ctypes.c_double
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_mxfp8_quantize.restype = None
            lib.orc_mxfp8_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.orc_ue4m3_value.restype = ctypes.c_double
            lib.orc_ue4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_pair_pattern.restype = ctypes.c_int
            lib.orc_pair_pattern.argtypes = [ctypes.c_uint8, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_int)]
            lib.orc_nvfp4s_quantize.restype = None
            lib.orc_nvfp4s_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p]
            lib.orc_topk_softmax.restype = None
            lib.orc_topk_softmax.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_align.restype = ctypes.c_int
            lib.orc_align.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_void_p]
            lib.orc_dequant_row.restype = ctypes.c_int
            lib.orc_dequant_row.argtypes = [ctypes.POINTER(_Weights), ctypes.c_int32,
                                            ctypes.c_int64, ctypes.c_void_p]
            lib.orc_moe_layer.restype = ctypes.c_int
            lib.orc_moe_layer.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.POINTER(_Weights), ctypes.POINTER(_Weights), ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_nvfp4_act_quantize.restype = None
            lib.orc_nvfp4_act_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_moe_layer_a4.restype = ctypes.c_int
            lib.orc_moe_layer_a4.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                ctypes.POINTER(_Weights), ctypes.POINTER(_Weights), ctypes.c_float, ctypes.c_float,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def e4m3_value(codes) -> np.ndarray:
    """Exact value of OCP E4M3 codes (NaN for S.1111.111)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_e4m3_value(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e8m0_value(codes) -> np.ndarray:
    """Exact value 2^(c-127) of OCP E8M0 scale bytes (NaN for 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_e8m0_value(i) for i in range(256)], dtype=np.float64)
    return table[c]


def fp16_value(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    table = np.array([lib.orc_fp16_value(i) for i in range(65536)], dtype=np.float64)
    return table[b]


def bf16_value(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    table = np.array([lib.orc_bf16_value(i) for i in range(65536)], dtype=np.float64)
    return table[b]


def e2m1_value(codes) -> np.ndarray:
    """Exact value of FP4 E2M1 codes (low nibble) [SQ App. A, Figure 3]."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_e2m1_value(i & 0xF) for i in range(256)], dtype=np.float64)
    return table[c]


def ue4m3_value(codes) -> np.ndarray:
    """Exact value of UE4M3 scale codes (NaN for 0x7F and codes >= 0x80)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_ue4m3_value(i) for i in range(256)], dtype=np.float64)
    return table[c]


def pair_pattern(nibble: int):
    """(p0, p1), the kept pair indices of a paired 4:8 metadata nibble, or
    None when the nibble is not one of the six patterns."""
    a, b = ctypes.c_int(), ctypes.c_int()
    return (a.value, b.value) if _load().orc_pair_pattern(nibble, ctypes.byref(a), ctypes.byref(b)) else None


def nvfp4s_quantize(W) -> dict:
    """Paired 4:8 sparse NVFP4 packing of W [N, K] (K % 32 == 0) [SQ App. A,
    Eq. 5-7]: {"v": [N, K/4] kept E2M1 codes, "m": [N, K/16] pattern nibbles,
    "s": [N, K/32] UE4M3 codes, "alpha": float32 per-matrix constant}."""
    lib = _load()
    W = np.ascontiguousarray(W, dtype=np.float64)
    N, K = W.shape
    assert K % 32 == 0
    v = np.empty((N, K // 4), dtype=np.uint8)
    m = np.empty((N, K // 16), dtype=np.uint8)
    sc = np.empty((N, K // 32), dtype=np.uint8)
    alpha = np.empty(1, dtype=np.float32)
    lib.orc_nvfp4s_quantize(_ptr(W), N, K, _ptr(v), _ptr(m), _ptr(sc), _ptr(alpha))
    return {"v": v, "m": m, "s": sc, "alpha": alpha[0]}


def nvfp4s_quantize_3d(W) -> dict:
    """nvfp4s_quantize of each expert's matrix of W [E, N, K]; the format
    dict the layer takes ({"fmt": "nvfp4s", "v", "m", "s", "alpha" [E]})."""
    parts = [nvfp4s_quantize(W[e]) for e in range(W.shape[0])]
    return {"fmt": "nvfp4s", "v": np.stack([p["v"] for p in parts]), "m": np.stack([p["m"] for p in parts]),
            "s": np.stack([p["s"] for p in parts]),
            "alpha": np.array([p["alpha"] for p in parts], dtype=np.float32)}


def nvfp4_act_quantize(v, alpha: float) -> tuple[np.ndarray, np.ndarray]:
    """Run-time activation quantizer Q_a [SQ Sec. 3.4, App. D.1, Eq. 5] of
    v [rows, K] (taken as binary32, K % 32 == 0) with the tensor-wide scale
    alpha: E2M1 codes [rows, K] (one per byte) and UE4M3 block scales
    [rows, K/32]; the decisions are binary32 (see moe_oracle.c)."""
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, K = v.shape
    assert K % 32 == 0 and alpha > 0
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    lib.orc_nvfp4_act_quantize(_ptr(v), rows, K, ctypes.c_float(alpha), _ptr(codes), _ptr(scales))
    return codes, scales


def nvfp4_act_values(codes, scales) -> np.ndarray:
    """S * E2M1(code) per element (the quantized activation without its
    tensor-wide scale alpha), exact in binary64."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    return e2m1_value(codes) * np.repeat(ue4m3_value(scales), 32, axis=1)[:, :K]


def mxfp8_quantize(v) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8 codes [rows, K] and E8M0 scales [rows, K/32] of v [rows, K]."""
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, K = v.shape
    assert K % 32 == 0
    q = np.empty((rows, K), dtype=np.uint8)
    s = np.empty((rows, K // 32), dtype=np.uint8)
    lib.orc_mxfp8_quantize(_ptr(v), rows, K, _ptr(q), _ptr(s))
    return q, s


def mxfp8_quantize_3d(v) -> tuple[np.ndarray, np.ndarray]:
    """Per-slab MXFP8 quantization of v [S, N, K]."""
    S, N, K = v.shape
    q, s = mxfp8_quantize(np.asarray(v).reshape(S * N, K))
    return q.reshape(S, N, K), s.reshape(S, N, K // 32)


# --------------------------------------------------------------------------
# Routing and alignment
# --------------------------------------------------------------------------

def topk_softmax(logits, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k routing: ids [M,k] int32 and renormalised weights [M,k] float64."""
    lib = _load()
    l = np.ascontiguousarray(logits, dtype=np.float32)
    M, E = l.shape
    ids = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    lib.orc_topk_softmax(_ptr(l), M, E, k, _ptr(ids), _ptr(w))
    return ids, w


def align_capacity(M: int, k: int, E: int, b: int) -> tuple[int, int]:
    """Worst-case rows / blocks: every active expert wastes at most b-1 rows."""
    mk = M * k
    cap_rows = mk + min(E, mk) * (b - 1)
    cap_rows = -(-cap_rows // b) * b
    return cap_rows, cap_rows // b


def align(ids, E: int, b: int, cap_rows: int | None = None, cap_blocks: int | None = None):
    """Stable-construction alignment [RB].

    Returns (sorted_route_ids [cap_rows], expert_ids [cap_blocks],
    num_rows_post_pad, n_invalid)."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M, k = ids.shape
    cr, cb = align_capacity(M, k, E, b)
    cap_rows = cr if cap_rows is None else cap_rows
    cap_blocks = cb if cap_blocks is None else cap_blocks
    sorted_ids = np.empty(cap_rows, dtype=np.int32)
    expert_ids = np.empty(cap_blocks, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    ninv = np.zeros(1, dtype=np.int32)
    rc = lib.orc_align(_ptr(ids), M, k, E, b, _ptr(sorted_ids), _ptr(expert_ids), _ptr(npp),
                       cap_rows, cap_blocks, _ptr(ninv))
    if rc != 0:
        raise ValueError("alignment capacity too small")
    return sorted_ids, expert_ids, int(npp[0]), int(ninv[0])


def align_fixed_capacity(ids, E: int, b: int, C: int):
    """Fixed-capacity (batched) layout [SQ App. D.1]: expert e owns rows
    e*C .. e*C + C - 1; its valid routes in route-id order fill the first
    min(N_e, C) of them, the sentinel M*k the rest; the active blocks, the
    first ceil(min(N_e, C) / b) of each expert in expert order, are listed
    compacted.  Returns (sorted_route_ids [E*C], expert_ids [E*C/b],
    block_rows [E*C/b], num_rows_post_pad, n_dropped_or_invalid).  A plain
    statement of the definition in Python loops (small cases only)."""
    ids = np.asarray(ids, dtype=np.int64)
    M, k = ids.shape
    sentinel = M * k
    flat = ids.reshape(-1)
    sorted_ids = np.full(E * C, sentinel, dtype=np.int32)
    expert_ids = np.full(E * C // b, -1, dtype=np.int32)
    block_rows = np.zeros(E * C // b, dtype=np.int32)
    bad = int(np.sum((flat < 0) | (flat >= E)))
    j = 0
    for e in range(E):
        routes = [r for r in range(M * k) if flat[r] == e]
        kept = routes[:C]
        bad += len(routes) - len(kept)
        for i, r in enumerate(kept):
            sorted_ids[e * C + i] = r
        for t in range(-(-len(kept) // b)):
            expert_ids[j] = e
            block_rows[j] = e * C + t * b
            j += 1
    return sorted_ids, expert_ids, block_rows, j * b, bad


def block_identity(sorted_route_ids, expert_ids, num_rows_post_pad: int, b: int, sentinel: int):
    """Mode identity of an aligned sequence [RB, block-membership paragraph].

    Consecutive groups of b aligned rows form blocks; B(e, j) is the set of
    valid routes in block j (whose expert is e); padding sentinels are excluded
    and the order inside a block is ignored.  The identity is the ordered
    sequence of (e, j, sorted(B(e, j))).  Reading: j is the global block index
    (the page labels a block both ways; both label the same sets)."""
    ident = []
    for j in range(num_rows_post_pad // b):
        rows = [int(r) for r in sorted_route_ids[j * b:(j + 1) * b] if int(r) != sentinel]
        ident.append((int(expert_ids[j]), j, tuple(sorted(rows))))
    return tuple(ident)


def split_k_schedule(n_moe_blocks: int, N: int, K: int, thread_n: int, thread_k: int, grid: int):
    """The page's derivation of the packed-AWQ split-K schedule [RB, schedule
    paragraphs], kept to document why a membership-dependent reduction makes
    results depend on block membership.

    The first 2*grid global (MoE block, N-tile) tiles run direct over the full
    K; the remaining tiles start at MoE block floor(direct / n_tiles) and are
    split into `slices` K-slices, where slices = floor(grid / remaining) (at
    least 1) -- a reading that reproduces both of the page's cases."""
    n_tiles = N // thread_n
    k_tiles = K // thread_k
    total = n_moe_blocks * n_tiles
    direct = min(total, 2 * grid)
    remaining = total - direct
    first_split_block = direct // n_tiles
    slices = max(1, grid // remaining) if remaining > 0 else 0
    return {
        "n_tiles": n_tiles, "k_tiles": k_tiles, "total_tiles": total,
        "direct_tiles": direct, "remainder_start_block": first_split_block,
        "slices": slices, "k_tiles_per_slice": (k_tiles // slices) if slices else 0,
    }


# --------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------

# the six paired 4:8 patterns as metadata nibbles p0 | p1 << 2, p0 < p1
_PAIR_NIBBLES = np.array([a | (b << 2) for a in range(4) for b in range(a + 1, 4)], dtype=np.uint8)


def _weights_struct(w: dict, E: int, keep: list):
    st = _Weights()
    fmt = w["fmt"]
    if fmt == "mxfp8":
        q = np.ascontiguousarray(w["q"], dtype=np.uint8)
        s = np.ascontiguousarray(w["s"], dtype=np.uint8)
        S, N, K = q.shape
        assert s.shape == (S, N, K // 32)
        st.fmt, st.q8, st.s8 = 0, _ptr(q), _ptr(s)
        keep += [q, s]
    elif fmt == "awq4":
        q = np.ascontiguousarray(w["q"], dtype=np.int32)
        s = np.ascontiguousarray(w["s"], dtype=np.uint16)
        z = np.ascontiguousarray(w["z"], dtype=np.int32)
        S, N, K8 = q.shape
        K = K8 * 8
        assert s.shape == (S, N, K // 128) and z.shape == (S, N // 8, K // 128)
        st.fmt, st.q4, st.s16, st.z4 = 1, _ptr(q), _ptr(s), _ptr(z)
        keep += [q, s, z]
    elif fmt == "nvfp4s":
        v = np.ascontiguousarray(w["v"], dtype=np.uint8)
        m = np.ascontiguousarray(w["m"], dtype=np.uint8)
        sc = np.ascontiguousarray(w["s"], dtype=np.uint8)
        alpha = np.ascontiguousarray(w["alpha"], dtype=np.float32)
        S, N, K4 = v.shape
        K = K4 * 4
        assert m.shape == (S, N, K // 16) and sc.shape == (S, N, K // 32) and alpha.shape == (S,)
        nib = np.stack([m & 0xF, m >> 4], axis=-1)
        if not np.isin(nib, _PAIR_NIBBLES).all():
            raise ValueError("a paired 4:8 metadata nibble is not one of the six patterns")
        st.fmt, st.v4, st.m4, st.sc8, st.alpha = 2, _ptr(v), _ptr(m), _ptr(sc), _ptr(alpha)
        keep += [v, m, sc, alpha]
    else:
        raise ValueError(fmt)
    st.E, st.N, st.K = E, N, K
    slot = w.get("slot")
    if slot is not None:
        slot = np.ascontiguousarray(slot, dtype=np.int32)
        assert slot.shape == (E,)
        st.slot = _ptr(slot)
        keep.append(slot)
    else:
        st.slot = None
    return st


def dequant_row(w: dict, E: int, e: int, n: int) -> np.ndarray:
    lib = _load()
    keep = []
    st = _weights_struct(w, E, keep)
    out = np.empty(st.K, dtype=np.float64)
    if lib.orc_dequant_row(ctypes.byref(st), e, n, _ptr(out)) != 0:
        raise KeyError(f"expert {e} not supplied")
    return out


def moe_layer(x, ids, w, E: int, w13: dict, w2: dict, mode: int = MODE_EXACT,
              hq_in=None, hs_in=None, want_h: bool = False, want_hq: bool = False):
    """Routed expert-FFN layer in binary64 [WD, SQ].

    x [M,d] exact values (float64); ids [M,k]; w [M,k]; w13 N=2I, K=d;
    w2 N=d, K=I.  Returns dict(y=[M,d], h=[M*k,I]?, hq=[M*k,I]?, hs=[M*k,I/32]?)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    M, d = x.shape
    k = ids.shape[1]
    keep = []
    s13 = _weights_struct(w13, E, keep)
    s2 = _weights_struct(w2, E, keep)
    I = s2.K
    assert s13.N == 2 * I and s13.K == d and s2.N == d
    y = np.empty((M, d), dtype=np.float64)
    h = np.empty((M * k, I), dtype=np.float64) if want_h else None
    hq = hs = None
    if want_hq:
        hq = np.zeros((M * k, I), dtype=np.uint8)
        hs = np.zeros((M * k, I // 32), dtype=np.uint8)
    if hq_in is not None:
        hq_in = np.ascontiguousarray(hq_in, dtype=np.uint8).reshape(M * k, I)
        hs_in = np.ascontiguousarray(hs_in, dtype=np.uint8).reshape(M * k, I // 32)
    rc = lib.orc_moe_layer(_ptr(x), M, d, I, _ptr(ids), _ptr(w), k, E,
                           ctypes.byref(s13), ctypes.byref(s2), mode,
                           _ptr(y), _ptr(h), _ptr(hq_in), _ptr(hs_in), _ptr(hq), _ptr(hs))
    if rc != 0:
        raise KeyError("a routed expert's weights were not supplied")
    return {"y": y, "h": h, "hq": hq, "hs": hs}


def moe_layer_a4(x, ids, w, E: int, w13: dict, w2: dict, alpha_x: float, alpha_h: float,
                 hv_in=None, want_xv: bool = False, want_h: bool = False, want_hv: bool = False):
    """Routed expert-FFN layer with NVFP4-quantized activations, the W4A4
    grouped path [SQ Sec. 3.4, App. D.1]: Q_a(x; alpha_x) before the first
    projection, Q_a(h; alpha_h) before the second, exact weights, binary64
    sums.  Returns dict(y [M,d], xv [M,d]?, h [M*k,I]?, hv [M*k,I]?), xv / hv
    the quantized values without alpha; hv_in replaces the oracle's own
    Q_a(h) (stage-wise check)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    M, d = x.shape
    k = ids.shape[1]
    keep = []
    s13 = _weights_struct(w13, E, keep)
    s2 = _weights_struct(w2, E, keep)
    I = s2.K
    assert s13.N == 2 * I and s13.K == d and s2.N == d and d % 32 == 0 and I % 32 == 0
    y = np.empty((M, d), dtype=np.float64)
    xv = np.empty((M, d), dtype=np.float64) if want_xv else None
    h = np.empty((M * k, I), dtype=np.float64) if want_h else None
    hv = np.empty((M * k, I), dtype=np.float64) if want_hv else None
    if hv_in is not None:
        hv_in = np.ascontiguousarray(hv_in, dtype=np.float64).reshape(M * k, I)
    rc = lib.orc_moe_layer_a4(_ptr(x), M, d, I, _ptr(ids), _ptr(w), k, E, ctypes.byref(s13), ctypes.byref(s2),
                              ctypes.c_float(alpha_x), ctypes.c_float(alpha_h), _ptr(y), _ptr(xv), _ptr(h),
                              _ptr(hv_in), _ptr(hv))
    if rc != 0:
        raise KeyError("a routed expert's weights were not supplied")
    return {"y": y, "xv": xv, "h": h, "hv": hv}
