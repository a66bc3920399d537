"""top_moe_expert_gb300 -- GB300 (sm_103a) routed MoE expert-FFN layer.

A thin ctypes binding over the C ABI of ``libmoe_ffn.so`` (declared in
``include/moe_ffn.h``).  The functions here carry the same names as the C
entry points and only marshal arguments: PyTorch supplies device memory and
the current CUDA stream; every step of the layer runs in the library's CUDA
kernels.  There is no fallback: if the library is not built, or no GPU is
present, calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import dataclasses
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ffn.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_CAPACITY", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_BOUNDS"}
MOE_W_MXFP8, MOE_W_AWQ4, MOE_W_NVFP4S = 0, 1, 3
MOE_BF16, MOE_FP16, MOE_FP32 = 0, 1, 2
MOE_PATH_DECODE, MOE_PATH_GROUPED = 0, 1

_DT = {torch.bfloat16: MOE_BF16, torch.float16: MOE_FP16, torch.float32: MOE_FP32}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class moe_weights_t(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("E", ctypes.c_int32), ("N", ctypes.c_int32),
                ("K", ctypes.c_int32), ("q", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("zero", ctypes.c_void_p), ("alpha", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None

_I32, _I64, _P, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
_PROTOS = {
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_abi_version": (_I32, []),
    "moe_ffn_select_path": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_topk_softmax": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P]),
    "moe_align_capacity": (_I32, [_I32, _I32, _I32, _I32, _P, _P]),
    "moe_align_workspace_size": (_I32, [_I32, _I32, _I32, _I32, _P]),
    "moe_align_block_size": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _I32, _I32, _P, _SZ, _P, _P]),
    "moe_mxfp8_quantize": (_I32, [_P, _I32, _I64, _I32, _P, _P, _P]),
    "moe_ffn_decode_workspace_size": (_I32, [_I32, _I32, _I32, _I32, _P]),
    "moe_ffn_decode": (_I32, [_P, _I32, _I32, _I32, _P, _P, _I32, ctypes.POINTER(moe_weights_t),
                              ctypes.POINTER(moe_weights_t), _P, _I32, _P, _SZ, _P, _P]),
    "moe_ffn_decode_logits": (_I32, [_P, _P, _I32, _I32, _I32, _I32, ctypes.POINTER(moe_weights_t),
                                     ctypes.POINTER(moe_weights_t), _P, _P, _P, _I32, _P, _SZ, _P, _P]),
    "moe_grouped_prepare_size": (_I32, [ctypes.POINTER(moe_weights_t), ctypes.POINTER(moe_weights_t), _P, _P]),
    "moe_grouped_prepare": (_I32, [ctypes.POINTER(moe_weights_t), ctypes.POINTER(moe_weights_t), _P, _P, _P]),
    "moe_grouped_prepare_nvfp4s": (_I32, [ctypes.POINTER(moe_weights_t), ctypes.POINTER(moe_weights_t),
                                          ctypes.c_float, ctypes.c_float, _P, _P, _P]),
    "moe_ffn_grouped_workspace_size": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "moe_ffn_grouped": (_I32, [_P, _I32, _I32, _I32, _P, _P, _I32, ctypes.POINTER(moe_weights_t),
                               ctypes.POINTER(moe_weights_t), _P, _P, _P, _P, _P, _I32, _I32, _P, _I32,
                               _P, _SZ, _P, _P]),
    "moe_ffn_decode_noalloc": (_I32, [_P, _I32, _I32, _I32, _P, _P, _I32, ctypes.POINTER(moe_weights_t),
                                      ctypes.POINTER(moe_weights_t), _P, _I32, _P, _P]),
    "moe_debug_exchange_stall": (_I32, [_I32]),
    "moe_ep_local_routes": (_I32, [_P, _I64, _I32, _I32, _P, _P]),
    "moe_align_fixed_capacity": (_I32, [_P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "moe_ffn_grouped_batched": (_I32, [_P, _I32, _I32, _I32, _P, _P, _I32, ctypes.POINTER(moe_weights_t),
                                       ctypes.POINTER(moe_weights_t), _P, _P, _P, _P, _P, _P, _I32, _I32, _P,
                                       _I32, _P, _SZ, _P, _P]),
}


def use_library(path: str) -> None:
    """Load the library at `path` for the calls that follow (for example the
    debug bounds-check build, build.LIB_DEBUG); the same entry points."""
    global _lib, LIB_PATH
    with _lock:
        LIB_PATH = path
        _lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe_ffn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m top_moe_expert_gb300.build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _PROTOS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# Every pointer handed to the library is checked first: a host tensor, a
# tensor on another GPU, a strided view, a wrong element type or a short
# output buffer would otherwise reach a kernel as a bad address or a bad
# size.  The checks raise ValueError; nothing is launched.

def _is_gpu(t: torch.Tensor) -> bool:
    return t.device.type == "cuda"


def _need(t, name: str, dtypes=None, shape=None, min_numel=None, device=None):
    """Check one tensor argument: a contiguous CUDA tensor on `device`, of one
    of `dtypes`, of exactly `shape` or at least `min_numel` elements."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor, not {type(t).__name__}")
    if not _is_gpu(t):
        raise ValueError(f"{name} must be a CUDA tensor (it is on {t.device})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}; the call's tensors are on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}; expected {' or '.join(str(d) for d in dtypes)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple(shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs at least {min_numel}")
    return t


def _dev(t: torch.Tensor, name: str):
    _need(t, name)


def _opt(t, name: str, **kw):
    """_need for an optional argument (None passes)."""
    return None if t is None else _need(t, name, **kw)


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _guard(device):
    """Make the tensors' GPU current for the call (the library launches on
    the current device)."""
    return torch.cuda.device(device) if device.type == "cuda" else contextlib.nullcontext()


def _stream(stream=None, device=None):
    """The stream handle: `stream`, or the current stream of `device`."""
    if stream is None:
        s = torch.cuda.current_stream(device)
    else:
        s = stream
        sd = getattr(s, "device", None)
        if device is not None and sd is not None and sd != device:
            raise ValueError(f"stream is on {sd}; the call's tensors are on {device}")
    return ctypes.c_void_p(s.cuda_stream)


_IDS = (torch.int32,)
_F32 = (torch.float32,)
_U8 = (torch.uint8,)
_YDT = (torch.bfloat16, torch.float32)


@dataclasses.dataclass(frozen=True)
class Weights:
    """One projection of all experts: MXFP8 (q uint8 [E,N,K], scale uint8
    [E,N,K/32]) or AWQ4 (q int32 [E,N,K/8], scale fp16 [E,N,K/128],
    zero int32 [E,N/8,K/128]) or NVFP4S, paired 4:8 sparse NVFP4 (q uint8
    [E,N,K/4] kept E2M1 codes, scale uint8 [E,N,K/32] UE4M3, zero uint8
    [E,N,K/16] pattern nibbles, alpha float32 [E]).  The tensors are checked against the format
    when the object is made (device, contiguity, dtype, shapes), and the
    object is immutable, so the layer calls only compare its device."""
    fmt: int
    q: torch.Tensor
    scale: torch.Tensor
    zero: torch.Tensor | None = None
    alpha: torch.Tensor | None = None

    def __post_init__(self):
        object.__setattr__(self, "device", self._check())
        object.__setattr__(self, "_struct", moe_weights_t(
            self.fmt, self.E, self.N, self.K, self.q.data_ptr(), self.scale.data_ptr(),
            self.zero.data_ptr() if self.zero is not None else None,
            self.alpha.data_ptr() if self.alpha is not None else None))

    @property
    def E(self):
        return self.q.shape[0]

    @property
    def N(self):
        return self.q.shape[1]

    @property
    def K(self):
        return self.q.shape[2] * {MOE_W_AWQ4: 8, MOE_W_NVFP4S: 4}.get(self.fmt, 1)

    def _check(self):
        q = _need(self.q, "weights.q")
        device = q.device
        if q.dim() != 3:
            raise ValueError(f"weights.q must be 3-D [E, ., .], not {tuple(q.shape)}")
        E, N, K = self.E, self.N, self.K
        if self.fmt == MOE_W_MXFP8:
            _need(q, "weights.q", _U8)
            if K % 32:
                raise ValueError(f"weights: K = {K} is not a multiple of 32")
            _need(self.scale, "weights.scale", _U8, (E, N, K // 32), device=device)
        elif self.fmt == MOE_W_AWQ4:
            _need(q, "weights.q", _IDS)
            if K % 128 or N % 8:
                raise ValueError(f"weights: AWQ needs K % 128 == 0 and N % 8 == 0 (K = {K}, N = {N})")
            _need(self.scale, "weights.scale", (torch.float16,), (E, N, K // 128), device=device)
            if self.zero is None:
                raise ValueError("weights.zero is required for AWQ weights")
            _need(self.zero, "weights.zero", _IDS, (E, N // 8, K // 128), device=device)
        elif self.fmt == MOE_W_NVFP4S:
            _need(q, "weights.q", _U8)
            if K % 64:
                raise ValueError(f"weights: NVFP4S needs K % 64 == 0 (K = {K})")
            _need(self.scale, "weights.scale", _U8, (E, N, K // 32), device=device)
            if self.zero is None or self.alpha is None:
                raise ValueError("weights.zero (patterns) and weights.alpha are required for NVFP4S weights")
            _need(self.zero, "weights.zero", _U8, (E, N, K // 16), device=device)
            _need(self.alpha, "weights.alpha", _F32, (E,), device=device)
        else:
            raise ValueError(f"weights: unknown format {self.fmt}")
        if self.fmt not in (MOE_W_AWQ4, MOE_W_NVFP4S) and self.zero is not None:
            raise ValueError("weights.zero must be None for MXFP8 weights")
        if self.fmt != MOE_W_NVFP4S and self.alpha is not None:
            raise ValueError("weights.alpha is only for NVFP4S weights")
        return device

    def on(self, name: str, device):
        """Raise unless the weights live on `device`."""
        if self.device != device:
            raise ValueError(f"{name} is on {self.device}; the call's tensors are on {device}")

    def c_struct(self) -> moe_weights_t:
        return self._struct


# ---------------------------------------------------------------- routing

def moe_topk_softmax(logits: torch.Tensor, k: int, topk_ids=None, topk_w=None, stream=None):
    _need(logits, "logits", _F32)
    if logits.dim() != 2:
        raise ValueError(f"logits must be [M, E], not {tuple(logits.shape)}")
    dev = logits.device
    M, E = logits.shape
    ids = topk_ids if topk_ids is not None else torch.empty((M, k), dtype=torch.int32, device=dev)
    w = topk_w if topk_w is not None else torch.empty((M, k), dtype=torch.float32, device=dev)
    _need(ids, "topk_ids", _IDS, (M, k), device=dev)
    _need(w, "topk_w", _F32, (M, k), device=dev)
    with _guard(dev):
        _check(lib().moe_topk_softmax(_ptr(logits), M, E, k, _ptr(ids), _ptr(w), _stream(stream, dev)),
               "moe_topk_softmax")
    return ids, w


def moe_ep_local_routes(topk_ids: torch.Tensor, e_lo: int, e_hi: int, local_ids=None, stream=None):
    """The routing as seen by the rank that owns experts [e_lo, e_hi): ids
    of its experts shifted to 0 .. e_hi - e_lo - 1, every other id -1 (an
    invalid route the layer skips)."""
    _need(topk_ids, "topk_ids", _IDS)
    dev = topk_ids.device
    out = local_ids if local_ids is not None else torch.empty_like(topk_ids)
    _need(out, "local_ids", _IDS, tuple(topk_ids.shape), device=dev)
    with _guard(dev):
        _check(lib().moe_ep_local_routes(_ptr(topk_ids), topk_ids.numel(), int(e_lo), int(e_hi), _ptr(out),
                                         _stream(stream, dev)), "moe_ep_local_routes")
    return out


# ---------------------------------------------------------------- alignment

def moe_ffn_select_path(M: int, k: int, E: int, d: int, I: int, fmt: int = None):
    """(path, b): MOE_PATH_DECODE with b = 0, or MOE_PATH_GROUPED with the
    block size for alignment, at the measured crossover of the two paths."""
    fmt = MOE_W_MXFP8 if fmt is None else fmt
    p, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_ffn_select_path(M, k, E, d, I, fmt, ctypes.byref(p), ctypes.byref(b)), "moe_ffn_select_path")
    return p.value, b.value


def moe_debug_exchange_stall(on: bool) -> None:
    """Failure-detection test hook: the single-token one-kernel launches that
    follow wait for h values tagged with a tag no CTA writes, so their bounded
    wait runs out and reports MOE_ERR_TIMEOUT in dev_status[1]; False
    restores normal operation."""
    _check(lib().moe_debug_exchange_stall(1 if on else 0), "moe_debug_exchange_stall")


def moe_align_capacity(M: int, k: int, E: int, b: int):
    cr, cb = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_align_capacity(M, k, E, b, ctypes.byref(cr), ctypes.byref(cb)), "moe_align_capacity")
    return cr.value, cb.value


def moe_align_workspace_size(M: int, k: int, E: int, b: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_align_workspace_size(M, k, E, b, ctypes.byref(n)), "moe_align_workspace_size")
    return n.value


def moe_align_block_size(topk_ids: torch.Tensor, E: int, b: int, cap_rows=None, cap_blocks=None,
                         out=None, ws=None, dev_status=None, stream=None):
    """Returns (sorted_route_ids [cap_rows], expert_ids [cap_blocks],
    num_rows_post_pad [1]) as int32 device tensors."""
    _need(topk_ids, "topk_ids", _IDS)
    if topk_ids.dim() != 2:
        raise ValueError(f"topk_ids must be [M, k], not {tuple(topk_ids.shape)}")
    M, k = topk_ids.shape
    dev = topk_ids.device
    if out is None:
        cr, cb = moe_align_capacity(M, k, E, b)
        cap_rows = cr if cap_rows is None else cap_rows
        cap_blocks = cb if cap_blocks is None else cap_blocks
        out = (torch.empty(cap_rows, dtype=torch.int32, device=dev),
               torch.empty(cap_blocks, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    else:
        # capacities default to the given buffers' lengths
        cap_rows = out[0].numel() if cap_rows is None else cap_rows
        cap_blocks = out[1].numel() if cap_blocks is None else cap_blocks
    _need(out[0], "sorted_route_ids", _IDS, min_numel=cap_rows, device=dev)
    _need(out[1], "expert_ids", _IDS, min_numel=cap_blocks, device=dev)
    _need(out[2], "num_rows_post_pad", _IDS, min_numel=1, device=dev)
    need = moe_align_workspace_size(M, k, E, b)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    _opt(ws, "ws", device=dev)
    _opt(dev_status, "dev_status", dtypes=_IDS, min_numel=2, device=dev)
    with _guard(dev):
        _check(lib().moe_align_block_size(_ptr(topk_ids), M, k, E, b, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                          cap_rows, cap_blocks, _ptr(ws), _nbytes(ws), _ptr(dev_status),
                                          _stream(stream, dev)), "moe_align_block_size")
    return out


def moe_align_fixed_capacity(topk_ids: torch.Tensor, E: int, b: int, C: int, out=None, dev_status=None,
                             stream=None):
    """Fixed-capacity layout: returns (sorted_route_ids [E*C], expert_ids
    [E*C/b], block_rows [E*C/b], num_rows_post_pad [1]) as int32 device
    tensors; C (a multiple of b) must be at least every expert's route count."""
    _need(topk_ids, "topk_ids", _IDS)
    if topk_ids.dim() != 2:
        raise ValueError(f"topk_ids must be [M, k], not {tuple(topk_ids.shape)}")
    if b < 1 or C < b or C % b:
        raise ValueError(f"capacity C = {C} must be a positive multiple of b = {b}")
    M, k = topk_ids.shape
    dev = topk_ids.device
    rows, blocks = E * C, E * C // b
    if out is None:
        out = (torch.empty(rows, dtype=torch.int32, device=dev), torch.empty(blocks, dtype=torch.int32, device=dev),
               torch.empty(blocks, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.int32, device=dev))
    _need(out[0], "sorted_route_ids", _IDS, (rows,), device=dev)
    _need(out[1], "expert_ids", _IDS, (blocks,), device=dev)
    _need(out[2], "block_rows", _IDS, (blocks,), device=dev)
    _need(out[3], "num_rows_post_pad", _IDS, min_numel=1, device=dev)
    _opt(dev_status, "dev_status", dtypes=_IDS, min_numel=2, device=dev)
    with _guard(dev):
        _check(lib().moe_align_fixed_capacity(_ptr(topk_ids), M, k, E, b, C, _ptr(out[0]), _ptr(out[1]),
                                              _ptr(out[2]), _ptr(out[3]), _ptr(dev_status), _stream(stream, dev)),
               "moe_align_fixed_capacity")
    return out


# ---------------------------------------------------------------- quantization

def moe_mxfp8_quantize(v: torch.Tensor, q=None, s=None, stream=None):
    """MXFP8 codes and E8M0 scales of v [rows, K] (fp32 or bf16)."""
    _need(v, "v", (torch.float32, torch.bfloat16))
    dev = v.device
    K = v.shape[-1]
    if K % 32:
        raise ValueError(f"v's last dimension ({K}) is not a multiple of 32")
    rows = v.numel() // K if K else 0
    q = q if q is not None else torch.empty(v.shape, dtype=torch.uint8, device=dev)
    s = s if s is not None else torch.empty((*v.shape[:-1], K // 32), dtype=torch.uint8, device=dev)
    _need(q, "q", _U8, min_numel=rows * K, device=dev)
    _need(s, "s", _U8, min_numel=rows * (K // 32), device=dev)
    with _guard(dev):
        _check(lib().moe_mxfp8_quantize(_ptr(v), _DT[v.dtype], rows, K, _ptr(q), _ptr(s), _stream(stream, dev)),
               "moe_mxfp8_quantize")
    return q, s


def _layer_args(x, topk_ids, topk_w, w13: Weights, w2: Weights, y, out_dtype, dev_status):
    """Check the common arguments of the layer calls; returns (device, M, d,
    k, y) with y allocated when not given."""
    _need(x, "x", tuple(_DT))
    if x.dim() != 2:
        raise ValueError(f"x must be [M, d], not {tuple(x.shape)}")
    dev = x.device
    M, d = x.shape
    _need(topk_ids, "topk_ids", _IDS, device=dev)
    if topk_ids.dim() != 2 or topk_ids.shape[0] != M:
        raise ValueError(f"topk_ids must be [M={M}, k], not {tuple(topk_ids.shape)}")
    k = topk_ids.shape[1]
    _need(topk_w, "topk_w", _F32, (M, k), device=dev)
    w13.on("w13", dev)
    w2.on("w2", dev)
    y = y if y is not None else torch.empty((M, d), dtype=out_dtype, device=dev)
    _need(y, "y", _YDT, (M, d), device=dev)
    _opt(dev_status, "dev_status", dtypes=_IDS, min_numel=2, device=dev)
    return dev, M, d, k, y


def moe_ffn_decode_workspace_size(M: int, k: int, d: int, I: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_ffn_decode_workspace_size(M, k, d, I, ctypes.byref(n)), "moe_ffn_decode_workspace_size")
    return n.value


def moe_ffn_decode(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, w13: Weights, w2: Weights,
                   out_dtype=torch.bfloat16, y=None, ws=None, dev_status=None, stream=None):
    """Output-centric decode path: y [M, d] = sum_j w_j * FFN_{e_j}(x)."""
    dev, M, d, k, y = _layer_args(x, topk_ids, topk_w, w13, w2, y, out_dtype, dev_status)
    I = w2.K
    if ws is None:
        # zeroed: the single-token path keeps its grid-barrier counters in the
        # first 256 bytes and needs them zero before the first call
        ws = torch.zeros(moe_ffn_decode_workspace_size(M, k, d, I), dtype=torch.uint8, device=dev)
    _need(ws, "ws", device=dev)
    a, b = w13.c_struct(), w2.c_struct()
    with _guard(dev):
        _check(lib().moe_ffn_decode(_ptr(x), _DT[x.dtype], M, d, _ptr(topk_ids), _ptr(topk_w), k,
                                    ctypes.byref(a), ctypes.byref(b), _ptr(y), _DT[y.dtype], _ptr(ws),
                                    _nbytes(ws), _ptr(dev_status), _stream(stream, dev)), "moe_ffn_decode")
    return y


def moe_ffn_decode_logits(logits: torch.Tensor, x: torch.Tensor, k: int, w13: Weights, w2: Weights,
                          out_dtype=torch.bfloat16, y=None, topk_ids=None, topk_w=None, ws=None, dev_status=None,
                          stream=None):
    """Routing + decode layer in one call (one kernel for a single token on the
    single-pass layout): returns (y, topk_ids, topk_w), identical to
    moe_topk_softmax followed by moe_ffn_decode."""
    _need(x, "x", tuple(_DT))
    if x.dim() != 2:
        raise ValueError(f"x must be [M, d], not {tuple(x.shape)}")
    dev = x.device
    M, d = x.shape
    _need(logits, "logits", _F32, device=dev)
    if logits.dim() != 2 or logits.shape[0] != M or logits.shape[1] != w13.E:
        raise ValueError(f"logits must be [M={M}, E={w13.E}], not {tuple(logits.shape)}")
    topk_ids = topk_ids if topk_ids is not None else torch.empty((M, k), dtype=torch.int32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty((M, k), dtype=torch.float32, device=dev)
    _need(topk_ids, "topk_ids", _IDS, (M, k), device=dev)
    dev, M, d, k, y = _layer_args(x, topk_ids, topk_w, w13, w2, y, out_dtype, dev_status)
    I = w2.K
    if ws is None:
        ws = torch.zeros(moe_ffn_decode_workspace_size(M, k, d, I), dtype=torch.uint8, device=dev)
    _need(ws, "ws", device=dev)
    a, b = w13.c_struct(), w2.c_struct()
    with _guard(dev):
        _check(lib().moe_ffn_decode_logits(_ptr(logits), _ptr(x), _DT[x.dtype], M, d, k, ctypes.byref(a),
                                           ctypes.byref(b), _ptr(topk_ids), _ptr(topk_w), _ptr(y), _DT[y.dtype],
                                           _ptr(ws), _nbytes(ws), _ptr(dev_status), _stream(stream, dev)),
               "moe_ffn_decode_logits")
    return y, topk_ids, topk_w


def moe_ffn_decode_noalloc(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, w13: Weights,
                           w2: Weights, out_dtype=torch.bfloat16, y=None, dev_status=None, stream=None):
    """moe_ffn_decode without a workspace, for callers that cannot give the
    library device memory: the intermediate lives in a fixed 4 MiB array
    inside the library (MXFP8 two-kernel path only; first call on a device
    outside stream capture; calls must not overlap on the GPU)."""
    dev, M, d, k, y = _layer_args(x, topk_ids, topk_w, w13, w2, y, out_dtype, dev_status)
    a, b = w13.c_struct(), w2.c_struct()
    with _guard(dev):
        _check(lib().moe_ffn_decode_noalloc(_ptr(x), _DT[x.dtype], M, d, _ptr(topk_ids), _ptr(topk_w), k,
                                            ctypes.byref(a), ctypes.byref(b), _ptr(y), _DT[y.dtype],
                                            _ptr(dev_status), _stream(stream, dev)), "moe_ffn_decode_noalloc")
    return y


# ---------------------------------------------------------------- grouped path

def moe_grouped_prepare(w13: Weights, w2: Weights, stream=None):
    """Scale atoms of both projections in the tensor-core layout."""
    dev = w13.device
    w2.on("w2", dev)
    a, b = w13.c_struct(), w2.c_struct()
    n13, n2 = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().moe_grouped_prepare_size(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n13), ctypes.byref(n2)),
           "moe_grouped_prepare_size")
    sfa13 = torch.empty(n13.value, dtype=torch.uint8, device=dev)
    sfa2 = torch.empty(n2.value, dtype=torch.uint8, device=dev)
    with _guard(dev):
        _check(lib().moe_grouped_prepare(ctypes.byref(a), ctypes.byref(b), _ptr(sfa13), _ptr(sfa2),
                                         _stream(stream, dev)), "moe_grouped_prepare")
    return sfa13, sfa2


def moe_grouped_prepare_nvfp4s(w13: Weights, w2: Weights, alpha_x: float, alpha_h: float, stream=None):
    """Prepared buffers (p13, p2) of paired 4:8 sparse NVFP4 weights for the
    W4A4 grouped path: the activations' tensor-wide scales alpha_x (block
    input) and alpha_h (SwiGLU output), the per-expert factors and the
    per-k-step side records; pass them to moe_ffn_grouped as sfa13 / sfa2."""
    dev = w13.device
    w2.on("w2", dev)
    if w13.fmt != MOE_W_NVFP4S or w2.fmt != MOE_W_NVFP4S:
        raise ValueError("moe_grouped_prepare_nvfp4s takes NVFP4S weights")
    if not (alpha_x > 0 and alpha_h > 0 and math.isfinite(alpha_x) and math.isfinite(alpha_h)):
        raise ValueError(f"alpha_x = {alpha_x}, alpha_h = {alpha_h}: both must be finite and > 0")
    a, b = w13.c_struct(), w2.c_struct()
    n13, n2 = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().moe_grouped_prepare_size(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n13), ctypes.byref(n2)),
           "moe_grouped_prepare_size")
    p13 = torch.empty(n13.value, dtype=torch.uint8, device=dev)
    p2 = torch.empty(n2.value, dtype=torch.uint8, device=dev)
    with _guard(dev):
        _check(lib().moe_grouped_prepare_nvfp4s(ctypes.byref(a), ctypes.byref(b), float(alpha_x), float(alpha_h),
                                                _ptr(p13), _ptr(p2), _stream(stream, dev)),
               "moe_grouped_prepare_nvfp4s")
    return p13, p2


def _round256(n):
    return (n + 255) // 256 * 256


def grouped_workspace_layout(M, k, d, I, b, cap_rows):
    """Byte offsets of Xq, Xs, Hq, Hs, Yr and D inside the MXFP8 grouped
    workspace (the layout include/moe_ffn.h documents) and its total."""
    n_mma = (b + 15) // 16 * 16
    nsf = (n_mma + 127) // 128
    cap_blocks = cap_rows // b
    off, out = 0, {}
    for name, size in (("xq", cap_rows * d), ("xs", cap_blocks * (d // 128) * nsf * 512),
                       ("hq", cap_rows * I), ("hs", cap_blocks * (I // 128) * nsf * 512),
                       ("yr", M * k * d * 4), ("done", cap_blocks * 4)):
        out[name] = off
        off += _round256(size)
    out["total"] = off
    out["nsf"] = nsf
    return out


def moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows, ctypes.byref(n)),
           "moe_ffn_grouped_workspace_size")
    return n.value


def moe_ffn_grouped(x, topk_ids, topk_w, w13: Weights, w2: Weights, sfa13, sfa2, aligned, b: int,
                    out_dtype=torch.bfloat16, y=None, ws=None, dev_status=None, stream=None):
    """Expert-centric grouped path; `aligned` = (sorted_route_ids,
    expert_ids, num_rows_post_pad) from moe_align_block_size with the same b,
    or (sorted_route_ids, expert_ids, block_rows, num_rows_post_pad) from
    moe_align_fixed_capacity (the fixed-capacity layout, MXFP8 only)."""
    dev, M, d, k, y = _layer_args(x, topk_ids, topk_w, w13, w2, y, out_dtype, dev_status)
    I = w2.K
    if b < 1:
        raise ValueError(f"block size b = {b} must be positive")
    if len(aligned) == 4:
        sorted_ids, expert_ids, block_rows, npp = aligned
    else:
        (sorted_ids, expert_ids, npp), block_rows = aligned, None
    _need(sorted_ids, "sorted_route_ids", _IDS, device=dev)
    cap_rows = sorted_ids.numel()
    _need(expert_ids, "expert_ids", _IDS, min_numel=cap_rows // b, device=dev)
    _opt(block_rows, "block_rows", dtypes=_IDS, min_numel=cap_rows // b, device=dev)
    _need(npp, "num_rows_post_pad", _IDS, min_numel=1, device=dev)
    a, bb = w13.c_struct(), w2.c_struct()
    if w13.fmt == w2.fmt and w13.fmt in (MOE_W_MXFP8, MOE_W_NVFP4S):
        # the block-scaled MMA reads the scale atoms moe_grouped_prepare wrote;
        # the NVFP4S path, what moe_grouped_prepare_nvfp4s wrote
        n13, n2 = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().moe_grouped_prepare_size(ctypes.byref(a), ctypes.byref(bb), ctypes.byref(n13),
                                              ctypes.byref(n2)), "moe_grouped_prepare_size")
        _need(sfa13, "sfa13", _U8, min_numel=n13.value, device=dev)
        _need(sfa2, "sfa2", _U8, min_numel=n2.value, device=dev)
    else:
        _opt(sfa13, "sfa13", device=dev)
        _opt(sfa2, "sfa2", device=dev)
    if ws is None:
        ws = torch.empty(moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows), dtype=torch.uint8, device=dev)
    _need(ws, "ws", device=dev)
    with _guard(dev):
        if block_rows is None:
            _check(lib().moe_ffn_grouped(_ptr(x), _DT[x.dtype], M, d, _ptr(topk_ids), _ptr(topk_w), k,
                                         ctypes.byref(a), ctypes.byref(bb), _ptr(sfa13), _ptr(sfa2),
                                         _ptr(sorted_ids), _ptr(expert_ids), _ptr(npp), b, cap_rows,
                                         _ptr(y), _DT[y.dtype], _ptr(ws), _nbytes(ws), _ptr(dev_status),
                                         _stream(stream, dev)), "moe_ffn_grouped")
        else:
            _check(lib().moe_ffn_grouped_batched(_ptr(x), _DT[x.dtype], M, d, _ptr(topk_ids), _ptr(topk_w), k,
                                                 ctypes.byref(a), ctypes.byref(bb), _ptr(sfa13), _ptr(sfa2),
                                                 _ptr(sorted_ids), _ptr(expert_ids), _ptr(block_rows), _ptr(npp),
                                                 b, cap_rows, _ptr(y), _DT[y.dtype], _ptr(ws), _nbytes(ws),
                                                 _ptr(dev_status), _stream(stream, dev)), "moe_ffn_grouped_batched")
    return y
