"""fp64 CPU oracle for the INT4 block-quantized MoE FFN layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the
bench's CPU-baseline / reference arm may import this module; the library's
product path never does.  It shares no code with the CUDA path and does not
import the library package.

The arithmetic lives in qmoe_oracle.c (plain C, double precision, one
thread).  This wrapper only marshals arrays.  Activations, router weights
and scales are passed as their 16-bit storage patterns together with a
dtype code (F16 = 0, BF16 = 1); torch fp16/bf16 tensors are accepted and
reinterpreted bit for bit.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16 = 0
BF16 = 1

_lib = None


def _load(path=None):
    global _lib
    if _lib is None or path is not None:
        path = path or _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_round_to_bf16.restype = ctypes.c_double
        lib.oracle_round_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_dequant_one.restype = ctypes.c_double
        lib.oracle_dequant_one.argtypes = [vp, vp, i32, vp, i32, i32, i32, i64, i64]
        lib.oracle_dequant.restype = None
        lib.oracle_dequant.argtypes = [vp, vp, i32, vp, i32, i32, i32, dp]
        lib.oracle_matmul_nbits.restype = None
        lib.oracle_matmul_nbits.argtypes = [vp, i32, vp, vp, i32, vp, i32, i32, i32, i32, dp]
        lib.oracle_router_probs.restype = None
        lib.oracle_router_probs.argtypes = [vp, i32, vp, vp, i32, i32, i32, dp]
        lib.oracle_topk.restype = None
        lib.oracle_topk.argtypes = [dp, i32, i32, i32, vp, dp]
        lib.oracle_group_by_expert.restype = None
        lib.oracle_group_by_expert.argtypes = [vp, i32, i32, i32, vp, vp]
        lib.oracle_qmoe_forward.restype = ctypes.c_int
        lib.oracle_qmoe_forward.argtypes = [vp, i32, vp, vp] + [vp] * 9 + [i32] * 7 + [vp, dp, dp, vp, dp, dp]
        lib.oracle_shared_expert.restype = ctypes.c_int
        lib.oracle_shared_expert.argtypes = [vp, i32, vp] + [vp] * 9 + [i32] * 5 + [dp, dp]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rmsnorm.argtypes = [vp, i32, i32, i32, ctypes.c_double, i32, dp]
        _lib = lib
    return _lib


class using_library:
    """Context manager: run the wrapper against another build of the oracle
    (the pin tests use it to load deliberately wrong variants)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self._saved = _load()
        _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _np(a, dtype):
    """Contiguous numpy array of `dtype`; torch tensors are viewed bit for bit."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype in (torch.float16, torch.bfloat16):
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def dtype_code(t):
    """F16/BF16 code of a torch tensor's dtype (or pass an int through)."""
    if isinstance(t, int):
        return t
    import torch
    return BF16 if t.dtype == torch.bfloat16 else F16


def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(bits)


def round_to_bf16(v: float) -> float:
    return _load().oracle_round_to_bf16(v)


def dequant(w, scales, scale_dtype, zp, N, K, block_size):
    """[N, K] float64: (q - zp) * scale per block of `block_size` along K."""
    w = _np(w, np.uint8)
    s = _np(scales, np.uint16)
    z = _np(zp, np.uint8)
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_dequant(_ptr(w), _ptr(s), scale_dtype, _ptr(z), N, K, block_size, _dptr(out))
    return out


def dequant_one(w, scales, scale_dtype, zp, N, K, block_size, n, k):
    w = _np(w, np.uint8)
    s = _np(scales, np.uint16)
    z = _np(zp, np.uint8)
    return _load().oracle_dequant_one(_ptr(w), _ptr(s), scale_dtype, _ptr(z), N, K, block_size, n, k)


def matmul_nbits(x, x_dtype, w, scales, scale_dtype, zp, M, N, K, block_size):
    """[M, N] float64: x[M, K] times the dequantised [N, K] matrix, transposed."""
    x = _np(x, np.uint16)
    w = _np(w, np.uint8)
    s = _np(scales, np.uint16)
    z = _np(zp, np.uint8)
    y = np.empty((M, N), dtype=np.float64)
    _load().oracle_matmul_nbits(_ptr(x), x_dtype, _ptr(w), _ptr(s), scale_dtype, _ptr(z),
                                M, N, K, block_size, _dptr(y))
    return y


def router_probs(x, x_dtype, router_w, bias, T, H, E):
    x = _np(x, np.uint16)
    r = _np(router_w, np.uint16)
    b = _np(bias, np.float32)
    p = np.empty((T, E), dtype=np.float64)
    _load().oracle_router_probs(_ptr(x), x_dtype, _ptr(r), _ptr(b), T, H, E, _dptr(p))
    return p


def topk(probs, k):
    probs = np.ascontiguousarray(probs, dtype=np.float64)
    T, E = probs.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _load().oracle_topk(_dptr(probs), T, E, k, _ptr(ids), _dptr(w))
    return ids, w


def group_by_expert(ids, E):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    _load().oracle_group_by_expert(_ptr(ids), T, k, E, _ptr(offsets), _ptr(perm))
    return offsets, perm


def qmoe_forward(layer, forced_ids=None, forced_w=None):
    """Whole layer in fp64.  `layer` is a dict with keys x, router_w,
    router_bias, gate_w, gate_s, gate_zp, up_*, down_*, and ints T, H, I, E,
    k, block_size plus dtype codes act_dtype / scale_dtype.  Returns
    (out [T, H] float64, ids [T, k] int32, w [T, k] float64, probs [T, E])."""
    L = layer
    T, H, I, E, k, bs = (int(L[n]) for n in ("T", "H", "I", "E", "k", "block_size"))
    arrs = {}
    for n in ("x", "router_w"):
        arrs[n] = _np(L[n], np.uint16)
    arrs["router_bias"] = _np(L.get("router_bias"), np.float32)
    for p in ("gate", "up", "down"):
        arrs[p + "_w"] = _np(L[p + "_w"], np.uint8)
        arrs[p + "_s"] = _np(L[p + "_s"], np.uint16)
        arrs[p + "_zp"] = _np(L.get(p + "_zp"), np.uint8)
    fi = None if forced_ids is None else np.ascontiguousarray(forced_ids, dtype=np.int32)
    fw = None if forced_w is None else np.ascontiguousarray(forced_w, dtype=np.float64)
    out = np.empty((T, H), dtype=np.float64)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    probs = np.empty((T, E), dtype=np.float64)
    rc = _load().oracle_qmoe_forward(
        _ptr(arrs["x"]), int(L["act_dtype"]), _ptr(arrs["router_w"]), _ptr(arrs["router_bias"]),
        _ptr(arrs["gate_w"]), _ptr(arrs["gate_s"]), _ptr(arrs["gate_zp"]),
        _ptr(arrs["up_w"]), _ptr(arrs["up_s"]), _ptr(arrs["up_zp"]),
        _ptr(arrs["down_w"]), _ptr(arrs["down_s"]), _ptr(arrs["down_zp"]),
        int(L["scale_dtype"]), T, H, I, E, k, bs,
        _ptr(fi), None if fw is None else _dptr(fw),
        _dptr(out), _ptr(ids), _dptr(w), _dptr(probs))
    if rc != 0:
        raise ValueError("oracle_qmoe_forward rejected its arguments")
    return out, ids, w, probs


def shared_expert(layer, x=None):
    """Gated shared expert in fp64.  `layer` holds shared_gate_w [H] (x's
    dtype), gate_/up_/down_ w, s, zp of a single expert (E = 1), ints H, I,
    block_size and dtype codes.  Returns (out [T, H] float64, gate [T])."""
    L = layer
    x = _np(L["x"] if x is None else x, np.uint16)
    T = x.shape[0]
    H, I, bs = (int(L[n]) for n in ("H", "I", "block_size"))
    arrs = {}
    for p in ("gate", "up", "down"):
        arrs[p + "_w"] = _np(L[p + "_w"], np.uint8)
        arrs[p + "_s"] = _np(L[p + "_s"], np.uint16)
        arrs[p + "_zp"] = _np(L.get(p + "_zp"), np.uint8)
    gw = _np(L["shared_gate_w"], np.uint16)
    out = np.empty((T, H), dtype=np.float64)
    gate = np.empty(T, dtype=np.float64)
    rc = _load().oracle_shared_expert(
        _ptr(x), int(L["act_dtype"]), _ptr(gw),
        _ptr(arrs["gate_w"]), _ptr(arrs["gate_s"]), _ptr(arrs["gate_zp"]),
        _ptr(arrs["up_w"]), _ptr(arrs["up_s"]), _ptr(arrs["up_zp"]),
        _ptr(arrs["down_w"]), _ptr(arrs["down_s"]), _ptr(arrs["down_zp"]),
        int(L["scale_dtype"]), T, H, I, bs, _dptr(out), _dptr(gate))
    if rc != 0:
        raise ValueError("oracle_shared_expert rejected its arguments")
    return out, gate


def rmsnorm(x, x_dtype, T, H, eps=1e-6, round_bf16=False):
    x = _np(x, np.uint16)
    out = np.empty((T, H), dtype=np.float64)
    _load().oracle_rmsnorm(_ptr(x), x_dtype, T, H, float(eps), int(bool(round_bf16)), _dptr(out))
    return out
