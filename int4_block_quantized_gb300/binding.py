"""Thin Python binding of the C ABI (include/qmoe.h) over ctypes.

Argument marshalling only: every step of the layer runs in the CUDA library
libqmoe.so.  Tensors are torch CUDA tensors (device memory and streams come
from PyTorch); calls are enqueued on torch's current stream.  There is no
fallback: if the library is missing this module raises on import use.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmoe.so")

F16, BF16 = 0, 1
PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_DECODE_SPLIT, PATH_DECODE_FUSED = 0, 1, 2, 4, 5
DECODE_MAX_TOKENS = 16
AUTO_DECODE_MAX_TOKENS = 5
DIAG_STALL_GEMM = 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported device or shape",
           3: "workspace missing or too small", 4: "CUDA runtime error",
           5: "device wait timed out", 6: "device index check failed"}


class QMoEError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, _STATUS.get(code, "unknown"), code))


class QWeight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zp", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libqmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libqmoe.so not built (run int4_block_quantized_gb300/build.py); "
                               "there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qmoe_status_string.restype = ctypes.c_char_p
        L.qmoe_status_string.argtypes = [i32]
        L.qmoe_last_cuda_error.restype = ctypes.c_char_p
        L.qmoe_last_cuda_error.argtypes = []
        L.qmoe_workspace_size.restype = sz
        L.qmoe_workspace_size.argtypes = [i32] * 5
        L.qmoe_workspace_init.restype = i32
        L.qmoe_workspace_init.argtypes = [vp, sz, vp]
        L.qmoe_workspace_set_diagnostics.restype = i32
        L.qmoe_workspace_set_diagnostics.argtypes = [vp, sz, ctypes.c_uint32, ctypes.c_uint32, vp]
        L.qmoe_route.restype = i32
        L.qmoe_route.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.matmul_nbits.restype = i32
        L.matmul_nbits.argtypes = [vp, i32, vp, vp, i32, vp, i32, i32, i32, i32, vp, vp]
        L.matmul_nbits_ex.restype = i32
        L.matmul_nbits_ex.argtypes = [vp, i32, vp, vp, i32, vp, i32, i32, i32, i32, vp, i32, vp, sz, vp]
        L.qmoe_forward.restype = i32
        L.qmoe_forward.argtypes = [vp, i32, vp, vp, QWeight, QWeight, QWeight] + [i32] * 7 + \
            [vp, vp, vp, i32, vp, sz, vp]
        L.qmoe_forward_ex.restype = i32
        L.qmoe_forward_ex.argtypes = [vp, i32, vp, vp, QWeight, QWeight, QWeight] + [i32] * 7 + \
            [vp, vp, vp, i32, i32, vp, sz, vp]
        L.qmoe_forward_kernels.restype = i32
        L.qmoe_forward_kernels.argtypes = [i32] * 11
        L.qmoe_forward_profiled.restype = i32
        L.qmoe_forward_profiled.argtypes = [vp, i32, vp, vp, QWeight, QWeight, QWeight] + [i32] * 7 + \
            [vp, i32, vp, sz, vp, ctypes.POINTER(ctypes.c_void_p), i32]
        L.qmoe_forward_noalloc.restype = i32
        L.qmoe_forward_noalloc.argtypes = [vp, i32, vp, vp, QWeight, QWeight, QWeight] + [i32] * 7 + \
            [vp, vp, vp, i32, vp]
        L.qmoe_noalloc_status.restype = i32
        L.qmoe_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.qmoe_shared_expert.restype = i32
        L.qmoe_shared_expert.argtypes = [vp, i32, vp, QWeight, QWeight, QWeight] + [i32] * 5 + \
            [vp, i32, vp, sz, vp]
        L.qmoe_dequant.restype = i32
        L.qmoe_dequant.argtypes = [vp, vp, i32, vp, i32, i32, i32, vp, vp]
        L.qmoe_rmsnorm.restype = i32
        L.qmoe_rmsnorm.argtypes = [vp, vp, i32, i32, i32, ctypes.c_float, vp]
        L.qmoe_repack_gptq.restype = i32
        L.qmoe_repack_gptq.argtypes = [vp, vp, vp] + [i32] * 5 + [vp, vp, vp, vp, vp, vp]
        L.qmoe_gptq_zero_offset.restype = i32
        L.qmoe_gptq_zero_offset.argtypes = [vp, sz, vp, vp]
        L.qmoe_unpack_zero_points.restype = i32
        L.qmoe_unpack_zero_points.argtypes = [vp, i32, i32, vp, vp]
        L.qmoe_get_device_status.restype = i32
        L.qmoe_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t):
    return BF16 if t.dtype == torch.bfloat16 else F16


def _check(rc, where):
    if rc != 0:
        if rc == 4:
            where = "%s [%s]" % (where, lib().qmoe_last_cuda_error().decode())
        raise QMoEError(rc, where)


def qmoe_status_string(code):
    return lib().qmoe_status_string(code).decode()


def qmoe_workspace_size(T, H, I, E, k):
    return int(lib().qmoe_workspace_size(T, H, I, E, k))


class Workspace:
    """Caller-owned device workspace sized for (T, H, I, E, k), initialised once."""

    def __init__(self, T, H, I, E, k, device=None):
        self.nbytes = qmoe_workspace_size(T, H, I, E, k)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check(lib().qmoe_workspace_init(_p(self.buf), self.nbytes, _stream()), "qmoe_workspace_init")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def set_diagnostics(self, wait_limit_kilocycles=0, flags=0):
        """Diagnostics of the failure path: the grouped GEMM's waits give up
        after wait_limit_kilocycles x 1024 SM cycles (0: about 2 s); flags
        DIAG_STALL_GEMM makes its dequantisers wait for a copy that cannot
        arrive.  (0, 0) restores normal operation."""
        _check(lib().qmoe_workspace_set_diagnostics(self.ptr, self.nbytes, int(wait_limit_kilocycles), int(flags),
                                                    _stream()), "qmoe_workspace_set_diagnostics")

    def status(self):
        bits = ctypes.c_uint32(0)
        rc = lib().qmoe_get_device_status(self.ptr, ctypes.byref(bits), _stream())
        return rc, bits.value


def qmoe_route(x, router_w, k, router_bias=None, ws=None, grouping=True):
    """(topk_w [T,k] fp32, topk_ids [T,k] int32, offsets [E+1], perm [T*k])."""
    T, H = x.shape
    E = router_w.shape[1]
    ws = ws or Workspace(T, H, 32, E, k, device=x.device)
    tw = torch.empty((T, k), dtype=torch.float32, device=x.device)
    ti = torch.empty((T, k), dtype=torch.int32, device=x.device)
    off = torch.empty(E + 1, dtype=torch.int32, device=x.device) if grouping else None
    perm = torch.empty(T * k, dtype=torch.int32, device=x.device) if grouping else None
    _check(lib().qmoe_route(_p(x), _p(router_w), _dt(x), _p(router_bias), T, H, E, k, _p(tw), _p(ti),
                            _p(off), _p(perm), ws.ptr, ws.nbytes, _stream()), "qmoe_route")
    return tw, ti, off, perm


def matmul_nbits(x, w, scales, zp, block_size, out=None):
    """y[M,N] = x[M,K] . dequant(W)[N,K]^T for one packed [N, K/2] matrix."""
    M, K = x.shape
    N = w.shape[-2]
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    _check(lib().matmul_nbits(_p(x), _dt(x), _p(w), _p(scales), _dt(scales), _p(zp), M, N, K,
                              block_size, _p(y), _stream()), "matmul_nbits")
    return y


def matmul_nbits_ex(x, w, scales, zp, block_size, out=None, path=PATH_AUTO, ws=None):
    """matmul_nbits for any M: tensor cores above the decode token limit."""
    M, K = x.shape
    N = w.shape[-2]
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    ws = ws or Workspace(M, N, K, 1, 1, device=x.device)
    _check(lib().matmul_nbits_ex(_p(x), _dt(x), _p(w), _p(scales), _dt(scales), _p(zp), M, N, K,
                                 block_size, _p(y), path, ws.ptr, ws.nbytes, _stream()),
           "matmul_nbits_ex")
    return y


def _qw(L, p):
    return QWeight(L[p + "_w"].data_ptr(), L[p + "_s"].data_ptr(),
                   None if L.get(p + "_zp") is None else L[p + "_zp"].data_ptr())


def qmoe_forward(layer, x=None, out=None, ws=None, accumulate=False, path=PATH_AUTO,
                 return_routing=False):
    """The whole layer.  `layer` holds router_w, router_bias, gate_/up_/down_ w, s,
    zp (device tensors) and ints H, I, E, k, block_size; x [T, H] defaults to
    layer['x'].  Returns out [T, H] (and (topk_w, topk_ids) if asked)."""
    L = layer
    x = L["x"] if x is None else x
    T = x.shape[0]
    H, I, E, k, bs = (int(L[n]) for n in ("H", "I", "E", "k", "block_size"))
    ws = ws or Workspace(T, H, I, E, k, device=x.device)
    o = out if out is not None else torch.empty((T, H), dtype=x.dtype, device=x.device)
    tw = ti = None
    if return_routing:
        tw = torch.empty((T, k), dtype=torch.float32, device=x.device)
        ti = torch.empty((T, k), dtype=torch.int32, device=x.device)
    rc = lib().qmoe_forward_ex(_p(x), _dt(x), _p(L["router_w"]), _p(L.get("router_bias")),
                               _qw(L, "gate"), _qw(L, "up"), _qw(L, "down"), _dt(L["gate_s"]),
                               T, H, I, E, k, bs, _p(o), _p(tw), _p(ti), int(bool(accumulate)),
                               int(path), ws.ptr, ws.nbytes, _stream())
    _check(rc, "qmoe_forward")
    return (o, tw, ti) if return_routing else o


def qmoe_shared_expert(layer, x=None, out=None, ws=None, accumulate=False):
    """out (+)= sigmoid(x . shared_gate_w) * FFN(x) for a shared expert dict
    (make_shared_expert layout: E = 1 weights plus shared_gate_w [H])."""
    L = layer
    x = L["x"] if x is None else x
    T = x.shape[0]
    H, I, bs = (int(L[n]) for n in ("H", "I", "block_size"))
    ws = ws or Workspace(T, H, I, 1, 1, device=x.device)
    o = out if out is not None else torch.empty((T, H), dtype=x.dtype, device=x.device)
    rc = lib().qmoe_shared_expert(_p(x), _dt(x), _p(L["shared_gate_w"]), _qw(L, "gate"), _qw(L, "up"),
                                  _qw(L, "down"), _dt(L["gate_s"]), T, H, I, bs, _p(o),
                                  int(bool(accumulate)), ws.ptr, ws.nbytes, _stream())
    _check(rc, "qmoe_shared_expert")
    return o


def qmoe_forward_noalloc(layer, x=None, out=None, accumulate=False, return_routing=False):
    """qmoe_forward with the library's static device workspace (no caller
    workspace; calls on one device must not overlap)."""
    L = layer
    x = L["x"] if x is None else x
    T = x.shape[0]
    H, I, E, k, bs = (int(L[n]) for n in ("H", "I", "E", "k", "block_size"))
    o = out if out is not None else torch.empty((T, H), dtype=x.dtype, device=x.device)
    tw = ti = None
    if return_routing:
        tw = torch.empty((T, k), dtype=torch.float32, device=x.device)
        ti = torch.empty((T, k), dtype=torch.int32, device=x.device)
    rc = lib().qmoe_forward_noalloc(_p(x), _dt(x), _p(L["router_w"]), _p(L.get("router_bias")),
                                    _qw(L, "gate"), _qw(L, "up"), _qw(L, "down"), _dt(L["gate_s"]),
                                    T, H, I, E, k, bs, _p(o), _p(tw), _p(ti), int(bool(accumulate)),
                                    _stream())
    _check(rc, "qmoe_forward_noalloc")
    return (o, tw, ti) if return_routing else o


def qmoe_noalloc_status():
    """(status code, raw bits) of the static scratch's device status word on
    the current device; reads and clears it (synchronises the stream)."""
    bits = ctypes.c_uint32(0)
    rc = lib().qmoe_noalloc_status(ctypes.byref(bits), _stream())
    return rc, bits.value


def qmoe_forward_kernels(layer, T, path=PATH_AUTO):
    """Kernels one qmoe_forward call on this layer with T tokens launches on
    the current device (1 fused decode, 3 decode, 5 prefill)."""
    L = layer
    H, I, E, k, bs = (int(L[n]) for n in ("H", "I", "E", "k", "block_size"))
    n = lib().qmoe_forward_kernels(T, H, I, E, k, bs, _dt(L["router_w"]), _dt(L["gate_s"]),
                                   int(L.get("gate_zp") is not None), int(L.get("down_zp") is not None),
                                   int(path))
    if n < 0:
        _check(-n, "qmoe_forward_kernels")
    return n


def qmoe_forward_profiled(layer, events, x=None, out=None, ws=None, path=PATH_AUTO):
    """qmoe_forward that records torch.cuda.Event objects `events` before the
    first kernel and after each kernel (kernels serialised)."""
    L = layer
    x = L["x"] if x is None else x
    T = x.shape[0]
    H, I, E, k, bs = (int(L[n]) for n in ("H", "I", "E", "k", "block_size"))
    ws = ws or Workspace(T, H, I, E, k, device=x.device)
    o = out if out is not None else torch.empty((T, H), dtype=x.dtype, device=x.device)
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    rc = lib().qmoe_forward_profiled(_p(x), _dt(x), _p(L["router_w"]), _p(L.get("router_bias")),
                                     _qw(L, "gate"), _qw(L, "up"), _qw(L, "down"), _dt(L["gate_s"]),
                                     T, H, I, E, k, bs, _p(o), int(path), ws.ptr, ws.nbytes, _stream(),
                                     arr, len(events))
    _check(rc, "qmoe_forward_profiled")
    return o


def qmoe_dequant(w, scales, zp, block_size):
    """fp32 [N, K] = (q - zp) * scale of one packed [N, K/2] matrix."""
    N, K2 = w.shape[-2], w.shape[-1]
    out = torch.empty((N, 2 * K2), dtype=torch.float32, device=w.device)
    _check(lib().qmoe_dequant(_p(w), _p(scales), _dt(scales), _p(zp), N, 2 * K2, block_size, _p(out),
                              _stream()), "qmoe_dequant")
    return out


def qmoe_rmsnorm(x, eps=1e-6, out=None):
    T, H = x.shape
    o = out if out is not None else torch.empty_like(x)
    _check(lib().qmoe_rmsnorm(_p(x), _p(o), _dt(x), T, H, float(eps), _stream()), "qmoe_rmsnorm")
    return o


def qmoe_gptq_zero_offset(qzeros):
    """Device int32 [1]: 1 if the median stored GPTQ zero point is 7, else 0."""
    off = torch.empty(1, dtype=torch.int32, device=qzeros.device)
    _check(lib().qmoe_gptq_zero_offset(_p(qzeros), qzeros.numel(), _p(off), _stream()), "qmoe_gptq_zero_offset")
    return off


def qmoe_repack_gptq(qweight, qzeros, scales, block_size, zero_offset=0, zero_offset_dev=None, check=True,
                     status=None):
    """GPTQ (qweight [E, K/8, N] int32, qzeros [E, K/bs, N/8] int32 or None,
    scales [E, K/bs, N]) -> canonical (w [E, N, K/2] u8, scales [E, N, K/bs],
    zp [E, N, K/bs] u8 or None).  A zero point above 15 (stored 15 with
    offset 1) sets QMOE_ST_RANGE in the status word: with check=True (the
    default) this synchronises and raises QMoEError; with check=False the
    caller's own int32 device tensor `status` (if given) collects the bit."""
    E, K8, N = qweight.shape
    K = 8 * K8
    nb = K // block_size
    w = torch.empty((E, N, K // 2), dtype=torch.uint8, device=qweight.device)
    s = torch.empty((E, N, nb), dtype=scales.dtype, device=qweight.device)
    zp = torch.empty((E, N, nb), dtype=torch.uint8, device=qweight.device) if qzeros is not None else None
    st = status if status is not None else (torch.zeros(1, dtype=torch.int32, device=qweight.device) if check else None)
    _check(lib().qmoe_repack_gptq(_p(qweight), _p(qzeros), _p(scales), E, K, N, block_size, int(zero_offset),
                                  _p(zero_offset_dev), _p(w), _p(s), _p(zp), _p(st), _stream()), "qmoe_repack_gptq")
    if check and status is None:
        _check(lib().qmoe_get_device_status(_p(st), None, _stream()),
               "qmoe_repack_gptq (a GPTQ zero point above 15 does not fit the 4-bit format)")
    return w, s, zp


def qmoe_unpack_zero_points(zp_packed, nb):
    """[rows, ceil(nb/2)] packed zero points -> [rows, nb] uint8."""
    rows = zp_packed.shape[0]
    out = torch.empty((rows, nb), dtype=torch.uint8, device=zp_packed.device)
    _check(lib().qmoe_unpack_zero_points(_p(zp_packed), rows, nb, _p(out), _stream()), "qmoe_unpack_zero_points")
    return out
