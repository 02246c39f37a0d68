"""GB300 (sm_103a) low-bit attention for training: the SageBwd scheme.

The compute path is the CUDA library libsage_attn.so (include/sage_attn.h).  This
module only marshals arguments to it: the ctypes functions carry the C names
(sage_attn_quantize, sage_attn_fwd, sage_attn_bwd, ...), and the torch helpers
below allocate device memory, read the current stream and call them.  There is
no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import workloads  # noqa: F401  (seeded synthetic inputs)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsage_attn.so")

SAGE_OK, SAGE_ERR_INVALID_ARG, SAGE_ERR_UNSUPPORTED, SAGE_ERR_CUDA, SAGE_ERR_TIMEOUT = 0, 1, 2, 3, 4

# names declared in include/sage_attn.h
ABI_FUNCTIONS = ("sage_attn_ws_bytes", "sage_attn_bwd_ws_bytes", "sage_attn_quantize", "sage_attn_fwd",
                 "sage_attn_bwd", "sage_attn_ws_views", "sage_attn_get_status", "sage_attn_selftest_wait",
                 "sage_attn_status_str", "sage_attn_timer_enable", "sage_attn_timer_read",
                 "sage_attn_bwd_noalloc", "sage_attn_step_host_bytes", "sage_attn_step_host",
                 "sage_attn_timer_only", "sage_attn_bwd_o32", "sage_attn_gqa_ws_bytes",
                 "sage_attn_gqa_bwd_ws_bytes", "sage_attn_gqa_quantize", "sage_attn_gqa_fwd", "sage_attn_gqa_bwd",
                 "sage_attn_gqa_ws_views", "sage_attn_qs_ws_bytes", "sage_attn_qs_quantize", "sage_attn_qs_fwd",
                 "sage_attn_qs_bwd", "sage_attn_qs_ws_views", "sage_attn_thrift_ws_bytes",
                 "sage_attn_thrift_quantize", "sage_attn_thrift_fwd", "sage_attn_thrift_sel",
                 "sage_attn_fp4_ws_bytes", "sage_attn_fp4_quantize", "sage_attn_fp4_fwd",
                 "sage_attn_fp4_ws_views", "sage_attn_fp4_bwd_ws_bytes", "sage_attn_fp4_bwd")


class SageError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({status_str(code)})")
        self.code = code


class sage_ws_views(ctypes.Structure):
    _fields_ = [("qc", ctypes.c_void_p), ("kc", ctypes.c_void_p), ("v8t", ctypes.c_void_p),
                ("sq", ctypes.c_void_p), ("sk", ctypes.c_void_p), ("sv", ctypes.c_void_p),
                ("kmean", ctypes.c_void_p), ("qr", ctypes.c_void_p), ("kr", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("n_pad", ctypes.c_int), ("qmean", ctypes.c_void_p),
                ("dsb", ctypes.c_void_p), ("vg", ctypes.c_void_p), ("v4", ctypes.c_void_p),
                ("v4sf", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
            L = ctypes.CDLL(LIB_PATH)
            i, sz, vp, fp, u64 = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float, ctypes.c_ulonglong
            L.sage_attn_ws_bytes.restype = sz
            L.sage_attn_ws_bytes.argtypes = [i, i, i, i]
            L.sage_attn_bwd_ws_bytes.restype = sz
            L.sage_attn_bwd_ws_bytes.argtypes = [i, i, i, i]
            L.sage_attn_quantize.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
            L.sage_attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, fp, vp]
            L.sage_attn_bwd.argtypes = [vp] * 11 + [sz] + [i] * 7 + [fp, vp]
            L.sage_attn_bwd_o32.argtypes = [vp] * 11 + [sz] + [i] * 7 + [fp, vp]
            L.sage_attn_gqa_ws_bytes.restype = sz
            L.sage_attn_gqa_ws_bytes.argtypes = [i] * 5
            L.sage_attn_gqa_bwd_ws_bytes.restype = sz
            L.sage_attn_gqa_bwd_ws_bytes.argtypes = [i] * 5
            L.sage_attn_gqa_quantize.argtypes = [vp, vp, vp] + [i] * 7 + [vp, sz, vp]
            L.sage_attn_gqa_fwd.argtypes = [vp, vp, vp, vp] + [i] * 6 + [fp, vp]
            L.sage_attn_gqa_bwd.argtypes = [vp] * 11 + [sz] + [i] * 8 + [fp, vp]
            L.sage_attn_gqa_ws_views.argtypes = [vp] + [i] * 5 + [ctypes.POINTER(sage_ws_views)]
            L.sage_attn_qs_ws_bytes.restype = sz
            L.sage_attn_qs_ws_bytes.argtypes = [i] * 5
            L.sage_attn_qs_quantize.argtypes = [vp, vp, vp] + [i] * 7 + [vp, sz, vp]
            L.sage_attn_qs_fwd.argtypes = [vp, vp, vp, vp] + [i] * 6 + [fp, vp]
            L.sage_attn_qs_bwd.argtypes = [vp] * 11 + [sz] + [i] * 8 + [fp, vp]
            L.sage_attn_qs_ws_views.argtypes = [vp] + [i] * 5 + [ctypes.POINTER(sage_ws_views)]
            L.sage_attn_fp4_ws_bytes.restype = sz
            L.sage_attn_fp4_ws_bytes.argtypes = [i] * 4
            L.sage_attn_fp4_quantize.argtypes = [vp, vp, vp] + [i] * 6 + [vp, sz, vp]
            L.sage_attn_fp4_fwd.argtypes = [vp, vp, vp, vp] + [i] * 5 + [fp, vp]
            L.sage_attn_fp4_ws_views.argtypes = [vp] + [i] * 4 + [ctypes.POINTER(sage_ws_views)]
            L.sage_attn_fp4_bwd_ws_bytes.restype = sz
            L.sage_attn_fp4_bwd_ws_bytes.argtypes = [i] * 4
            L.sage_attn_fp4_bwd.argtypes = [vp] * 11 + [sz] + [i] * 7 + [fp, vp]
            L.sage_attn_thrift_ws_bytes.restype = sz
            L.sage_attn_thrift_ws_bytes.argtypes = [i] * 4
            L.sage_attn_thrift_quantize.argtypes = [vp, vp, vp] + [i] * 7 + [ctypes.c_double, vp, sz, vp, sz, vp]
            L.sage_attn_thrift_fwd.argtypes = [vp] * 5 + [i] * 5 + [fp, vp]
            L.sage_attn_thrift_sel.restype = vp
            L.sage_attn_thrift_sel.argtypes = [vp] + [i] * 4
            L.sage_attn_ws_views.argtypes = [vp, i, i, i, i, ctypes.POINTER(sage_ws_views)]
            L.sage_attn_get_status.argtypes = [vp, vp]
            L.sage_attn_selftest_wait.argtypes = [vp, u64, vp]
            L.sage_attn_bwd_noalloc.argtypes = [vp] * 10 + [i] * 7 + [fp, vp]
            L.sage_attn_step_host_bytes.restype = sz
            L.sage_attn_step_host_bytes.argtypes = [i, i, i, i, i]
            L.sage_attn_step_host.argtypes = [vp] * 10 + [sz] + [i] * 7 + [fp, i, vp]
            L.sage_attn_timer_enable.argtypes = [i]
            L.sage_attn_timer_only.argtypes = [ctypes.c_char_p]
            L.sage_attn_timer_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(ctypes.c_int)]
            L.sage_attn_status_str.restype = ctypes.c_char_p
            L.sage_attn_status_str.argtypes = [i]
            _lib = L
    return _lib


# ----------------------------------------------------------- C names, as is

def sage_attn_ws_bytes(B, H, N, D):
    return lib().sage_attn_ws_bytes(B, H, N, D)


def sage_attn_bwd_ws_bytes(B, H, N, D):
    return lib().sage_attn_bwd_ws_bytes(B, H, N, D)


def sage_attn_quantize(Q, K, V, B, H, N, D, qk_norm, k_smooth, ws, ws_bytes, stream):
    return lib().sage_attn_quantize(Q, K, V, B, H, N, D, int(qk_norm), int(k_smooth), ws, ws_bytes, stream)


def sage_attn_fwd(ws, O, LSE, O32, B, H, N, D, causal, sm_scale, stream):
    return lib().sage_attn_fwd(ws, O, LSE, O32, B, H, N, D, int(causal), float(sm_scale), stream)


def sage_attn_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D, causal, qk_norm,
                  k_smooth, sm_scale, stream):
    return lib().sage_attn_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D,
                               int(causal), int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_bwd_o32(Q, K, V, O32, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D, causal, qk_norm,
                      k_smooth, sm_scale, stream):
    return lib().sage_attn_bwd_o32(Q, K, V, O32, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D,
                                   int(causal), int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_fp4_ws_bytes(B, H, N, D):
    return lib().sage_attn_fp4_ws_bytes(B, H, N, D)


def sage_attn_fp4_quantize(Q, K, V, B, H, N, D, qk_norm, k_smooth, ws, ws_bytes, stream):
    return lib().sage_attn_fp4_quantize(Q, K, V, B, H, N, D, int(qk_norm), int(k_smooth), ws, ws_bytes, stream)


def sage_attn_fp4_fwd(ws, O, LSE, O32, B, H, N, D, causal, sm_scale, stream):
    return lib().sage_attn_fp4_fwd(ws, O, LSE, O32, B, H, N, D, int(causal), float(sm_scale), stream)


def sage_attn_fp4_bwd_ws_bytes(B, H, N, D):
    return lib().sage_attn_fp4_bwd_ws_bytes(B, H, N, D)


def sage_attn_fp4_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D, causal, qk_norm,
                      k_smooth, sm_scale, stream):
    return lib().sage_attn_fp4_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, N, D,
                                   int(causal), int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_fp4_ws_views(ws, B, H, N, D) -> sage_ws_views:
    v = sage_ws_views()
    rc = lib().sage_attn_fp4_ws_views(ws, B, H, N, D, ctypes.byref(v))
    if rc != SAGE_OK:
        raise SageError("sage_attn_fp4_ws_views", rc)
    return v


def sage_attn_thrift_ws_bytes(B, H, N, D):
    return lib().sage_attn_thrift_ws_bytes(B, H, N, D)


def sage_attn_thrift_quantize(Q, K, V, B, H, N, D, qk_norm, k_smooth, causal, budget, ws, ws_bytes, tws, tws_bytes,
                              stream):
    return lib().sage_attn_thrift_quantize(Q, K, V, B, H, N, D, int(qk_norm), int(k_smooth), int(causal),
                                           float(budget), ws, ws_bytes, tws, tws_bytes, stream)


def sage_attn_thrift_fwd(ws, tws, O, LSE, O32, B, H, N, D, causal, sm_scale, stream):
    return lib().sage_attn_thrift_fwd(ws, tws, O, LSE, O32, B, H, N, D, int(causal), float(sm_scale), stream)


def sage_attn_thrift_sel(tws, B, H, N, D):
    return lib().sage_attn_thrift_sel(tws, B, H, N, D)


def sage_attn_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, B, H, N, D, causal, qk_norm, k_smooth, sm_scale,
                          stream):
    return lib().sage_attn_bwd_noalloc(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, B, H, N, D, int(causal),
                                       int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_step_host_bytes(B, H, N, D, groups):
    return lib().sage_attn_step_host_bytes(B, H, N, D, int(groups))


def sage_attn_step_host(Q, K, V, dO, O, LSE, dQ, dK, dV, dev, dev_bytes, B, H, N, D, causal, qk_norm, k_smooth,
                        sm_scale, groups, stream):
    return lib().sage_attn_step_host(Q, K, V, dO, O, LSE, dQ, dK, dV, dev, dev_bytes, B, H, N, D, int(causal),
                                     int(qk_norm), int(k_smooth), float(sm_scale), int(groups), stream)


def sage_attn_gqa_ws_bytes(B, H, Hkv, N, D):
    return lib().sage_attn_gqa_ws_bytes(B, H, Hkv, N, D)


def sage_attn_gqa_bwd_ws_bytes(B, H, Hkv, N, D):
    return lib().sage_attn_gqa_bwd_ws_bytes(B, H, Hkv, N, D)


def sage_attn_gqa_quantize(Q, K, V, B, H, Hkv, N, D, qk_norm, k_smooth, ws, ws_bytes, stream):
    return lib().sage_attn_gqa_quantize(Q, K, V, B, H, Hkv, N, D, int(qk_norm), int(k_smooth), ws, ws_bytes, stream)


def sage_attn_gqa_fwd(ws, O, LSE, O32, B, H, Hkv, N, D, causal, sm_scale, stream):
    return lib().sage_attn_gqa_fwd(ws, O, LSE, O32, B, H, Hkv, N, D, int(causal), float(sm_scale), stream)


def sage_attn_gqa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, Hkv, N, D, causal, qk_norm,
                      k_smooth, sm_scale, stream):
    return lib().sage_attn_gqa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, Hkv, N, D,
                                   int(causal), int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_gqa_ws_views(ws, B, H, Hkv, N, D) -> sage_ws_views:
    v = sage_ws_views()
    rc = lib().sage_attn_gqa_ws_views(ws, B, H, Hkv, N, D, ctypes.byref(v))
    if rc:
        raise SageError("sage_attn_gqa_ws_views", rc)
    return v


def sage_attn_qs_ws_bytes(B, H, Hkv, N, D):
    return lib().sage_attn_qs_ws_bytes(B, H, Hkv, N, D)


def sage_attn_qs_quantize(Q, K, V, B, H, Hkv, N, D, qk_norm, k_smooth, ws, ws_bytes, stream):
    return lib().sage_attn_qs_quantize(Q, K, V, B, H, Hkv, N, D, int(qk_norm), int(k_smooth), ws, ws_bytes, stream)


def sage_attn_qs_fwd(ws, O, LSE, O32, B, H, Hkv, N, D, causal, sm_scale, stream):
    return lib().sage_attn_qs_fwd(ws, O, LSE, O32, B, H, Hkv, N, D, int(causal), float(sm_scale), stream)


def sage_attn_qs_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, Hkv, N, D, causal, qk_norm,
                     k_smooth, sm_scale, stream):
    return lib().sage_attn_qs_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, bwd_ws_bytes, B, H, Hkv, N, D,
                                  int(causal), int(qk_norm), int(k_smooth), float(sm_scale), stream)


def sage_attn_qs_ws_views(ws, B, H, Hkv, N, D) -> sage_ws_views:
    v = sage_ws_views()
    rc = lib().sage_attn_qs_ws_views(ws, B, H, Hkv, N, D, ctypes.byref(v))
    if rc != SAGE_OK:
        raise SageError("sage_attn_qs_ws_views", rc)
    return v


def sage_attn_ws_views(ws, B, H, N, D) -> sage_ws_views:
    v = sage_ws_views()
    rc = lib().sage_attn_ws_views(ws, B, H, N, D, ctypes.byref(v))
    if rc:
        raise SageError("sage_attn_ws_views", rc)
    return v


def sage_attn_get_status(ws, stream):
    return lib().sage_attn_get_status(ws, stream)


def sage_attn_selftest_wait(ws, budget_ns, stream):
    return lib().sage_attn_selftest_wait(ws, int(budget_ns), stream)


def sage_attn_timer_enable(on):
    return lib().sage_attn_timer_enable(int(on))


def sage_attn_timer_only(kernel):
    """Time only the launch group `kernel` (None: every group)."""
    return lib().sage_attn_timer_only(kernel.encode() if kernel else None)


def sage_attn_timer_read(kernel: str):
    """(total ms, launches) of the timed launches of `kernel` since the last read."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
    rc = lib().sage_attn_timer_read(kernel.encode(), ctypes.byref(ms), ctypes.byref(n))
    if rc:
        raise SageError("sage_attn_timer_read", rc)
    return ms.value, n.value


def status_str(code) -> str:
    try:
        return lib().sage_attn_status_str(int(code)).decode()
    except RuntimeError:
        return str(code)


# ------------------------------------------------------------- torch helpers

def _check(fn, rc):
    if rc != SAGE_OK:
        raise SageError(fn, rc)


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _shape(q):
    B, H, N, D = q.shape
    return B, H, N, D


def alloc_ws(B, H, N, D, device="cuda", hkv=None, q_smooth=False):
    import torch
    if q_smooth:
        n = sage_attn_qs_ws_bytes(B, H, H if hkv is None else hkv, N, D)
    else:
        n = sage_attn_ws_bytes(B, H, N, D) if hkv in (None, H) else sage_attn_gqa_ws_bytes(B, H, hkv, N, D)
    if n == 0:
        raise SageError("sage_attn_ws_bytes", SAGE_ERR_UNSUPPORTED)
    return torch.empty(n, dtype=torch.uint8, device=device)


def alloc_bwd_ws(B, H, N, D, device="cuda", hkv=None):
    import torch
    n = sage_attn_bwd_ws_bytes(B, H, N, D) if hkv in (None, H) else sage_attn_gqa_bwd_ws_bytes(B, H, hkv, N, D)
    if n == 0:
        raise SageError("sage_attn_bwd_ws_bytes", SAGE_ERR_UNSUPPORTED)
    return torch.empty(n, dtype=torch.uint8, device=device)


def quantize(q, k, v, qk_norm=False, k_smooth=True, ws=None, stream=None, q_smooth=False):
    """Quantize pass on bf16 [B, H, N, D] CUDA tensors (k, v: [B, Hkv, N, D], Hkv dividing H, for
    grouped-query attention); returns the workspace tensor.  q_smooth: Q-smoothing
    (sage_attn_qs_quantize; forward and backward then take q_smooth=True too)."""
    B, H, N, D = _shape(q)
    hkv = k.shape[1]
    if ws is None:
        ws = alloc_ws(B, H, N, D, q.device, hkv, q_smooth)
    if q_smooth:
        _check("sage_attn_qs_quantize",
               sage_attn_qs_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, hkv, N, D, qk_norm, k_smooth, _ptr(ws),
                                     ws.numel(), _stream_ptr(stream)))
    elif hkv == H:
        _check("sage_attn_quantize", sage_attn_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, qk_norm, k_smooth,
                                                        _ptr(ws), ws.numel(), _stream_ptr(stream)))
    else:
        _check("sage_attn_gqa_quantize",
               sage_attn_gqa_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, hkv, N, D, qk_norm, k_smooth, _ptr(ws),
                                      ws.numel(), _stream_ptr(stream)))
    return ws


def forward(ws, B, H, N, D, causal, sm_scale=None, o=None, lse=None, o32=False, device="cuda", stream=None,
            hkv=None, q_smooth=False):
    """Forward from a quantize workspace; returns (O bf16, LSE fp32[, O32 fp32]).  hkv: key/value
    heads of a grouped-query workspace; q_smooth: a workspace quantized with Q-smoothing."""
    import torch
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    O32 = torch.empty((B, H, N, D), dtype=torch.float32, device=device) if o32 is True else (o32 or None)
    if q_smooth:
        _check("sage_attn_qs_fwd", sage_attn_qs_fwd(_ptr(ws), _ptr(o), _ptr(lse), _ptr(O32), B, H,
                                                    H if hkv is None else hkv, N, D, causal, sm_scale,
                                                    _stream_ptr(stream)))
    elif hkv in (None, H):
        _check("sage_attn_fwd", sage_attn_fwd(_ptr(ws), _ptr(o), _ptr(lse), _ptr(O32), B, H, N, D, causal,
                                              sm_scale, _stream_ptr(stream)))
    else:
        _check("sage_attn_gqa_fwd", sage_attn_gqa_fwd(_ptr(ws), _ptr(o), _ptr(lse), _ptr(O32), B, H, hkv, N, D,
                                                      causal, sm_scale, _stream_ptr(stream)))
    return (o, lse, O32) if O32 is not None else (o, lse)


def fp4_quantize(q, k, v, qk_norm=False, k_smooth=True, ws=None, stream=None):
    """Quantize pass of the NVFP4 variant: the INT8 codes of Q and K and V's NVFP4 codes and
    block scales; returns the workspace tensor."""
    import torch
    B, H, N, D = _shape(q)
    if ws is None:
        n = sage_attn_fp4_ws_bytes(B, H, N, D)
        if n == 0:
            raise SageError("sage_attn_fp4_ws_bytes", SAGE_ERR_UNSUPPORTED)
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check("sage_attn_fp4_quantize", sage_attn_fp4_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, qk_norm,
                                                            k_smooth, _ptr(ws), ws.numel(), _stream_ptr(stream)))
    return ws


def fp4_forward(ws, B, H, N, D, causal, sm_scale=None, o=None, lse=None, o32=False, device="cuda", stream=None):
    """Forward of the NVFP4 variant; returns (O bf16, LSE fp32[, O32 fp32])."""
    import torch
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    O32 = torch.empty((B, H, N, D), dtype=torch.float32, device=device) if o32 is True else (o32 or None)
    _check("sage_attn_fp4_fwd", sage_attn_fp4_fwd(_ptr(ws), _ptr(o), _ptr(lse), _ptr(O32), B, H, N, D, causal,
                                                  sm_scale, _stream_ptr(stream)))
    return (o, lse, O32) if O32 is not None else (o, lse)


def fp4_backward(q, k, v, o, lse, do, ws, causal, qk_norm=False, k_smooth=True, sm_scale=None, bwd_ws=None,
                 dq=None, dk=None, dv=None, stream=None):
    """Backward of the NVFP4 variant (P^ recomputed in NVFP4); returns (dQ, dK, dV) bf16."""
    import torch
    B, H, N, D = _shape(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if bwd_ws is None:
        n = sage_attn_fp4_bwd_ws_bytes(B, H, N, D)
        if n == 0:
            raise SageError("sage_attn_fp4_bwd_ws_bytes", SAGE_ERR_UNSUPPORTED)
        bwd_ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check("sage_attn_fp4_bwd",
           sage_attn_fp4_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                             _ptr(ws), _ptr(bwd_ws), bwd_ws.numel(), B, H, N, D, causal, qk_norm, k_smooth, sm_scale,
                             _stream_ptr(stream)))
    return dq, dk, dv


def thrift_quantize(q, k, v, causal, budget, qk_norm=False, k_smooth=True, ws=None, tws=None, stream=None):
    """ThriftAttention's quantize pass: the low-bit codes (ws) and the selection of ceil(budget x
    visible pairs) promoted (query block, key tile) pairs with the fp16 operands of the
    high-precision path (tws).  Returns (ws, tws)."""
    import torch
    B, H, N, D = _shape(q)
    if ws is None:
        ws = alloc_ws(B, H, N, D, q.device)
    if tws is None:
        n = sage_attn_thrift_ws_bytes(B, H, N, D)
        if n == 0:
            raise SageError("sage_attn_thrift_ws_bytes", SAGE_ERR_UNSUPPORTED)
        tws = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check("sage_attn_thrift_quantize",
           sage_attn_thrift_quantize(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, qk_norm, k_smooth, causal, budget,
                                     _ptr(ws), ws.numel(), _ptr(tws), tws.numel(), _stream_ptr(stream)))
    return ws, tws


def thrift_forward(ws, tws, B, H, N, D, causal, sm_scale=None, o=None, lse=None, o32=False, device="cuda",
                   stream=None):
    """ThriftAttention's forward; returns (O bf16, LSE fp32[, O32 fp32])."""
    import torch
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    O32 = torch.empty((B, H, N, D), dtype=torch.float32, device=device) if o32 is True else (o32 or None)
    _check("sage_attn_thrift_fwd", sage_attn_thrift_fwd(_ptr(ws), _ptr(tws), _ptr(o), _ptr(lse), _ptr(O32), B, H, N,
                                                        D, causal, sm_scale, _stream_ptr(stream)))
    return (o, lse, O32) if O32 is not None else (o, lse)


def thrift_sel(tws, B, H, N, D):
    """The promoted pairs as a uint8 CUDA tensor [B*H, nb, nb] viewing the scratch."""
    nb = (N + 127) // 128
    off = sage_attn_thrift_sel(_ptr(tws), B, H, N, D) - tws.data_ptr()
    return tws[off:off + B * H * nb * nb].view(B * H, nb, nb)


def backward(q, k, v, o, lse, do, ws, causal, qk_norm=False, k_smooth=True, sm_scale=None, bwd_ws=None,
             dq=None, dk=None, dv=None, stream=None, o32=None, q_smooth=False):
    """Backward; returns (dQ, dK, dV) bf16.  With o32 (the forward's fp32 output) the row
    terms D_i take it instead of the bf16 o (sage_attn_bwd_o32); q_smooth: a workspace quantized
    with Q-smoothing (sage_attn_qs_bwd)."""
    import torch
    B, H, N, D = _shape(q)
    hkv = k.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if bwd_ws is None:
        bwd_ws = alloc_bwd_ws(B, H, N, D, q.device, hkv)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if q_smooth:
        if o32 is not None:
            raise ValueError("the fp32 auxiliary output is not offered with Q-smoothing")
        _check("sage_attn_qs_bwd",
               sage_attn_qs_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(ws), _ptr(bwd_ws), bwd_ws.numel(), B, H, hkv, N, D, causal,
                                qk_norm, k_smooth, sm_scale, _stream_ptr(stream)))
        return dq, dk, dv
    if hkv != H:
        if o32 is not None:
            raise ValueError("the fp32 auxiliary output is not offered with grouped key/value heads")
        _check("sage_attn_gqa_bwd",
               sage_attn_gqa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(ws), _ptr(bwd_ws), bwd_ws.numel(), B, H, hkv, N, D, causal,
                                 qk_norm, k_smooth, sm_scale, _stream_ptr(stream)))
        return dq, dk, dv
    if o32 is not None:
        _check("sage_attn_bwd_o32",
               sage_attn_bwd_o32(_ptr(q), _ptr(k), _ptr(v), _ptr(o32), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(ws), _ptr(bwd_ws), bwd_ws.numel(), B, H, N, D, causal, qk_norm,
                                 k_smooth, sm_scale, _stream_ptr(stream)))
        return dq, dk, dv
    _check("sage_attn_bwd", sage_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                                          _ptr(dk), _ptr(dv), _ptr(ws), _ptr(bwd_ws), bwd_ws.numel(), B, H, N,
                                          D, causal, qk_norm, k_smooth, sm_scale, _stream_ptr(stream)))
    return dq, dk, dv


def alloc_step_host(B, H, N, D, groups=0, device="cuda"):
    """Device scratch for step_host (its status word: get_status(scratch))."""
    import torch
    n = sage_attn_step_host_bytes(B, H, N, D, groups)
    if n == 0:
        raise SageError("sage_attn_step_host_bytes", SAGE_ERR_UNSUPPORTED)
    return torch.empty(n, dtype=torch.uint8, device=device)


def step_host(q, k, v, do, out, scratch, causal, qk_norm=False, k_smooth=True, sm_scale=None, groups=0,
              stream=None):
    """Quantize + forward + backward of host (CPU, ideally pinned) bf16 [B, H, N, D] tensors with the copies
    overlapped with the computation.  `out` holds host tensors o, lse, dq, dk, dv that receive the results;
    they are complete once `stream` has completed."""
    B, H, N, D = _shape(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    _check("sage_attn_step_host",
           sage_attn_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(out["o"]), _ptr(out["lse"]),
                               _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(scratch), scratch.numel(),
                               B, H, N, D, causal, qk_norm, k_smooth, sm_scale, groups, _stream_ptr(stream)))
    return out


def get_status(ws, stream=None) -> int:
    return sage_attn_get_status(_ptr(ws), _stream_ptr(stream))


def ws_tensors(ws, B, H, N, D, hkv=None, q_smooth=False, fp4=False) -> dict:
    """Views of a quantize workspace as torch tensors (for inspection and tests); hkv: key/value
    heads of a grouped-query workspace (K and V sections then hold B*hkv heads); q_smooth: a
    Q-smoothing workspace (adds qmean [B, H, Np/128, D] and dsb [B, H, Np/128, Np]); fp4: an
    NVFP4 workspace (adds vg [B, H], v4 [B, H, D, Np/2] and v4sf [B, H, Np/64, 512])."""
    import torch
    hk = H if hkv is None else hkv
    if fp4:
        v = sage_attn_fp4_ws_views(_ptr(ws), B, H, N, D)
    elif q_smooth:
        v = sage_attn_qs_ws_views(_ptr(ws), B, H, hk, N, D)
    elif hk == H:
        v = sage_attn_ws_views(_ptr(ws), B, H, N, D)
    else:
        v = sage_attn_gqa_ws_views(_ptr(ws), B, H, hk, N, D)
    base = ws.data_ptr()
    np_ = v.n_pad
    bh, bk = B * H, B * hk

    def view(ptr, n_bytes, dtype, shape):
        off = ptr - base
        return ws[off:off + n_bytes].view(dtype).view(shape)

    extra = {}
    if fp4:
        extra = {"vg": view(v.vg, bk * 4, torch.float32, (B, hk)),
                 "v4": view(v.v4, bk * D * np_ // 2, torch.uint8, (B, hk, D, np_ // 2)),
                 "v4sf": view(v.v4sf, bk * (np_ // 64) * 512, torch.uint8, (B, hk, np_ // 64, 512))}
    if q_smooth:
        nb = np_ // 128
        extra = {"qmean": view(v.qmean, bh * nb * D * 4, torch.float32, (B, H, nb, D)),
                 "dsb": view(v.dsb, bh * nb * np_ * 4, torch.float32, (B, H, nb, np_))}
    return extra | {
        "qc": view(v.qc, bh * np_ * D * 2, torch.bfloat16, (B, H, np_, D)),
        "kc": view(v.kc, bk * np_ * D * 2, torch.bfloat16, (B, hk, np_, D)),
        "v8t": view(v.v8t, bk * D * np_, torch.uint8, (B, hk, D, np_)),
        "sq": view(v.sq, bh * (np_ // 128) * 4, torch.float32, (B, H, np_ // 128)),
        "sk": view(v.sk, bk * (np_ // 64) * 4, torch.float32, (B, hk, np_ // 64)),
        "sv": view(v.sv, bk * D * 4, torch.float32, (B, hk, D)),
        "kmean": view(v.kmean, bk * D * 4, torch.float32, (B, hk, D)),
        "qr": view(v.qr, bh * np_ * 4, torch.float32, (B, H, np_)),
        "kr": view(v.kr, bk * np_ * 4, torch.float32, (B, hk, np_)),
        "n_pad": np_,
    }
