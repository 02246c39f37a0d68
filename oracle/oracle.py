"""ctypes front end of the CPU oracle (sage_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the bench's
CPU-baseline leg, never by the library.  It shares no code with the CUDA path.

All arrays are float64 numpy arrays of one head, [N, D] token-major.  The
quantizer mask selects which quantizers are on (QM_ALL = the low-bit scheme,
0 = exact fp64 attention through the same code).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

QM_QK, QM_V, QM_P, QM_DO, QM_DS, QM_F32 = 1, 2, 4, 8, 16, 32
QM_ALL = 63
QM_FP4 = 64  # NVFP4 for V and P (with QM_ALL: the FP4 variant of the scheme)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libsage_oracle.so")
_lock = threading.Lock()
_lib = None


_CMD = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard", "-fPIC",
        "-shared"]


def _fingerprint() -> str:
    """Source bytes, flags and host machine: a library built otherwise is rebuilt."""
    import hashlib
    import platform
    h = hashlib.sha256(open(_SRC, "rb").read())
    h.update(" ".join(_CMD).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, OpenMP, IEEE operations only)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    stamp = _OUT + ".stamp"
    fp = _fingerprint()
    fresh = os.path.exists(_OUT) and os.path.exists(stamp) and open(stamp).read().strip() == fp
    if force or not fresh:
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.run(_CMD + ["-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _OUT)
        with open(stamp, "w") as f:
            f.write(fp + "\n")
    return _OUT


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            fp = ctypes.POINTER(ctypes.c_float)
            i = ctypes.c_int
            L.sage_oracle_e4m3.restype = ctypes.c_double
            L.sage_oracle_e4m3.argtypes = [ctypes.c_double]
            L.sage_oracle_e4m3_f32.argtypes = [fp, fp, ctypes.c_long]
            L.sage_oracle_e2m1.restype = ctypes.c_double
            L.sage_oracle_e2m1.argtypes = [ctypes.c_double]
            L.sage_oracle_e2m1_f64.argtypes = [dp, dp, ctypes.c_long]
            L.sage_oracle_fp16_f64.argtypes = [dp, dp, ctypes.c_long]
            L.sage_oracle_fwd_thrift.argtypes = ([i, i, i, ctypes.c_double, i] + [dp] * 6 +
                                                 [ctypes.POINTER(ctypes.c_ubyte)] + [dp] * 3 + [dp, fp, dp])
            L.sage_oracle_to_bf16.argtypes = [dp, dp, ctypes.c_long]
            L.sage_oracle_quantize.argtypes = [i, i, dp, dp, dp, i, i, i] + [dp] * 11
            L.sage_oracle_fwd.argtypes = [i, i, i, ctypes.c_double, i] + [dp] * 6 + [dp, fp, dp]
            L.sage_oracle_bwd.argtypes = [i, i, i, ctypes.c_double, i, i] + [dp] * 12 + [dp] * 4
            L.sage_oracle_bwd_sdo.argtypes = [i, i, i, ctypes.c_double, i, i] + [dp] * 12 + [dp] * 5
            L.sage_oracle_quantize_qs.argtypes = [i, i, dp, dp, dp, i, i, i] + [dp] * 13
            L.sage_oracle_fwd_qs.argtypes = [i, i, i, ctypes.c_double, i] + [dp] * 7 + [dp, fp, dp]
            L.sage_oracle_bwd_qs.argtypes = [i, i, i, ctypes.c_double, i, i] + [dp] * 12 + [dp] * 7
            _lib = L
    return _lib


def _d(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _c64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def e4m3(x: np.ndarray) -> np.ndarray:
    """e4m3 rounding (nearest even, saturating) of fp32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().sage_oracle_e4m3_f32(_f(x), _f(y), x.size)
    return y


def e2m1(x: np.ndarray) -> np.ndarray:
    """e2m1 (FP4) rounding (nearest, ties to the even mantissa, saturating at 6)."""
    x = _c64(x)
    y = np.empty_like(x)
    lib().sage_oracle_e2m1_f64(_d(x), _d(y), x.size)
    return y


def fp16(x: np.ndarray) -> np.ndarray:
    """fp16 rounding (nearest even) as the oracle forms it."""
    x = _c64(x)
    y = np.empty_like(x)
    lib().sage_oracle_fp16_f64(_d(x), _d(y), x.size)
    return y


def _block_means(x: np.ndarray) -> np.ndarray:
    """Channel means of the 128-token blocks [ceil(N/128), D]: fp64 sums over the block's
    tokens in token order, divided by the block's token count."""
    N, D = x.shape
    nb = -(-N // 128)
    out = np.empty((nb, D))
    for b in range(nb):
        blk = x[b * 128:(b + 1) * 128]
        s = np.zeros(D)
        for t in range(blk.shape[0]):
            s = s + blk[t]
        out[b] = s / blk.shape[0]
    return out


def thrift_select(q, k, causal, budget) -> np.ndarray:
    """ThriftAttention's selection ("ThriftAttention" (gist.science summary), Methodology
    step 1): the importance of the pair (128-query block I, 128-key tile J) is the dot
    product of the blocks' token means, qbar_I . kbar_J, over the raw inputs; the
    ceil(budget * pairs) most important of the pairs the mask lets through (causal: J <= I)
    are promoted, ties taken in (I, J) order.  Returns uint8 [nI, nJ], 1 = promoted."""
    q, k = _c64(q), _c64(k)
    N = q.shape[0]
    nb = -(-N // 128)
    qm, km = _block_means(q), _block_means(k)
    # the dot products in a fixed order: fp64 products added over the channels one by one
    score = np.zeros((nb, nb))
    for d in range(q.shape[1]):
        score = score + qm[:, d, None] * km[None, :, d]
    vis = np.tril(np.ones((nb, nb), dtype=bool)) if causal else np.ones((nb, nb), dtype=bool)
    idx = np.flatnonzero(vis.ravel())
    n = int(math.ceil(budget * idx.size - 1e-12))
    order = idx[np.lexsort((idx, -score.ravel()[idx]))]
    sel = np.zeros(nb * nb, dtype=np.uint8)
    sel[order[:n]] = 1
    return sel.reshape(nb, nb)


def thrift_inputs(qz: dict, v) -> dict:
    """The high-precision path's operands: the softmax's q' and k'' (the smoothed keys,
    RN32(k' - kmean), which K's quantizer takes) and V, rounded to fp16."""
    ks = (qz["kn"] - qz["kmean"]).astype(np.float32).astype(np.float64)
    return {"qh": fp16(qz["qn"]), "kh": fp16(ks), "vh": fp16(_c64(v))}


def to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (both nearest even), returned as float64 values."""
    x = _c64(x)
    y = np.empty_like(x)
    lib().sage_oracle_to_bf16(_d(x), _d(y), x.size)
    return y


def quantize(q, k, v, qk_norm, k_smooth, qmask=QM_ALL, q_smooth=False) -> dict:
    """One head's codes and scales.  q_smooth adds "qmean" [ceil(N/128), D] (the query
    blocks' channel means, removed before the INT8 quantizer) and "dsb" [ceil(N/128), N]
    (the logit term they carry back), see sage_oracle.c."""
    q, k, v = _c64(q), _c64(k), _c64(v)
    N, D = q.shape
    nI = max(1, -(-N // 128))
    o = {n: np.zeros((N, D)) for n in ("qn", "kn", "qx", "kx", "vx")}
    o.update(qr=np.zeros(N), kr=np.zeros(N), kmean=np.zeros(D),
             sq=np.zeros(nI), sk=np.zeros(max(1, -(-N // 64))), sv=np.zeros(D))
    args = [N, D, _d(q), _d(k), _d(v), int(qk_norm), int(k_smooth), int(qmask),
            _d(o["qn"]), _d(o["qr"]), _d(o["kn"]), _d(o["kr"]), _d(o["kmean"]),
            _d(o["qx"]), _d(o["sq"]), _d(o["kx"]), _d(o["sk"]), _d(o["vx"]), _d(o["sv"])]
    if q_smooth:
        o.update(qmean=np.zeros((nI, D)), dsb=np.zeros((nI, max(N, 1))))
        rc = lib().sage_oracle_quantize_qs(*args, _d(o["qmean"]), _d(o["dsb"]))
    else:
        rc = lib().sage_oracle_quantize(*args)
    if rc:
        raise RuntimeError(f"oracle quantize failed ({rc})")
    return o


def forward(qz: dict, causal, sm_scale, qmask=QM_ALL, thrift=None) -> dict:
    """One head's forward; with Q-smoothing when qz carries "dsb".  thrift: ThriftAttention's
    mixed precision, {"sel": thrift_select(...), **thrift_inputs(...)}."""
    N, D = qz["qx"].shape
    O64 = np.zeros((N, D))
    O32 = np.zeros((N, D), dtype=np.float32)
    L = np.zeros(N)
    args = [N, D, int(causal), float(sm_scale), int(qmask), _d(qz["qx"]), _d(qz["sq"]), _d(qz["kx"]),
            _d(qz["sk"]), _d(qz["vx"]), _d(qz["sv"])]
    if thrift is not None:
        if "dsb" in qz:
            raise ValueError("ThriftAttention is not combined with Q-smoothing")
        sel = np.ascontiguousarray(thrift["sel"], dtype=np.uint8)
        th = {n: _c64(thrift[n]) for n in ("qh", "kh", "vh")}
        rc = lib().sage_oracle_fwd_thrift(*args, sel.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                          _d(th["qh"]), _d(th["kh"]), _d(th["vh"]), _d(O64), _f(O32), _d(L))
    elif "dsb" in qz:
        rc = lib().sage_oracle_fwd_qs(*args, _d(qz["dsb"]), _d(O64), _f(O32), _d(L))
    else:
        rc = lib().sage_oracle_fwd(*args, _d(O64), _f(O32), _d(L))
    if rc:
        raise RuntimeError(f"oracle forward failed ({rc})")
    return {"O64": O64, "O32": O32, "Obf": to_bf16(O64), "LSE64": L,
            "LSE32": L.astype(np.float32)}


def backward(qz: dict, v, do, O, LSE, causal, sm_scale, qk_norm, qmask=QM_ALL, sdo=None) -> dict:
    """One head's backward; sdo (optional, [D]) gives the e4m3 channel scales of dO instead of
    taking them from this head's dO (grouped-query attention, see run_group).  With
    Q-smoothing when qz carries "dsb" and "qmean"."""
    v, do, O, LSE = _c64(v), _c64(do), _c64(O), _c64(LSE)
    N, D = v.shape
    dQ, dK, dV = np.zeros((N, D)), np.zeros((N, D)), np.zeros((N, D))
    Dv = np.zeros(N)
    common = (N, D, int(causal), float(sm_scale), int(qk_norm), int(qmask),
              _d(v), _d(do), _d(O), _d(LSE),
              _d(qz["qx"]), _d(qz["sq"]), _d(qz["kx"]), _d(qz["sk"]),
              _d(qz["qn"]), _d(qz["qr"]), _d(qz["kn"]), _d(qz["kr"]))
    if "dsb" in qz:
        sdo_a = _c64(sdo) if sdo is not None else None
        rc = lib().sage_oracle_bwd_qs(*common, _d(sdo_a) if sdo_a is not None else None, _d(qz["dsb"]),
                                      _d(qz["qmean"]), _d(dQ), _d(dK), _d(dV), _d(Dv))
    elif sdo is None:
        rc = lib().sage_oracle_bwd(*common, _d(dQ), _d(dK), _d(dV), _d(Dv))
    else:
        sdo = _c64(sdo)
        rc = lib().sage_oracle_bwd_sdo(*common, _d(sdo), _d(dQ), _d(dK), _d(dV), _d(Dv))
    if rc:
        raise RuntimeError(f"oracle backward failed ({rc})")
    return {"dQ64": dQ, "dK64": dK, "dV64": dV, "dQbf": to_bf16(dQ), "dKbf": to_bf16(dK),
            "dVbf": to_bf16(dV), "Dvec": Dv}


def run_head(q, k, v, do, causal, sm_scale, qk_norm=False, k_smooth=True, qmask=QM_ALL,
             backward_pass=True, o_aux="bf16", q_smooth=False) -> dict:
    """Quantize, forward and (optionally) backward of one head.

    In the low-bit scheme (F32 bit on) the backward consumes the forward's bf16 O
    and fp32 LSE, as a training step would; with exact arithmetic it consumes
    the fp64 values.  o_aux="fp32" gives the backward the forward's fp32 O instead
    of the bf16 one for D_i = rowsum(dO * O): the high-precision auxiliary output of
    "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science
    summary), Methodology, principle 2.  q_smooth: Q-smoothing (see quantize).
    """
    qz = quantize(q, k, v, qk_norm, k_smooth, qmask, q_smooth)
    fw = forward(qz, causal, sm_scale, qmask)
    out = dict(qz)
    out.update(fw)
    if backward_pass:
        if qmask & QM_F32:
            O_used = fw["O32"].astype(np.float64) if o_aux == "fp32" else fw["Obf"]
            L_used = fw["LSE32"].astype(np.float64)
        else:
            O_used, L_used = fw["O64"], fw["LSE64"]
        out.update(backward(qz, v, do, O_used, L_used, causal, sm_scale, qk_norm, qmask))
    return out


def run_group(qs, k, v, dos, causal, sm_scale, qk_norm=False, k_smooth=True, qmask=QM_ALL,
              q_smooth=False) -> dict:
    """Grouped-query attention: the G query heads qs[g] (with upstream gradients dos[g])
    share the key/value head k, v.  Each query head is quantized (Q block scales of its
    own; K and V codes, the same for every head of the group), run forward and backward
    as one head, except that the e4m3 channel scale of dO spans the group's tokens: dV of
    the shared head sums P^T dO over all of them, so one scale per channel keeps that sum
    a single FP8 accumulation.  dK and dV of the shared head are the sums over the group.
    Returns {"heads": [run_head-like dicts], "dK64", "dV64", "dKbf", "dVbf", "sdo"}.
    """
    qs = [_c64(q) for q in qs]
    dos = [_c64(d) for d in dos]
    N, D = _c64(v).shape
    if qmask & QM_DO:
        a = np.max(np.abs(np.stack(dos)), axis=(0, 1))  # per channel over the group's tokens
        s = (a / 448.0).astype(np.float32).astype(np.float64) if qmask & QM_F32 else a / 448.0
        sdo = np.where(a > 0.0, s, 0.0)
    else:
        sdo = np.ones(D)
    heads = []
    dK, dV = np.zeros((N, D)), np.zeros((N, D))
    for q, do in zip(qs, dos):
        qz = quantize(q, k, v, qk_norm, k_smooth, qmask, q_smooth)
        fw = forward(qz, causal, sm_scale, qmask)
        out = dict(qz)
        out.update(fw)
        if qmask & QM_F32:
            O_used, L_used = fw["Obf"], fw["LSE32"].astype(np.float64)
        else:
            O_used, L_used = fw["O64"], fw["LSE64"]
        out.update(backward(qz, v, do, O_used, L_used, causal, sm_scale, qk_norm, qmask, sdo=sdo))
        heads.append(out)
        dK += out["dK64"]
        dV += out["dV64"]
    return {"heads": heads, "dK64": dK, "dV64": dV, "dKbf": to_bf16(dK), "dVbf": to_bf16(dV), "sdo": sdo}
