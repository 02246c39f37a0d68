"""Shared helpers of the parity tests: run the CUDA path through the C ABI and the
CPU oracle on the same seeded inputs, and compare.  Imported by tests only."""
from __future__ import annotations

import numpy as np
import torch

import bit_trainable_attention_sagebwd_gb300 as sa
from bit_trainable_attention_sagebwd_gb300 import workloads as wl
from oracle import oracle as orc

O_ATOL = 2e-3       # max |O32_gpu - O32_oracle|, the stated forward tolerance
LSE_ATOL = 1e-4     # LSE differs only through ~1 ulp exp2/log2 differences
GRAD_RTOL = 1e-2    # relative L2 of dQ, dK, dV against the oracle


def to_dev(x: dict, dev="cuda") -> dict:
    return {n: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
            for n, a in x.items()}


def head_f64(x: dict, w, bh) -> dict:
    b, h = divmod(bh, w.H)
    return {n: wl.bf16_bits_to_f32(a[b, h]).astype(np.float64) for n, a in x.items()}


def e4m3_decode(u8: torch.Tensor) -> np.ndarray:
    return u8.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def run_gpu(w, x: dict, backward=True, o32_aux=False) -> dict:
    t = to_dev(x)
    B, H, N, D = w.B, w.H, w.N, w.D
    ws = sa.quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth)
    o, lse, o32 = sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o32=True)
    out = {"ws": ws, "O": o, "LSE": lse, "O32": o32, "in": t}
    if backward:
        dq, dk, dv = sa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], ws, w.causal, w.qk_norm,
                                 w.k_smooth, w.sm_scale, o32=o32 if o32_aux else None)
        out.update(dQ=dq, dK=dk, dV=dv)
    torch.cuda.synchronize()
    st = sa.get_status(ws)
    assert st == sa.SAGE_OK, f"device status {st}"
    out["views"] = sa.ws_tensors(ws, B, H, N, D)
    return out


def check_quantize_head(w, g: dict, bh: int, r: dict):
    """Bit-exact comparison of one head's codes and scales."""
    b, h = divmod(bh, w.H)
    v = g["views"]
    N, np_ = w.N, v["n_pad"]
    qc = v["qc"][b, h].float().cpu().numpy().astype(np.float64)
    kc = v["kc"][b, h].float().cpu().numpy().astype(np.float64)
    assert np.array_equal(qc[:N], r["qx"]), f"q codes differ at head {bh}: {np.sum(qc[:N] != r['qx'])}"
    assert np.array_equal(kc[:N], r["kx"]), f"k codes differ at head {bh}: {np.sum(kc[:N] != r['kx'])}"
    assert not qc[N:].any() and not kc[N:].any(), "padded code rows must be zero"
    nq, nk = -(-N // 128), -(-N // 64)
    assert np.array_equal(v["sq"][b, h].cpu().numpy()[:nq].astype(np.float64), r["sq"][:nq])
    assert np.array_equal(v["sk"][b, h].cpu().numpy()[:nk].astype(np.float64), r["sk"][:nk])
    assert np.array_equal(v["sv"][b, h].cpu().numpy().astype(np.float64), r["sv"])
    assert np.array_equal(v["kmean"][b, h].cpu().numpy().astype(np.float64), r["kmean"])
    if w.qk_norm:
        assert np.array_equal(v["qr"][b, h].cpu().numpy()[:N].astype(np.float64), r["qr"])
        assert np.array_equal(v["kr"][b, h].cpu().numpy()[:N].astype(np.float64), r["kr"])
    v8 = e4m3_decode(v["v8t"][b, h])  # [D, Np]
    assert np.array_equal(v8[:, :N].T, r["vx"]), f"v codes differ at head {bh}: {np.sum(v8[:, :N].T != r['vx'])}"
    assert not v8[:, N:].any()


def check_forward_head(w, g: dict, bh: int, r: dict) -> dict:
    b, h = divmod(bh, w.H)
    o32 = g["O32"][b, h].cpu().numpy()
    err = float(np.abs(o32.astype(np.float64) - r["O32"].astype(np.float64)).max())
    assert err <= O_ATOL, f"O32 max abs error {err} at head {bh}"
    obf = g["O"][b, h]
    assert torch.equal(obf, g["O32"][b, h].to(torch.bfloat16)), "bf16 O must be the rounding of O32"
    lse = g["LSE"][b, h].cpu().numpy().astype(np.float64)
    lerr = float(np.abs(lse - r["LSE64"]).max())
    assert lerr <= LSE_ATOL * max(1.0, float(np.abs(r["LSE64"]).max())), f"LSE error {lerr} at head {bh}"
    return {"o_err": err, "lse_err": lerr}


def full_size_heads(w) -> list:
    """Heads the full-size checks compare: every head of a small workload; otherwise the first,
    the last and one in the middle.  The forward and backward launch their CTAs in groups of
    heads whose operands fit in L2 (heads in order, longest tiles first within a group), so
    the first and last heads sit in the first and last groups and B*H/2 + 1 in a middle one
    (long_32k: backward groups of 4 heads, forward groups of 7)."""
    if w.bh <= 4:
        return list(range(w.bh))
    return sorted({0, w.bh // 2 + 1, w.bh - 1})


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def check_backward_head(w, g: dict, bh: int, r: dict) -> dict:
    b, h = divmod(bh, w.H)
    out = {}
    for name, key in (("dQ", "dQbf"), ("dK", "dKbf"), ("dV", "dVbf")):
        got = g[name][b, h].float().cpu().numpy().astype(np.float64)
        e = rel_l2(got, r[key])
        assert e <= GRAD_RTOL, f"{name} relative L2 error {e} at head {bh}"
        out[name] = e
    return out


def oracle_head(w, x, bh, backward=True, o_aux="bf16", qmask=None) -> dict:
    hx = head_f64(x, w, bh)
    return orc.run_head(hx["q"], hx["k"], hx["v"], hx["do"], w.causal, w.sm_scale, w.qk_norm, w.k_smooth,
                        qmask=orc.QM_ALL if qmask is None else qmask, backward_pass=backward, o_aux=o_aux)
