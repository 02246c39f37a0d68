"""NVFP4 variant (sage_attn_fp4_*) on the GPU against the CPU oracle's QM_FP4 mode
("Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science summary),
Methodology principle 1; "ThriftAttention" (gist.science summary), Methodology step 2).

V's NVFP4 values (e2m1 code x e4m3 block scale x tensor scale) must equal the oracle's bit
for bit, the INT8 codes of Q and K too; O32 within the forward's 2e-3, LSE within 1e-4
(relative to max(1, |LSE|)), and the bf16 O the rounding of O32.  P's codes and block
scales are formed in the softmax, where a code or scale near a rounding boundary is redone
from an accurate 2^t; heavy-tailed logits put many of them there."""
import numpy as np
import pytest

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# The backward recomputes P^ in NVFP4 from the saved LSE (the forward's blocks); dQ, dK, dV
# are held to the backward's relative-L2 tolerance of 1e-2 against the oracle.

SMALL = [
    wl.custom(1, 2, 333, 64, True, seed=90, kind="k_offset2", name="n333_d64_causal"),
    wl.custom(1, 2, 700, 128, True, qk_norm=True, sm_scale=16.0, seed=91, name="n700_d128_causal_qknorm"),
    wl.custom(2, 1, 250, 128, False, seed=92, kind="k_outlier20", name="n250_d128_outliers"),
    wl.custom(1, 1, 1, 64, False, seed=93, name="n1_d64"),
    wl.custom(1, 2, 640, 128, True, seed=94, kind="student_t3", name="n640_d128_student"),
    wl.custom(1, 1, 512, 64, False, seed=95, kind="k_offset3", name="n512_d64_offset3"),
]

_E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])


def _v_values(views, b, h, N, D):
    """V's NVFP4 values [N, D] from the workspace: code x block scale x tensor scale."""
    import torch
    codes = views["v4"][b, h].cpu().numpy()  # [D, Np/2]
    lo, hi = codes & 15, codes >> 4
    c = np.empty((D, codes.shape[1] * 2), dtype=np.int64)
    c[:, 0::2], c[:, 1::2] = lo, hi
    atoms = views["v4sf"][b, h].cpu().numpy()  # [Np/64, 512]
    d = np.arange(D)[:, None]
    b16 = np.arange(c.shape[1] // 16)[None, :]
    sb = atoms[b16 // 4, (d % 32) * 16 + (d // 32) * 4 + (b16 % 4)]  # [D, Np/16]
    s = torch.from_numpy(sb.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    g = float(views["vg"][b, h].item())
    vals = _E2M1[c] * np.repeat(s, 16, axis=1) * g
    return vals[:, :N].T


def _run(w, x, backward=False):
    import torch
    import bit_trainable_attention_sagebwd_gb300 as sa
    import parity
    t = parity.to_dev(x)
    B, H, N, D = w.B, w.H, w.N, w.D
    ws = sa.fp4_quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth)
    o, lse, o32 = sa.fp4_forward(ws, B, H, N, D, w.causal, w.sm_scale, o32=True)
    out = {"O": o, "LSE": lse, "O32": o32}
    if backward:
        dq, dk, dv = sa.fp4_backward(t["q"], t["k"], t["v"], o, lse, t["do"], ws, w.causal, w.qk_norm, w.k_smooth,
                                     w.sm_scale)
        out.update(dQ=dq, dK=dk, dV=dv)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == sa.SAGE_OK
    out["views"] = sa.ws_tensors(ws, B, H, N, D, fp4=True)
    return out


def _check_head(w, x, g, bh, backward=False):
    import parity
    from oracle import oracle as orc
    b, h = divmod(bh, w.H)
    r = parity.oracle_head(w, x, bh, backward=backward, qmask=orc.QM_ALL | orc.QM_FP4)
    if backward:
        parity.check_backward_head(w, g, bh, r)
    v = g["views"]
    N = w.N
    qc = v["qc"][b, h].float().cpu().numpy().astype(np.float64)
    kc = v["kc"][b, h].float().cpu().numpy().astype(np.float64)
    assert np.array_equal(qc[:N], r["qx"]) and np.array_equal(kc[:N], r["kx"]), f"Q/K codes differ at head {bh}"
    vv = _v_values(v, b, h, N, w.D)
    assert np.array_equal(vv, r["vx"]), f"V NVFP4 values differ at head {bh}: {np.sum(vv != r['vx'])}"
    return parity.check_forward_head(w, g, bh, r)


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_fp4_forward_small(w):
    x = wl.all_inputs(w)
    g = _run(w, x)
    for bh in range(w.bh):
        _check_head(w, x, g, bh)


@pytest.mark.parametrize("name", ["pretrain_8k", "long_32k", "video_dit"])
def test_fp4_forward_full_size(name):
    """Full-size workloads; the oracle computes the first, a middle and the last head."""
    import parity
    w = wl.WORKLOADS[name]
    x = wl.all_inputs(w)
    g = _run(w, x)
    for bh in parity.full_size_heads(w):
        _check_head(w, x, g, bh)


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_fp4_backward_small(w):
    x = wl.all_inputs(w)
    g = _run(w, x, backward=True)
    for bh in range(w.bh):
        _check_head(w, x, g, bh, backward=True)


@pytest.mark.parametrize("name", ["pretrain_8k", "long_32k"])
def test_fp4_backward_full_size(name):
    """Full-size workloads; the oracle computes the first, a middle and the last head."""
    import parity
    w = wl.WORKLOADS[name]
    x = wl.all_inputs(w)
    g = _run(w, x, backward=True)
    for bh in parity.full_size_heads(w):
        _check_head(w, x, g, bh, backward=True)
