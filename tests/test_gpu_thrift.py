"""ThriftAttention's selective mixed precision on the GPU (sage_attn_thrift_*) against the CPU
oracle ("ThriftAttention" (gist.science summary), Methodology steps 1-2).

The promoted pairs must equal the oracle's selection bit for bit (index work); O32 within the
forward's 2e-3, LSE within 1e-4 (relative to max(1, |LSE|)), and the bf16 O the rounding of
O32.  The promoted tiles' fp16 logits are summed in fp32 on the tensor core rather than
rounded once from the exact sum, so the running maximum can differ in its last bit from the
oracle's; the low-bit tiles' codes follow it, which the tolerance covers."""
import numpy as np
import pytest

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    (wl.custom(1, 2, 640, 128, True, seed=80, kind="k_offset2", name="n640_d128_causal"), 0.2),
    (wl.custom(1, 2, 700, 64, False, qk_norm=True, sm_scale=8.0, seed=81, name="n700_d64_qknorm"), 0.3),
    (wl.custom(2, 1, 1000, 128, True, seed=82, kind="student_t3", name="n1000_d128_student"), 0.05),
    (wl.custom(1, 1, 129, 128, False, k_smooth=False, seed=83, name="n129_nosmooth"), 0.5),
    (wl.custom(1, 2, 512, 64, True, seed=84, name="n512_budget0"), 0.0),
    (wl.custom(1, 2, 384, 128, True, seed=85, kind="k_offset3", name="n384_budget1"), 1.0),
    # block means whose values span more than 38 binades take the fp64 sum in order; the
    # others the exact integer sum (the same bits either way)
    (wl.custom(1, 2, 515, 128, True, seed=86, kind="exp_spread", name="n515_exp_spread"), 0.1),
]


def _run(w, x, budget):
    import torch
    import bit_trainable_attention_sagebwd_gb300 as sa
    import parity
    t = parity.to_dev(x)
    B, H, N, D = w.B, w.H, w.N, w.D
    ws, tws = sa.thrift_quantize(t["q"], t["k"], t["v"], w.causal, budget, w.qk_norm, w.k_smooth)
    o, lse, o32 = sa.thrift_forward(ws, tws, B, H, N, D, w.causal, w.sm_scale, o32=True)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == sa.SAGE_OK
    return {"O": o, "LSE": lse, "O32": o32, "sel": sa.thrift_sel(tws, B, H, N, D).cpu().numpy()}


def _check_head(w, x, g, bh, budget):
    import parity
    from oracle import oracle as orc
    hx = parity.head_f64(x, w, bh)
    sel = orc.thrift_select(hx["q"], hx["k"], w.causal, budget)
    assert np.array_equal(g["sel"][bh], sel), f"promoted pairs differ at head {bh}"
    qz = orc.quantize(hx["q"], hx["k"], hx["v"], w.qk_norm, w.k_smooth)
    th = dict(sel=sel, **orc.thrift_inputs(qz, hx["v"]))
    r = orc.forward(qz, w.causal, w.sm_scale, thrift=th)
    parity.check_forward_head(w, g, bh, r)
    return int(sel.sum())


@pytest.mark.parametrize("w,budget", CASES, ids=[c[0].name for c in CASES])
def test_thrift_forward_small(w, budget):
    x = wl.all_inputs(w)
    g = _run(w, x, budget)
    for bh in range(w.bh):
        _check_head(w, x, g, bh, budget)


@pytest.mark.parametrize("name", ["pretrain_8k", "long_32k"])
def test_thrift_forward_full_size(name):
    """The page's 5 % budget on full-size causal workloads; the oracle computes the first, a
    middle and the last head."""
    import parity
    w = wl.WORKLOADS[name]
    x = wl.all_inputs(w)
    g = _run(w, x, 0.05)
    for bh in parity.full_size_heads(w):
        assert _check_head(w, x, g, bh, 0.05) > 0
