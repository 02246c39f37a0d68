"""Q-smoothing (sage_attn_qs_*) against the oracle's Q-smoothed run_group: the query blocks'
channel means and the codes of the smoothed queries bit-exact, the logit terms within fp32
summation error, O32 and LSE within the forward tolerances, dQ, dK, dV within the gradient
tolerance.  Covers plain heads, multi-query attention with QK-norm and grouped heads, ragged
and causal."""
import numpy as np
import pytest
import torch

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (workload with H query heads, key/value heads Hkv)
CASES = [
    (wl.custom(1, 2, 333, 64, True, seed=60, kind="q_offset3", name="qs_h2_n333_d64_causal"), 2),
    (wl.custom(2, 3, 256, 128, False, qk_norm=True, sm_scale=16.0, seed=61, name="qs_b2_h3_mqa_qknorm"), 1),
    (wl.custom(1, 4, 600, 128, True, seed=62, kind="q_offset3", name="qs_h4_kv2_n600_d128_causal"), 2),
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("w,hkv", CASES, ids=[c[0].name for c in CASES])
def test_q_smoothing_matches_oracle(w, hkv):
    import bit_trainable_attention_sagebwd_gb300 as sa
    import parity
    from oracle import oracle as orc
    x = wl.all_inputs(w)
    B, H, N, D = w.B, w.H, w.N, w.D
    G = H // hkv
    kx, vx = x["k"][:, :hkv], x["v"][:, :hkv]
    q, k, v, do = _dev(x["q"]), _dev(kx), _dev(vx), _dev(x["do"])
    ws = sa.quantize(q, k, v, w.qk_norm, w.k_smooth, q_smooth=True)
    o, lse, o32 = sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o32=True, hkv=hkv, q_smooth=True)
    dq, dk, dv = sa.backward(q, k, v, o, lse, do, ws, w.causal, w.qk_norm, w.k_smooth, w.sm_scale, q_smooth=True)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == sa.SAGE_OK
    views = sa.ws_tensors(ws, B, H, N, D, hkv=hkv, q_smooth=True)
    f64 = lambda a: wl.bf16_bits_to_f32(a).astype(np.float64)  # noqa: E731
    nI = -(-N // 128)
    for b in range(B):
        for kh in range(hkv):
            heads = [kh * G + g for g in range(G)]
            r = orc.run_group([f64(x["q"][b, h]) for h in heads], f64(kx[b, kh]), f64(vx[b, kh]),
                              [f64(x["do"][b, h]) for h in heads], w.causal, w.sm_scale, w.qk_norm, w.k_smooth,
                              q_smooth=True)
            r0 = r["heads"][0]
            kc = views["kc"][b, kh].float().cpu().numpy().astype(np.float64)
            assert np.array_equal(kc[:N], r0["kx"])
            for g, h in enumerate(heads):
                rh = r["heads"][g]
                qm = views["qmean"][b, h].cpu().numpy().astype(np.float64)
                assert np.array_equal(qm[:nI], rh["qmean"]), f"query block means differ at head {h}"
                qc = views["qc"][b, h].float().cpu().numpy().astype(np.float64)
                assert np.array_equal(qc[:N], rh["qx"]), f"q codes differ at head {h}"
                assert np.array_equal(views["sq"][b, h].cpu().numpy()[:nI].astype(np.float64), rh["sq"])
                dsb = views["dsb"][b, h].cpu().numpy().astype(np.float64)[:nI, :N]
                bound = 1e-5 * (np.abs(rh["qmean"]) @ np.abs(rh["kn"] - rh["kmean"]).T) + 1e-30
                assert np.all(np.abs(dsb - rh["dsb"]) <= bound), f"logit terms differ at head {h}"
                e = float(np.abs(o32[b, h].cpu().numpy().astype(np.float64) - rh["O32"].astype(np.float64)).max())
                assert e <= parity.O_ATOL, f"O32 error {e} at head {h}"
                lerr = float(np.abs(lse[b, h].cpu().numpy().astype(np.float64) - rh["LSE64"]).max())
                assert lerr <= parity.LSE_ATOL * max(1.0, float(np.abs(rh["LSE64"]).max()))
                eq = parity.rel_l2(dq[b, h].float().cpu().numpy().astype(np.float64), rh["dQbf"])
                assert eq <= parity.GRAD_RTOL, f"dQ relative L2 {eq} at head {h}"
            for name, got in (("dK", dk), ("dV", dv)):
                e = parity.rel_l2(got[b, kh].float().cpu().numpy().astype(np.float64), r[name + "bf"])
                assert e <= parity.GRAD_RTOL, f"{name} relative L2 {e} at key/value head {kh}"


def test_q_smoothing_zero_means_match_the_plain_path():
    """Query blocks whose every channel mean is exactly zero (each token paired with its
    negation inside the block): the Q-smoothed codes and scales equal the plain path's, the
    logit terms are zero, and O and the gradients agree with the plain path to the rounding
    of the logit (RN(acc RN(s_q s_k)) alpha against acc RN(RN(s_q s_k) alpha))."""
    import bit_trainable_attention_sagebwd_gb300 as sa
    w = wl.custom(1, 2, 256, 128, True, seed=63, name="qs_zero_mean")
    x = wl.all_inputs(w)
    qb = x["q"].copy()
    qb[:, :, 64:128] = qb[:, :, 0:64] ^ np.uint16(0x8000)  # negation of the first 64 tokens
    qb[:, :, 192:256] = qb[:, :, 128:192] ^ np.uint16(0x8000)
    q, k, v, do = _dev(qb), _dev(x["k"]), _dev(x["v"]), _dev(x["do"])
    B, H, N, D = w.B, w.H, w.N, w.D
    out = {}
    for qs in (False, True):
        ws = sa.quantize(q, k, v, False, True, q_smooth=qs)
        o, lse = sa.forward(ws, B, H, N, D, True, w.sm_scale, q_smooth=qs)
        grads = sa.backward(q, k, v, o, lse, do, ws, True, False, True, w.sm_scale, q_smooth=qs)
        torch.cuda.synchronize()
        assert sa.get_status(ws) == sa.SAGE_OK
        out[qs] = (sa.ws_tensors(ws, B, H, N, D, q_smooth=qs), o, grads)
    vs, vp = out[True][0], out[False][0]
    assert torch.equal(vs["qmean"], torch.zeros_like(vs["qmean"]))
    assert torch.equal(vs["dsb"][..., :N], torch.zeros_like(vs["dsb"][..., :N]))
    assert torch.equal(vs["qc"], vp["qc"]) and torch.equal(vs["sq"], vp["sq"])
    rel = lambda a, b: float((a.float() - b.float()).norm() / b.float().norm())  # noqa: E731
    assert rel(out[True][1], out[False][1]) < 5e-3
    for a, b in zip(out[True][2], out[False][2]):
        assert rel(a, b) < 5e-3
