"""Grouped-query attention (sage_attn_gqa_*) against the oracle's run_group: query heads
sharing one key/value head.  Codes and scales bit-exact per head, O32 and LSE per query head
within the forward tolerances, dQ per query head and dK, dV per key/value head (summed over
the group) within the gradient tolerance."""
import numpy as np
import pytest
import torch

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (workload with H query heads, key/value heads Hkv).  The backward splits a key block's query
# heads over `split` CTAs (a divisor of the group, at most 2 x SMs / key tiles); the last two
# cases have enough key tiles (32 and 40 per head) that split stays below the group on 148 or
# 152 SMs, so every CTA loops over two query heads (16 / 8 and 8 / 4).
CASES = [
    (wl.custom(1, 4, 333, 64, True, seed=50, kind="k_offset2", name="h4_kv2_n333_d64_causal"), 2),
    (wl.custom(2, 3, 256, 128, False, qk_norm=True, sm_scale=16.0, seed=51, name="b2_h3_mqa_qknorm"), 1),
    (wl.custom(1, 8, 640, 128, True, seed=52, kind="student_t3", name="h8_kv2_n640_d128_causal"), 2),
    (wl.custom(1, 16, 4000, 64, True, seed=53, kind="k_offset2", name="h16_mqa_n4000_d64_causal"), 1),
    (wl.custom(1, 8, 5000, 128, True, seed=54, name="h8_mqa_n5000_d128_causal"), 1),
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("w,hkv", CASES, ids=[c[0].name for c in CASES])
def test_gqa_matches_oracle_group(w, hkv):
    import bit_trainable_attention_sagebwd_gb300 as sa
    import parity
    from oracle import oracle as orc
    x = wl.all_inputs(w)
    B, H, N, D = w.B, w.H, w.N, w.D
    G = H // hkv
    kx, vx = x["k"][:, :hkv], x["v"][:, :hkv]  # the key/value heads: [B, Hkv, N, D]
    q, k, v, do = _dev(x["q"]), _dev(kx), _dev(vx), _dev(x["do"])
    ws = sa.quantize(q, k, v, w.qk_norm, w.k_smooth)
    o, lse, o32 = sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o32=True, hkv=hkv)
    dq, dk, dv = sa.backward(q, k, v, o, lse, do, ws, w.causal, w.qk_norm, w.k_smooth, w.sm_scale)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == sa.SAGE_OK
    assert dk.shape == (B, hkv, N, D) and dv.shape == (B, hkv, N, D)
    views = sa.ws_tensors(ws, B, H, N, D, hkv=hkv)
    f64 = lambda a: wl.bf16_bits_to_f32(a).astype(np.float64)
    for b in range(B):
        for kh in range(hkv):
            heads = [kh * G + g for g in range(G)]
            r = orc.run_group([f64(x["q"][b, h]) for h in heads], f64(kx[b, kh]), f64(vx[b, kh]),
                              [f64(x["do"][b, h]) for h in heads], w.causal, w.sm_scale, w.qk_norm, w.k_smooth)
            # K and V codes and scales of the shared head
            r0 = r["heads"][0]
            kc = views["kc"][b, kh].float().cpu().numpy().astype(np.float64)
            assert np.array_equal(kc[:N], r0["kx"])
            assert np.array_equal(views["sv"][b, kh].cpu().numpy().astype(np.float64), r0["sv"])
            assert np.array_equal(views["kmean"][b, kh].cpu().numpy().astype(np.float64), r0["kmean"])
            v8 = parity.e4m3_decode(views["v8t"][b, kh])
            assert np.array_equal(v8[:, :N].T, r0["vx"])
            for g, h in enumerate(heads):
                rh = r["heads"][g]
                qc = views["qc"][b, h].float().cpu().numpy().astype(np.float64)
                assert np.array_equal(qc[:N], rh["qx"]), f"q codes differ at head {h}"
                e = float(np.abs(o32[b, h].cpu().numpy().astype(np.float64) - rh["O32"].astype(np.float64)).max())
                assert e <= parity.O_ATOL, f"O32 error {e} at head {h}"
                lerr = float(np.abs(lse[b, h].cpu().numpy().astype(np.float64) - rh["LSE64"]).max())
                assert lerr <= parity.LSE_ATOL * max(1.0, float(np.abs(rh["LSE64"]).max()))
                eq = parity.rel_l2(dq[b, h].float().cpu().numpy().astype(np.float64), rh["dQbf"])
                assert eq <= parity.GRAD_RTOL, f"dQ relative L2 {eq} at head {h}"
            for name, got in (("dK", dk), ("dV", dv)):
                e = parity.rel_l2(got[b, kh].float().cpu().numpy().astype(np.float64), r[name + "bf"])
                assert e <= parity.GRAD_RTOL, f"{name} relative L2 {e} at key/value head {kh}"
