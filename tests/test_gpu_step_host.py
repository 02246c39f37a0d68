"""sage_attn_step_host (host tensors, copies overlapped with compute) against the three
device calls on the same inputs: identical O, LSE, dK, dV; dQ within the order of its
fp32 reductions."""
import numpy as np
import pytest

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    (wl.custom(2, 3, 333, 64, True, seed=41, kind="k_offset2", name="b2h3_n333_d64"), 4),   # 3 ranges of 2 heads
    (wl.custom(1, 5, 256, 128, False, qk_norm=True, sm_scale=16.0, seed=42, name="h5_qknorm"), 2),  # 3 + 2 heads
    (wl.custom(1, 2, 129, 128, True, k_smooth=False, seed=43, name="h2_nosmooth"), 0),
]


@pytest.mark.parametrize("w,groups", CASES, ids=[c[0].name for c in CASES])
def test_step_host_matches_device_calls(w, groups):
    import torch
    import bit_trainable_attention_sagebwd_gb300 as sa
    x = wl.all_inputs(w)
    host = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for n, a in x.items()}
    dev = {n: v.cuda() for n, v in host.items()}
    B, H, N, D = w.B, w.H, w.N, w.D
    ws = sa.quantize(dev["q"], dev["k"], dev["v"], w.qk_norm, w.k_smooth)
    o, lse = sa.forward(ws, B, H, N, D, w.causal, w.sm_scale)
    dq, dk, dv = sa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], ws, w.causal, w.qk_norm, w.k_smooth,
                             w.sm_scale)
    out = {"o": torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
           "lse": torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True),
           "dq": torch.empty(dq.shape, dtype=dq.dtype, pin_memory=True),
           "dk": torch.empty(dk.shape, dtype=dk.dtype, pin_memory=True),
           "dv": torch.empty(dv.shape, dtype=dv.dtype, pin_memory=True)}
    scratch = sa.alloc_step_host(B, H, N, D, groups)
    sa.step_host(host["q"], host["k"], host["v"], host["do"], out, scratch, w.causal, w.qk_norm, w.k_smooth,
                 w.sm_scale, groups)
    torch.cuda.synchronize()
    assert sa.get_status(scratch) == sa.SAGE_OK
    assert torch.equal(out["o"], o.cpu())
    assert torch.equal(out["lse"], lse.cpu())
    assert torch.equal(out["dk"], dk.cpu())
    assert torch.equal(out["dv"], dv.cpu())
    ref = dq.float().cpu()
    rel = float((out["dq"].float() - ref).norm() / ref.norm())
    assert rel < 1e-5, rel

