"""The backward entry point that allocates nothing (sage_attn_bwd_noalloc).

Some callers cannot allocate device memory: code running inside CUDA graph
capture, hosts whose memory pool owns the whole device, deployments that
allocate nothing after start-up.  For them the backward keeps its scratch in one
fixed array inside the library.  This test calls that entry point through the C
ABI twice in a row and checks each result against the ordinary sage_attn_bwd
(which takes caller-allocated scratch) on the same inputs.  Both run the same
kernels, so dK and dV must be identical bit for bit; dQ is summed over key blocks
by fp32 reductions whose order varies from run to run, so it must agree to a
relative L2 of 1e-5.  The outputs are filled with NaN before the first call and
with a large constant before the second, so neither a skipped write nor scratch
left over from the first call (the second call would double dQ if the shared
array were not cleared) can pass.  It also checks that a shape too large for the
array is refused before any launch.
"""
import numpy as np
import pytest
import torch

import bit_trainable_attention_sagebwd_gb300 as sa
from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DQ_RTOL = 1e-5  # dQ: the same sums in another order (fp32 reductions), then bf16


def _rel(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_noalloc_backward_matches_allocating_backward_twice():
    w = wl.custom(1, 2, 1000, 128, True, qk_norm=True, sm_scale=16.0, seed=31, name="noalloc")
    x = wl.all_inputs(w)
    t = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda() for n, a in x.items()}
    B, H, N, D = w.B, w.H, w.N, w.D
    assert sa.sage_attn_bwd_ws_bytes(B, H, N, D) <= 32 << 20  # fits the library's array
    ws = sa.quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth)
    o, lse = sa.forward(ws, B, H, N, D, w.causal, w.sm_scale)
    ref = sa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], ws, w.causal, w.qk_norm, w.k_smooth, w.sm_scale)
    P = sa._ptr
    s = sa._stream_ptr()
    for fill in (float("nan"), 1.0e4):
        dq, dk, dv = (torch.full_like(t["q"], fill) for _ in range(3))
        rc = sa.sage_attn_bwd_noalloc(P(t["q"]), P(t["k"]), P(t["v"]), P(o), P(lse), P(t["do"]), P(dq), P(dk),
                                      P(dv), P(ws), B, H, N, D, w.causal, w.qk_norm, w.k_smooth, w.sm_scale, s)
        assert rc == sa.SAGE_OK, sa.status_str(rc)
        torch.cuda.synchronize()
        assert sa.get_status(ws) == sa.SAGE_OK
        assert torch.isfinite(dq.float()).all()
        assert torch.equal(dk, ref[1]), "dK differs from sage_attn_bwd"
        assert torch.equal(dv, ref[2]), "dV differs from sage_attn_bwd"
        assert _rel(dq, ref[0]) <= DQ_RTOL


def test_noalloc_backward_refuses_oversize_shapes():
    q = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    ws = sa.alloc_ws(1, 1, 128, 128)
    P = sa._ptr
    B, H, N, D = 1, 64, 8192, 128  # scratch of this shape is far above the array's size
    assert sa.sage_attn_bwd_ws_bytes(B, H, N, D) > 32 << 20
    rc = sa.sage_attn_bwd_noalloc(P(q), P(q), P(q), P(q), P(lse), P(q), P(q), P(q), P(q), P(ws), B, H, N, D,
                                  1, 0, 1, 0.0, sa._stream_ptr())
    assert rc == sa.SAGE_ERR_UNSUPPORTED
