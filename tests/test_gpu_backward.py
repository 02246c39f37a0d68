"""Backward parity of the CUDA path (through the C ABI) against the CPU oracle:
relative L2 error of dQ, dK, dV at most 1e-2 per head (the stated tolerance),
plus the forward checks on the same run."""
import pytest

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SMALL = [
    wl.custom(1, 2, 333, 64, True, seed=20, kind="k_offset2", name="n333_d64_causal"),
    wl.custom(1, 2, 700, 128, True, qk_norm=True, sm_scale=16.0, seed=21, name="n700_d128_causal_qknorm"),
    wl.custom(2, 1, 250, 128, False, seed=22, kind="k_outlier20", name="n250_d128_outliers"),
    wl.custom(1, 1, 1, 64, False, seed=23, name="n1_d64"),
    wl.custom(1, 1, 64, 128, True, seed=24, name="n64_d128_causal"),
    wl.custom(1, 1, 512, 64, False, qk_norm=True, sm_scale=8.0, seed=25, kind="k_offset3", name="n512_d64_qknorm"),
    wl.custom(1, 2, 640, 128, True, seed=26, kind="student_t3", name="n640_d128_student"),
    wl.custom(1, 1, 129, 128, False, k_smooth=False, seed=27, name="n129_d128_nosmooth"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_backward_small(w):
    import parity
    x = wl.all_inputs(w)
    g = parity.run_gpu(w, x, backward=True)
    for bh in range(w.bh):
        r = parity.oracle_head(w, x, bh, backward=True)
        parity.check_forward_head(w, g, bh, r)
        parity.check_backward_head(w, g, bh, r)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_backward_full_size(name):
    """Full-size workloads in the bench's launch configuration; the oracle computes the
    first, a middle and the last head (every head of the small workload)."""
    import parity
    w = wl.WORKLOADS[name]
    x = wl.all_inputs(w)
    g = parity.run_gpu(w, x, backward=True)
    for bh in parity.full_size_heads(w):
        r = parity.oracle_head(w, x, bh, backward=True)
        parity.check_backward_head(w, g, bh, r)


AUX = [
    wl.custom(1, 2, 640, 128, True, seed=26, kind="student_t3", name="n640_d128_student"),
    wl.custom(1, 2, 700, 128, True, qk_norm=True, sm_scale=16.0, seed=21, name="n700_d128_causal_qknorm"),
    wl.custom(1, 1, 512, 64, False, seed=15, kind="k_offset3", name="n512_d64_offset3"),
]


@pytest.mark.parametrize("w", AUX, ids=[w.name for w in AUX])
def test_backward_fp32_auxiliary_output(w):
    """sage_attn_bwd_o32: D_i from the forward's fp32 output.  Parity with the oracle fed the
    same fp32 O; and, against the exact (unquantized, fp64) gradients, its error is reported
    next to that of the bf16-O backward."""
    import numpy as np
    import parity
    from oracle import oracle as orc
    x = wl.all_inputs(w)
    g32 = parity.run_gpu(w, x, backward=True, o32_aux=True)
    gbf = parity.run_gpu(w, x, backward=True)
    for bh in range(w.bh):
        r = parity.oracle_head(w, x, bh, backward=True, o_aux="fp32")
        parity.check_backward_head(w, g32, bh, r)
        exact = parity.oracle_head(w, x, bh, backward=True, qmask=0)
        b, h = divmod(bh, w.H)
        for name, key in (("dQ", "dQ64"), ("dK", "dK64"), ("dV", "dV64")):
            e32 = parity.rel_l2(g32[name][b, h].float().cpu().numpy().astype(np.float64), exact[key])
            ebf = parity.rel_l2(gbf[name][b, h].float().cpu().numpy().astype(np.float64), exact[key])
            print(f"{w.name} head {bh} {name}: rel L2 vs exact, D from fp32 O {e32:.3e}, from bf16 O {ebf:.3e}")
            # the low-bit scheme's own error dominates; the auxiliary output must not add to it
            assert e32 <= ebf * 1.1 + 1e-4
