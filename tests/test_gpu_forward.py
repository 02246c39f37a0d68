"""Quantize + forward parity of the CUDA path (through the C ABI) against the CPU oracle.

Codes and scales must match bit for bit; O32 within 2e-3 max abs error; LSE
within 1e-4 (relative to max(1, |LSE|)); bf16 O must be the rounding of O32."""
import pytest

from bit_trainable_attention_sagebwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SMALL = [
    wl.custom(1, 2, 333, 64, True, seed=10, kind="k_offset2", name="n333_d64_causal"),
    wl.custom(1, 2, 700, 128, True, qk_norm=True, sm_scale=16.0, seed=11, name="n700_d128_causal_qknorm"),
    wl.custom(2, 1, 250, 128, False, seed=12, kind="k_outlier20", name="n250_d128_outliers"),
    wl.custom(1, 1, 1, 64, False, seed=13, name="n1_d64"),
    wl.custom(1, 1, 64, 128, True, seed=14, name="n64_d128_causal"),
    wl.custom(1, 1, 512, 64, False, seed=15, kind="k_offset3", name="n512_d64_offset3"),
    wl.custom(1, 2, 640, 128, True, seed=16, kind="student_t3", name="n640_d128_student"),
    wl.custom(1, 1, 129, 128, False, k_smooth=False, seed=17, name="n129_d128_nosmooth"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_quantize_forward_small(w):
    import parity
    x = wl.all_inputs(w)
    g = parity.run_gpu(w, x, backward=False)
    for bh in range(w.bh):
        r = parity.oracle_head(w, x, bh, backward=False)
        parity.check_quantize_head(w, g, bh, r)
        parity.check_forward_head(w, g, bh, r)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_quantize_forward_full_size(name):
    """Full-size workloads in the bench's launch configuration; the oracle computes the
    first, a middle and the last head (every head of the small workload)."""
    import parity
    w = wl.WORKLOADS[name]
    x = wl.all_inputs(w)
    g = parity.run_gpu(w, x, backward=False)
    for bh in parity.full_size_heads(w):
        r = parity.oracle_head(w, x, bh, backward=False)
        parity.check_quantize_head(w, g, bh, r)
        parity.check_forward_head(w, g, bh, r)


# Heavy-tailed logits put many probabilities next to e4m3 rounding midpoints.  With every
# P code equal to the oracle's, O32 differs from the oracle only through fp32 accumulation
# order (about 1e-6 here); one flipped code on a large probability moves a row by ~1e-3.
EXACT_P = [
    wl.custom(1, 2, 640, 128, True, seed=26, kind="student_t3", name="n640_d128_student"),
    wl.custom(1, 4, 2048, 128, True, seed=13, kind="student_t3", name="n2048_d128_student"),
    wl.custom(1, 4, 2048, 64, False, seed=7, kind="k_offset3", name="n2048_d64_offset3"),
]
O_EXACT_ATOL = 1e-4


@pytest.mark.parametrize("w", EXACT_P, ids=[w.name for w in EXACT_P])
def test_forward_p_codes_exact(w):
    import numpy as np
    import parity
    x = wl.all_inputs(w)
    g = parity.run_gpu(w, x, backward=False)
    for bh in range(w.bh):
        r = parity.oracle_head(w, x, bh, backward=False)
        b, h = divmod(bh, w.H)
        err = float(np.abs(g["O32"][b, h].cpu().numpy().astype(np.float64) - r["O32"]).max())
        assert err <= O_EXACT_ATOL, f"O32 error {err} at head {bh}: a P code differs from the oracle's"


def _boundary_inputs():
    """Q, K and V values whose quotients by their scales sit exactly on rounding boundaries:
    INT8 half-integers (k + 1/2) and e4m3 midpoints, normal and subnormal."""
    import numpy as np
    w = wl.custom(1, 1, 256, 128, False, k_smooth=False, seed=31, name="boundaries")
    x = wl.all_inputs(w)
    rng = np.random.default_rng(5)
    # INT8: block max 127/8 gives the scale 1/8 exactly; (k + 1/2)/8 are exact bf16 values
    half = (np.arange(-127, 127) + 0.5) / 8.0
    for name in ("q", "k"):
        t = rng.choice(half, size=(256, 128))
        t[0, 0] = t[64, 0] = t[128, 0] = t[192, 0] = 127.0 / 8.0
        x[name][0, 0] = wl.f32_to_bf16_bits(t.astype(np.float32))
    # e4m3: channel max 28 gives the scale 1/16 exactly; midpoints / 16 are exact bf16 values
    mids = [(1 + (m + 0.5) / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    mids = [v for v in mids if v < 448] + [(k + 0.5) * 2.0 ** -9 for k in range(8)]
    vals = np.array(mids + [-v for v in mids]) / 16.0
    t = rng.choice(vals, size=(256, 128))
    t[0, :] = 28.0
    x["v"][0, 0] = wl.f32_to_bf16_bits(t.astype(np.float32))
    return w, x


def test_codes_on_rounding_boundaries():
    import parity
    w, x = _boundary_inputs()
    g = parity.run_gpu(w, x, backward=False)
    r = parity.oracle_head(w, x, 0, backward=False)
    parity.check_quantize_head(w, g, 0, r)
