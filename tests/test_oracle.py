"""Pins of the CPU oracle to things other than itself (no GPU needed).

- e4m3 rounding: exhaustive over every positive fp32 in [2^-11, 448] against
  torch's float8_e4m3fn cast (a library routine), plus signs, underflow and
  saturation.
- bf16 and fp16 rounding (every bf16 output and reference gradient, the D_i of
  the backward, the fp16 path of ThriftAttention): every mantissa of every fp32
  binade where the rounding rule changes, against torch's bfloat16 / float16
  casts (library routines), plus a random sample over all bit patterns.
- exact mode (every quantizer off): forward against torch scaled-dot-product
  attention in float64, backward against torch autograd, and against central
  finite differences of the oracle's own forward.
- invariants: softmax invariance to a per-channel shift of K (K-smoothing), the
  FlashAttention identity rowsum(P*dP) = rowsum(dO*O) seen through
  sum_j dK_j = 0, unit-norm q' and k' under QK-norm.
- the full low-bit scheme on inputs its quantizers must represent exactly:
  it must then equal exact attention.
- one quantizer at a time: exact relations (QK, V, dO quantizers) or rigorous
  error bounds (P and dS quantizers) against library attention.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc

torch.set_default_dtype(torch.float64)


def ref_attention(q, k, v, causal, sm_scale, qk_norm=False, k_smooth=False):
    """Textbook attention in float64 with torch (library SDPA + logsumexp)."""
    qq = F.normalize(q, dim=-1) if qk_norm else q
    kk = F.normalize(k, dim=-1) if qk_norm else k
    if k_smooth:
        kk = kk - kk.mean(0, keepdim=True)
    O = F.scaled_dot_product_attention(qq[None, None], kk[None, None], v[None, None],
                                       is_causal=causal, scale=sm_scale)[0, 0]
    s = sm_scale * (qq @ kk.T)
    if causal:
        n = s.shape[0]
        s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
    return O, torch.logsumexp(s, -1), s


def ref_grads(q, k, v, do, causal, sm_scale, qk_norm=False, k_smooth=False):
    q = torch.tensor(q, requires_grad=True)
    k = torch.tensor(k, requires_grad=True)
    v = torch.tensor(v, requires_grad=True)
    O, lse, _ = ref_attention(q, k, v, causal, sm_scale, qk_norm, k_smooth)
    (O * torch.tensor(do)).sum().backward()
    return O.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


# ---------------------------------------------------------------- e4m3 rounding

def test_e4m3_exhaustive_against_torch_cast():
    lo = int(np.array(2.0 ** -11, dtype=np.float32).view(np.uint32))
    hi = int(np.array(448.0, dtype=np.float32).view(np.uint32))
    chunk = 1 << 24
    for start in range(lo, hi + 1, chunk):
        bits = np.arange(start, min(start + chunk, hi + 1), dtype=np.uint32)
        x = bits.view(np.float32)
        y = orc.e4m3(x)
        t = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy()
        assert np.array_equal(y, t), f"mismatch in chunk starting at {start:#x}"
        assert np.array_equal(orc.e4m3(-x), -t)


def _binade(e: int, sign: int = 0) -> np.ndarray:
    """Every fp32 with biased exponent e (all 2^23 mantissas) and the given sign."""
    bits = (np.uint32(sign) << np.uint32(31)) | (np.uint32(e) << np.uint32(23)) | \
        np.arange(1 << 23, dtype=np.uint32)
    return bits.view(np.float32)


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    return bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


def test_bf16_rounding_against_torch_cast():
    """The oracle's bf16 rounding (nearest even; inf and NaN kept) equals torch's fp32 ->
    bfloat16 cast on every mantissa of the binades where the rule changes (subnormals, the
    smallest normals, around 1, the two largest finite binades, where rounding reaches
    infinity, and inf/NaN), both signs, and on 2^24 random bit patterns."""
    for e in (0, 1, 2, 126, 127, 128, 253, 254, 255):
        for sign in (0, 1):
            x = _binade(e, sign)
            y = orc.to_bf16(x.astype(np.float64))
            t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
            assert _same(y, t), f"bf16 rounding differs in binade {e}, sign {sign}"
    x = np.random.default_rng(1).integers(0, 1 << 32, size=1 << 24, dtype=np.uint64).astype(np.uint32)
    x = x.view(np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
    assert _same(orc.to_bf16(x.astype(np.float64)), t)


def test_fp16_rounding_against_torch_cast():
    """The oracle's fp16 rounding (nearest even, subnormal below 2^-14) equals torch's
    fp32 -> float16 cast on every positive fp32 from 2^-26 (below it both give 0) up to the
    largest finite binade [2^15, 2^16) except past 65520 (where IEEE rounds to infinity and
    the oracle saturates at 65504, a range its inputs never reach), on negative values, and
    on 2^24 random bit patterns with |x| < 65520."""
    for e in range(101, 143):
        x = _binade(e)
        if e == 142:
            x = x[x < 65520.0]
        y = orc.fp16(x.astype(np.float64))
        t = torch.from_numpy(x).to(torch.float16).to(torch.float32).numpy().astype(np.float64)
        assert np.array_equal(y, t), f"fp16 rounding differs in binade {e}"
        assert np.array_equal(orc.fp16(-x.astype(np.float64)), -t)
    tiny = _binade(100)
    assert np.all(orc.fp16(tiny.astype(np.float64)) == 0.0)
    x = np.random.default_rng(2).integers(0, 1 << 32, size=1 << 24, dtype=np.uint64).astype(np.uint32)
    x = x.view(np.float32)
    x = x[np.abs(x) < 65520.0]
    t = torch.from_numpy(x).to(torch.float16).to(torch.float32).numpy().astype(np.float64)
    assert np.array_equal(orc.fp16(x.astype(np.float64)), t)
    assert np.all(orc.fp16(np.array([65520.0, 1e6, 3e38])) == 65504.0)


def test_e4m3_underflow_and_saturation():
    rng = np.random.default_rng(0)
    tiny = (rng.random(10000) * 2.0 ** -11).astype(np.float32)
    assert np.all(orc.e4m3(tiny) == 0.0)
    big = np.concatenate([np.float32([448.0, 460.0, 463.99, 464.0, 1e6, np.inf]),
                          (448 + rng.random(1000) * 1e5).astype(np.float32)])
    assert np.all(orc.e4m3(big) == 448.0)
    assert np.all(orc.e4m3(-big) == -448.0)
    # the e4m3 value set: 2^-9 * {1..7} subnormals, (1 + m/8) 2^e normals up to 448
    grid = np.concatenate([np.linspace(0, 0.1, 100001), np.linspace(0, 448, 200001)]).astype(np.float32)
    vals = np.unique(orc.e4m3(grid))
    assert len(vals) == 127  # 0, 7 subnormals, 15 binades x 8 - 1 (NaN code)


# ---------------------------------------------------------- exact-mode pins

CASES = [  # N, D, causal, qk_norm, k_smooth
    (1, 16, False, False, True),
    (5, 16, True, True, True),
    (64, 64, True, False, False),
    (130, 32, False, True, True),
    (300, 32, True, False, True),
]


def _rand(rng, N, D, offset=0.0):
    return rng.standard_normal((N, D)) + offset


@pytest.mark.parametrize("N,D,causal,qk_norm,k_smooth", CASES)
def test_exact_mode_matches_library_attention(N, D, causal, qk_norm, k_smooth):
    rng = np.random.default_rng(N * 7 + D)
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    k = k + rng.normal(0, 2.0, size=(1, D))
    sm = 1.0 / math.sqrt(D) if not qk_norm else 4.0
    r = orc.run_head(q, k, v, do, causal, sm, qk_norm, k_smooth, qmask=0)
    O, lse, dq, dk, dv = ref_grads(q, k, v, do, causal, sm, qk_norm, k_smooth)
    np.testing.assert_allclose(r["O64"], O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["LSE64"], lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dV64"], dv, rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dQ64"], dq, rtol=0, atol=1e-11)
    # with K-smoothing the exact gradient carries the (I - 11^T/N) projection;
    # the oracle applies none, which is exact because dS rows sum to zero
    np.testing.assert_allclose(r["dK64"], dk, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal,qk_norm", [(False, False), (True, False), (True, True), (False, True)])
def test_exact_mode_finite_differences(causal, qk_norm):
    rng = np.random.default_rng(5)
    N, D = 48, 16
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    sm = 0.3 if not qk_norm else 3.0

    def loss(q_, k_, v_):
        r = orc.run_head(q_, k_, v_, do, causal, sm, qk_norm, True, qmask=0, backward_pass=False)
        return float((r["O64"] * do).sum())

    g = orc.run_head(q, k, v, do, causal, sm, qk_norm, True, qmask=0)
    h = 1e-6
    for name, grad in (("q", g["dQ64"]), ("k", g["dK64"]), ("v", g["dV64"])):
        for _ in range(10):
            i, d = rng.integers(N), rng.integers(D)
            xs = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            xs[name][i, d] += h
            fp = loss(xs["q"], xs["k"], xs["v"])
            xs[name][i, d] -= 2 * h
            fm = loss(xs["q"], xs["k"], xs["v"])
            fd = (fp - fm) / (2 * h)
            assert abs(fd - grad[i, d]) <= 1e-7 + 1e-6 * abs(fd), (name, i, d, fd, grad[i, d])


def test_exact_mode_invariants():
    rng = np.random.default_rng(11)
    N, D = 200, 32
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    shift = rng.normal(0, 5.0, size=(1, D))
    for causal in (False, True):
        for smooth in (False, True):
            a = orc.run_head(q, k, v, do, causal, 0.2, False, smooth, qmask=0)
            b = orc.run_head(q, k + shift, v, do, causal, 0.2, False, smooth, qmask=0)
            np.testing.assert_allclose(a["O64"], b["O64"], atol=1e-12, rtol=0)
        # sum_j dS_ij = 0 (rowsum(P*dP) = rowsum(dO*O)) makes every column of dK sum to 0
        r = orc.run_head(q, k, v, do, causal, 0.2, False, True, qmask=0)
        assert np.abs(r["dK64"].sum(0)).max() < 1e-11


def test_qk_norm_unit_vectors_in_scheme():
    rng = np.random.default_rng(3)
    q, k, v = (_rand(rng, 256, 128) for _ in range(3))
    qz = orc.quantize(q, k, v, True, False, orc.QM_ALL)
    for x in (qz["qn"], qz["kn"]):
        assert np.abs(np.linalg.norm(x, axis=1) - 1.0).max() < 1e-6


# ---------------------------------------------- the scheme on lossless inputs

def _lossless_inputs(N, D, seed):
    """Inputs that every quantizer of the scheme represents exactly.

    q, k: sparse +-1 entries (3 per token) so logits are small integers; one
    channel per tensor holds a 127 at the first token of each block (scale 1),
    in a channel the other tensor leaves at zero.  k has zero column means
    (second half = -first half) so K-smoothing is the identity.  v, do: values
    on the e4m3 grid with one 448 per channel (scale 1).
    """
    rng = np.random.default_rng(seed)
    q = np.zeros((N, D))
    k = np.zeros((N // 2, D))
    for x in (q, k):
        for t in range(x.shape[0]):
            dims = rng.choice(np.arange(2, D), 3, replace=False)
            x[t, dims] = rng.choice([-1.0, 1.0], 3)
    q[::128, 0] = 127.0
    k[::64, 1] = 127.0
    k = np.concatenate([k, -k])
    grid = np.array([0.25, 0.5, 1.0, 1.5, 2.0, 3.0])
    v = rng.choice(grid, (N, D)) * rng.choice([-1.0, 1.0], (N, D))
    do = rng.choice(grid, (N, D)) * rng.choice([-1.0, 1.0], (N, D))
    v[rng.integers(N, size=D), np.arange(D)] = 448.0
    do[rng.integers(N, size=D), np.arange(D)] = -448.0
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_scheme_is_exact_on_representable_inputs(causal):
    N, D = 256, 64
    q, k, v, do = _lossless_inputs(N, D, 1)
    sm = math.log(2.0)  # alpha = RN32(ln2 * log2 e) = 1: logits stay integers
    r = orc.run_head(q, k, v, do, causal, sm, False, True, qmask=orc.QM_ALL, backward_pass=False)
    assert np.all(r["sq"] == 1.0) and np.all(r["sk"] == 1.0) and np.all(r["sv"] == 1.0)
    assert np.array_equal(r["qx"], q) and np.array_equal(r["kx"], k) and np.array_equal(r["vx"], v)
    O, lse, _ = ref_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v), causal, sm)
    np.testing.assert_allclose(r["O64"], O.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(r["LSE64"], lse.numpy(), rtol=0, atol=1e-12)


def test_uniform_attention_closed_form():
    rng = np.random.default_rng(2)
    N, D = 256, 64
    q = np.zeros((N, D))
    k, v, do = (_rand(rng, N, D) for _ in range(3))
    for causal in (False, True):
        r = orc.run_head(q, k, v, do, causal, 0.125, False, True, qmask=orc.QM_ALL)
        vhat = r["vx"] * r["sv"][None, :]
        if causal:
            expect = np.cumsum(vhat, 0) / np.arange(1, N + 1)[:, None]
            lse = np.log(np.arange(1, N + 1))
        else:
            expect = np.broadcast_to(vhat.mean(0), (N, D))
            lse = np.full(N, math.log(N))
        np.testing.assert_allclose(r["O64"], expect, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["LSE64"], lse, atol=1e-6)  # LSE enters fp32
    # non-causal uniform P = 1/256 is an e4m3 value: every dV row is the mean dO
    r = orc.run_head(q, k, v, do, False, 0.125, False, True, qmask=orc.QM_ALL)
    assert np.abs(r["dV64"] - r["dV64"][0]).max() == 0.0
    np.testing.assert_allclose(r["dV64"][0], do.mean(0), atol=2.0 ** -4 * np.abs(do).mean(0).max() * 2)


# ------------------------------------------------------ one quantizer at a time

def _dequant(r, N):
    qh = r["qx"] * np.repeat(r["sq"], 128)[:N, None]
    kh = r["kx"] * np.repeat(r["sk"], 64)[:N, None]
    return qh, kh


@pytest.mark.parametrize("causal", [False, True])
def test_qk_quantizer_equals_attention_on_dequantized_inputs(causal):
    rng = np.random.default_rng(21)
    N, D = 200, 32  # ragged: Q blocks of 128 + 72 tokens, K blocks 64,64,64,8
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    k = k + rng.normal(0, 2.0, size=(1, D))
    sm = 0.2
    r = orc.run_head(q, k, v, do, causal, sm, False, True, qmask=orc.QM_QK)
    qh, kh = _dequant(r, N)
    # the codes: integers in [-127, 127], error at most half a step, 127 reached per block
    for x, codes, sc, blk in ((q, r["qx"], r["sq"], 128), (k - k.mean(0), r["kx"], r["sk"], 64)):
        assert np.array_equal(codes, np.round(codes)) and np.abs(codes).max() <= 127
        steps = np.repeat(sc, blk)[:N, None]
        assert np.all(np.abs(x - codes * steps) <= steps / 2 * (1 + 1e-12))
        for b in range(len(sc)):
            assert np.abs(codes[b * blk:(b + 1) * blk]).max() == 127
    O, lse, dq, dk, dv = ref_grads(qh, kh, v, do, causal, sm)
    np.testing.assert_allclose(r["O64"], O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["LSE64"], lse, atol=1e-12, rtol=0)
    np.testing.assert_allclose(r["dV64"], dv, atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dQ64"], dq, atol=1e-11, rtol=0)
    np.testing.assert_allclose(r["dK64"], dk, atol=1e-11, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_v_quantizer_equals_attention_on_dequantized_v(causal):
    rng = np.random.default_rng(22)
    N, D = 200, 32
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    r = orc.run_head(q, k, v, do, causal, 0.2, False, True, qmask=orc.QM_V, backward_pass=False)
    vh = r["vx"] * r["sv"][None, :]
    assert np.all(np.abs(r["vx"]).max(0) == 448.0)  # per-channel scale reaches the top code
    O, _, _ = ref_attention(torch.tensor(q), torch.tensor(k), torch.tensor(vh), causal, 0.2)
    np.testing.assert_allclose(r["O64"], O.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_do_quantizer_is_identity_on_representable_do(causal):
    """Per-channel e4m3 of dO loses nothing when each channel is on the grid
    with a 448 in it; a per-token scale (the wrong axis) would not."""
    N, D = 256, 64
    _, _, _, do = _lossless_inputs(N, D, 4)
    rng = np.random.default_rng(4)
    q, k, v = (_rand(rng, N, D) for _ in range(3))
    a = orc.run_head(q, k, v, do, causal, 0.2, False, True, qmask=orc.QM_DO)
    b = orc.run_head(q, k, v, do, causal, 0.2, False, True, qmask=0)
    for n in ("dQ64", "dK64", "dV64"):
        np.testing.assert_allclose(a[n], b[n], atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_p_quantizer_error_bound(causal):
    """e4m3 P: |p^ - p| <= 2^-4 p + 2^-10/448 for every weight, so
    |O_d - O*_d| <= (2^-4 sum_j p_j |v_jd| + 2^-10/448 sum_j |v_jd|) / l."""
    rng = np.random.default_rng(23)
    N, D = 300, 32
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    sm = 0.5
    r = orc.run_head(q, k, v, do, causal, sm, False, False, qmask=orc.QM_P, backward_pass=False)
    O, lse, s = ref_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v), causal, sm)
    m = s.max(-1, keepdim=True).values
    p = torch.exp(s - m).numpy()  # unnormalised, max 1 per row
    l = p.sum(-1, keepdims=True)
    valid = np.isfinite(s.numpy())
    bound = (2.0 ** -4 * p @ np.abs(v) + 2.0 ** -10 / 448 * (valid @ np.abs(v))) / l
    err = np.abs(r["O64"] - O.numpy())
    assert np.all(err <= bound * (1 + 1e-9) + 1e-14)
    assert err.max() > 0  # the quantizer did act


@pytest.mark.parametrize("causal", [False, True])
def test_ds_quantizer_error_bound(causal):
    """INT8 dS per (128 query x 64 key) tile: |dS^ - dS| <= s_tile/2 <= max|dS|/254,
    so |dQ_id - dQ*_id| <= sm (max|dS|/254) sum_j |k_jd| (and likewise dK)."""
    rng = np.random.default_rng(24)
    N, D = 200, 32
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    sm = 0.3
    a = orc.run_head(q, k, v, do, causal, sm, False, False, qmask=orc.QM_DS)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    O, _, s = ref_attention(qt, kt, vt, causal, sm)
    (O * torch.tensor(do)).sum().backward()
    P = torch.softmax(s, -1).detach().numpy()
    dP = do @ v.T
    dS = P * (dP - (do * O.detach().numpy()).sum(-1, keepdims=True))
    step = np.abs(dS).max() / 254
    bq = sm * step * (np.ones((N, N)) @ np.abs(k))
    bk = sm * step * (np.ones((N, N)) @ np.abs(q))
    eq = np.abs(a["dQ64"] - qt.grad.numpy())
    ek = np.abs(a["dK64"] - kt.grad.numpy())
    assert np.all(eq <= bq + 1e-12) and np.all(ek <= bk + 1e-12)
    assert eq.max() > 0
    np.testing.assert_allclose(a["dV64"], vt.grad.numpy(), atol=1e-12, rtol=0)


def test_fp32_rounding_alone_is_small():
    rng = np.random.default_rng(25)
    N, D = 256, 64
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    b = orc.run_head(q, k, v, do, True, 0.125, True, True, qmask=0)
    qz = orc.quantize(q, k, v, True, True, orc.QM_F32)
    fa = orc.forward(qz, True, 0.125, orc.QM_F32)
    np.testing.assert_allclose(fa["O64"], b["O64"], rtol=0, atol=1e-5 * np.abs(b["O64"]).max())
    # the scheme feeds its backward the bf16 O; here it gets the exact O and LSE so
    # that only the fp32 roundings inside the backward differ
    a = orc.backward(qz, v, do, b["O64"], b["LSE64"], True, 0.125, True, orc.QM_F32)
    for n in ("dQ64", "dK64", "dV64"):
        np.testing.assert_allclose(a[n], b[n], rtol=0, atol=1e-5 * np.abs(b[n]).max())


def test_full_scheme_error_is_modest():
    """All quantizers on against exact attention: the scheme's own error (reported
    by the bench; asserted loosely here as a sanity bound)."""
    rng = np.random.default_rng(26)
    N, D = 384, 64
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    k = k + rng.normal(0, 2.0, size=(1, D))
    a = orc.run_head(q, k, v, do, True, 0.125, False, True, qmask=orc.QM_ALL)
    b = orc.run_head(q, k, v, do, True, 0.125, False, True, qmask=0)

    def rel(x, y):
        return np.linalg.norm(x - y) / np.linalg.norm(y)

    assert rel(a["O64"], b["O64"]) < 0.05
    for n in ("dQ64", "dK64", "dV64"):
        assert rel(a[n], b[n]) < 0.1, n


def test_fp32_auxiliary_output_feeds_the_row_terms():
    """o_aux="fp32" ("Attn-QAT" summary, Methodology, principle 2): the backward's row terms
    are rowsum(dO * O) with the forward's fp32 O instead of its bf16 rounding; dV does not
    depend on them, dQ and dK do."""
    rng = np.random.default_rng(27)
    N, D = 192, 64
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    a = orc.run_head(q, k, v, do, True, 0.125, False, True)
    b = orc.run_head(q, k, v, do, True, 0.125, False, True, o_aux="fp32")
    np.testing.assert_allclose(a["Dvec"], (do * a["Obf"]).sum(1), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["Dvec"], (do * b["O32"].astype(np.float64)).sum(1), rtol=1e-12, atol=1e-14)
    assert not np.allclose(a["Dvec"], b["Dvec"], rtol=1e-6, atol=0)
    np.testing.assert_array_equal(a["dV64"], b["dV64"])
    assert not np.array_equal(a["dQ64"], b["dQ64"]) and not np.array_equal(a["dK64"], b["dK64"])


# ---------------------------------------------------------------- grouped-query attention

@pytest.mark.parametrize("causal,qk_norm", [(True, False), (False, True)])
def test_group_exact_mode_matches_library_attention(causal, qk_norm):
    """Exact arithmetic: G query heads on one key/value head equal torch attention with the
    key/value head repeated, and dK, dV are the sums of the per-head gradients."""
    rng = np.random.default_rng(40)
    G, N, D = 3, 160, 64
    qs = [_rand(rng, N, D) for _ in range(G)]
    dos = [_rand(rng, N, D) for _ in range(G)]
    k, v = _rand(rng, N, D), _rand(rng, N, D)
    r = orc.run_group(qs, k, v, dos, causal, 0.2, qk_norm, True, qmask=0)
    dK, dV = np.zeros((N, D)), np.zeros((N, D))
    for g in range(G):
        O, lse, dq, dk, dv = ref_grads(qs[g], k, v, dos[g], causal, 0.2, qk_norm, True)
        np.testing.assert_allclose(r["heads"][g]["O64"], O, rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["heads"][g]["dQ64"], dq, rtol=0, atol=1e-10)
        dK += dk
        dV += dv
    np.testing.assert_allclose(r["dK64"], dK, rtol=0, atol=1e-10)
    np.testing.assert_allclose(r["dV64"], dV, rtol=0, atol=1e-10)


def test_group_do_scale_spans_the_group():
    """In the low-bit scheme the group's dO channel scale is max |dO| over all of its heads'
    tokens / 448 (fp32): with one head the group is that head, and a head with larger dO
    sets the scale of the others."""
    rng = np.random.default_rng(41)
    N, D = 128, 64
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    one = orc.run_group([q], k, v, [do], True, 0.125)
    single = orc.run_head(q, k, v, do, True, 0.125)
    for n in ("dQ64", "dK64", "dV64"):
        np.testing.assert_array_equal(one["heads"][0][n], single[n])
    np.testing.assert_array_equal(one["dV64"], single["dV64"])
    big = 8.0 * do
    two = orc.run_group([q, q], k, v, [do, big], True, 0.125)
    np.testing.assert_array_equal(two["sdo"], (np.abs(big).max(0) / 448.0).astype(np.float32).astype(np.float64))
    # the first head's dO is coded with the larger scale: its dV differs from the lone head's
    assert not np.array_equal(two["heads"][0]["dV64"], single["dV64"])


# ---------------------------------------------------------------- Q-smoothing

def _bf16(x):
    return torch.tensor(x).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("causal,qk_norm", [(False, False), (True, False), (True, True)])
def test_q_smoothing_exact_mode_matches_library_attention(causal, qk_norm):
    """Exact arithmetic: (q' - qmean_I) k'' + qmean_I k'' is q' k'', so the Q-smoothed path
    equals torch attention, and its dK (the per-tile qmean term included) equals autograd's.
    N = 300 leaves a ragged last query block of 44 tokens, whose mean is over those alone."""
    rng = np.random.default_rng(50)
    N, D = 300, 64
    q, k, v, do = (_rand(rng, N, D) for _ in range(4))
    q = q + rng.normal(0, 3.0, size=(1, D))  # a common query component for the mean to carry
    sm = 0.125 if not qk_norm else 4.0
    r = orc.run_head(q, k, v, do, causal, sm, qk_norm, True, qmask=0, q_smooth=True)
    O, lse, dq, dk, dv = ref_grads(q, k, v, do, causal, sm, qk_norm, True)
    np.testing.assert_allclose(r["O64"], O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["LSE64"], lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dQ64"], dq, rtol=0, atol=1e-10)
    np.testing.assert_allclose(r["dK64"], dk, rtol=0, atol=1e-10)
    np.testing.assert_allclose(r["dV64"], dv, rtol=0, atol=1e-10)


def test_q_smoothing_quantizer_parts():
    """The block means are fp32 roundings of the exact means over each block's valid
    tokens; the INT8 codes reconstruct q' - qmean to half a step; dsb is qmean . k'' with
    k'' the smoothed keys K's quantizer takes (fp32 rounding of the fp64 dot product)."""
    rng = np.random.default_rng(51)
    N, D = 200, 64
    q = _bf16(_rand(rng, N, D, offset=2.0))
    k, v = _bf16(_rand(rng, N, D)), _bf16(_rand(rng, N, D))
    z = orc.quantize(q, k, v, False, True, q_smooth=True)
    assert z["qmean"].shape == (2, D) and z["dsb"].shape == (2, N)
    for I, (t0, t1) in enumerate([(0, 128), (128, 200)]):
        exact = np.array([math.fsum(q[t0:t1, d]) / (t1 - t0) for d in range(D)])
        np.testing.assert_array_equal(z["qmean"][I], exact.astype(np.float32).astype(np.float64))
        qs = (q[t0:t1] - z["qmean"][I]).astype(np.float32).astype(np.float64)
        s = z["sq"][I]
        assert s == np.float32(np.abs(qs).max() / 127.0)
        assert np.abs(z["qx"][t0:t1]).max() == 127
        assert np.all(np.abs(z["qx"][t0:t1] * s - qs) <= 0.5 * s * (1 + 1e-6))
    ks = (k - z["kmean"]).astype(np.float32).astype(np.float64)
    want = (z["qmean"] @ ks.T).astype(np.float32).astype(np.float64)
    np.testing.assert_allclose(z["dsb"], want, rtol=2 ** -22, atol=1e-12)
    # no Q-smoothing: the same K, V codes, and the unsmoothed Q codes
    z0 = orc.quantize(q, k, v, False, True)
    for n in ("kx", "sk", "vx", "sv", "kmean"):
        np.testing.assert_array_equal(z[n], z0[n])
    assert not np.array_equal(z["qx"], z0["qx"])


def test_q_smoothing_zero_mean_blocks_keep_the_codes():
    """Query blocks whose channel means are exactly zero (each token paired with its
    negation) keep their unsmoothed codes and scales, and dsb is zero; the outputs then differ
    from the plain scheme only by where the logit rounds (RN(acc RN(sq sk)) alpha against
    acc RN(RN(sq sk) alpha))."""
    rng = np.random.default_rng(52)
    N, D = 256, 64
    half = _bf16(_rand(rng, 64, D))
    q = np.concatenate([half, -half, half[::-1], -half[::-1]])
    k, v, do = (_bf16(_rand(rng, N, D)) for _ in range(3))
    zq = orc.quantize(q, k, v, False, True, q_smooth=True)
    z0 = orc.quantize(q, k, v, False, True)
    assert np.all(zq["qmean"] == 0) and np.all(zq["dsb"] == 0)
    np.testing.assert_array_equal(zq["qx"], z0["qx"])
    np.testing.assert_array_equal(zq["sq"], z0["sq"])
    a = orc.run_head(q, k, v, do, True, 0.125, q_smooth=True)
    b = orc.run_head(q, k, v, do, True, 0.125)
    for n in ("O64", "dQ64", "dK64", "dV64"):
        rel = np.linalg.norm(a[n] - b[n]) / np.linalg.norm(b[n])
        assert rel < 2e-3, (n, rel)


def test_q_smoothing_constant_blocks_reduce_to_high_precision_logits():
    """Every token of a query block equal: q' - qmean = 0, so the block's scale and codes are
    0 and its logits are dsb alone, a high-precision product.  With only the Q/K quantizer on,
    the forward then equals exact attention to fp32 rounding, however coarse K's codes."""
    rng = np.random.default_rng(53)
    N, D = 256, 64
    q = np.repeat(_bf16(_rand(rng, 2, D, offset=1.0)), 128, axis=0)
    k, v, do = (_bf16(_rand(rng, N, D)) for _ in range(3))
    qm = orc.QM_QK | orc.QM_F32
    r = orc.run_head(q, k, v, do, False, 0.125, qmask=qm, backward_pass=False, q_smooth=True)
    assert np.all(r["sq"] == 0) and np.all(r["qx"] == 0)
    O, lse, *_ = ref_grads(q, k, v, do, False, 0.125, False, True)
    np.testing.assert_allclose(r["O64"], O, rtol=0, atol=1e-5)
    np.testing.assert_allclose(r["LSE64"], lse, rtol=0, atol=1e-5)


def test_q_smoothing_lowers_the_error_of_offset_queries():
    """Queries with a large common component: removing each block's mean before INT8 leaves
    the codes the varying part.  With the quantizer that Q-smoothing acts on (Q/K INT8) as the
    only one on, O and dK (which reads the Q codes) land several times closer to exact
    attention, and dQ no farther.  (With every quantizer on, the e4m3 P and dO codes dominate
    the gradients' error, and the difference drowns in it.)"""
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)  # noqa: E731
    qm = orc.QM_QK | orc.QM_F32
    for seed in (54, 55, 56):
        rng = np.random.default_rng(seed)
        N, D = 256, 64
        q, k, v, do = (_rand(rng, N, D) for _ in range(4))
        q = q + 6.0
        ex = orc.run_head(q, k, v, do, True, 0.125, qmask=0)
        plain = orc.run_head(q, k, v, do, True, 0.125, qmask=qm)
        smooth = orc.run_head(q, k, v, do, True, 0.125, qmask=qm, q_smooth=True)
        for n in ("O64", "dK64"):
            assert rel(smooth[n], ex[n]) < 0.5 * rel(plain[n], ex[n]), (seed, n)
        assert rel(smooth["dQ64"], ex["dQ64"]) <= rel(plain["dQ64"], ex["dQ64"]), seed


# ---------------------------------------------------------------- NVFP4 (the FP4 variant)

def _e2m1_brute(x):
    """Nearest value of the e2m1 magnitude grid; a tie takes the value whose mantissa bit is
    0 (0, 1, 2, 4); beyond 6, 6."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    even = {0.0, 1.0, 2.0, 4.0}
    out = np.empty_like(x)
    for i, v in enumerate(x):
        a = abs(v)
        d = np.abs(grid - a)
        best = grid[d == d.min()]
        r = best[0] if len(best) == 1 else [b for b in best if b in even][0]
        out[i] = math.copysign(min(r, 6.0), v)
    return out


def test_e2m1_rounding_against_the_grid():
    """Every multiple of 1/128 in [-8, 8] (all midpoints included) and random values: the
    oracle's arithmetic rounding equals the nearest-grid-value definition."""
    x = np.concatenate([np.arange(-1024, 1025) / 128.0, np.random.default_rng(60).normal(0, 3, 4000)])
    np.testing.assert_array_equal(orc.e2m1(x), _e2m1_brute(x))


def _nvfp4_exact_values(rng, N, D, m):
    """Values that NVFP4 holds exactly: per (channel, 16-token block) e2m1 grid values times
    2^k (k per block, the block's largest magnitude 6 * 2^k), the tensor's largest 2688 * 2^m."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    v = rng.choice(grid, size=(N, D)) * rng.choice([-1.0, 1.0], size=(N, D))
    for t0 in range(0, N, 16):
        v[t0, :] = 6.0  # every block's largest magnitude is 6 before its power of two
    k = rng.integers(-6, 3, size=(N // 16, D))
    v *= np.repeat(2.0 ** k, 16, axis=0)
    v[0, 0] = 2688.0 * 2.0 ** m  # the tensor scale becomes 2^m; its block's scale is 448
    v[1:16, 0] = rng.choice(grid, size=15) * 448.0 * 2.0 ** m
    return v


def test_nvfp4_v_keeps_representable_values_and_its_block_axis():
    """V whose 16-token blocks (per channel) are e2m1 values times a power of two per block,
    with the head's largest |V| = 2688 * 2^m: the tensor scale is 2^m, every block scale is
    exact, and the quantized V equals V.  The blocks' powers of two differ along tokens, so
    blocks taken along another axis, or one scale per channel, would not reproduce it."""
    rng = np.random.default_rng(61)
    N, D = 64, 64
    v = _nvfp4_exact_values(rng, N, D, -4)
    q, k = _rand(rng, N, D), _rand(rng, N, D)
    z = orc.quantize(q, k, v, False, True, qmask=orc.QM_ALL | orc.QM_FP4)
    np.testing.assert_array_equal(z["vx"], v)
    assert np.all(z["sv"] == 1.0)
    # generic values: each value within one e2m1 half-spacing (at most 1) of its block's step
    w = _rand(rng, N, D)
    zw = orc.quantize(q, k, w, False, True, qmask=orc.QM_ALL | orc.QM_FP4)
    blk = np.abs(w).reshape(N // 16, 16, D).max(axis=1)
    step = np.repeat(blk / 6.0 * (1 + 1.0 / 16), 16, axis=0)
    assert np.all(np.abs(zw["vx"] - w) <= step * 1.0 + 1e-12)
    assert np.mean(zw["vx"] == 0.0) < 0.2


@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_uniform_rows_reduce_to_means(causal):
    """Identical keys: every visible logit of a row is equal, so p~ = 1 on each of them, its
    block scale is 448 and its code 6: P^ is exact.  With V exactly representable, O is the
    mean of V over the visible keys (with causal masking, the running mean) to rounding."""
    rng = np.random.default_rng(62)
    N, D = 64, 64
    v = _nvfp4_exact_values(rng, N, D, -3)
    q = _rand(rng, N, D)
    k = np.repeat(_rand(rng, 1, D), N, axis=0)
    r = orc.run_head(q, k, v, _rand(rng, N, D), causal, 0.125, qmask=orc.QM_FP4 | orc.QM_F32,
                     backward_pass=False)
    want = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None] if causal else np.repeat(v.mean(0, keepdims=True), N, 0)
    np.testing.assert_allclose(r["O64"], want, rtol=1e-12, atol=1e-12)


def test_nvfp4_backward_exact_when_p_is_representable():
    """Non-causal, identical keys, 64 keys: P = 1/64 everywhere, which NVFP4 holds exactly
    (block scale e4m3(448/64) = 7, code 6), and V is representable.  The FP4 variant (only
    that quantizer on) then computes what the unquantized path computes: O, LSE, dK, dV agree
    with it to fp32 rounding.  (The backward's P is 2^-6 (1 + ~1e-6) from the fp32 LSE, which
    the block scale rounds back to 2^-6; dQ, zero in exact arithmetic for identical keys, is
    all cancellation here and is left out.)"""
    rng = np.random.default_rng(63)
    N, D = 64, 64
    v = _nvfp4_exact_values(rng, N, D, -3)
    q, do = _rand(rng, N, D), _rand(rng, N, D)
    k = np.repeat(_rand(rng, 1, D), N, axis=0)
    r = orc.run_head(q, k, v, do, False, 0.125, k_smooth=False, qmask=orc.QM_FP4 | orc.QM_F32)
    p = orc.run_head(q, k, v, do, False, 0.125, k_smooth=False, qmask=orc.QM_F32)
    for name in ("O64", "LSE64", "dK64", "dV64"):
        scale = float(np.abs(p[name]).max())
        assert float(np.abs(r[name] - p[name]).max()) <= 1e-5 * scale, name
    # and a P that NVFP4 cannot hold (1/48: block scale 9.333 rounds to 9) moves dV by percents
    r48 = orc.run_head(q[:48], k[:48], v[:48], do[:48], False, 0.125, k_smooth=False, qmask=orc.QM_FP4 | orc.QM_F32)
    p48 = orc.run_head(q[:48], k[:48], v[:48], do[:48], False, 0.125, k_smooth=False, qmask=orc.QM_F32)
    assert np.linalg.norm(r48["dV64"] - p48["dV64"]) > 1e-3 * np.linalg.norm(p48["dV64"])


def test_nvfp4_p_blocks_follow_the_keys():
    """Keys 0-15 with large logits and keys 16-31 with logits 10 lower, V = 1 on the second
    block only: that block's own scale keeps its small P (about 2^-10 of the first block's),
    so O's channel stays within a few percent of exact attention; one scale for the whole row
    would flush those P to zero."""
    rng = np.random.default_rng(64)
    N, D = 32, 64
    q = np.zeros((N, D))
    q[:, 0] = 1.0
    k = np.zeros((N, D))
    k[:16, 0] = 80.0
    k[16:, 0] = 80.0 - 10.0 / (0.125 * math.log2(math.e))
    v = np.zeros((N, D))
    v[16:, 1] = 1.0
    ex = orc.run_head(q, k, v, _rand(rng, N, D), False, 0.125, k_smooth=False, qmask=0, backward_pass=False)
    r = orc.run_head(q, k, v, _rand(rng, N, D), False, 0.125, k_smooth=False, qmask=orc.QM_FP4 | orc.QM_F32,
                     backward_pass=False)
    assert ex["O64"][0, 1] > 1e-4
    np.testing.assert_allclose(r["O64"][:, 1], ex["O64"][:, 1], rtol=0.05)


# ---------------------------------------------------------------- ThriftAttention

def _thrift_case(seed, N=640, D=64):
    rng = np.random.default_rng(seed)
    q, k, v = (_rand(rng, N, D) for _ in range(3))
    k = k + rng.normal(0, 2.0, size=(1, D))
    return q, k, v


def test_thrift_selection_invariants():
    """The promoted pairs are the ceil(budget * visible) pairs of largest block-mean score
    qbar_I . kbar_J among the pairs the causal mask lets through, ties in index order."""
    q, k, _ = _thrift_case(70)
    nb = 5
    qm = np.stack([q[b * 128:(b + 1) * 128].mean(0) for b in range(nb)])
    km = np.stack([k[b * 128:(b + 1) * 128].mean(0) for b in range(nb)])
    score = qm @ km.T
    for causal in (False, True):
        vis = np.tril(np.ones((nb, nb), bool)) if causal else np.ones((nb, nb), bool)
        for budget in (0.0, 0.05, 0.3, 1.0):
            sel = orc.thrift_select(q, k, causal, budget).astype(bool)
            assert sel.sum() == math.ceil(budget * vis.sum() - 1e-12)
            assert not np.any(sel & ~vis)
            if 0 < sel.sum() < vis.sum():
                assert score[sel].min() >= score[vis & ~sel].max()


def _bf16_values(rng, n, lo, hi):
    """n bf16 values of random sign and significand whose biased exponents lie in [lo, hi],
    with both ends present."""
    e = rng.integers(lo, hi + 1, size=n)
    e[0], e[1] = lo, hi
    bits = (rng.integers(0, 2, size=n) << 15) | (e << 7) | rng.integers(0, 128, size=n)
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()


def test_thrift_block_means_are_exact_within_the_exponent_bound():
    """The block means are fp64 sums in token order divided by the count.  When a 128-token
    block's bf16 values span at most 38 binades every partial sum is an integer multiple of
    the smallest value's ulp below 2^53 of them, so the in-order sum is the exact sum and the
    mean is the exact mean rounded once (checked against rational arithmetic); one binade
    more and an in-order sum can round."""
    from fractions import Fraction
    rng = np.random.default_rng(73)
    for lo in (1, 60, 127 - 19, 254 - 38):
        x = np.stack([_bf16_values(rng, 128, lo, lo + 38) for _ in range(4)], axis=1)
        got = orc._block_means(x)
        for d in range(x.shape[1]):
            exact = sum(Fraction(float(t)) for t in x[:, d]) / 128
            assert got[0, d] == float(exact)
    # ragged tail block: the count is the block's own
    x = np.stack([_bf16_values(rng, 128 + 37, 100, 138)], axis=1)
    got = orc._block_means(x)
    assert got[1, 0] == float(sum(Fraction(float(t)) for t in x[128:, 0]) / 37)
    # 39 binades: 1.0078125 first (odd in units of its ulp 2^-7), then 127 copies of 255 * 2^32
    # (exponent 39 above); the exact sum needs 54 significant bits
    lead = float.fromhex("0x1.02p+0")
    big = 255.0 * 2.0 ** 32
    s = 0.0
    for t in [lead] + [big] * 127:
        s += t
    assert Fraction(s) != Fraction(lead) + 127 * Fraction(big)
    # and at 38 binades the same construction stays exact
    s = 0.0
    for t in [lead] + [big / 2] * 127:
        s += t
    assert Fraction(s) == Fraction(lead) + 127 * Fraction(big / 2)


@pytest.mark.parametrize("causal", [False, True])
def test_thrift_budget_zero_is_the_low_bit_forward(causal):
    q, k, v = _thrift_case(71)
    qz = orc.quantize(q, k, v, False, True)
    plain = orc.forward(qz, causal, 0.125)
    th = dict(sel=orc.thrift_select(q, k, causal, 0.0), **orc.thrift_inputs(qz, v))
    mixed = orc.forward(qz, causal, 0.125, thrift=th)
    np.testing.assert_array_equal(mixed["O64"], plain["O64"])
    np.testing.assert_array_equal(mixed["LSE64"], plain["LSE64"])


def _fp16_attention(qh, kh, vh, causal, sm_scale):
    s = (qh @ kh.T) * sm_scale
    if causal:
        s = np.where(np.tril(np.ones(s.shape, bool)), s, -np.inf)
    s = s - s.max(1, keepdims=True)
    p = np.exp(s)
    return (p @ vh) / p.sum(1, keepdims=True)


@pytest.mark.parametrize("causal", [False, True])
def test_thrift_promoted_tiles_are_fp16_attention(causal):
    """Every pair promoted: the forward is attention on the fp16-rounded q', k'', V, whose
    only other rounding is P's fp16 rounding (relative 2^-11): O within 2^-11 max|V|."""
    q, k, v = _thrift_case(72)
    qz = orc.quantize(q, k, v, False, True)
    th = dict(sel=orc.thrift_select(q, k, causal, 1.0), **orc.thrift_inputs(qz, v))
    r = orc.forward(qz, causal, 0.125, thrift=th)
    ref = _fp16_attention(th["qh"], th["kh"], th["vh"], causal, 0.125)
    assert np.abs(r["O64"] - ref).max() <= 2.0 ** -11 * np.abs(th["vh"]).max() * 1.01 + 1e-6


@pytest.mark.parametrize("budget", [0.1, 0.4])
def test_thrift_mixed_tiles_merge_in_one_softmax(budget):
    """With the low-bit path made exact (quantizers off) any mix of promoted and other tiles
    must give exact attention up to the promoted tiles' fp16 rounding: the two paths share
    the running maximum and row sum.  The low-bit scheme then moves toward exact attention
    as the budget grows."""
    q, k, v = _thrift_case(73)
    ex = orc.run_head(q, k, v, v, True, 0.125, qmask=0, backward_pass=False)
    qz0 = orc.quantize(q, k, v, False, True, qmask=0)
    th0 = dict(sel=orc.thrift_select(q, k, True, budget), **orc.thrift_inputs(qz0, v))
    r0 = orc.forward(qz0, True, 0.125, qmask=0, thrift=th0)
    assert np.abs(r0["O64"] - ex["O64"]).max() <= 2.0 ** -10 * np.abs(v).max()
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)  # noqa: E731
    qz = orc.quantize(q, k, v, False, True)
    errs = []
    for b in (0.0, budget, 1.0):
        th = dict(sel=orc.thrift_select(q, k, True, b), **orc.thrift_inputs(qz, v))
        errs.append(rel(orc.forward(qz, True, 0.125, thrift=th)["O64"], ex["O64"]))
    assert errs[0] > errs[1] > errs[2]
