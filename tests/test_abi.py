"""The C ABI library loads without a GPU, exports every function include/sage_attn.h
declares, sizes its workspaces, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

import bit_trainable_attention_sagebwd_gb300 as sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_trainable_attention_sagebwd_gb300 import build
    build.build()
    return sa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sage_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sage_attn_\w+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) == set(sa.ABI_FUNCTIONS)


def test_workspace_sizes(lib):
    for (B, H, N, D) in [(1, 2, 256, 64), (4, 16, 2048, 128), (1, 32, 32768, 128), (1, 1, 1, 64), (2, 3, 333, 128)]:
        n = sa.sage_attn_ws_bytes(B, H, N, D)
        np_ = (N + 127) // 128 * 128
        # at least the codes: two bf16 containers and one e4m3 tensor
        assert n >= B * H * np_ * D * 5
        assert n % 256 == 0
        assert sa.sage_attn_bwd_ws_bytes(B, H, N, D) >= B * H * np_ * D * 5
    for bad in [(1, 1, 128, 96), (0, 1, 128, 64), (1, 1, 0, 64), (1, 1, 128, 256)]:
        assert sa.sage_attn_ws_bytes(*bad) == 0
        assert sa.sage_attn_bwd_ws_bytes(*bad) == 0


def test_argument_errors_return_before_launch(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: the checks fail first
    odd = ctypes.c_void_p(0x10001)
    assert sa.sage_attn_quantize(null, fake, fake, 1, 1, 128, 64, 0, 1, fake, 1 << 30, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_quantize(odd, fake, fake, 1, 1, 128, 64, 0, 1, fake, 1 << 30, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_quantize(fake, fake, fake, 1, 1, 128, 96, 0, 1, fake, 1 << 30, null) == sa.SAGE_ERR_UNSUPPORTED
    assert sa.sage_attn_quantize(fake, fake, fake, 1, 1, 128, 64, 0, 1, fake, 16, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fwd(fake, fake, null, null, 1, 1, 128, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fwd(fake, fake, fake, odd, 1, 1, 128, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fwd(fake, fake, fake, null, 1, 1, 128, 64, 1, float("nan"), null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fwd(fake, fake, fake, null, 1, 1, 128, 80, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED
    args = [fake] * 11
    assert sa.sage_attn_bwd(*args[:10], fake, 16, 1, 1, 128, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    a2 = list(args)
    a2[6] = odd
    assert sa.sage_attn_bwd(*a2[:10], fake, 1 << 40, 1, 1, 128, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    # the fp32-auxiliary backward: same checks, O32 in place of O
    assert sa.sage_attn_bwd_o32(*args[:3], null, *args[4:10], fake, 1 << 40, 1, 1, 128, 64, 1, 0, 1, 0.125,
                                null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_bwd_o32(*args[:10], fake, 16, 1, 1, 128, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_bwd_o32(*args[:10], fake, 1 << 40, 1, 1, 128, 80, 1, 0, 1, 0.125,
                                null) == sa.SAGE_ERR_UNSUPPORTED
    with pytest.raises(sa.SageError):
        sa.sage_attn_ws_views(fake, 1, 1, 128, 96)
    assert sa.status_str(sa.SAGE_ERR_TIMEOUT) == "device wait timed out"


def test_ws_views_offsets(lib):
    base = 1 << 20
    v = sa.sage_attn_ws_views(ctypes.c_void_p(base), 2, 3, 333, 128)
    assert v.n_pad == 384
    ptrs = [v.status, v.qc, v.kc, v.v8t, v.sq, v.sk, v.sv, v.kmean, v.qr, v.kr]
    assert ptrs == sorted(ptrs) and all((p - base) % 256 == 0 for p in ptrs)
    assert v.kc - v.qc >= 6 * 384 * 128 * 2


def test_step_host_sizes_and_argument_errors(lib):
    """Scratch of the host-tensor step: inputs and outputs of the whole batch plus the
    workspaces of the largest head range; smaller ranges need less; bad arguments are
    refused before any CUDA call."""
    B, H, N, D = 4, 16, 2048, 128
    t = B * H * N * D * 2
    sizes = {g: sa.sage_attn_step_host_bytes(B, H, N, D, g) for g in (1, 2, 5, 8, 64)}
    for g, n in sizes.items():
        assert n >= 8 * t + B * H * N * 4 and n % 256 == 0
    assert sizes[1] > sizes[2] > sizes[5] > sizes[8] > sizes[64]
    assert sa.sage_attn_step_host_bytes(B, H, N, D, 0) == sizes[5]  # automatic: five ranges
    assert sa.sage_attn_step_host_bytes(1, 1, 128, 96, 0) == 0
    n = sizes[5]
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)
    host = [fake] * 9
    assert sa.sage_attn_step_host(*host, null, n, B, H, N, D, 1, 0, 1, 0.0, 0, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_step_host(*host, ctypes.c_void_p(0x10010), n, B, H, N, D, 1, 0, 1, 0.0, 0,
                                  null) == sa.SAGE_ERR_INVALID_ARG  # scratch not 256-byte aligned
    assert sa.sage_attn_step_host(*host, fake, n - 256, B, H, N, D, 1, 0, 1, 0.0, 0, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_step_host(*host, fake, n, B, H, N, D, 1, 0, 1, float("inf"), 0,
                                  null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_step_host(*host, fake, n, B, H, N, 96, 1, 0, 1, 0.0, 0, null) == sa.SAGE_ERR_UNSUPPORTED
    host[4] = null  # no O buffer
    assert sa.sage_attn_step_host(*host, fake, n, B, H, N, D, 1, 0, 1, 0.0, 0, null) == sa.SAGE_ERR_INVALID_ARG


def test_timer_filter_needs_no_gpu(lib):
    assert sa.sage_attn_timer_only("bwd_main") == sa.SAGE_OK
    assert sa.sage_attn_timer_only(None) == sa.SAGE_OK
    assert sa.sage_attn_timer_read("bwd_main") == (0.0, 0)


def test_q_smoothing_workspace_and_argument_errors(lib):
    """The Q-smoothing workspace is the grouped one plus the query block means and the logit
    terms (4 bytes each, [B*H][Np/128][D] and [B*H][Np/128][Np]); its views point into it in
    order, and its calls refuse bad arguments before any launch."""
    for (B, H, Hkv, N, D) in [(1, 2, 2, 256, 64), (4, 16, 4, 2048, 128), (2, 3, 1, 333, 128)]:
        np_ = (N + 127) // 128 * 128
        nb = np_ // 128
        base = sa.sage_attn_gqa_ws_bytes(B, H, Hkv, N, D)
        n = sa.sage_attn_qs_ws_bytes(B, H, Hkv, N, D)
        extra = B * H * nb * (D + np_) * 4
        assert base + extra <= n <= base + extra + 512 and n % 256 == 0
        v = sa.sage_attn_qs_ws_views(ctypes.c_void_p(1 << 20), B, H, Hkv, N, D)
        ptrs = [v.status, v.qc, v.kc, v.v8t, v.sq, v.sk, v.sv, v.kmean, v.qr, v.kr, v.qmean, v.dsb]
        assert ptrs == sorted(ptrs) and v.dsb - v.qmean >= B * H * nb * D * 4
        assert (1 << 20) + n - v.dsb >= B * H * nb * np_ * 4
    # the other layouts have no Q-smoothing sections
    v = sa.sage_attn_ws_views(ctypes.c_void_p(1 << 20), 1, 2, 256, 64)
    assert v.qmean is None and v.dsb is None
    assert sa.sage_attn_qs_ws_bytes(1, 4, 3, 128, 64) == 0  # Hkv must divide H
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)
    n = sa.sage_attn_qs_ws_bytes(1, 4, 2, 256, 64)
    assert sa.sage_attn_qs_quantize(null, fake, fake, 1, 4, 2, 256, 64, 0, 1, fake, n, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_qs_quantize(fake, fake, fake, 1, 4, 2, 256, 64, 0, 1, fake, n - 256,
                                    null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_qs_quantize(fake, fake, fake, 1, 4, 3, 256, 64, 0, 1, fake, n, null) == sa.SAGE_ERR_UNSUPPORTED
    assert sa.sage_attn_qs_fwd(fake, fake, null, null, 1, 4, 2, 256, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_qs_fwd(fake, fake, fake, null, 1, 4, 2, 256, 96, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED
    nbw = sa.sage_attn_gqa_bwd_ws_bytes(1, 4, 2, 256, 64)
    args = [fake] * 11
    assert sa.sage_attn_qs_bwd(*args, nbw - 256, 1, 4, 2, 256, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_qs_bwd(*args, nbw, 1, 4, 2, 256, 64, 1, 0, 1, float("nan"), null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_qs_bwd(*args, nbw, 1, 4, 3, 256, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED


def test_nvfp4_workspace_and_argument_errors(lib):
    """The NVFP4 workspace is the plain one plus V's packed e2m1 codes (half a byte per value),
    their e4m3 block scales (one per 16 tokens, in 512-byte atoms of 128 channel rows x 4
    blocks, as the tensor core reads them) and one fp32 tensor scale per head; its views point
    there, the plain workspace's do not, and its calls refuse bad arguments before any launch."""
    for (B, H, N, D) in [(1, 2, 256, 64), (4, 16, 2048, 128), (2, 3, 333, 128)]:
        np_ = (N + 127) // 128 * 128
        base = sa.sage_attn_ws_bytes(B, H, N, D)
        n = sa.sage_attn_fp4_ws_bytes(B, H, N, D)
        extra = B * H * (D * np_ // 2 + np_ // 64 * 512 + 4)
        assert base + extra <= n <= base + extra + 1024 and n % 256 == 0
        v = sa.sage_attn_fp4_ws_views(ctypes.c_void_p(1 << 20), B, H, N, D)
        assert v.v4 is not None and v.v4sf is not None and v.vg is not None
        assert v.v4sf - v.v4 >= B * H * D * np_ // 2
        assert (1 << 20) + n - v.v4sf >= B * H * np_ // 64 * 512
        assert sa.sage_attn_fp4_bwd_ws_bytes(B, H, N, D) >= sa.sage_attn_bwd_ws_bytes(B, H, N, D) + B * H * np_ * D * 2
    v = sa.sage_attn_ws_views(ctypes.c_void_p(1 << 20), 1, 2, 256, 64)
    assert v.v4 is None and v.v4sf is None and v.vg is None
    assert sa.sage_attn_fp4_ws_bytes(1, 1, 128, 96) == 0 and sa.sage_attn_fp4_bwd_ws_bytes(1, 1, 128, 96) == 0
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10001)
    n = sa.sage_attn_fp4_ws_bytes(1, 2, 256, 64)
    assert sa.sage_attn_fp4_quantize(null, fake, fake, 1, 2, 256, 64, 0, 1, fake, n, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_quantize(fake, fake, fake, 1, 2, 256, 64, 0, 1, fake, n - 256,
                                     null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_quantize(fake, fake, fake, 1, 2, 256, 96, 0, 1, fake, n, null) == sa.SAGE_ERR_UNSUPPORTED
    assert sa.sage_attn_fp4_fwd(fake, fake, null, null, 1, 2, 256, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_fwd(fake, fake, fake, odd, 1, 2, 256, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_fwd(fake, fake, fake, null, 1, 2, 256, 64, 1, float("inf"), null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_fwd(fake, fake, fake, null, 1, 2, 256, 80, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED
    nbw = sa.sage_attn_fp4_bwd_ws_bytes(1, 2, 256, 64)
    args = [fake] * 11
    assert sa.sage_attn_fp4_bwd(*args, nbw - 256, 1, 2, 256, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_bwd(*args, nbw, 1, 2, 256, 64, 1, 0, 1, float("nan"), null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_fp4_bwd(*args, nbw, 1, 2, 256, 96, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED
    bad = list(args)
    bad[4] = null  # LSE
    assert sa.sage_attn_fp4_bwd(*bad, nbw, 1, 2, 256, 64, 1, 0, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG


def test_thrift_workspace_and_argument_errors(lib):
    """ThriftAttention's scratch holds the block means (fp64), the pair keys (8 bytes) and the
    promoted pairs (1 byte) per (query block, key tile), the fp16 copies of q', k'' and V, and the
    low-bit pass's hand-over (fp32 output and two fp32 per row); the selection pointer lies
    after the means and keys; the calls refuse bad arguments (a budget outside [0, 1] too)."""
    for (B, H, N, D) in [(1, 2, 256, 64), (4, 16, 2048, 128), (2, 3, 333, 128)]:
        np_ = (N + 127) // 128 * 128
        nb = np_ // 128
        bh = B * H
        need = 2 * bh * nb * D * 8 + bh * nb * nb * 9 + 3 * bh * np_ * D * 2 + bh * np_ * D * 4 + bh * np_ * 8
        n = sa.sage_attn_thrift_ws_bytes(B, H, N, D)
        assert need <= n <= need + 9 * 256 and n % 256 == 0
        sel = sa.sage_attn_thrift_sel(ctypes.c_void_p(1 << 20), B, H, N, D)
        assert sel - (1 << 20) >= 2 * bh * nb * D * 8 + bh * nb * nb * 8
        assert (1 << 20) + n - sel >= bh * nb * nb
    assert sa.sage_attn_thrift_ws_bytes(1, 1, 128, 96) == 0
    assert sa.sage_attn_thrift_sel(ctypes.c_void_p(0), 1, 1, 128, 64) is None
    assert sa.sage_attn_thrift_sel(ctypes.c_void_p(1 << 20), 1, 1, 128, 96) is None
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10001)
    n = sa.sage_attn_ws_bytes(1, 2, 256, 64)
    nt = sa.sage_attn_thrift_ws_bytes(1, 2, 256, 64)

    def tq(q=fake, budget=0.05, D=64, ws_bytes=n, tws=fake, tws_bytes=nt):
        return sa.sage_attn_thrift_quantize(q, fake, fake, 1, 2, 256, D, 0, 1, 1, budget, fake, ws_bytes, tws,
                                            tws_bytes, null)
    assert tq(q=null) == sa.SAGE_ERR_INVALID_ARG
    assert tq(tws=odd) == sa.SAGE_ERR_INVALID_ARG
    for budget in (-0.01, 1.01, float("nan")):
        assert tq(budget=budget) == sa.SAGE_ERR_INVALID_ARG
    assert tq(D=96) == sa.SAGE_ERR_UNSUPPORTED
    assert tq(ws_bytes=n - 256) == sa.SAGE_ERR_INVALID_ARG
    assert tq(tws_bytes=nt - 256) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_thrift_fwd(fake, fake, fake, null, null, 1, 2, 256, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_thrift_fwd(fake, null, fake, fake, null, 1, 2, 256, 64, 1, 0.125, null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_thrift_fwd(fake, fake, fake, fake, null, 1, 2, 256, 64, 1, float("nan"),
                                   null) == sa.SAGE_ERR_INVALID_ARG
    assert sa.sage_attn_thrift_fwd(fake, fake, fake, fake, null, 1, 2, 256, 80, 1, 0.125, null) == sa.SAGE_ERR_UNSUPPORTED
