"""Seeded synthetic inputs for the low-bit attention path.

This module is the one piece shared by the CUDA path's callers (tests, bench) and
the CPU oracle's callers: it draws the inputs and nothing else.  It holds none of
the method's arithmetic (no quantization, no softmax, no scales).

Every tensor is [B, H, N, D], drawn in fp32 from numpy's PCG64 generator and
rounded to bf16 (round to nearest, ties to even).  Each (tensor, head) pair has
its own stream, seeded with (seed, tensor id, b*H + h), so a single head can be
regenerated without drawing the others; the CPU oracle uses that to compute
sampled heads of the full-size workloads.

The five named workloads follow the training shapes the SageBwd pages discuss
(8k and 64k tokens per step, long context, a bidirectional video-DiT-like layer)
with synthetic values; no dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# tensor ids for the per-head streams
_TQ, _TK, _TV, _TDO, _TEXTRA = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    causal: bool
    qk_norm: bool
    k_smooth: bool
    sm_scale: float          # softmax temperature applied to q.k
    kind: str                # value recipe, see head_inputs()
    seed: int
    note: str = ""

    @property
    def bh(self) -> int:
        return self.B * self.H

    def ops(self) -> dict:
        """Causal-adjusted operation counts (FlashAttention convention).

        forward = 4*B*H*N^2*D (QK^T and PV), backward = 2.5x forward, both halved
        when causal.
        """
        f = 4.0 * self.B * self.H * self.N * self.N * self.D
        if self.causal:
            f *= 0.5
        return {"fwd": f, "bwd": 2.5 * f, "fwd_bwd": 3.5 * f}


WORKLOADS = {
    # B=1,H=2,N=256,D=64 non-causal; K carries a per-(b,h,d) offset shared by all tokens
    "pr1_ref": Workload("pr1_ref", 1, 2, 256, 64, False, False, True, 1.0 / 8.0,
                        "k_offset2", 0, "B1 H2 N256 D64, non-causal, K offset N(0,2^2)"),
    # pretraining layer, 8k tokens/step; 4 outlier K channels per head scaled by 20
    "pretrain_8k": Workload("pretrain_8k", 4, 16, 2048, 128, True, False, True,
                            1.0 / math.sqrt(128.0), "k_outlier20", 1,
                            "B4 H16 N2048 D128, causal, 4 K outlier channels x20"),
    # same layer with QK-norm, 64k tokens/step, logits scaled by a fixed 16
    "qknorm_64k": Workload("qknorm_64k", 16, 16, 4096, 128, True, True, True, 16.0,
                           "normal", 2, "B16 H16 N4096 D128, causal, QK-norm, scale 16"),
    # long context; Q and K Student-t (nu=3) scaled to unit variance
    "long_32k": Workload("long_32k", 1, 32, 32768, 128, True, False, True,
                         1.0 / math.sqrt(128.0), "student_t3", 3,
                         "B1 H32 N32768 D128, causal, Student-t(3) Q/K"),
    # bidirectional video-DiT-like layer; K offset N(0,3^2)
    "video_dit": Workload("video_dit", 2, 24, 16384, 64, False, False, True, 1.0 / 8.0,
                          "k_offset3", 4, "B2 H24 N16384 D64, non-causal, K offset N(0,3^2)"),
}

BENCH_WORKLOAD = "long_32k"


def custom(B, H, N, D, causal, qk_norm=False, k_smooth=True, sm_scale=None,
           kind="normal", seed=0, name="custom") -> Workload:
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    return Workload(name, B, H, N, D, bool(causal), bool(qk_norm), bool(k_smooth),
                    float(sm_scale), kind, int(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed, tid, bh):
    return np.random.default_rng([int(seed), int(tid), int(bh)])


def head_inputs(w: Workload, bh: int) -> dict:
    """bf16 bit patterns (uint16 [N, D]) of q, k, v, do for head index bh = b*H + h."""
    N, D = w.N, w.D
    out = {}
    if w.kind == "student_t3":
        q = _rng(w.seed, _TQ, bh).standard_t(3, size=(N, D)) / math.sqrt(3.0)
        k = _rng(w.seed, _TK, bh).standard_t(3, size=(N, D)) / math.sqrt(3.0)
    else:
        q = _rng(w.seed, _TQ, bh).standard_normal((N, D))
        k = _rng(w.seed, _TK, bh).standard_normal((N, D))
    v = _rng(w.seed, _TV, bh).standard_normal((N, D))
    do = _rng(w.seed, _TDO, bh).standard_normal((N, D))
    ex = _rng(w.seed, _TEXTRA, bh)
    if w.kind == "k_offset2":
        k = k + ex.normal(0.0, 2.0, size=(1, D))
    elif w.kind == "k_offset3":
        k = k + ex.normal(0.0, 3.0, size=(1, D))
    elif w.kind == "q_offset3":
        q = q + ex.normal(0.0, 3.0, size=(1, D))  # a common query component (Q-smoothing cases)
    elif w.kind == "k_outlier20":
        ch = ex.permutation(D)[:4]
        k[:, ch] *= 20.0
    elif w.kind == "exp_spread":
        # Q and K magnitudes spread over about 48 binades (each element scaled down by 2^u, u a
        # whole number in [0, 44)): block sums whose values span more than 38 binades, logits
        # no larger than the plain recipe's
        q = q * np.exp2(-ex.integers(0, 44, size=(N, D)))
        k = k * np.exp2(-ex.integers(0, 44, size=(N, D)))
    elif w.kind in ("normal", "student_t3"):
        pass
    else:
        raise ValueError(f"unknown input recipe {w.kind!r}")
    for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
        out[name] = f32_to_bf16_bits(x.astype(np.float32))
    return out


def all_inputs(w: Workload) -> dict:
    """bf16 bit patterns (uint16 [B, H, N, D]) of q, k, v, do for every head.

    Heads are drawn on a thread pool (numpy's generators release the GIL while they fill
    arrays); every head has its own stream, so the result does not depend on the order."""
    import concurrent.futures as cf
    import os
    shape = (w.B, w.H, w.N, w.D)
    out = {n: np.empty(shape, dtype=np.uint16) for n in ("q", "k", "v", "do")}

    def one(bh):
        hi = head_inputs(w, bh)
        b, h = divmod(bh, w.H)
        for n in out:
            out[n][b, h] = hi[n]

    workers = min(16, os.cpu_count() or 1, w.bh)
    if workers <= 1 or w.N * w.D < (1 << 16):
        for bh in range(w.bh):
            one(bh)
    else:
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, range(w.bh)))
    return out


def sample_heads(w: Workload, every: int = 8, limit: int | None = None) -> list:
    """Deterministic head subset: first, last and every `every`-th head."""
    hs = sorted(set([0, w.bh - 1] + list(range(0, w.bh, every))))
    if limit is not None:
        hs = hs[:limit - 1] + [w.bh - 1] if limit < len(hs) else hs
    return hs
