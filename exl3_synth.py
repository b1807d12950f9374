"""Seeded synthetic inputs for the EXL3 trellis-quantized linear layer.

This module only draws random arrays with the shapes and distributions of the
workloads described on the source pages; it holds none of the layer's
arithmetic (no decoding, no transforms, no contraction).  Both the CPU oracle
and the CUDA library consume exactly the arrays produced here, so every
comparison between them starts from identical bytes.

Recipe (all numpy PCG64, seed = 20260000 + 100 * config + sub_case):

* trellis: uniform uint16 words, shape [k/16, n/16, 16*K] (the per-linear
  trellis tensor shape of the Arc 140V MoE post, section 2.A).  With uniform
  bits every 16-bit trellis state is uniform.
* suh / svh: +1 or -1 with equal probability, stored as IEEE binary16.
* x: N(0, 1) drawn in float64 and rounded to binary16, with the outlier rule
  of the workload (rows scaled x20 or channels scaled x30).
* bias (linears with an output bias): N(0, 4^2) rounded to binary16, from
  its own seed stream (config 6).
* MoE routing: logits N(0, 1) [T, E]; the top-k logits by value (ties toward
  the lower expert id) and the softmax of those k logits as routing weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20260000


def seed_for(config: int, sub: int = 0) -> int:
    """Seed of sub-case ``sub`` of workload ``config``."""
    return SEED_BASE + 100 * config + sub


def rng_for(config: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(config, sub)))


def trellis(rng: np.random.Generator, k: int, n: int, K: int) -> np.ndarray:
    """Uniform packed trellis words, uint16 [k/16, n/16, 16*K]."""
    if k % 16 or n % 16:
        raise ValueError("k and n must be multiples of 16")
    return rng.integers(0, 1 << 16, size=(k // 16, n // 16, 16 * K), dtype=np.uint16)


def signs(rng: np.random.Generator, length: int) -> np.ndarray:
    """Random +-1 vector as float16."""
    return np.where(rng.integers(0, 2, size=length) == 1, 1.0, -1.0).astype(np.float16)


def activations(rng: np.random.Generator, M: int, k: int, *, outlier_rows: float = 0.0,
                row_scale: float = 20.0, outlier_channels: float = 0.0,
                channel_scale: float = 30.0) -> np.ndarray:
    """x ~ N(0,1) in float64, optionally with outliers, rounded to float16 [M, k].

    outlier_rows: fraction of rows (at least one when > 0) scaled by row_scale,
    chosen by a seeded permutation.  outlier_channels: fraction of the k input
    channels (at least one when > 0) scaled by channel_scale.
    """
    x = rng.standard_normal((M, k))
    if outlier_rows > 0:
        cnt = max(1, math.ceil(outlier_rows * M))
        rows = rng.permutation(M)[:cnt]
        x[rows] *= row_scale
    if outlier_channels > 0:
        cnt = max(1, math.ceil(outlier_channels * k))
        cols = rng.permutation(k)[:cnt]
        x[:, cols] *= channel_scale
    return x.astype(np.float16)


def bias(rng: np.random.Generator, n: int, scale: float = 4.0) -> np.ndarray:
    """Output bias, N(0, scale^2) in float64 rounded to float16 [n]."""
    return (rng.standard_normal(n) * scale).astype(np.float16)


BIAS_CONFIG = 6   # seed stream of the bias vectors (kept apart from the five workloads)


def bias_for(sub: int, n: int) -> np.ndarray:
    """The bias vector of sub-case ``sub`` (seed 20260000 + 600 + sub)."""
    return bias(rng_for(BIAS_CONFIG, sub), n)


def routing(rng: np.random.Generator, T: int, E: int, topk: int):
    """Router draw: (ids int32 [T, topk], weights float32 [T, topk]).

    Logits ~ N(0,1) [T, E]; the topk largest per token (ties toward the lower
    id, via a stable sort of the negated logits); weights are the softmax of
    the selected logits (so they sum to one per token).
    """
    logits = rng.standard_normal((T, E))
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(logits, order, axis=1)
    sel = sel - sel.max(axis=1, keepdims=True)
    w = np.exp(sel)
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


# --------------------------------------------------------------------------
# The five workloads (shapes of the pages' dense 27B family and 256-expert MoE)
# --------------------------------------------------------------------------

@dataclass
class LinearCase:
    """One linear: x [M,k] fp16, trellis [k/16,n/16,16K] u16, suh [k], svh [n]."""
    name: str
    M: int
    k: int
    n: int
    K: int
    x: np.ndarray
    trellis: np.ndarray
    suh: np.ndarray
    svh: np.ndarray
    meta: dict = field(default_factory=dict)


def linear_case(config: int, sub: int, M: int, k: int, n: int, K: int, *,
                outlier_rows: float = 0.0, outlier_channels: float = 0.0,
                name: str = "") -> LinearCase:
    rng = rng_for(config, sub)
    tr = trellis(rng, k, n, K)
    suh = signs(rng, k)
    svh = signs(rng, n)
    x = activations(rng, M, k, outlier_rows=outlier_rows, outlier_channels=outlier_channels)
    return LinearCase(name or f"cfg{config}.{sub}", M, k, n, K, x, tr, suh, svh)


def config1() -> LinearCase:
    """Single linear k=2048, n=512, K=4, x [1, 2048]."""
    return linear_case(1, 0, 1, 2048, 512, 4, name="cfg1 k2048 n512 K4 M1")


CONFIG2_N = (5120, 17408, 25600)
CONFIG2_M = (1, 4, 16)


def config2(n: int, M: int) -> LinearCase:
    """Dense decode sweep: k=5120, n in CONFIG2_N, K=4, M in CONFIG2_M."""
    sub = CONFIG2_N.index(n) * 10 + CONFIG2_M.index(M)
    return linear_case(2, sub, M, 5120, n, 4, name=f"cfg2 k5120 n{n} K4 M{M}")


CONFIG3_K = (2, 3, 4, 5, 6, 7, 8)
CONFIG3_M = (1, 8, 64)


def config3(K: int, M: int) -> LinearCase:
    """Mixed-width layer: k=n=4096, one tensor per K, 5% outlier rows x20."""
    sub = CONFIG3_K.index(K) * 10 + CONFIG3_M.index(M)
    return linear_case(3, sub, M, 4096, 4096, K, outlier_rows=0.05,
                       name=f"cfg3 k4096 n4096 K{K} M{M}")


def config4(M: int = 4096) -> LinearCase:
    """Prefill: M=4096, k=5120, n=17408, K=4, 1% of channels x30."""
    return linear_case(4, 0, M, 5120, 17408, 4, outlier_channels=0.01,
                       name=f"cfg4 k5120 n17408 K4 M{M}")


@dataclass
class ExpertProj:
    """One projection kind for all E experts (contiguous arenas)."""
    trellis: np.ndarray  # [E, nslots, k/16, n/16, 16K] uint16
    suh: np.ndarray      # [E, nslots, k] fp16
    svh: np.ndarray      # [E, nslots, n] fp16
    k: int
    n: int
    K: int
    nslots: int


@dataclass
class MoECase:
    name: str
    T: int
    hidden: int
    inter: int
    E: int
    topk: int
    K: int
    x: np.ndarray         # [T, hidden] fp16
    ids: np.ndarray       # [T, topk] int32
    weights: np.ndarray   # [T, topk] float32
    w13: ExpertProj
    w2: ExpertProj


def expert_proj(rng: np.random.Generator, E: int, nslots: int, k: int, n: int, K: int) -> ExpertProj:
    tr = rng.integers(0, 1 << 16, size=(E, nslots, k // 16, n // 16, 16 * K), dtype=np.uint16)
    suh = np.where(rng.integers(0, 2, size=(E, nslots, k)) == 1, 1.0, -1.0).astype(np.float16)
    svh = np.where(rng.integers(0, 2, size=(E, nslots, n)) == 1, 1.0, -1.0).astype(np.float16)
    return ExpertProj(tr, suh, svh, k, n, K, nslots)


CONFIG5_T = (1, 128, 4096)


def moe_case(config: int, sub: int, T: int, *, E: int = 256, topk: int = 8, hidden: int = 2048,
             inter: int = 512, K: int = 3, K2: int = 0, name: str = "") -> MoECase:
    """Routed experts: gate+up (nslots=2, hidden->inter each, K bits) and down
    (inter->hidden, K2 bits; K2 = 0 means K)."""
    rng = rng_for(config, sub)
    w13 = expert_proj(rng, E, 2, hidden, inter, K)
    w2 = expert_proj(rng, E, 1, inter, hidden, K2 or K)
    ids, w = routing(rng, T, E, topk)
    x = activations(rng, T, hidden)
    return MoECase(name or f"moe{config}.{sub}", T, hidden, inter, E, topk, K, x, ids, w, w13, w2)


@dataclass
class MixedExpertProj:
    """One projection kind with a width per expert: the trellis arena packs
    expert e's nslots tensors ([k/16, n/16, 16*K[e]] each) right after expert
    e-1's, as one flat uint16 array."""
    trellis: np.ndarray  # flat uint16, sum over e of nslots * k * n * K[e] / 16 words
    suh: np.ndarray      # [E, nslots, k] fp16
    svh: np.ndarray      # [E, nslots, n] fp16
    K: np.ndarray        # [E] int32 widths
    k: int
    n: int
    nslots: int


@dataclass
class MixedMoECase:
    name: str
    T: int
    hidden: int
    inter: int
    E: int
    topk: int
    x: np.ndarray
    ids: np.ndarray
    weights: np.ndarray
    w13: MixedExpertProj
    w2: MixedExpertProj


def mixed_expert_proj(rng: np.random.Generator, K: np.ndarray, nslots: int, k: int, n: int) -> MixedExpertProj:
    K = np.asarray(K, dtype=np.int32)
    E = len(K)
    words = int(sum(nslots * (k // 16) * (n // 16) * 16 * int(w) for w in K))
    tr = rng.integers(0, 1 << 16, size=words, dtype=np.uint16)
    suh = np.where(rng.integers(0, 2, size=(E, nslots, k)) == 1, 1.0, -1.0).astype(np.float16)
    svh = np.where(rng.integers(0, 2, size=(E, nslots, n)) == 1, 1.0, -1.0).astype(np.float16)
    return MixedExpertProj(tr, suh, svh, K, k, n, nslots)


def mixed_moe_case(config: int, sub: int, T: int, K13, K2, *, topk: int = 8, hidden: int = 2048,
                   inter: int = 512, name: str = "") -> MixedMoECase:
    """Routed experts with a width per expert: K13[e] for gate+up, K2[e] for
    down (E = len(K13)); otherwise the recipe of moe_case."""
    rng = rng_for(config, sub)
    E = len(K13)
    w13 = mixed_expert_proj(rng, K13, 2, hidden, inter)
    w2 = mixed_expert_proj(rng, K2, 1, inter, hidden)
    ids, w = routing(rng, T, E, topk)
    x = activations(rng, T, hidden)
    return MixedMoECase(name or f"moe-mixed{config}.{sub}", T, hidden, inter, E, topk, x, ids, w, w13, w2)


def config5(T: int) -> MoECase:
    """Grouped MoE: E=256, top-8, hidden 2048, inter 512, K=3."""
    return moe_case(5, CONFIG5_T.index(T), T, name=f"cfg5 E256 top8 h2048 i512 K3 T{T}")
