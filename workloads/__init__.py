"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and lays out the MoE routing metadata; it
holds none of the GEMM's or the quantiser's arithmetic.  The shapes are the
five workloads of the FP8 fine-grained-scaled GEMM:

  tiny      dense    M=128  N=256   K=512
  skinny    dense    M=256  N=7168  K=2048, 1% of activation entries x20
  sweep     dense    M=4096 (N,K) in (7168,18432) (24576,1536) (2112,7168)
  contig    MoE contiguous, G=8, 32768 routed tokens, N=4096, K=7168
  masked    MoE masked, G=16, max_m=256, N=7168, K=2048

Expert popularity for the contiguous workload spans 10x, after the remark that
MoE expert activation frequencies differ by more than ten times
("DeepGEMM：面向大模型的高效矩阵计算加速方案", 一.1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QBLOCK = 128          # granularity of the fine-grained scales
SENTINEL_BF16 = 0x7FBF  # fill for rows a grouped GEMM must leave untouched


@dataclass(frozen=True)
class Workload:
    name: str
    layout: str            # "dense" | "contiguous" | "masked"
    M: int = 0             # dense rows
    N: int = 0
    K: int = 0
    G: int = 1
    tokens: int = 0        # contiguous: routed tokens before padding
    max_m: int = 0         # masked: rows per expert buffer
    outliers: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", "dense", M=128, N=256, K=512, seed=0),
    "skinny": Workload("skinny", "dense", M=256, N=7168, K=2048, outliers=True, seed=1),
    "sweep_n7168_k18432": Workload("sweep_n7168_k18432", "dense", M=4096, N=7168, K=18432, seed=2),
    "sweep_n24576_k1536": Workload("sweep_n24576_k1536", "dense", M=4096, N=24576, K=1536, seed=2),
    "sweep_n2112_k7168": Workload("sweep_n2112_k7168", "dense", M=4096, N=2112, K=7168, seed=2),
    "contig": Workload("contig", "contiguous", N=4096, K=7168, G=8, tokens=32768, seed=3),
    "masked": Workload("masked", "masked", N=7168, K=2048, G=16, max_m=256, seed=4),
}


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# --------------------------------------------------------------- dense -----
def normal_matrix(g: np.random.Generator, shape, outliers: bool = False) -> np.ndarray:
    """fp32 N(0,1); with ``outliers`` each entry is multiplied by 20 with
    probability 0.01 (Bernoulli from the same generator)."""
    x = g.standard_normal(shape, dtype=np.float32)
    if outliers:
        hit = g.random(shape, dtype=np.float32) < 0.01
        x[hit] *= np.float32(20.0)
    return x


def dense_inputs(M: int, N: int, K: int, seed: int, outliers: bool = False):
    """(x fp32 [M,K], w fp32 [N,K]) for a dense workload."""
    g = rng(seed)
    x = normal_matrix(g, (M, K), outliers)
    w = normal_matrix(g, (N, K))
    return x, w


# ---------------------------------------------------------- MoE routing -----
def contiguous_routing(G: int, tokens: int, seed: int, align: int = QBLOCK):
    """Per-expert token counts from a multinomial whose expert probabilities
    are p_g proportional to 10^(g/(G-1)) (a 10x span), each count padded up to a
    multiple of ``align`` with rows whose expert index is -1.

    Returns (counts int64 [G], m_indices int32 [sum_M], seg_start int64 [G])."""
    g = rng(seed)
    p = 10.0 ** (np.arange(G) / max(G - 1, 1))
    p = p / p.sum()
    counts = g.multinomial(tokens, p)
    padded = (counts + align - 1) // align * align
    sum_M = int(padded.sum())
    m_indices = np.full(sum_M, -1, dtype=np.int32)
    seg_start = np.zeros(G, dtype=np.int64)
    off = 0
    for e in range(G):
        seg_start[e] = off
        m_indices[off:off + counts[e]] = e
        off += int(padded[e])
    return counts, m_indices, seg_start


def masked_counts(G: int, max_m: int, seed: int) -> np.ndarray:
    """masked_m[g] ~ U{0..max_m}, int32 [G]."""
    return rng(seed).integers(0, max_m + 1, G).astype(np.int32)


def contiguous_inputs(w: Workload):
    """(x fp32 [sum_M,K], weights fp32 [G,N,K], m_indices, counts)."""
    counts, m_indices, _ = contiguous_routing(w.G, w.tokens, w.seed)
    g = rng(w.seed + 1000)
    x = normal_matrix(g, (len(m_indices), w.K))
    wt = normal_matrix(g, (w.G, w.N, w.K))
    return x, wt, m_indices, counts


def masked_inputs(w: Workload):
    """(x fp32 [G,max_m,K], weights fp32 [G,N,K], masked_m int32 [G])."""
    masked_m = masked_counts(w.G, w.max_m, w.seed)
    g = rng(w.seed + 1000)
    x = normal_matrix(g, (w.G, w.max_m, w.K))
    wt = normal_matrix(g, (w.G, w.N, w.K))
    return x, wt, masked_m


# ------------------------------------------------------ exact-arithmetic ----
def exact_operands(g: np.random.Generator, shape, vmax: int = 2) -> np.ndarray:
    """Small integers in [-vmax, vmax] (int8).  Every such value and every
    product and 128-term sum of them is exact in any float format that the
    path uses, so results built from them are unique."""
    return g.integers(-vmax, vmax + 1, shape).astype(np.int8)


def exact_scales(g: np.random.Generator, shape, emin: int = -3, emax: int = 0) -> np.ndarray:
    """Power-of-two fp32 scales 2^e, e ~ U{emin..emax}."""
    e = g.integers(emin, emax + 1, shape)
    return np.ldexp(np.ones(shape, dtype=np.float32), e).astype(np.float32)


def sample_rows(n_rows: int, count: int, seed: int, must=()) -> np.ndarray:
    """A sorted sample of distinct row indices that always contains ``must``
    (first/last rows, tile edges) plus ``count`` random rows."""
    g = rng(seed + 777)
    pick = set(int(r) for r in must if 0 <= r < n_rows)
    extra = g.choice(n_rows, size=min(count, n_rows), replace=False)
    pick.update(int(r) for r in extra)
    return np.array(sorted(pick), dtype=np.int32)
