"""Seeded synthetic inputs for the TT-EmbeddingBag workloads.

This module only draws random numbers and lays them out; it holds none of the
TT-EmbeddingBag arithmetic (no decode, no contraction, no pooling).  Both the
float64 oracle (``oracle/``) and the CUDA path take their inputs from here, so
the two sides read identical bytes.

Workloads (TT-Rec / FBTT-Embedding pages: the README's parameter list and its
sample benchmark line, and the TT-Rec abstract's DLRM setting):

==== =================================================================
id   workload
==== =================================================================
1    tiny: p=[4,5,6], q=[2,2,2], r=[4,4], cores ~N(0,0.3), B=8 bags of
     length U{1..4}, indices uniform, sum pooling, lr=0.1
2    p=[200,220,250], q=[4,4,4], r=[32,32], cores ~N(0,0.1), B=512 bags
     of exactly 20 lookups, indices uniform, sum pooling, lr=0.1 (the
     FBTT README sample configuration)
3    same table as 2; B=4096 bags of length max(1, Poisson(20)); indices
     Zipf(1.05) over a random permutation of [0,E); weights U(0,1); mean
     pooling; a hot-row cache of the 110,000 lowest-Zipf-rank rows
4    p=[200,200,1000], q=[4,4,8], r=[64,64], cores ~N(0,0.05), B=65536
     bags of length max(1, Poisson(30)), indices Zipf(1.1) over a random
     permutation, sum pooling, lr=0.05
5    26 tables, E0 log-uniform in [1e3, 4e7], p1=p2=round(E0^(1/3)),
     p3=ceil(E0/(p1 p2)), q=[4,4,4], r1=r2 in {16,32,64}, cores
     ~N(0,0.1), B=32768 one-hot bags per table, indices Zipf(1.05) over a
     per-table permutation, sum pooling, lr=0.1
==== =================================================================

Every workload is drawn from ``numpy.random.default_rng(seed)`` (PCG64) in a
fixed order: table parameters, cores, bag lengths, indices, weights, then the
upstream gradient ``grad_out`` (N(0,1), one row per bag).

Layout conventions shared by both sides:

* core k of a table is a float32 array of shape ``[p_k, r_{k-1}, q_k, r_k]``
  (r_0 = r_3 = 1), C-contiguous, so one slice ``G_k[i_k]`` is contiguous;
* bags are CSR: ``offsets`` has ``num_bags + 1`` int64 entries, bag g holds
  ``indices[offsets[g]:offsets[g+1]]``;
* with several tables, bags are ordered table-major: bag ``g = t*B + b`` is
  sample b of table t, and its indices are row ids of table t.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

__all__ = [
    "TableSpec",
    "Workload",
    "zipf_ranks",
    "make_cores",
    "config",
    "CONFIG_NAMES",
]

CONFIG_NAMES = {
    1: "tiny p=[4,5,6] q=[2,2,2] r=[4,4] B=8",
    2: "11M x 64 rank-32 uniform, B=512 x 20 (nnz=10240), sum",
    3: "11M x 64 rank-32 Zipf(1.05), B=4096 x Poisson(20), weights, mean, hot-row cache",
    4: "40M x 128 rank-64 Zipf(1.1), B=65536 x Poisson(30), sum",
    5: "26 tables one-hot, E0 log-uniform [1e3,4e7], q=[4,4,4], r in {16,32,64}, B=32768",
}


@dataclasses.dataclass
class TableSpec:
    """Shape of one TT table: E rows, p/q factorisations and the two inner ranks."""

    num_embeddings: int
    p: List[int]
    q: List[int]
    ranks: List[int]

    @property
    def embedding_dim(self) -> int:
        return int(self.q[0] * self.q[1] * self.q[2])

    def core_shapes(self):
        r = [1, self.ranks[0], self.ranks[1], 1]
        return [(self.p[k], r[k], self.q[k], r[k + 1]) for k in range(3)]


@dataclasses.dataclass
class Workload:
    """One seeded workload: tables with their cores, the bags and grad_out."""

    name: str
    tables: List[TableSpec]
    cores: List[List[np.ndarray]]  # cores[t][k], float32
    indices: np.ndarray  # int64 [nnz]
    offsets: np.ndarray  # int64 [num_bags + 1]
    weights: Optional[np.ndarray]  # float32 [nnz] or None
    mode: str  # "sum" | "mean"
    lr: float
    batch: int  # B, bags per table
    grad_out: np.ndarray  # float32 [num_bags, D]
    cache_rows: Optional[np.ndarray] = None  # int64 rows of table 0 to cache

    @property
    def num_tables(self) -> int:
        return len(self.tables)

    @property
    def num_bags(self) -> int:
        return int(self.offsets.shape[0] - 1)

    @property
    def nnz(self) -> int:
        return int(self.indices.shape[0])

    @property
    def embedding_dim(self) -> int:
        return self.tables[0].embedding_dim


def zipf_ranks(rng: np.random.Generator, n: int, support: int, s: float) -> np.ndarray:
    """Draw ``n`` ranks k in [1, support] with P(k) proportional to k**-s.

    Rejection-inversion for monotone discrete distributions (Hoermann and
    Derflinger, 1996): with h(x) = x**-s and its antiderivative H, rank k owns
    the interval [H(k+1/2) - h(k), H(k+1/2)] of length h(k); the intervals are
    disjoint because h is convex.  A uniform u over [H(3/2) - h(1),
    H(support + 1/2)] is inverted, rounded to the nearest integer k, and kept
    iff it falls in k's interval.
    """
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    a = 1.0 - s

    def H(x):
        lx = np.log(x)
        return lx if a == 0.0 else np.expm1(a * lx) / a

    def Hinv(y):
        return np.exp(y) if a == 0.0 else np.exp(np.log1p(a * y) / a)

    lo = float(H(1.5)) - 1.0
    hi = float(H(support + 0.5))
    out = np.empty(n, dtype=np.int64)
    filled = 0
    while filled < n:
        m = max(1024, int((n - filled) * 1.25))
        u = lo + rng.random(m) * (hi - lo)
        x = Hinv(u)
        k = np.clip(np.floor(x + 0.5), 1, support)
        keep = u >= H(k + 0.5) - np.power(k, -s)
        k = k[keep].astype(np.int64)
        take = min(k.shape[0], n - filled)
        out[filled : filled + take] = k[:take]
        filled += take
    return out


def make_cores(rng: np.random.Generator, spec: TableSpec, sigma: float) -> List[np.ndarray]:
    """i.i.d. N(0, sigma) float32 cores in the [p_k, r_{k-1}, q_k, r_k] layout."""
    return [rng.normal(0.0, sigma, size=shape).astype(np.float32) for shape in spec.core_shapes()]


def _offsets_from_lengths(lengths: np.ndarray) -> np.ndarray:
    off = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return off


def _grad_out(rng, num_bags, dim):
    return rng.standard_normal((num_bags, dim), dtype=np.float32)


def config(cid: int, seed: int = 0, batch: Optional[int] = None) -> Workload:
    """Build workload ``cid`` (1..5).

    ``batch`` overrides B (bags per table) while keeping every distribution,
    table shape and value scale; it gives scaled-down cases of the large
    workloads that a float64 CPU oracle finishes in seconds.
    """
    rng = np.random.default_rng(seed)
    if cid == 1:
        spec = TableSpec(120, [4, 5, 6], [2, 2, 2], [4, 4])
        cores = make_cores(rng, spec, 0.3)
        B = batch or 8
        lengths = rng.integers(1, 5, size=B)
        idx = rng.integers(0, spec.num_embeddings, size=int(lengths.sum()), dtype=np.int64)
        return Workload(
            CONFIG_NAMES[1], [spec], [cores], idx, _offsets_from_lengths(lengths), None,
            "sum", 0.1, B, _grad_out(rng, B, spec.embedding_dim),
        )
    if cid == 2:
        spec = TableSpec(11_000_000, [200, 220, 250], [4, 4, 4], [32, 32])
        cores = make_cores(rng, spec, 0.1)
        B = batch or 512
        lengths = np.full(B, 20, dtype=np.int64)
        idx = rng.integers(0, spec.num_embeddings, size=int(lengths.sum()), dtype=np.int64)
        return Workload(
            CONFIG_NAMES[2], [spec], [cores], idx, _offsets_from_lengths(lengths), None,
            "sum", 0.1, B, _grad_out(rng, B, spec.embedding_dim),
        )
    if cid == 3:
        spec = TableSpec(11_000_000, [200, 220, 250], [4, 4, 4], [32, 32])
        cores = make_cores(rng, spec, 0.1)
        B = batch or 4096
        perm = rng.permutation(spec.num_embeddings).astype(np.int64)
        lengths = np.maximum(1, rng.poisson(20.0, size=B)).astype(np.int64)
        ranks = zipf_ranks(rng, int(lengths.sum()), spec.num_embeddings, 1.05)
        idx = perm[ranks - 1]
        w = rng.random(idx.shape[0], dtype=np.float32)
        hot = perm[:110_000].copy()
        return Workload(
            CONFIG_NAMES[3], [spec], [cores], idx, _offsets_from_lengths(lengths), w,
            "mean", 0.1, B, _grad_out(rng, B, spec.embedding_dim), cache_rows=hot,
        )
    if cid == 4:
        spec = TableSpec(40_000_000, [200, 200, 1000], [4, 4, 8], [64, 64])
        cores = make_cores(rng, spec, 0.05)
        B = batch or 65536
        perm = rng.permutation(spec.num_embeddings).astype(np.int64)
        lengths = np.maximum(1, rng.poisson(30.0, size=B)).astype(np.int64)
        ranks = zipf_ranks(rng, int(lengths.sum()), spec.num_embeddings, 1.1)
        idx = perm[ranks - 1]
        return Workload(
            CONFIG_NAMES[4], [spec], [cores], idx, _offsets_from_lengths(lengths), None,
            "sum", 0.05, B, _grad_out(rng, B, spec.embedding_dim),
        )
    if cid == 5:
        T = 26
        B = batch or 32768
        e0 = np.rint(np.exp(rng.uniform(math.log(1e3), math.log(4e7), size=T))).astype(np.int64)
        rank_choice = rng.choice(np.array([16, 32, 64]), size=T)
        specs, cores, parts = [], [], []
        for t in range(T):
            E = int(e0[t])
            p1 = int(round(E ** (1.0 / 3.0)))
            p3 = -(-E // (p1 * p1))
            r = int(rank_choice[t])
            spec = TableSpec(E, [p1, p1, p3], [4, 4, 4], [r, r])
            specs.append(spec)
            cores.append(make_cores(rng, spec, 0.1))
        for t in range(T):
            E = specs[t].num_embeddings
            perm = rng.permutation(E).astype(np.int64)
            parts.append(perm[zipf_ranks(rng, B, E, 1.05) - 1])
        idx = np.concatenate(parts)
        offsets = np.arange(T * B + 1, dtype=np.int64)
        return Workload(
            CONFIG_NAMES[5], specs, cores, idx, offsets, None, "sum", 0.1, B,
            _grad_out(rng, T * B, 64),
        )
    raise ValueError(f"unknown workload id {cid}")
