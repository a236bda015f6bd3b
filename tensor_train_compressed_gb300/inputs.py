"""Seeded synthetic inputs for the TT embedding-bag workloads.

This module draws random numbers and nothing else: TT cores, row indices,
bag offsets and output gradients.  It holds none of the method's arithmetic
(no index decomposition, no contraction, no pooling), so both the CPU oracle
and the CUDA path can be fed from it without sharing any computation.

Workloads (the five synthetic configurations of the TT embedding-bag
benchmark; the pages' own Meta-240/480/788 workloads are not described and
these stand in for them):

  1  1000 rows = 10x10x10, D=16 = 2x4x2, R1=R2=4, 64 bags of length U{1..4},
     indices uniform over rows, forward.
  2  1e6 rows = 100^3, D=64 = 4x4x4, R1=R2=16, 4096 bags of length 1,
     indices Zipf(1.05) over a seeded random row permutation, forward.
  3  12e6 rows = 200x240x250, D=128 = 4x8x4, R1=R2=32, 32768 bags of
     length 20, indices Zipf(1.2) (rank k -> row k-1), forward.
  4  8 tables, N = 1e5, 1e6, 4e6, 1e7, 2e7, 3e7, 4e7, 4e7 rows, each
     factored into three near-equal m_k, D=128 = 4x8x4, R1=R2=64, 32768 bags
     per table of length max(Poisson(20), 1), indices Zipf(1.4), forward.
  5  48e6 rows = 360x360x370 (47,952,000), D=128 = 4x8x4, R1=R2=32, 32768
     bags of length U{10..30}, indices Zipf(1.2), forward + backward with
     grad_out ~ N(0,1) + SGD at lr = 0.01.

Core layout: G_k is float32, contiguous [m_k][R_{k-1}][n_k][R_k] with
R_0 = R_3 = 1; every core is drawn i.i.d. N(0, s^2) with s = 1/sqrt(R1).
Seeds: cores 1000*cfg + table, indices/offsets 2000*cfg + table,
grad_out 3000*cfg + table.
"""
from __future__ import annotations

import functools
import math
from dataclasses import dataclass, field

import numpy as np

__all__ = ["CONFIGS", "TTInputs", "make_inputs", "factor3", "zipf_cdf"]


def factor3(N: int) -> tuple[int, int, int]:
    """Three near-equal row factors with product >= N.

    Start from c = ceil(N^(1/3)) for every factor, then for k = 3, 2, 1 lower
    m_k while the product stays >= N.
    """
    c = max(1, int(math.ceil(round(N ** (1.0 / 3.0), 9))))
    while c ** 3 < N:
        c += 1
    m = [c, c, c]
    for k in (2, 1, 0):
        while m[k] > 1:
            m[k] -= 1
            if m[0] * m[1] * m[2] < N:
                m[k] += 1
                break
    return tuple(m)


CONFIGS: dict[int, dict] = {
    1: dict(name="tiny 1000x16 R4", tables=[(10, 10, 10)], N=[1000], n=(2, 4, 2), R=4,
            B=64, bag=("uniform", 1, 4), dist=("uniform",), train=False),
    2: dict(name="1M-row gather D64 R16", tables=[(100, 100, 100)], N=[1_000_000], n=(4, 4, 4),
            R=16, B=4096, bag=("fixed", 1), dist=("zipf", 1.05, "permuted"), train=False),
    3: dict(name="12M-row bag D128 R32 batch 32768", tables=[(200, 240, 250)], N=[12_000_000],
            n=(4, 8, 4), R=32, B=32768, bag=("fixed", 20), dist=("zipf", 1.2, "identity"),
            train=False),
    4: dict(name="8 tables D128 R64 batch 32768",
            tables=[factor3(N) for N in (100_000, 1_000_000, 4_000_000, 10_000_000,
                                         20_000_000, 30_000_000, 40_000_000, 40_000_000)],
            N=[100_000, 1_000_000, 4_000_000, 10_000_000, 20_000_000, 30_000_000,
               40_000_000, 40_000_000],
            n=(4, 8, 4), R=64, B=32768, bag=("poisson", 20), dist=("zipf", 1.4, "identity"),
            train=False),
    5: dict(name="48M-row training step D128 R32 batch 32768", tables=[(360, 360, 370)],
            N=[360 * 360 * 370], n=(4, 8, 4), R=32, B=32768, bag=("uniform", 10, 30),
            dist=("zipf", 1.2, "identity"), train=True, lr=0.01),
}


@functools.lru_cache(maxsize=4)
def zipf_cdf(N: int, alpha: float) -> np.ndarray:
    """Unnormalised cumulative weights of P(rank k) ~ k^-alpha, k = 1..N (float64)."""
    w = np.arange(1, N + 1, dtype=np.float64)
    np.power(w, -alpha, out=w)
    np.cumsum(w, out=w)
    return w


@dataclass
class TTInputs:
    m: tuple
    n: tuple
    R: tuple                     # (1, R1, R2, 1)
    cores: list                  # [G1, G2, G3] float32, [m_k][R_{k-1}][n_k][R_k]
    indices: np.ndarray          # int64 [nnz]
    offsets: np.ndarray          # int64 [B+1], CSR
    grad_out: np.ndarray | None = None   # float32 [B][D] (training only)
    N: int = 0                   # rows the indices are drawn over (<= prod(m))
    cfg: int = 0
    table: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def D(self) -> int:
        return int(np.prod(self.n))

    @property
    def nnz(self) -> int:
        return int(self.indices.shape[0])

    @property
    def num_bags(self) -> int:
        return int(self.offsets.shape[0] - 1)


def _bag_lengths(rng: np.random.Generator, spec: tuple, B: int) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        return np.full(B, spec[1], dtype=np.int64)
    if kind == "uniform":          # inclusive integer range
        return rng.integers(spec[1], spec[2] + 1, size=B, dtype=np.int64)
    if kind == "poisson":
        return np.maximum(rng.poisson(spec[1], size=B).astype(np.int64), 1)
    raise ValueError(kind)


def _draw_rows(rng: np.random.Generator, spec: tuple, N: int, nnz: int) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(0, N, size=nnz, dtype=np.int64)
    if kind == "zipf":
        alpha, mapping = spec[1], spec[2]
        cdf = zipf_cdf(N, alpha)
        u = rng.random(nnz) * cdf[-1]
        rank0 = np.searchsorted(cdf, u, side="right").astype(np.int64)   # rank - 1
        np.minimum(rank0, N - 1, out=rank0)
        if mapping == "permuted":
            perm = rng.permutation(N).astype(np.int64)
            return perm[rank0]
        return rank0
    raise ValueError(kind)


def make_cores(m, n, R, seed: int, std: float) -> list:
    """Seeded Gaussian cores [m_k][R_k][n_k][R_{k+1}] of a chain of len(m) cores
    (R: the len(m) + 1 ranks, or one inner rank for three cores)."""
    rng = np.random.default_rng(seed)
    d = len(m)
    Rf = tuple(R) if not np.isscalar(R) else (1, R, R, 1)
    assert len(Rf) == d + 1
    shapes = [(m[k], Rf[k], n[k], Rf[k + 1]) for k in range(d)]
    return [(rng.standard_normal(s, dtype=np.float32) * np.float32(std)).astype(np.float32)
            for s in shapes]


def make_inputs(cfg: int, table: int = 0, num_bags: int | None = None,
                with_grad: bool | None = None, mapping: str | None = None) -> TTInputs:
    """Seeded inputs of workload ``cfg`` (table ``table``).

    ``num_bags`` overrides the batch size (a draw of that many bags from the
    workload's seed: a different draw from the full batch's, not its first
    bags; used for reduced-size parity cases).  ``mapping`` overrides how Zipf
    ranks become rows: "identity" (rank k -> row k - 1) or "permuted" (through a
    seeded random permutation of the rows), the sensitivity variant.
    """
    c = CONFIGS[cfg]
    m = tuple(int(v) for v in c["tables"][table])
    N = int(c["N"][table])
    n = tuple(int(v) for v in c["n"])
    R = (1, int(c["R"]), int(c["R"]), 1)
    cores = make_cores(m, n, R, seed=1000 * cfg + table, std=1.0 / math.sqrt(c["R"]))
    B = int(c["B"] if num_bags is None else num_bags)
    rng = np.random.default_rng(2000 * cfg + table)
    lengths = _bag_lengths(rng, c["bag"], B)
    offsets = np.zeros(B + 1, dtype=np.int64)
    np.cumsum(lengths, out=offsets[1:])
    nnz = int(offsets[-1])
    dist = c["dist"]
    if mapping is not None and dist[0] == "zipf":
        dist = (dist[0], dist[1], mapping)
    indices = _draw_rows(rng, dist, N, nnz)
    grad = None
    if with_grad if with_grad is not None else c.get("train", False):
        g = np.random.default_rng(3000 * cfg + table)
        grad = g.standard_normal((B, n[0] * n[1] * n[2]), dtype=np.float32)
    return TTInputs(m=m, n=n, R=R, cores=cores, indices=indices, offsets=offsets,
                    grad_out=grad, N=N, cfg=cfg, table=table)


def make_custom(m, n, R, num_bags: int, max_len: int, seed: int, dist=("uniform",),
                std: float = 0.5, with_grad: bool = True, empty_frac: float = 0.0) -> TTInputs:
    """Seeded inputs of an arbitrary shape (edge cases, ragged tails, tiny pins); any number
    of cores (len(m) = len(n) = len(R) - 1)."""
    m = tuple(int(v) for v in m)
    n = tuple(int(v) for v in n)
    R = tuple(int(v) for v in R)
    cores = make_cores(m, n, R, seed=seed, std=std)
    rng = np.random.default_rng(seed + 1)
    lengths = rng.integers(1, max_len + 1, size=num_bags, dtype=np.int64) if max_len > 0 \
        else np.zeros(num_bags, dtype=np.int64)
    if empty_frac > 0:
        lengths[rng.random(num_bags) < empty_frac] = 0
    offsets = np.zeros(num_bags + 1, dtype=np.int64)
    np.cumsum(lengths, out=offsets[1:])
    M = int(np.prod(m))
    indices = _draw_rows(rng, dist, M, int(offsets[-1]))
    grad = None
    if with_grad:
        grad = np.random.default_rng(seed + 2).standard_normal(
            (num_bags, int(np.prod(n))), dtype=np.float32)
    return TTInputs(m=m, n=n, R=R, cores=cores, indices=indices, offsets=offsets,
                    grad_out=grad, N=M)


def make_sample_weights(nnz: int, seed: int, low: float = 0.0, high: float = 2.0) -> np.ndarray:
    """Seeded per-sample weights of the weighted-sum pooling: float32 [nnz], uniform on
    [low, high)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(low, high, size=int(nnz)).astype(np.float32)
