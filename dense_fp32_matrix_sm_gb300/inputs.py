"""Seeded synthetic inputs for the SGEMM workloads, shared by the tests, the
bench and the oracle checks.

This module holds no GEMM arithmetic: it only draws matrices and picks which
output entries a large-size parity check samples.  Generator: numpy's PCG64
(``np.random.default_rng(seed)``), drawing A, then B, then C0, each directly
in float32, so the bytes are the same on every platform.

Workloads (the pages time square FP32 problems on uniform[-1, 1] inputs --
"Writing a Fast Matmul in CUDA, Step by Step", Step 1 -- at 4096 and 4092;
the MLP- and decode-shaped rows follow the transformer uses those pages
name):

  square128    128 x 128 x 128,       A,B ~ U[-1,1],             seed 0, alpha 1,   beta 0
  square4096   4096 x 4096 x 4096,    A,B ~ U[-1,1],             seed 1, alpha 1,   beta 0
  square4092   4092 x 4092 x 4092,    A,B ~ N(0,1), C0 ~ U[-1,1], seed 2, alpha 0.5, beta 3
  mlp          8192 x 14336 x 4096,   A ~ N(0,1), B ~ N(0,0.02),  seed 3, alpha 1,   beta 0
  decode16     16 x 16384 x 8192,     A ~ N(0,1), B ~ N(0,0.02), C0 ~ U[-1,1], seed 4, alpha 1, beta 1

Two more measured beside them: decode1 (the one-token case of decode16:
1 x 16384 x 8192, same distributions, seed 5) and square512 (512^3,
A,B ~ U[-1,1], seed 6: a small problem between 128^3 and 4096^3, where a
partial wave decides the speed -- "Writing a Fast Matmul in CUDA", "Size
effects").
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist_a: Tuple[str, float]      # ("uniform", half-width) or ("normal", sigma)
    dist_b: Tuple[str, float]
    dist_c: Optional[Tuple[str, float]]  # None: C starts zeroed and beta == 0
    seed: int
    alpha: float
    beta: float

    @property
    def flops(self) -> int:
        """2*M*N*K: one multiply and one add per inner step (epilogue not counted)."""
        return 2 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """A and B read once, C written once, plus C read once when beta != 0."""
        c_passes = 2 if self.beta != 0.0 else 1
        return 4 * (self.M * self.K + self.K * self.N + c_passes * self.M * self.N)

    def describe(self) -> str:
        def d(x):
            if x is None:
                return "zero"
            kind, p = x
            return f"U[-{p:g},{p:g}]" if kind == "uniform" else f"N(0,{p:g})"
        return (f"sgemm {self.M}x{self.N}x{self.K} fp32 row-major alpha={self.alpha:g} beta={self.beta:g} "
                f"A~{d(self.dist_a)} B~{d(self.dist_b)} C0~{d(self.dist_c)} seed={self.seed}")


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("square128", 128, 128, 128, ("uniform", 1.0), ("uniform", 1.0), None, 0, 1.0, 0.0),
        Workload("square4096", 4096, 4096, 4096, ("uniform", 1.0), ("uniform", 1.0), None, 1, 1.0, 0.0),
        Workload("square4092", 4092, 4092, 4092, ("normal", 1.0), ("normal", 1.0), ("uniform", 1.0), 2,
                 0.5, 3.0),
        Workload("mlp", 8192, 14336, 4096, ("normal", 1.0), ("normal", 0.02), None, 3, 1.0, 0.0),
        Workload("decode16", 16, 16384, 8192, ("normal", 1.0), ("normal", 0.02), ("uniform", 1.0), 4,
                 1.0, 1.0),
        Workload("decode1", 1, 16384, 8192, ("normal", 1.0), ("normal", 0.02), ("uniform", 1.0), 5,
                 1.0, 1.0),
        Workload("square512", 512, 512, 512, ("uniform", 1.0), ("uniform", 1.0), None, 6, 1.0, 0.0),
    )
}


def _draw(rng: np.random.Generator, shape, dist) -> np.ndarray:
    kind, p = dist
    if kind == "uniform":
        # 24-bit float32 draws in [0, 1); 2r - 1 is exact in float32.
        x = rng.random(shape, dtype=np.float32)
        x *= np.float32(2.0)
        x -= np.float32(1.0)
        if p != 1.0:
            x *= np.float32(p)
        return x
    if kind == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
        if p != 1.0:
            x *= np.float32(p)
        return x
    if kind == "int":
        # integers in [-p, p]: every product and partial sum is exact in fp32 for small K
        return rng.integers(-int(p), int(p) + 1, size=shape).astype(np.float32)
    raise ValueError(f"unknown distribution {kind}")


def make_inputs(M: int, N: int, K: int, seed: int, dist_a=("uniform", 1.0), dist_b=("uniform", 1.0),
                dist_c=("uniform", 1.0)):
    """Draw (A, B, C0) as C-contiguous float32 arrays: A is M x K, B is K x N, C0 is M x N.

    dist_c None gives a zero C0.  The draw order (A, B, C0) is fixed, so a
    seed names one set of inputs.
    """
    rng = np.random.default_rng(seed)
    A = _draw(rng, (M, K), dist_a)
    B = _draw(rng, (K, N), dist_b)
    C0 = np.zeros((M, N), dtype=np.float32) if dist_c is None else _draw(rng, (M, N), dist_c)
    return A, B, C0


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.N, w.K, w.seed, w.dist_a, w.dist_b, w.dist_c)


def sample_entries(M: int, N: int, n: int, seed: int, tile_m: int = 128, tile_n: int = 128):
    """Output positions a large-size parity check compares.

    n uniform (i, j) draws from PCG64(seed + 1000), plus, always: the four
    corners, the whole last row and last column (in up to 4096 steps each),
    and one position inside every edge tile of a tile_m x tile_n grid, so
    ragged-tail bugs cannot hide between samples.  Returns (rows, cols) as
    int64 arrays without duplicates.
    """
    if M == 0 or N == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    rng = np.random.default_rng(seed + 1000)
    rows = [rng.integers(0, M, size=n, dtype=np.int64)]
    cols = [rng.integers(0, N, size=n, dtype=np.int64)]
    corners_r = np.array([0, 0, M - 1, M - 1], dtype=np.int64)
    corners_c = np.array([0, N - 1, 0, N - 1], dtype=np.int64)
    rows.append(corners_r)
    cols.append(corners_c)
    step_n = max(1, N // 4096)
    jj = np.arange(0, N, step_n, dtype=np.int64)
    rows.append(np.full(jj.size, M - 1, dtype=np.int64))
    cols.append(jj)
    step_m = max(1, M // 4096)
    ii = np.arange(0, M, step_m, dtype=np.int64)
    rows.append(ii)
    cols.append(np.full(ii.size, N - 1, dtype=np.int64))
    # one entry per tile in the last tile-row and the last tile-column
    tm = (M + tile_m - 1) // tile_m
    tn = (N + tile_n - 1) // tile_n
    for t in range(tn):
        rows.append(np.array([min(M - 1, (tm - 1) * tile_m + rng.integers(0, tile_m))], np.int64))
        cols.append(np.array([min(N - 1, t * tile_n + rng.integers(0, tile_n))], np.int64))
    for t in range(tm):
        rows.append(np.array([min(M - 1, t * tile_m + rng.integers(0, tile_m))], np.int64))
        cols.append(np.array([min(N - 1, (tn - 1) * tile_n + rng.integers(0, tile_n))], np.int64))
    r = np.concatenate(rows)
    c = np.concatenate(cols)
    key = np.unique(r * N + c)
    return key // N, key % N


def _sample_line(L: int, n: int, rng: np.random.Generator, tile: int) -> np.ndarray:
    """Up to n distinct indices in [0, L): both ends, one inside every tile
    of size `tile` (evenly thinned if there are more tiles than n/2), the
    rest uniform."""
    if n >= L:
        return np.arange(L, dtype=np.int64)
    picks = {0, L - 1}
    if L > 2:
        picks.add(L - 2)
    tiles = (L + tile - 1) // tile
    chosen = range(tiles) if tiles <= n // 2 else np.linspace(0, tiles - 1, n // 2).astype(int)
    for t in chosen:
        picks.add(int(min(L - 1, t * tile + rng.integers(0, tile))))
    while len(picks) < n:
        picks.update(int(x) for x in rng.integers(0, L, size=n - len(picks)))
    return np.array(sorted(picks)[:n] if len(picks) > n else sorted(picks), dtype=np.int64)


def sample_rows_cols(M: int, N: int, n_rows: int = 256, n_cols: int = 256, seed: int = 0,
                     tile_m: int = 128, tile_n: int = 128):
    """Row and column index sets whose cross product is a large-size parity
    sample (256 x 256 = 65,536 entries by default).  Both ends and one index
    inside every edge tile are always present.  Every entry (i, j) depends
    only on row i of A and column j of B, so the oracle can compute the whole
    sample as one small product A[rows] x B[:, cols]."""
    rng = np.random.default_rng(seed + 1000)
    if M <= n_rows:
        n_cols = max(n_cols, (n_rows * n_cols) // max(1, M))
    return _sample_line(M, n_rows, rng, tile_m), _sample_line(N, n_cols, rng, tile_n)
