"""The split-K GEMM the library runs as its ordered-reduction example (test infrastructure).

Only the test suite may use this module; it shares no code with the CUDA path. What the
library computes is the plain definition C = A B^T (fp64 here), whatever the split of K:
the Pith review of "DASH: Deterministic Attention Scheduling for High-throughput
Reproducible LLM Training" (section "Where Pith is reading between the lines") lists
split-K GEMMs among the kernels its reduction-order principle applies to, and the split
only changes the order in which the partial sums over K are added.
"""
from __future__ import annotations

import numpy as np

__all__ = ["gemm_nt", "gemm_nt_split_partials"]


def gemm_nt(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C[m, n] = sum_k A[m, k] B[n, k], in fp64."""
    return np.asarray(a, dtype=np.float64) @ np.asarray(b, dtype=np.float64).T


def gemm_nt_split_partials(a: np.ndarray, b: np.ndarray, splits: int) -> list[np.ndarray]:
    """The per-chunk partials A[:, chunk] B[:, chunk]^T of an even split of K (fp64)."""
    k = a.shape[1]
    if k % splits:
        raise ValueError("K must split evenly")
    w = k // splits
    return [gemm_nt(a[:, s * w:(s + 1) * w], b[:, s * w:(s + 1) * w]) for s in range(splits)]
