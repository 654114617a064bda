"""fp64 CPU oracle of softmax attention, forward and backward (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may use this
module. It imports nothing from the CUDA package.

What is computed
----------------
The pages ("DASH: Deterministic Attention Scheduling for High-throughput Reproducible
LLM Training": the Pith review, sections "The pith" and "Core claim", and the Figure 1
caption "Overview of the deterministic FlashAttention") describe the backward pass of
FlashAttention-3: each KV tile accumulates its dK/dV locally, and each dQ block is a sum
of per-KV-tile partials reduced in a fixed order. The schedule only reorders that work,
so the exact result is the plain attention gradient. The pages print no equations; this
file writes out the textbook definition, per (batch, head) slice, in float64:

    S    = scale * Q K^T                      (causal: S[i, j] = -inf for key j > query i)
    LSE  = log sum_j exp(S[i, j])              (natural log, one value per query row)
    P    = exp(S - LSE)
    O    = P V
    D    = rowsum(dO * O)
    dV   = P^T dO
    dP   = dO V^T
    dS   = P * (dP - D)
    dQ   = scale * dS K
    dK   = scale * dS^T Q

The causal mask is top-left aligned (query and key lengths are equal). Tensors use the
BSHD layout [batch, seqlen, heads, headdim]; LSE is [batch, heads, seqlen].

The backward takes O and LSE as inputs, so it can be fed either this module's own
forward (end-to-end parity) or the GPU forward's O/LSE (backward-only parity).

Query rows may be processed in blocks (``row_block``) so long sequences fit in memory.
That is a plain partition of the sum over query rows in dK = scale * sum_i dS[i]^T Q[i]
and dV = sum_i P[i]^T dO[i]; every row's own values do not depend on the partition.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "attn_fwd_slice",
    "attn_bwd_slice",
    "attn_fwd",
    "attn_bwd",
    "causal_mask",
]


def causal_mask(rows: np.ndarray, s: int) -> np.ndarray:
    """Boolean [len(rows), s]: True where query ``rows[r]`` may attend key ``j`` (j <= row)."""
    return np.arange(s)[None, :] <= rows[:, None]


def _scores(q_rows: np.ndarray, k: np.ndarray, scale: float, rows: np.ndarray, causal: bool) -> np.ndarray:
    """S = scale * Q K^T for the given query rows, with -inf where the causal mask forbids."""
    s = scale * (q_rows @ k.T)
    if causal:
        s = np.where(causal_mask(rows, k.shape[0]), s, -np.inf)
    return s


def attn_fwd_slice(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
                   row_block: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Forward for one (batch, head) slice. q, k, v: [s, d] float64. Returns O [s, d], LSE [s]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s_len = q.shape[0]
    rb = s_len if row_block is None else row_block
    o = np.empty_like(q)
    lse = np.empty(s_len, dtype=np.float64)
    for r0 in range(0, s_len, rb):
        rows = np.arange(r0, min(r0 + rb, s_len))
        sc = _scores(q[rows], k, scale, rows, causal)
        mx = sc.max(axis=1, keepdims=True)
        lse_blk = mx[:, 0] + np.log(np.exp(sc - mx).sum(axis=1))
        p = np.exp(sc - lse_blk[:, None])
        o[rows] = p @ v
        lse[rows] = lse_blk
    return o, lse


def attn_bwd_slice(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
                   lse: np.ndarray, scale: float, causal: bool,
                   row_block: int | None = None) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Backward for one (batch, head) slice.

    q, k, v, o, do: [s, d]; lse: [s]. P is recomputed from Q, K and the given LSE.
    Returns dQ, dK, dV as [s, d] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    s_len = q.shape[0]
    rb = s_len if row_block is None else row_block
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    d_row = (do * o).sum(axis=1)                      # D = rowsum(dO * O)
    for r0 in range(0, s_len, rb):
        rows = np.arange(r0, min(r0 + rb, s_len))
        sc = _scores(q[rows], k, scale, rows, causal)
        p = np.exp(sc - lse[rows][:, None])           # masked entries: exp(-inf) = 0
        dv += p.T @ do[rows]                          # dV = P^T dO
        dp = do[rows] @ v.T                           # dP = dO V^T
        ds = p * (dp - d_row[rows][:, None])          # dS = P * (dP - D)
        dq[rows] = scale * (ds @ k)                   # dQ = scale * dS K
        dk += scale * (ds.T @ q[rows])                # dK = scale * dS^T Q
    return dq, dk, dv


def _slices(x: np.ndarray):
    """Yield (b, h, x[b, :, h, :]) over a BSHD array."""
    for b in range(x.shape[0]):
        for h in range(x.shape[2]):
            yield b, h


def attn_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
             row_block: int | None = None, heads: list[tuple[int, int]] | None = None):
    """Forward over BSHD arrays [b, s, h, d]. Returns O (float64, BSHD) and LSE [b, h, s].

    ``heads`` restricts the work to the listed (b, h) slices; other entries are NaN.
    """
    bsz, s_len, nh, _ = q.shape
    o = np.full(q.shape, np.nan, dtype=np.float64)
    lse = np.full((bsz, nh, s_len), np.nan, dtype=np.float64)
    for b, h in (heads if heads is not None else list(_slices(q))):
        o[b, :, h, :], lse[b, h, :] = attn_fwd_slice(q[b, :, h, :], k[b, :, h, :], v[b, :, h, :],
                                                     scale, causal, row_block)
    return o, lse


def attn_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, do: np.ndarray,
             lse: np.ndarray, scale: float, causal: bool, row_block: int | None = None,
             heads: list[tuple[int, int]] | None = None):
    """Backward over BSHD arrays. lse is [b, h, s]. Returns dQ, dK, dV (float64, BSHD).

    ``heads`` restricts the work to the listed (b, h) slices; other entries are NaN.
    """
    dq = np.full(q.shape, np.nan, dtype=np.float64)
    dk = np.full(q.shape, np.nan, dtype=np.float64)
    dv = np.full(q.shape, np.nan, dtype=np.float64)
    for b, h in (heads if heads is not None else list(_slices(q))):
        dq[b, :, h, :], dk[b, :, h, :], dv[b, :, h, :] = attn_bwd_slice(
            q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], o[b, :, h, :], do[b, :, h, :],
            lse[b, h, :], scale, causal, row_block)
    return dq, dk, dv
