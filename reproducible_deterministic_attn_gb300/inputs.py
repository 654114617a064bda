"""Seeded synthetic inputs for the attention backward (shared by the tests, the oracle
checks and the benchmark; holds none of the method's arithmetic).

The benchmark on the pages is FlashAttention-3's backward-throughput benchmark on BF16
random inputs. The stand-in here: Q, K, V and dO drawn N(0, 1) in float32 from
``torch.Generator().manual_seed(seed)``, in the fixed order q, k, v, dO, each of shape
[batch, seqlen, heads, headdim] (BSHD), then rounded to bfloat16 (round to nearest even).
"""

from __future__ import annotations

import torch

__all__ = ["make_inputs", "make_gemm_inputs"]


def make_inputs(b: int, s: int, h: int, d: int, seed: int = 0) -> dict[str, torch.Tensor]:
    """Return {'q', 'k', 'v', 'do'}: contiguous bf16 CPU tensors of shape [b, s, h, d]."""
    gen = torch.Generator().manual_seed(seed)
    out = {}
    for name in ("q", "k", "v", "do"):
        out[name] = torch.randn((b, s, h, d), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_gemm_inputs(m: int, n: int, k: int, seed: int = 0) -> dict[str, torch.Tensor]:
    """Return {'a': [m, k], 'b': [n, k]}: N(0, 1) drawn in float32 in the order a, b from
    ``torch.Generator().manual_seed(seed)``, rounded to contiguous bf16 CPU tensors."""
    gen = torch.Generator().manual_seed(seed)
    a = torch.randn((m, k), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    b = torch.randn((n, k), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return {"a": a, "b": b}

