"""Helpers for the GPU tests: run the library on seeded inputs and compare with the oracle."""
import math

import numpy as np
import torch

import reproducible_deterministic_attn_gb300 as da
from oracle.attention import attn_bwd, attn_fwd
from reproducible_deterministic_attn_gb300.inputs import make_inputs

# Tolerance of the backward (and forward O) against the fp64 oracle: per tensor,
# max |gpu - ref| <= REL_TOL * max |ref|. bf16 operands with fp32 accumulation; P and dS
# are rounded to bf16 before their contractions.
REL_TOL = 2e-2
LSE_ATOL = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def run_case(B, S, H, D, causal, schedule, deterministic, seed=0, device="cuda:0"):
    x = make_inputs(B, S, H, D, seed)
    q, k, v, do = (x[n].to(device) for n in ("q", "k", "v", "do"))
    return run_tensors(q, k, v, do, causal, schedule, deterministic)


def run_tensors(q, k, v, do, causal, schedule, deterministic):
    """Forward and backward on given BSHD bf16 device tensors, scale 1/sqrt(d)."""
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = da.attn_forward(q, k, v, scale, causal)
    dq, dk, dv = da.attn_backward(q, k, v, o, do, lse, scale, causal, schedule, deterministic)
    torch.cuda.synchronize()
    return dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, scale=scale)


def max_rel(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def check_against_oracle(res, causal, heads=None, row_block=1024):
    """Both parity modes on the listed (b, h) slices (all when None)."""
    q, k, v, do = (to64(res[n]) for n in ("q", "k", "v", "do"))
    o_gpu, lse_gpu = to64(res["o"]), res["lse"].cpu().double().numpy()
    scale = res["scale"]
    if heads is None:
        heads = [(b, h) for b in range(q.shape[0]) for h in range(q.shape[2])]
    sel = lambda a: np.stack([a[b, :, h] for b, h in heads])
    sel_l = lambda a: np.stack([a[b, h] for b, h in heads])
    # mode A: everything from Q, K, V, dO in fp64
    o_ref, lse_ref = attn_fwd(q, k, v, scale, causal, row_block, heads)
    dq_a, dk_a, dv_a = attn_bwd(q, k, v, o_ref, do, lse_ref, scale, causal, row_block, heads)
    # mode B: backward only, from the GPU forward's O and LSE
    dq_b, dk_b, dv_b = attn_bwd(q, k, v, o_gpu, do, lse_gpu, scale, causal, row_block, heads)
    errs = {
        "o": max_rel(sel(o_gpu), sel(o_ref)),
        "lse_abs": float(np.abs(sel_l(lse_gpu) - sel_l(lse_ref)).max()),
    }
    for name, ra, rb in (("dq", dq_a, dq_b), ("dk", dk_a, dk_b), ("dv", dv_a, dv_b)):
        g = sel(to64(res[name]))
        errs[name + "_A"] = max_rel(g, sel(ra))
        errs[name + "_B"] = max_rel(g, sel(rb))
    return errs


def assert_within(errs):
    for key, val in errs.items():
        lim = LSE_ATOL if key == "lse_abs" else REL_TOL
        assert val <= lim, (key, val, errs)
