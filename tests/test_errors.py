"""Failure paths on the GPU, made on the host (no fault, trap or hang is ever caused):

* every ordered-reduction wait is bounded: with a skew on the awaited ordinals no wait
  can be satisfied, the kernel records DASH_ERR_SYNC_TIMEOUT and returns, and the context
  stays usable for a normal call right after;
* the forward's waits are bounded the same way, and its status word reports a wait that
  ran out (the testing hook withholds the K/V tiles);
* a head spread over many rounds of the persistent grid -- where a fixed per-schedule
  dQ order would wait on itself -- runs to the end, because shift's order is the order
  of arrival on the dealt grid.
"""
import math

import pytest
import torch

import reproducible_deterministic_attn_gb300 as da
from reproducible_deterministic_attn_gb300.inputs import make_inputs
from tests._lib import ensure_built, has_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("D,det", [(64, 1), (128, 1), (128, 2)])
def test_sync_timeout_is_reported_and_context_survives(D, det):
    B, S, H = 1, 512, 2
    x = make_inputs(B, S, H, D, 3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(D)
    o, lse = da.attn_forward(q, k, v, scale, False)
    ref = da.attn_backward(q, k, v, o, do, lse, scale, False, "shift", det)
    ws = da.new_workspace(B, S, H, D, q.device)
    try:
        da.dash_debug_set_sync(50_000_000, 1)          # 50 ms per wait, unreachable ordinals
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        da.dash_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, da.MASK_FULL,
                         da.SCHED_SHIFT, det)
        st = da.dash_attn_get_status(ws)
        assert st == da.DASH_ERR_SYNC_TIMEOUT
        assert "timed out" in da.dash_last_error()
    finally:
        da.dash_debug_set_sync(0, 0)
    again = da.attn_backward(q, k, v, o, do, lse, scale, False, "shift", det, workspace=ws)
    for a, b in zip(again, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("D", [64, 128])
def test_forward_timeout_is_reported_and_context_survives(D):
    """The forward's waits are bounded too: with the K/V tiles withheld (the testing hook)
    every wait for them runs out, the status word says so and the LSE rows are NaN; the
    next call, without the hook, computes the normal result."""
    B, S, H = 1, 512, 2
    x = make_inputs(B, S, H, D, 5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = 1 / math.sqrt(D)
    o_ref, lse_ref = da.attn_forward(q, k, v, scale, True)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    o, lse = torch.empty_like(q), torch.empty_like(lse_ref)
    try:
        da.dash_debug_set_sync(50_000_000, 1)          # 50 ms per wait, K/V withheld
        da.dash_attn_fwd_ex(q, k, v, o, lse, scale, da.MASK_CAUSAL, status)
        torch.cuda.synchronize()
        assert int(status.item()) == da.DASH_ERR_SYNC_TIMEOUT
        assert bool(torch.isnan(lse).all())
    finally:
        da.dash_debug_set_sync(0, 0)
    da.dash_attn_fwd_ex(q, k, v, o, lse, scale, da.MASK_CAUSAL, status)
    torch.cuda.synchronize()
    assert int(status.item()) == da.DASH_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_head_spread_over_many_rounds_of_the_grid_runs():
    # Shift with more KV tiles per head than the persistent grid holds: KV tile `grid` is
    # queued behind KV tile 0 on CTA 0. In the fixed step order KV_0's last reduction
    # would wait for it (a cycle); the order of arrival on the dealt grid puts it after,
    # so the ordered call runs to the end. All-zero inputs give exactly zero gradients
    # (P = 1, dO = 0: dV = P^T dO = 0, dP = 0 and D = 0, so dS = 0).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 8 * sms + 1
    B, S, H, D = 1, 128 * n, 1, 64
    q = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, S), dtype=torch.float32, device="cuda")
    ws = da.new_workspace(B, S, H, D, q.device)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    da.dash_attn_bwd(q, q, q, q, q, lse, dq, dk, dv, ws, 0.1, da.MASK_FULL, da.SCHED_SHIFT, 1)
    assert da.dash_attn_get_status(ws) == da.DASH_OK
    for t in (dq, dk, dv):
        assert int(torch.count_nonzero(t)) == 0
