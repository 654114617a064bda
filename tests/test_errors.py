"""Failure paths on the GPU, made on the host (no fault, trap or hang is ever caused):

* every ordered-reduction wait is bounded: with a skew on the awaited ordinals no wait
  can be satisfied, the kernel records DASH_ERR_SYNC_TIMEOUT and returns, and the context
  stays usable for a normal call right after;
* a schedule whose waits would form a cycle on the grid this GPU can hold is refused
  before anything is queued.
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


def test_deadlock_prone_grid_is_refused():
    # Shift with more KV tiles per head than the persistent grid holds: KV tile `grid` is
    # queued behind KV tile 0 on CTA 0, but KV_0's last reduction waits for it.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 8 * sms + 1
    B, S, H, D = 1, 128 * n, 1, 64
    q = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, S), dtype=torch.float32, device="cuda")
    ws = da.new_workspace(B, S, H, D, q.device)
    out = torch.empty_like(q)
    with pytest.raises(da.DashError) as ei:
        da.dash_attn_bwd(q, q, q, q, q, lse, out, out.clone(), out.clone(), ws, 0.1,
                         da.MASK_FULL, da.SCHED_SHIFT, 1)
    assert ei.value.status == da.DASH_ERR_DEADLOCK_RISK
