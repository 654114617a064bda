"""The allocation-free backward (dash_attn_bwd_static) against the regular one.

Some callers cannot allocate device memory when they run the backward (a runtime that
reserves all device memory for its own pool, code that must not enter the CUDA
allocator); dash_attn_bwd_static serves them from a fixed array in the library's device
image. This file is collected last on purpose: the entry point's first call on a device
sets up the array's address, and the test must pass both in a fresh process and after
every other test has run.
"""
import ctypes
import math

import pytest
import torch

import reproducible_deterministic_attn_gb300 as da
from reproducible_deterministic_attn_gb300.inputs import make_inputs
from tests._lib import ensure_built, has_gpu
from tests.gpu_common import REL_TOL

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


CASES = [
    # (B, S, H, D, causal, schedule, deterministic) -- all fit the 64 MiB static scratch
    (1, 1024, 4, 128, False, "shift", 1),
    (2, 512, 3, 64, True, "symmetric_shift", 1),
    (1, 768, 2, 128, True, "descending", 0),
    # 160 units on a 152-SM grid: full shift splits the last round's 8 KV tiles over two
    # CTAs each; causal symmetric shift at head dim 64 deals KV-tile pieces longest first
    (1, 2048, 10, 128, False, "shift", 2),
    (5, 1024, 8, 64, True, "symmetric_shift", 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_static_matches_regular_on_two_calls_in_a_row(case):
    B, S, H, D, causal, sched, det = case
    x = make_inputs(B, S, H, D, seed=4)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(D)
    mask = da.MASK_CAUSAL if causal else da.MASK_FULL
    o, lse = da.attn_forward(q, k, v, scale, causal)
    ref = da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lib = da.load()
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = lib.dash_attn_bwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                      dk.data_ptr(), dv.data_ptr(), status.data_ptr(),
                                      B, S, H, D, ctypes.c_float(scale), mask,
                                      da.SCHEDULES[sched], det,
                                      torch.cuda.current_stream().cuda_stream)
        assert st == da.DASH_OK, da.dash_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert not torch.isnan(got).any(), (call, name)
            assert _rel(got, want) <= REL_TOL, (call, name, _rel(got, want))
            if det:
                # same kernels and the same fixed order: the bits agree too
                assert torch.equal(got, want), (call, name)


def _static_call(lib, t, status, B, S, H, D, mask, sched, det):
    q, k, v, o, do, lse, dq, dk, dv = t
    return lib.dash_attn_bwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), status.data_ptr(), B, S, H, D,
                                    ctypes.c_float(1.0 / math.sqrt(D)), mask, sched, det,
                                    torch.cuda.current_stream().cuda_stream)


def _buffers(B, S, H, D):
    """Inputs and sentinel-filled outputs of the full claimed size, so that no refusal
    test could read or write out of bounds even if the call went ahead."""
    def bf():
        return torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, S), dtype=torch.float32, device="cuda")
    outs = [torch.full((B, S, H, D), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    return [bf(), bf(), bf(), bf(), bf(), lse] + outs


@pytest.mark.parametrize("refusal", ["beyond_scratch", "unsupported_pair"])
def test_static_refusal_queues_nothing(refusal):
    """A refused call returns its error before anything is queued: the outputs and the
    status word keep the values they had."""
    if refusal == "beyond_scratch":
        B, S, H, D, mask, sched = 2, 8192, 16, 128, da.MASK_FULL, da.SCHEDULES["shift"]
        want = da.DASH_ERR_WORKSPACE_TOO_SMALL
    else:
        B, S, H, D, mask, sched = 1, 256, 2, 64, da.MASK_CAUSAL, da.SCHEDULES["shift"]
        want = da.DASH_ERR_UNSUPPORTED
    t = _buffers(B, S, H, D)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    lib = da.load()
    st = _static_call(lib, t, status, B, S, H, D, mask, sched, 1)
    assert st == want
    if refusal == "beyond_scratch":
        assert "static scratch" in da.dash_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == 12345
    for out in t[6:]:
        assert bool((out == 7.0).all())
