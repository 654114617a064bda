"""The checked build on the GPU: libdash_attn_checked.so, whose backward checks every index
it reads from its schedule tables (a CTA's piece range, each piece, each task's tiles,
each dQ ordinal) before using it and records DASH_ERR_BOUNDS instead of going on.

* No false positives: on valid tables it runs clean and, in the deterministic modes,
  gives exactly the product build's bits (the checks change no arithmetic).
* The checks fire and are reported: the testing hook lowers only the bound the checks
  compare against (the kernel's own indexing is unchanged, so no access leaves its
  buffer), the call reports DASH_ERR_BOUNDS with the table, head, value and bound, and the
  next call without the hook computes the normal result.

A process loads one library, so the checked build runs in a child process.
"""
import hashlib
import json
import math
import os
import subprocess
import sys

import pytest
import torch

import reproducible_deterministic_attn_gb300 as da
from reproducible_deterministic_attn_gb300 import build as _build
from reproducible_deterministic_attn_gb300.inputs import make_inputs
from tests._lib import ensure_built, has_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (B, S, H, D), causal, schedule, deterministic (0 = unordered adds, 1 or 2 dQ chains)
CASES = [
    ((1, 512, 2, 64), False, "shift", 1),
    ((1, 512, 2, 64), True, "symmetric_shift", 2),
    ((1, 640, 2, 128), False, "ascending", 1),
    ((1, 512, 2, 128), True, "symmetric_shift", 2),
    ((1, 512, 2, 128), True, "descending", 1),
    ((1, 2048, 10, 128), False, "shift", 2),     # splits KV tiles on a 152-SM grid
    ((1, 512, 2, 128), False, "shift", 0),
]

CHILD = r"""
import hashlib, json, math, sys
sys.path.insert(0, ROOT)
import torch
import reproducible_deterministic_attn_gb300 as da
from reproducible_deterministic_attn_gb300.inputs import make_inputs
assert da.dash_bounds_checks_enabled()

def run(shape, causal, sched, det):
    B, S, H, D = shape
    x = make_inputs(B, S, H, D, 7)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(D)
    o, lse = da.attn_forward(q, k, v, scale, causal)
    return q, k, v, o, do, lse, scale

def digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.view(torch.int16).cpu().numpy().tobytes())
    return h.hexdigest()

out = {"clean": [], "narrowed": []}
for shape, causal, sched, det in CASES:
    q, k, v, o, do, lse, scale = run(shape, causal, sched, det)
    g = da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
    out["clean"].append(digest(g))
# the hook: the checks' tile bound one below the real one; short waits, should any wait
# be left to run out instead of seeing the failure
for shape, causal, sched, det in NARROW:
    q, k, v, o, do, lse, scale = run(shape, causal, sched, det)
    ref = da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
    da.dash_debug_set_sync(200_000_000, 0)
    assert da.dash_debug_narrow_checks(1) == da.DASH_OK
    try:
        da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
        status, msg = 0, ""
    except da.DashError as e:
        status, msg = e.status, str(e)
    finally:
        da.dash_debug_narrow_checks(0)
        da.dash_debug_set_sync(0, 0)
    again = da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
    same = all(torch.equal(a, b) for a, b in zip(again, ref)) if det else True
    out["narrowed"].append({"status": status, "msg": msg, "same_after": same})
print(json.dumps(out))
"""

NARROW = [
    ((1, 512, 2, 64), False, "shift", 1),
    ((1, 512, 2, 128), True, "symmetric_shift", 2),
    ((1, 512, 2, 128), False, "ascending", 0),
]


def _digest(ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.view(torch.int16).cpu().numpy().tobytes())
    return h.hexdigest()


@pytest.fixture(scope="module")
def checked_run():
    ensure_built()
    _build.build(checks=True)
    script = (f"ROOT = {ROOT!r}\nCASES = {CASES!r}\nNARROW = {NARROW!r}\n" + CHILD)
    env = dict(os.environ, DASH_ATTN_BOUNDS_CHECKS="1")
    res = subprocess.run([sys.executable, "-c", script], env=env, cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_checked_build_matches_the_product_build(checked_run):
    for (shape, causal, sched, det), got in zip(CASES, checked_run["clean"]):
        if not det:
            continue          # unordered adds: the bits may differ from run to run
        B, S, H, D = shape
        x = make_inputs(B, S, H, D, 7)
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        scale = 1 / math.sqrt(D)
        o, lse = da.attn_forward(q, k, v, scale, causal)
        ref = da.attn_backward(q, k, v, o, do, lse, scale, causal, sched, det)
        assert got == _digest(ref), (shape, causal, sched, det)


def test_failed_check_is_reported_and_context_survives(checked_run):
    for case, got in zip(NARROW, checked_run["narrowed"]):
        assert got["status"] == da.DASH_ERR_BOUNDS, (case, got)
        assert "bounds check failed" in got["msg"], (case, got)
        assert got["same_after"], (case, got)
