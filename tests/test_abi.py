"""The C ABI library loads, exports every function include/*.h declares, and rejects bad
arguments synchronously (no GPU needed: nothing reaches the device)."""
import ctypes
import glob
import json
import os
import re
import subprocess
import sys

import pytest

import reproducible_deterministic_attn_gb300 as da
from tests._lib import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(dash_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    return da.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    raw = ctypes.CDLL(da.dash_attn.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), name


def test_status_strings(lib):
    assert da.dash_status_string(0) == "DASH_OK"
    assert da.dash_status_string(5) == "DASH_ERR_SYNC_TIMEOUT"
    assert da.dash_status_string(6) == "DASH_ERR_DEADLOCK_RISK"
    assert da.dash_status_string(7) == "DASH_ERR_BOUNDS"
    assert da.dash_status_string(99) == "DASH_ERR_UNKNOWN"


def test_workspace_size(lib):
    B, S, H, D = 2, 256, 3, 64
    ws = da.dash_attn_bwd_workspace_size(B, S, H, D)
    # header, D and -LSE*log2e rows, the two score-offset block arrays (32 bytes per row
    # each), two fp32 dQ accumulator copies, one 128-byte line of semaphores per dQ block,
    # 256 x 4 split-tile flags and the split tiles' fp32 dK/dV partials (at most half the
    # B * H * S / 128 KV tiles, at most 256)
    splits = min(B * H * (S // 128) // 2, 256)
    need = (256 + 2 * B * H * S * 4 + 2 * B * H * S * 32 + 2 * B * H * S * D * 4
            + B * H * (S // 128) * 128 + 256 * 4 * 4 + splits * 2 * 128 * D * 4)
    assert need <= ws <= need + 8 * 256 and ws % 256 == 0
    assert da.dash_attn_bwd_workspace_size(1, 100, 1, 64) == 0      # S not a multiple of 128
    assert da.dash_attn_bwd_workspace_size(1, 128, 1, 96) == 0      # unsupported head dim


def _bwd(lib, **kw):
    a = dict(q=16, k=16, v=16, o=16, dO=16, lse=16, dq=16, dk=16, dv=16, ws=256, wsb=1 << 30,
             B=1, S=256, H=1, D=64, scale=0.125, mask=0, sched=0, det=1)
    a.update(kw)
    return lib.dash_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["dO"], a["lse"], a["dq"],
                             a["dk"], a["dv"], a["ws"], a["wsb"], a["B"], a["S"], a["H"],
                             a["D"], a["scale"], a["mask"], a["sched"], a["det"], None)


def test_bwd_rejects_bad_arguments_without_touching_the_device(lib):
    assert _bwd(lib, q=None) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, B=0) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, mask=2) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, sched=4) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, det=3) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, det=-1) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, scale=0.0) == da.DASH_ERR_INVALID_ARG
    assert _bwd(lib, D=96) == da.DASH_ERR_UNSUPPORTED
    assert _bwd(lib, S=200) == da.DASH_ERR_UNSUPPORTED
    assert _bwd(lib, q=17) == da.DASH_ERR_INVALID_ARG              # misaligned
    assert _bwd(lib, ws=128) == da.DASH_ERR_INVALID_ARG            # workspace not 256-aligned
    assert _bwd(lib, wsb=100) == da.DASH_ERR_WORKSPACE_TOO_SMALL
    assert _bwd(lib, sched=2, mask=1) == da.DASH_ERR_UNSUPPORTED   # shift needs the full mask
    assert _bwd(lib, sched=3, mask=0) == da.DASH_ERR_UNSUPPORTED   # symmetric shift: causal


def test_fwd_rejects_bad_arguments(lib):
    f = lib.dash_attn_fwd
    assert f(None, 16, 16, 16, 16, 1, 128, 1, 64, 0.1, 0, None) == da.DASH_ERR_INVALID_ARG
    assert f(16, 16, 16, 16, 16, 1, 128, 1, 32, 0.1, 0, None) == da.DASH_ERR_UNSUPPORTED
    assert f(16, 16, 16, 16, 16, 1, 128, 1, 64, 0.1, 7, None) == da.DASH_ERR_INVALID_ARG


def test_gemm_splitk_rejects_bad_arguments_without_touching_the_device(lib):
    f = lib.dash_gemm_splitk
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_size_t] + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    ws_need = da.dash_gemm_splitk_workspace_size(256, 256)
    assert ws_need == 256 + 4 * 4 or ws_need % 256 == 0
    def call(a=16, b=16, c=16, ws=256, wsb=1 << 20, M=256, N=256, K=512, splits=2, det=1):
        return f(a, b, c, ws, wsb, M, N, K, splits, det, None)
    assert call(a=None) == da.DASH_ERR_INVALID_ARG
    assert call(splits=0) == da.DASH_ERR_INVALID_ARG
    assert call(det=2) == da.DASH_ERR_INVALID_ARG
    assert call(ws=128) == da.DASH_ERR_INVALID_ARG                  # workspace not 256-aligned
    assert call(M=200) == da.DASH_ERR_UNSUPPORTED                   # M not a multiple of 128
    assert call(K=500) == da.DASH_ERR_UNSUPPORTED                   # K not 64 * splits aligned
    assert call(wsb=16) == da.DASH_ERR_WORKSPACE_TOO_SMALL
    assert da.dash_gemm_splitk_workspace_size(100, 128) == 0


def test_product_build_has_no_bounds_checks(lib):
    assert da.dash_bounds_checks_enabled() is False
    assert da.dash_debug_narrow_checks(1) == da.DASH_ERR_UNSUPPORTED


def test_checked_build_loads_and_exports_every_symbol():
    """The checked variant (compiled with DASH_BOUNDS_CHECKS=1) is selected by
    DASH_ATTN_BOUNDS_CHECKS=1, exports the same functions, reports itself and takes the
    narrowing hook; run in a child process because a process loads one library."""
    from reproducible_deterministic_attn_gb300 import build as _build

    _build.build(checks=True)
    script = (
        "import ctypes, json, sys; sys.path.insert(0, %r)\n"
        "import reproducible_deterministic_attn_gb300 as da\n"
        "from tests.test_abi import _declared\n"
        "raw = ctypes.CDLL(da.dash_attn.LIB_PATH)\n"
        "print(json.dumps({'path': da.dash_attn.LIB_PATH,\n"
        "  'missing': [n for n in _declared() if not hasattr(raw, n)],\n"
        "  'enabled': da.dash_bounds_checks_enabled(),\n"
        "  'neg': da.dash_debug_narrow_checks(-1), 'one': da.dash_debug_narrow_checks(1),\n"
        "  'zero': da.dash_debug_narrow_checks(0)}))\n" % ROOT)
    env = dict(os.environ, DASH_ATTN_BOUNDS_CHECKS="1")
    out = subprocess.run([sys.executable, "-c", script], env=env, cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    got = json.loads(out.stdout.strip().splitlines()[-1])
    assert got["path"].endswith("libdash_attn_checked.so")
    assert got["missing"] == []
    assert got["enabled"] is True
    assert (got["neg"], got["one"], got["zero"]) == (da.DASH_ERR_INVALID_ARG, da.DASH_OK, da.DASH_OK)
