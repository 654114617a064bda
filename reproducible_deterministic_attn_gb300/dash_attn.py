"""Thin Python binding of libdash_attn (ctypes). Argument marshalling only: every step of
the attention forward/backward runs in the library's CUDA kernels.

The functions keep the C names. Tensors are torch CUDA tensors (BSHD bf16, LSE fp32
[B, H, S]); the stream defaults to torch's current stream on the tensors' device. A
status other than DASH_OK raises DashError. There is no CPU path: calling into the
library without the built shared object raises immediately.
"""

from __future__ import annotations

import ctypes
import os

import torch

MASK_FULL, MASK_CAUSAL = 0, 1
SCHED_ASCENDING, SCHED_DESCENDING, SCHED_SHIFT, SCHED_SYMMETRIC_SHIFT = 0, 1, 2, 3
SCHEDULES = {"ascending": 0, "descending": 1, "shift": 2, "symmetric_shift": 3}
MASKS = {"full": 0, "causal": 1}

DASH_OK = 0
DASH_ERR_INVALID_ARG = 1
DASH_ERR_UNSUPPORTED = 2
DASH_ERR_WORKSPACE_TOO_SMALL = 3
DASH_ERR_CUDA = 4
DASH_ERR_SYNC_TIMEOUT = 5
DASH_ERR_DEADLOCK_RISK = 6
DASH_ERR_BOUNDS = 7

# DASH_ATTN_BOUNDS_CHECKS=1 selects the checked build (device-side bounds checks on every
# schedule-table index the backward reads; build it with build(checks=True)).
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libdash_attn_checked.so" if os.environ.get("DASH_ATTN_BOUNDS_CHECKS") == "1"
                        else "libdash_attn.so")

_lib = None

_c_int, _c_float, _c_double, _c_size, _vp = (ctypes.c_int, ctypes.c_float, ctypes.c_double,
                                             ctypes.c_size_t, ctypes.c_void_p)
_i32p = ctypes.POINTER(ctypes.c_int32)
_dblp = ctypes.POINTER(ctypes.c_double)

_SIGNATURES = {
    "dash_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_float,
                               _c_int, _vp]),
    "dash_attn_fwd_ex": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                  _c_float, _c_int, _vp, _vp]),
    "dash_attn_bwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "dash_attn_bwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_size,
                               _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int, _c_int,
                               _vp]),
    "dash_attn_bwd_static": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_int,
                                      _c_int, _vp]),
    "dash_attn_get_status": (_c_int, [_vp, _vp]),
    "dash_status_string": (ctypes.c_char_p, [_c_int]),
    "dash_last_error": (ctypes.c_char_p, []),
    "dash_attn_shutdown": (None, []),
    "dash_debug_set_sync": (None, [ctypes.c_longlong, _c_int]),
    "dash_bounds_checks_enabled": (_c_int, []),
    "dash_debug_narrow_checks": (_c_int, [_c_int]),
    "dash_debug_set_trace": (None, [_vp]),
    "dash_profile_enable": (_c_int, [_c_int]),
    "dash_profile_read": (_c_int, [_dblp, ctypes.POINTER(_c_int)]),
    "dash_sched_num_slots": (_c_int, [_c_int, _c_int, _c_int]),
    "dash_sched_table": (_c_int, [_c_int, _c_int, _c_int, _i32p, _i32p, _c_int, _i32p]),
    "dash_sched_dealt_table": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _i32p]),
    "dash_sched_deal": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _i32p, _i32p,
                                 _c_int]),
    "dash_sched_simulate": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_double,
                                     _c_double, _dblp, _dblp]),
    "dash_sched_simulate_ex": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                        _c_double, _c_double, _c_double, _c_int, _dblp, _dblp]),
    "dash_sched_select": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_double, _c_double,
                                   _c_double, _c_int, ctypes.POINTER(_c_int), _dblp]),
    "dash_gemm_splitk_workspace_size": (ctypes.c_size_t, [_c_int, _c_int]),
    "dash_gemm_splitk": (_c_int, [_vp, _vp, _vp, _vp, ctypes.c_size_t, _c_int, _c_int, _c_int,
                                  _c_int, _c_int, _vp]),
}


class DashError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        name = lib.dash_status_string(status).decode()
        detail = lib.dash_last_error().decode()
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


def load():
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != DASH_OK:
        raise DashError(status, where)


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("expected BSHD tensors [batch, seqlen, heads, headdim]")
    return tuple(int(x) for x in q.shape)


def dash_attn_fwd(q, k, v, o, lse, scale: float, mask: int, stream=None) -> None:
    """O and LSE of softmax attention (writes into o and lse)."""
    B, S, H, D = _shape(q)
    _check(load().dash_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, S, H, D, float(scale), int(mask),
                                _stream(q, stream)), "dash_attn_fwd")


def dash_attn_fwd_ex(q, k, v, o, lse, scale: float, mask: int, status=None, stream=None) -> None:
    """dash_attn_fwd with a device status word (an int32 CUDA tensor of one element, or
    None): cleared by the call, set to DASH_ERR_SYNC_TIMEOUT by the kernel if a wait ran
    out."""
    B, S, H, D = _shape(q)
    _check(load().dash_attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, S, H, D, float(scale), int(mask),
                                   status.data_ptr() if status is not None else None,
                                   _stream(q, stream)), "dash_attn_fwd_ex")


def dash_attn_bwd_workspace_size(B: int, S: int, H: int, D: int) -> int:
    return int(load().dash_attn_bwd_workspace_size(B, S, H, D))


def dash_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, workspace, scale: float, mask: int,
                  schedule: int, deterministic: int, stream=None) -> None:
    """dQ, dK, dV (written into dq, dk, dv). workspace: a uint8 CUDA tensor."""
    B, S, H, D = _shape(q)
    _check(load().dash_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                dO.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                B, S, H, D, float(scale), int(mask), int(schedule),
                                int(deterministic), _stream(q, stream)), "dash_attn_bwd")


def dash_attn_bwd_static(q, k, v, o, dO, lse, dq, dk, dv, scale: float, mask: int,
                         schedule: int, deterministic: int, status_out=None, stream=None) -> None:
    """dash_attn_bwd without a workspace: the scratch is the library's static device array
    (no device allocation). status_out: optional int32 CUDA tensor for the status word."""
    B, S, H, D = _shape(q)
    _check(load().dash_attn_bwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       dO.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(),
                                       None if status_out is None else status_out.data_ptr(),
                                       B, S, H, D, float(scale), int(mask), int(schedule),
                                       int(deterministic), _stream(q, stream)),
           "dash_attn_bwd_static")


def dash_attn_get_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the status the last backward recorded."""
    return int(load().dash_attn_get_status(workspace.data_ptr(), _stream(workspace, stream)))


def dash_status_string(status: int) -> str:
    return load().dash_status_string(int(status)).decode()


def dash_last_error() -> str:
    return load().dash_last_error().decode()


def dash_attn_shutdown() -> None:
    load().dash_attn_shutdown()


def dash_debug_set_sync(timeout_ns: int, ordinal_skew: int) -> None:
    load().dash_debug_set_sync(int(timeout_ns), int(ordinal_skew))


def dash_bounds_checks_enabled() -> bool:
    """True when the loaded library is the checked build."""
    return bool(load().dash_bounds_checks_enabled())


def dash_debug_narrow_checks(tiles: int) -> int:
    """Checked build's testing hook: lower the checks' tile bound by `tiles` (0 restores it)."""
    return int(load().dash_debug_narrow_checks(int(tiles)))


# dash_debug_set_trace sites with a fixed meaning (include/dash_attn.h)
TRACE_SITES = 32
TRACE_DQ_TURN_WAIT = 15     # waiting for a dQ block's turn (ordered mode)
TRACE_DQ_ADD = 16           # adding a dQ partial and handing the turn on
TRACE_TOTAL = 19            # the CTA's total cycles


def dash_debug_set_trace(counters) -> None:
    """counters: a zeroed uint64 CUDA tensor of 32 * SM-count entries, or None to stop."""
    load().dash_debug_set_trace(None if counters is None else counters.data_ptr())


def dash_profile_enable(on: bool) -> None:
    _check(load().dash_profile_enable(int(bool(on))), "dash_profile_enable")


def dash_profile_read():
    """Returns (summed main-kernel milliseconds, launches) since the last read."""
    ms, cnt = ctypes.c_double(0.0), ctypes.c_int(0)
    _check(load().dash_profile_read(ctypes.byref(ms), ctypes.byref(cnt)), "dash_profile_read")
    return ms.value, cnt.value


def dash_sched_num_slots(mask: int, schedule: int, n: int) -> int:
    return int(load().dash_sched_num_slots(int(mask), int(schedule), int(n)))


def dash_sched_table(mask: int, schedule: int, n: int):
    """Returns (slot_offsets, tasks as (kv, q) pairs, ordinals n x n) or raises."""
    slots = dash_sched_num_slots(mask, schedule, n)
    if slots < 0:
        raise DashError(-slots, "dash_sched_table")
    cap = n * n
    off = (ctypes.c_int32 * (slots + 1))()
    tasks = (ctypes.c_int32 * cap)()
    ords = (ctypes.c_int32 * (n * n))()
    cnt = load().dash_sched_table(int(mask), int(schedule), int(n), off, tasks, cap, ords)
    if cnt < 0:
        raise DashError(-cnt, "dash_sched_table")
    pairs = [(tasks[k] >> 16, tasks[k] & 0xFFFF) for k in range(cnt)]
    return list(off), pairs, [list(ords[i * n:(i + 1) * n]) for i in range(n)]


def dash_sched_deal(mask: int, schedule: int, n: int, heads: int, grid: int,
                    head_dim: int = 128):
    """Each CTA's work in run order at head dimension `head_dim`: per CTA a list of
    (head, [(kv, q), ...], part, split) pieces (part 0: whole KV tiles; 1 / 2: first /
    second half of split tile `split`)."""
    _, pairs, _ = dash_sched_table(mask, schedule, n)
    slots = dash_sched_num_slots(mask, schedule, n)
    cap = 2 * heads * slots              # a chain has at most two KV tiles
    off = (ctypes.c_int32 * (grid + 1))()
    pieces = (ctypes.c_int32 * (5 * cap))()
    cnt = load().dash_sched_deal(int(mask), int(schedule), int(n), int(heads), int(grid),
                                 int(head_dim), off, pieces, cap)
    if cnt < 0:
        raise DashError(-cnt, "dash_sched_deal")
    return [[(pieces[5 * k], pairs[pieces[5 * k + 1]:pieces[5 * k + 2]], pieces[5 * k + 3],
              pieces[5 * k + 4]) for k in range(off[c], off[c + 1])] for c in range(grid)]


def dash_sched_dealt_table(mask: int, schedule: int, n: int, heads: int, grid: int,
                           head_dim: int = 128):
    """The dQ orders the backward follows on `grid` CTAs at head dimension `head_dim`:
    ords[h][i][j] (-1 = masked)."""
    ords = (ctypes.c_int32 * (heads * n * n))()
    _check(load().dash_sched_dealt_table(int(mask), int(schedule), int(n), int(heads),
                                         int(grid), int(head_dim), ords),
           "dash_sched_dealt_table")
    return [[list(ords[(h * n + i) * n:(h * n + i + 1) * n]) for i in range(n)]
            for h in range(heads)]


def dash_sched_simulate(mask: int, schedule: int, n: int, heads: int, num_sms: int,
                        c: float, r: float, head_dim: int = 128):
    """Returns (makespan, per-SM finish times), or (None, None) on a deadlock."""
    mk = ctypes.c_double(0.0)
    ends = (ctypes.c_double * num_sms)()
    st = load().dash_sched_simulate(int(mask), int(schedule), int(n), int(heads), int(num_sms),
                                    int(head_dim), float(c), float(r), ctypes.byref(mk), ends)
    if st == DASH_ERR_DEADLOCK_RISK:
        return None, None
    _check(st, "dash_sched_simulate")
    return mk.value, list(ends)


def dash_sched_simulate_ex(mask: int, schedule: int, n: int, heads: int, num_sms: int,
                           c: float, r: float, h: float, overlapped: int, head_dim: int = 128):
    """Returns (makespan, per-SM finish times), or (None, None) on a deadlock."""
    mk = ctypes.c_double(0.0)
    ends = (ctypes.c_double * num_sms)()
    st = load().dash_sched_simulate_ex(int(mask), int(schedule), int(n), int(heads),
                                       int(num_sms), int(head_dim), float(c), float(r),
                                       float(h), int(overlapped), ctypes.byref(mk), ends)
    if st == DASH_ERR_DEADLOCK_RISK:
        return None, None
    _check(st, "dash_sched_simulate_ex")
    return mk.value, list(ends)


def dash_sched_select(mask: int, n: int, heads: int, num_sms: int, c: float, r: float,
                      h: float, overlapped: int, head_dim: int = 128):
    """Returns (schedule, makespan) chosen by the library's cost model."""
    sched = _c_int(-1)
    mk = ctypes.c_double(0.0)
    st = load().dash_sched_select(int(mask), int(n), int(heads), int(num_sms), int(head_dim),
                                  float(c), float(r), float(h), int(overlapped),
                                  ctypes.byref(sched), ctypes.byref(mk))
    _check(st, "dash_sched_select")
    return sched.value, mk.value


def dash_gemm_splitk_workspace_size(M: int, N: int) -> int:
    return int(load().dash_gemm_splitk_workspace_size(int(M), int(N)))


def dash_gemm_splitk(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor, workspace: torch.Tensor,
                     splits: int, deterministic: int, stream=None) -> None:
    """C = A B^T (a: bf16 [M, K], b: bf16 [N, K], c: fp32 [M, N]), K in `splits` chunks."""
    M, K = a.shape
    N = b.shape[0]
    _check(load().dash_gemm_splitk(a.data_ptr(), b.data_ptr(), c.data_ptr(), workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), int(M), int(N),
                                   int(K), int(splits), int(deterministic), _stream(a, stream)),
           "dash_gemm_splitk")


def gemm_splitk(a: torch.Tensor, b: torch.Tensor, splits: int, deterministic: int = 1,
                workspace=None, stream=None, check: bool = True) -> torch.Tensor:
    """Allocates C (and a workspace if none is given) and runs dash_gemm_splitk."""
    M, N = a.shape[0], b.shape[0]
    if workspace is None:
        workspace = torch.empty(dash_gemm_splitk_workspace_size(M, N), dtype=torch.uint8,
                                device=a.device)
    c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    dash_gemm_splitk(a, b, c, workspace, splits, deterministic, stream)
    if check:
        _check(dash_attn_get_status(workspace, stream), "dash_gemm_splitk (device status)")
    return c


# ---- conveniences (allocation through torch; the compute stays in the library) ----

def new_workspace(B: int, S: int, H: int, D: int, device) -> torch.Tensor:
    nbytes = dash_attn_bwd_workspace_size(B, S, H, D)
    if nbytes == 0:
        raise DashError(DASH_ERR_UNSUPPORTED, "dash_attn_bwd_workspace_size")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def attn_forward(q, k, v, scale: float, causal: bool, stream=None):
    """Allocates O and LSE and runs dash_attn_fwd. Returns (o, lse)."""
    B, S, H, D = _shape(q)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    dash_attn_fwd(q, k, v, o, lse, scale, MASK_CAUSAL if causal else MASK_FULL, stream)
    return o, lse


def attn_backward(q, k, v, o, dO, lse, scale: float, causal: bool, schedule="ascending",
                  deterministic=True, workspace=None, stream=None, check: bool = True):
    """Allocates dQ/dK/dV (and a workspace if none is given) and runs dash_attn_bwd.

    deterministic: False/0 (arrival order), True/1 (one fixed chain per dQ block) or 2 (the
    fixed order as two interleaved chains)."""
    B, S, H, D = _shape(q)
    if workspace is None:
        workspace = new_workspace(B, S, H, D, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sched = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    dash_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, workspace, scale,
                  MASK_CAUSAL if causal else MASK_FULL, sched, int(deterministic), stream)
    if check:
        _check(dash_attn_get_status(workspace, stream), "dash_attn_bwd (device status)")
    return dq, dk, dv
