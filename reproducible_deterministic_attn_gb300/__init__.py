"""GB300-native deterministic attention backward with DASH schedules.

The compute lives in libdash_attn.so (hand-written sm_103a CUDA behind a C ABI, see
include/dash_attn.h); this package is its ctypes binding. Importing the package does not
load the library; the first call does, and fails loudly if it has not been built.
"""

from .dash_attn import (  # noqa: F401
    DASH_ERR_BOUNDS, DASH_ERR_CUDA, DASH_ERR_DEADLOCK_RISK, DASH_ERR_INVALID_ARG, DASH_ERR_SYNC_TIMEOUT,
    DASH_ERR_UNSUPPORTED, DASH_ERR_WORKSPACE_TOO_SMALL, DASH_OK, MASK_CAUSAL, MASK_FULL,
    MASKS, SCHED_ASCENDING, SCHED_DESCENDING, SCHED_SHIFT, SCHED_SYMMETRIC_SHIFT, SCHEDULES,
    DashError, attn_backward, attn_forward, dash_attn_bwd, dash_attn_bwd_static,
    dash_attn_bwd_workspace_size,
    dash_attn_fwd, dash_attn_fwd_ex, dash_attn_get_status, dash_attn_shutdown, dash_debug_set_sync,
    dash_bounds_checks_enabled, dash_debug_narrow_checks,
    dash_debug_set_trace,
    dash_last_error, dash_profile_enable, dash_profile_read, dash_sched_num_slots, dash_sched_simulate, dash_sched_simulate_ex, dash_sched_select,
    dash_sched_table, dash_sched_deal, dash_sched_dealt_table, dash_gemm_splitk, dash_gemm_splitk_workspace_size, gemm_splitk,
    dash_status_string, load, new_workspace, TRACE_SITES, TRACE_DQ_TURN_WAIT, TRACE_DQ_ADD,
    TRACE_TOTAL,
)
