"""Exact tiled attention for GB300 (sm_103a): C-ABI library + thin binding."""

from .binding import (  # noqa: F401
    FAError,
    backward,
    backward_stage,
    backward_varlen,
    FA_NOALLOC_MAX_ROWS,
    fa_bwd,
    fa_bwd_noalloc,
    fa_bwd_stage,
    fa_bwd_varlen,
    fa_bwd_workspace_bytes,
    fa_fwd,
    fa_fwd_varlen,
    fa_last_failure,
    fa_sched_enumerate,
    fa_status_string,
    fa_sync_status,
    forward,
    forward_varlen,
    sync_status,
)
