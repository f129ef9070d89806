"""GB300 (sm_103a) exact attention: thin Python binding over libfa_gb300.so.

The functions here carry the names of the C ABI in ``include/fa.h`` and only
marshal arguments: they check dtypes/devices/shapes, allocate outputs and
workspaces with torch when the caller passes none, and pass raw device
pointers and the current CUDA stream to the library. Every step of the
computation runs in the library's CUDA kernels. There is no fallback: if the
library is missing or a call fails, a ``FAError`` is raised.
"""
from __future__ import annotations

from ._native import (  # noqa: F401
    FAError,
    FA_OK,
    FA_ERR_INVALID,
    FA_ERR_UNSUPPORTED,
    FA_ERR_CUDA,
    FA_ERR_TIMEOUT,
    FA_ERR_WORKSPACE,
    library,
    library_path,
    fa_version,
    fa_status_string,
    fa_fwd,
    fa_bwd,
    fa_bwd_workspace_size,
    fa_fwd_varlen,
    fa_bwd_varlen,
    fa_fwd_dropout,
    fa_bwd_dropout,
    fa_bwd_varlen_workspace_size,
    fa_decode_splitkv,
    fa_decode_paged,
    fa_decode_kvcache,
    fa_decode_workspace_size,
    fa_decode_num_splits,
    fa_device_status,
    fa_selftest_wait_timeout,
    fa_debug_set_fault,
    FA_FAULT_NONE,
    FA_FAULT_FWD_SKIP_KEY_TILE,
    FA_FAULT_BWD_SKIP_KEY_TILE,
    FA_SELFTEST_SITE,
)

__all__ = [
    "FAError",
    "library",
    "library_path",
    "fa_version",
    "fa_status_string",
    "fa_fwd",
    "fa_bwd",
    "fa_bwd_workspace_size",
    "fa_fwd_varlen",
    "fa_fwd_dropout",
    "fa_bwd_dropout",
    "fa_bwd_varlen",
    "fa_bwd_varlen_workspace_size",
    "fa_decode_splitkv",
    "fa_decode_paged",
    "fa_decode_kvcache",
    "fa_decode_workspace_size",
    "fa_decode_num_splits",
    "fa_device_status",
    "fa_selftest_wait_timeout",
    "fa_debug_set_fault",
    "FA_FAULT_NONE",
    "FA_FAULT_FWD_SKIP_KEY_TILE",
    "FA_FAULT_BWD_SKIP_KEY_TILE",
]
