"""GB300 (sm_103a) Mamba-1 selective scan, forward and backward.

The compute lives in ``libss.so`` (CUDA kernels behind the C ABI of
``include/ss.h``); ``binding`` marshals torch CUDA tensors into it.  The
library is loaded on first use and every entry point raises if it is
missing -- there is no other implementation to fall back on.
"""

from .binding import (SS_BF16, SS_ERR_DEVICE_TIMEOUT, SS_F16, SS_F32, SS_OK, SSError, bwd_saved_workspace_bytes,
                      bwd_workspace_bytes, device_status, fwd_workspace_bytes, lib, plan_info, saved_bytes,
                      selftest_wait_timeout, set_copies_only, ss_bwd, ss_bwd_ex, ss_bwd_saved, ss_decode_step, ss_fwd,
                      ss_fwd_ex, ss_fwd_noalloc, ss_fwd_save, staging_uses_tma, status_string)

__all__ = ["ss_fwd", "ss_fwd_save", "ss_fwd_ex", "ss_fwd_noalloc", "ss_bwd", "ss_bwd_saved", "ss_bwd_ex",
           "ss_decode_step",
           "fwd_workspace_bytes", "bwd_workspace_bytes", "saved_bytes", "bwd_saved_workspace_bytes", "status_string",
           "plan_info", "lib", "SSError", "SS_F32", "SS_F16", "SS_BF16", "SS_OK", "SS_ERR_DEVICE_TIMEOUT",
           "device_status", "selftest_wait_timeout", "set_copies_only", "staging_uses_tma"]
