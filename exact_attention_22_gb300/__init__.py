"""Exact attention forward and backward passes on GB300 (sm_103a).

The compute path is the CUDA library ``libfa.so`` (built from ``csrc/``); this
package only marshals arguments to its C ABI (``include/fa.h``).  There is no
CPU or PyTorch fallback: if the library is missing, importing the binding
raises.
"""
from .binding import (FA_BF16, FA_FP16, FA_OK, FaError, STATUS_NAMES, attention, attention_backward,  # noqa: F401
                      attention_backward_host, attention_fp8, attention_host, attention_kv, fa_bwd, fa_bwd_gqa, fa_bwd_host,
                      fa_bwd_host_workspace_bytes, fa_bwd_workspace_bytes, fa_fwd, fa_fwd_fp8, fa_fwd_fp8_host,
                      fa_fwd_fp8_host_workspace_bytes,
                      fa_fwd_gqa, fa_fwd_host, fa_fwd_host_workspace_bytes, fa_fwd_kv, fa_fwd_kv_splits_hint,
                      fa_fwd_kv_workspace_bytes,
                      fa_fwd_splitkv,
                      fa_fwd_splitkv_noalloc,
                      fa_get_device_status, fa_noalloc_scratch_bytes, fa_selftest_bwd_fault, fa_selftest_fwd_fault,
                      fa_selftest_wait_timeout,
                      fa_splitkv_workspace_bytes, fa_status_string, library_path, load_library)
