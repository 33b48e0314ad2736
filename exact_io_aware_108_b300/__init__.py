"""Exact IO-aware attention for B300 (sm_103a).

The compute path is the CUDA library ``libfa.so`` (C ABI in include/fa.h);
this package is its thin Python binding. Importing the package does not
load the library; the first call does, and fails loudly if it is missing.
"""
from ._binding import (  # noqa: F401
    FAError,
    FA_F16,
    FA_BF16,
    fa_bwd,
    fa_bwd_blocksparse,
    fa_bwd_finish,
    fa_bwd_gqa,
    fa_bwd_main,
    fa_bwd_noalloc,
    fa_bwd_noalloc_max_workspace,
    fa_bwd_prepare,
    fa_bwd_workspace_size,
    fa_decode_paged,
    fa_decode_paged_num_splits,
    fa_decode_paged_workspace_size,
    fa_fwd,
    fa_fwd_blocksparse,
    fa_fwd_ex,
    fa_fwd_fp8,
    fa_fwd_fp8_workspace_size,
    fa_fwd_gqa,
    fa_fwd_splitkv,
    fa_fwd_splitkv_num_splits,
    fa_fwd_splitkv_workspace_size,
    fa_debug_starve_pipelines,
    fa_get_device_error,
    fa_last_error_message,
    fa_set_wait_limit_ns,
    fa_status_str,
    fa_version,
    exported_symbols,
    library_path,
    load_library,
)
from .api import (  # noqa: F401
    attention_backward,
    attention_decode_paged,
    attention_forward,
    attention_forward_fp8,
)
