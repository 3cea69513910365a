"""Exact IO-aware attention (forward + backward) for one GB300 GPU.

The computation lives in ``libfa_sm103.so`` (hand-written CUDA for sm_103a, C ABI declared in
``include/fa.h``); this package holds the ctypes binding with the same names, the build step and
the seeded synthetic workloads.
"""

from .binding import (  # noqa: F401
    EXPORTED,
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_ERR_WORKSPACE,
    FA_OK,
    BlockIndex,
    FAError,
    default_scale,
    fa_block_index_build,
    fa_block_index_size,
    fa_bwd,
    fa_bwd_block_sparse,
    fa_bwd_deterministic,
    fa_bwd_dkdv,
    fa_bwd_dq_convert,
    fa_bwd_gqa,
    fa_bwd_varlen,
    fa_bwd_varlen_workspace_size,
    fa_bwd_noalloc,
    fa_bwd_preprocess,
    fa_bwd_workspace_size,
    fa_fwd,
    fa_fwd_block_sparse,
    fa_fwd_gqa,
    fa_fwd_varlen,
    fa_get_error,
    fa_status_string,
    load_library,
    workspace_for,
)
from .build_lib import LIB_PATH, build  # noqa: F401
