"""Fused causal / sliding-window GQA flash attention for GB300 (sm_103a).

The compute lives in ``libfa_gb300.so`` (hand-written CUDA, C ABI in
``include/fa.h``); this package is its Python binding.  Importing the package
does not load the library: the first call does, and fails loudly if it has
not been built.
"""
from ._binding import (  # noqa: F401
    FA_DTYPE_BF16,
    FA_DTYPE_FP16,
    FA_DTYPE_FP32,
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_ERR_WORKSPACE,
    FA_OK,
    FA_OP_BWD,
    FA_OP_BWD_FUSED,
    FA_OP_FWD,
    FaError,
    attention_bwd,
    attention_fwd,
    check_status,
    fa_bwd,
    fa_bwd_cross,
    fa_bwd_dkdv,
    fa_bwd_dkdv_dq,
    fa_bwd_dq,
    fa_bwd_preprocess,
    fa_check_status,
    fa_debug_config,
    fa_debug_fwd_tiles,
    fa_debug_max_ctas,
    fa_fwd,
    fa_fwd_cross,
    fa_plan_block_mask,
    fa_plan_kv_range,
    fa_plan_q_range,
    fa_qk_norm_rope_bwd,
    fa_qk_norm_rope_bwd_opt,
    fa_qk_norm_rope_fwd,
    fa_qk_norm_rope_fwd_opt,
    fa_status_string,
    fa_tile_m,
    fa_tile_n,
    fa_workspace_size,
    load,
    qk_norm_rope_bwd,
    qk_norm_rope_bwd_opt,
    qk_norm_rope_fwd,
    qk_norm_rope_fwd_opt,
)

__all__ = [n for n in dir() if not n.startswith("_")]
