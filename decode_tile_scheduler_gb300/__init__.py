"""decode_tile_scheduler_gb300 -- fused inference attention over a paged KV
cache for NVIDIA GB300 (sm_103a): split-KV decode with a GPU tile scheduler,
tcgen05 prefill, FP8 E4M3 KV with fp32 tile scales, and the shared-KV sparse
variant, behind the C ABI of include/fia.h (libfia.so).

Python here marshals arguments only; the CUDA library does every step of the
computation and there is no CPU fallback.
"""
from ._abi import (  # noqa: F401
    EXPORTS, FIA_ERR_BAD_DTYPE, FIA_ERR_BAD_SHAPE, FIA_ERR_CUDA, FIA_ERR_NULL_ARG, FIA_ERR_UNSUPPORTED,
    FIA_ERR_WORKSPACE_TOO_SMALL, FIA_OK, KV_BF16, KV_FP8_E4M3, LAYOUT_BSND, LAYOUT_TND, MASK_BAND,
    MASK_NONE, MASK_RIGHT_DOWN_CAUSAL, MASK_ALL, MASK_LEFT_UP_CAUSAL, KV_LAYOUT_BNBSH,
    KV_LAYOUT_BNNBSD, SPARSE_KV_BF16, SPARSE_KV_FP8_PACKED, CombineParams, FiaError, FiaParams,
    FiaPlanLayout, SparseParams, fia_decode_run_noalloc, fia_lse_combine, fia_execute, fia_get_plan_layout, fia_get_workspace_size, fia_plan, fia_run, lib, lib_path,
    sparse_attn_metadata, sparse_attn_run, status_string)
from ._build import build  # noqa: F401
from .api import (  # noqa: F401
    FiaCall, SparseCall, fused_infer_attention, lse_combine, lse_shape, make_fia_params,
    params_from_problem, sparse_params_from_problem)
