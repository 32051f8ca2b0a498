"""Deterministic gated BF16 FFN for GB300 (sm_103a): Python binding of libdetffn.

The compute path is the C-ABI library ``libdetffn.so`` built from ``csrc/``;
the binding in ``detffn.py`` only marshals arguments (tensor pointers, sizes,
the current CUDA stream).  Importing the package does not load the library;
the first call does, and raises if the library is missing -- there is no CPU
fallback.
"""
from .detffn import (  # noqa: F401
    BF16, F16, F32, FLAG_HOST_IO, FLAG_OVERLAP_DHIDDEN, FLAG_SPLIT_FORWARD, FLAG_TEST_STALL, OP_BACKWARD, OP_FORWARD, OP_FORWARD_SHARDED, OP_WGRAD_CHUNKED, PATH_AUTO,
    PATH_EXACT, PATH_TENSOR, DetFFNError, detffn_backward, detffn_forward,
    detffn_forward_sharded, detffn_get_status, detffn_rank_tree_reduce, detffn_silu_tables,
    detffn_cvt_f32_bf16, detffn_forward_decode_noalloc, detffn_forward_decode_noalloc_status,
    detffn_forward_decode_noalloc_test_waits,
    detffn_profile_read, detffn_profiling, detffn_selfcheck_fused_schedule, detffn_selfcheck_node_add,
    detffn_selfcheck_pieces,
    detffn_tree_gemm, detffn_tree_gemm_leaves,
    detffn_wgrad_chunked,
    detffn_workspace_size, workspace,
)
