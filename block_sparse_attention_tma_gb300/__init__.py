"""Fused block-sparse scaled-dot-product attention for GB300 (sm_103a).

The compute lives in the C-ABI library ``libgbattn.so`` (hand-written CUDA);
``binding`` marshals PyTorch tensors into its entry points. Importing the
package does not load the library; the first call does, and raises if the
library is missing or the GPU is not compute capability 10.3.
"""
from .binding import (  # noqa: F401
    MaskSpec, BlockLists, GbattnError,
    NONE, CAUSAL, SLIDING, BLOCK_DIAG, PREFIX_LM, DYNAMIC_TOPK, MINI_CAUSAL, TABLE, pack_mask_table,
    build_block_mask, alloc_block_lists, attn_fwd, attn_bwd, attn_fwd_splitkv, attn_fwd_splitkv_paged,
    attn_fwd_splitkv_noalloc, attn_bwd_workspace_bytes, attn_fwd_splitkv_workspace_bytes, load_library,
    set_dkdv_cta_pair, last_device_error,
)
