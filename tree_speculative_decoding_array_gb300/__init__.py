"""GB300-native tree speculative-decoding verify step.

One verify round is five calls of the C ABI in ``include/tsv.h`` (built from
``csrc/`` into ``libtsv.so``): ``tree_mask`` -> ``tree_verify_attention`` ->
``lm_head_argmax`` -> ``tree_accept_walk`` -> ``kv_gather_positions``.  This
package is only the Python binding (argument marshalling over ctypes); it has
no fallback and raises if the library is not built.
"""
from ._abi import (ATTN_AUTO, ATTN_SIMT, ATTN_TCGEN05, BF16, DEV_TIMEOUT, DEV_BAD_KV_LEN, DEV_BAD_PARENT, DEV_BAD_PATH, DEV_BAD_ROOT, DEV_OK, F16, I8_SCALED,
                   MAX_LAYERS, MAX_T, Q4_G64, AttnDesc, KvDesc, TsvError, load)
from .api import (VerifyRound, append_desc, draft_children, tree_select, attention_workspace_size, attn_desc, kv_desc, kv_gather_positions, gather_positions, lm_head_argmax,
                  lm_head_logits, lm_head_workspace_size, sample_nucleus, sample_workspace_size, sliding_band_mask, tree_accept_walk, tree_append, tree_mask,
                  tree_verify_attention)

__all__ = [
    "load", "TsvError", "ATTN_AUTO", "ATTN_SIMT", "ATTN_TCGEN05", "DEV_TIMEOUT", "AttnDesc", "KvDesc", "F16", "BF16", "I8_SCALED", "Q4_G64", "MAX_T", "MAX_LAYERS",
    "DEV_OK", "DEV_BAD_ROOT", "DEV_BAD_PARENT", "DEV_BAD_PATH", "DEV_BAD_KV_LEN",
    "draft_children", "tree_select", "tree_mask", "sliding_band_mask", "append_desc", "tree_append", "attn_desc", "attention_workspace_size", "tree_verify_attention", "lm_head_workspace_size",
    "lm_head_argmax", "lm_head_logits", "sample_workspace_size", "sample_nucleus", "tree_accept_walk", "kv_desc", "kv_gather_positions", "gather_positions", "VerifyRound",
]
