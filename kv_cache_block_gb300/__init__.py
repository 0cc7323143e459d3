"""Key-Key Semantic Affinity KV-cache block selector for GB300 (sm_103a).

The compute lives in ``libkk.so`` (C ABI, include/kk.h); ``kk`` is its thin
Python binding. The binding loads the library on first use and raises when
it has not been built (``python -m kv_cache_block_gb300.build``); there is no
other code path.
"""
import importlib

_BINDING = (
    "BlockTable", "KKError", "kcache_desc", "kk_anchor", "kk_coarse_means", "kk_device_error",
    "kk_head_variance", "kk_head_variance_workspace_bytes", "kk_pool_blocks", "kk_pool_blocks_weighted", "kk_pool_blocks_weighted_static",
    "kk_score", "kk_score_pool_batched", "kk_score_pool_batched_workspace_bytes", "kk_score_topk",
    "kk_select_step", "kk_topk", "AnchorRing", "kk_anchor_ring_fill", "kk_append_tokens",
    "kk_select_step_workspace_bytes",
)
__all__ = ["kk", *_BINDING]


def __getattr__(name):
    if name == "kk":
        return importlib.import_module(".kk", __name__)
    if name in _BINDING:
        return getattr(importlib.import_module(".kk", __name__), name)
    raise AttributeError(name)
