"""Key-Key Semantic Affinity KV-cache block selector for GB300 (sm_103a).

The compute lives in ``libkk.so`` (C ABI, include/kk.h); ``kk`` is its thin
Python binding. Import fails loudly when the library has not been built.
"""
from . import kk  # noqa: F401
from .kk import (  # noqa: F401
    BlockTable,
    KKError,
    kcache_desc,
    kk_anchor,
    kk_coarse_means,
    kk_device_error,
    kk_head_variance,
    kk_head_variance_workspace_bytes,
    kk_pool_blocks,
    kk_pool_blocks_weighted,
    kk_score,
    kk_score_pool_batched,
    kk_score_pool_batched_workspace_bytes,
    kk_score_topk,
    kk_select_step,
    kk_topk,
)
