"""The C-ABI library loads, exports every entry point include/kk.h declares,
and rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kk.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kk_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def kk():
    from kv_cache_block_gb300 import kk as mod

    return mod


def test_header_declares_the_method_steps():
    names = declared_functions()
    for n in ("kk_pool_blocks", "kk_anchor", "kk_score", "kk_topk", "kk_select_step",
              "kk_head_variance", "kk_pool_blocks_weighted", "kk_score_pool_batched", "kk_coarse_means"):
        assert n in names


def test_library_exports_every_declared_symbol(kk):
    lib = ctypes.CDLL(kk.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) <= set(kk.EXPORTS)


def test_status_strings(kk):
    assert kk.status_str(0) == "ok"
    assert "invalid" in kk.status_str(1)
    assert kk.status_str(99) == "unknown status"


def _desc(kk, **kw):
    d = dict(base=4096, dtype=kk.KK_BF16, num_layers=2, num_kv_heads=2, head_dim=128, block_size=16,
             num_pages=8, stride_layer=8 * 2 * 16 * 128, stride_page=2 * 16 * 128, stride_head=16 * 128,
             stride_token=128)
    d.update(kw)
    return kk.kk_kcache_desc(*[d[f] for f, _ in kk.kk_kcache_desc._fields_])


def _table(kk, R=1, max_blocks=4, ptrs=True):
    p = 4096 if ptrs else None
    return kk.kk_block_table(p, p, p, R, max_blocks)


def test_host_argument_errors(kk):
    lib = kk._lib
    d = _desc(kk)
    t = _table(kk)
    B = ctypes.byref
    # kk_pool_blocks: null descriptor, negative n, missing pointers, weights without sets
    assert lib.kk_pool_blocks(None, 1, 1, 1, None, 0, None, 1, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks(B(d), 1, 1, -1, None, 0, None, 1, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks(B(d), None, 1, 1, None, 0, None, 1, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks(B(d), 16, 16, 1, 16, 0, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks(B(d), 16, 16, 0, None, 0, None, 16, None) == kk.KK_OK  # nothing to do
    # unsupported layouts: head_dim, alignment, strides, too many heads
    assert lib.kk_pool_blocks(B(_desc(kk, head_dim=96)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, base=4100)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, stride_token=130)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, stride_head=-128)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, dtype=kk.KK_F32, head_dim=256)), 16, 16, 1, None, 0, None, 16,
                              None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, num_layers=40, num_kv_heads=32)), 16, 16, 1, None, 0, None, 16,
                              None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks(B(_desc(kk, dtype=7)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks(B(_desc(kk, block_size=0)), 16, 16, 1, None, 0, None, 16, None) == kk.KK_ERR_INVALID
    # kk_anchor: W out of range, missing output, bad tables
    assert lib.kk_anchor(B(d), B(t), 0, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor(B(d), B(t), 1025, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor(B(d), B(t), 8, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor(B(d), B(_table(kk, R=-1)), 8, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor(B(d), B(_table(kk, ptrs=False)), 8, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor(B(d), None, 8, None, 16, None) == kk.KK_ERR_INVALID
    # kk_score / kk_score_topk: dims and K
    assert lib.kk_score(16, 100, 8, B(t), 16, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_score(None, 128, 8, B(t), 16, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_score(16, 128, 8, B(t), 16, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score(20, 128, 8, B(t), 16, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_score_topk(16, 128, 8, B(t), 16, 0, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk(16, 128, 8, B(t), 16, 257, 16, None, None, None, None) == kk.KK_ERR_INVALID
    # kk_topk: K range, R range, empty
    assert lib.kk_topk(16, 16, 1, 4, 0, 16, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_topk(16, 16, 1, 4, 300, 16, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_topk(16, 16, -1, 4, 4, 16, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_topk(None, None, 0, 4, 4, None, None, None, None) == kk.KK_OK
    # kk_select_step
    assert lib.kk_select_step(B(d), B(t), 8, None, None, 4, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_select_step(B(d), B(t), 8, None, 16, 0, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    # stability filter: window, history words, threshold, table size
    f = float
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 0, f(0.5), 16, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 33, f(0.5), 16, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 20, f(0.5), None, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 20, f("nan"), 16, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 20, f("inf"), 16, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(t), 16, 4, 20, f(0.5), 18, None, 16, None, None, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_score_topk_stable(16, 128, 8, B(_table(kk, max_blocks=1 << 27)), 16, 4, 20, f(0.5), 16, None, 16,
                                    None, None, None, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_select_step_stable(B(d), B(t), 8, None, 16, 4, 0, f(0.5), 16, None, None, 16, None, None, None,
                                     None) == kk.KK_ERR_INVALID
    assert lib.kk_select_step_stable(B(d), B(t), 8, None, 16, 4, 20, f(0.5), None, None, None, 16, None, None, None,
                                     None) == kk.KK_ERR_INVALID
    # decode-step options: workspace too small or misaligned, ring on a score-only call, bad rings
    ws_need = lib.kk_select_step_workspace_bytes(1, 65536, 32)
    assert ws_need > 0
    assert lib.kk_select_step_workspace_bytes(1, 300, 32) == 0  # too short to split
    assert lib.kk_select_step_workspace_bytes(1, 65536, 0) == 0
    big = _table(kk, max_blocks=65536)
    small_ws = kk.kk_step_options(None, 4096, ws_need - 8)
    assert lib.kk_score_topk(16, 128, 8, B(big), 16, 32, 16, None, None, B(small_ws), None) == kk.KK_ERR_INVALID
    odd_ws = kk.kk_step_options(None, 4100, ws_need)
    assert lib.kk_score_topk(16, 128, 8, B(big), 16, 32, 16, None, None, B(odd_ws), None) == kk.KK_ERR_UNSUPPORTED
    ring = kk.kk_anchor_ring(4096, 4096, 16)
    with_ring = kk.kk_step_options(ctypes.pointer(ring), None, 0)
    assert lib.kk_score_topk(16, 128, 8, B(t), 16, 4, 16, None, None, B(with_ring), None) == kk.KK_ERR_INVALID
    assert lib.kk_topk(16, 16, 1, 4, 4, 16, None, B(with_ring), None) == kk.KK_ERR_INVALID
    # W above the ring's slots, empty ring, missing positions
    assert lib.kk_select_step(B(d), B(t), 17, None, 16, 4, None, 16, None, None, B(with_ring), None) == \
        kk.KK_ERR_INVALID
    for bad in (kk.kk_anchor_ring(4096, 4096, 0), kk.kk_anchor_ring(4096, None, 16),
                kk.kk_anchor_ring(None, 4096, 16), kk.kk_anchor_ring(4096, 4096, 1025)):
        o = kk.kk_step_options(ctypes.pointer(bad), None, 0)
        assert lib.kk_select_step(B(d), B(t), 8, None, 16, 4, None, 16, None, None, B(o), None) == kk.KK_ERR_INVALID
        assert lib.kk_anchor_ring_fill(B(d), B(t), None, B(bad), None) == kk.KK_ERR_INVALID
        assert lib.kk_append_tokens(B(d), B(t), 16, None, 16, 16, B(bad), None) == kk.KK_ERR_INVALID
    assert lib.kk_anchor_ring_fill(B(d), B(t), None, None, None) == kk.KK_ERR_INVALID
    # the fused write side and table: k_new needs block_sum and a ring (select steps only), 16-byte
    # alignment, and no fp32 cache of D 256; a table needs a block table (not kk_topk)
    O = kk.kk_step_options
    rp = ctypes.pointer(ring)
    assert lib.kk_select_step(B(d), B(t), 8, None, 16, 4, None, 16, None, None, B(O(rp, None, 0, 4096, None)),
                              None) == kk.KK_ERR_INVALID
    assert lib.kk_select_step(B(d), B(t), 8, None, 16, 4, None, 16, None, None, B(O(None, None, 0, 4096, 4096)),
                              None) == kk.KK_ERR_INVALID
    assert lib.kk_select_step(B(d), B(t), 8, None, 16, 4, None, 16, None, None, B(O(rp, None, 0, 4100, 4096)),
                              None) == kk.KK_ERR_UNSUPPORTED
    d256 = _desc(kk, dtype=kk.KK_F32, head_dim=256, stride_layer=8 * 2 * 16 * 256, stride_page=2 * 16 * 256,
                 stride_head=16 * 256, stride_token=256)
    assert lib.kk_select_step(B(d256), B(t), 8, None, 16, 4, None, 16, None, None,
                              B(O(ctypes.pointer(kk.kk_anchor_ring(4096, 4096, 16)), None, 0, 4096, 4096)),
                              None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_score_topk(16, 128, 8, B(t), 16, 4, 16, None, None, B(O(None, None, 0, 4096, 4096)), None) == \
        kk.KK_ERR_INVALID
    assert lib.kk_topk(16, 16, 1, 4, 4, 16, None, B(O(None, None, 0, None, None, 4096)), None) == kk.KK_ERR_INVALID
    # kk_head_variance: workspace too small / missing output
    assert lib.kk_head_variance(B(d), B(t), 4, 16, 256, 1, None) == kk.KK_ERR_INVALID
    assert lib.kk_head_variance(B(d), B(t), 4, None, 256, 1 << 30, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted(B(d), B(t), 4, 16, None, 256, 1 << 30, None) == kk.KK_ERR_INVALID
    # kk_pool_blocks_weighted_static: missing outputs, negative size, scratch above its 32 MiB
    # (rejected before any CUDA call)
    assert lib.kk_pool_blocks_weighted_static(B(d), B(t), 4, None, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted_static(B(d), B(t), 4, 16, None, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted_static(B(d), B(t), -1, 16, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted_static(None, B(t), 4, 16, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted_static(B(d), None, 4, 16, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_pool_blocks_weighted_static(B(d), B(t), 1 << 20, 16, 16, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_pool_blocks_weighted_static(B(d), B(_table(kk, R=0)), 4, 16, 16, None) == kk.KK_OK
    ws = lib.kk_head_variance_workspace_bytes(B(d), 4, 1)
    assert ws >= 4 * 4 * 128 * 4 + 4 * 4 * 4 + 4 * 8
    assert lib.kk_head_variance(B(d), B(t), 4, 16, 256 + 8, ws, None) == kk.KK_ERR_UNSUPPORTED
    # kk_coarse_means
    assert lib.kk_coarse_means(16, 128, 8, B(t), 0, 16, None) == kk.KK_ERR_INVALID
    assert lib.kk_coarse_means(16, 48, 8, B(t), 4, 16, None) == kk.KK_ERR_UNSUPPORTED
    # kk_device_error needs an output pointer
    assert lib.kk_device_error(None, None) == kk.KK_ERR_INVALID


def test_binding_rejects_host_tensors(kk):
    import torch

    with pytest.raises(ValueError):
        kk._ptr(torch.zeros(4), torch.float32, "x")


def test_hier_host_errors(kk):
    """kk_hier_select rejects bad shares, fan-outs, dims and oversized levels on the host."""
    lib = kk._lib
    t = kk.kk_block_table(4096, 4096, None, 1, 4)
    B = __import__("ctypes").byref
    assert lib.kk_hier_select(16, 128, 8, B(t), 16, 16, 16, 64, 8, 0, 200, 100, 4, 16, None, None, None, None) == \
        kk.KK_ERR_INVALID
    assert lib.kk_hier_select(16, 128, 8, B(t), 16, 16, 16, 64, 8, 500, 1001, 100, 4, 16, None, None, None, None) == \
        kk.KK_ERR_INVALID
    assert lib.kk_hier_select(16, 128, 8, B(t), 16, 16, 16, 0, 8, 500, 200, 100, 4, 16, None, None, None, None) == \
        kk.KK_ERR_INVALID
    assert lib.kk_hier_select(16, 96, 8, B(t), 16, 16, 16, 64, 8, 500, 200, 100, 4, 16, None, None, None, None) == \
        kk.KK_ERR_UNSUPPORTED
    big = kk.kk_block_table(4096, 4096, None, 1, 1 << 22)
    assert lib.kk_hier_select(16, 128, 8, B(big), 16, 16, 16, 64, 8, 1000, 1000, 1000, 4, 16, None, None, None, None) == \
        kk.KK_ERR_UNSUPPORTED


def test_hier_pool_host_errors(kk):
    """The shared-pool hierarchy: coarse row counts, and bad shares, sizes and dims rejected on the host."""
    lib = kk._lib
    assert lib.kk_hier_pool_coarse_rows(65536, 64, 8) == 1152  # 128 Grids + 1024 Chunks
    assert lib.kk_hier_pool_coarse_rows(300, 8, 3) == 128      # 13 + 38, padded to a tile
    assert lib.kk_hier_pool_coarse_rows(0, 64, 8) == 0
    assert lib.kk_hier_pool_coarse_rows(1 << 20, 16, 8) == -1  # 65536 Chunks: too many
    assert lib.kk_hier_pool_coarse_rows(10, 0, 8) == -1
    assert lib.kk_hier_select_pool_workspace_bytes(4, 1 << 20, 16, 8) == 0
    ok = (16, 16, 16)
    args = lambda R, N, D, cp, gc, pm, K: (*ok, R, N, D, cp, gc, *pm, K, 16, None, None, 16, 1 << 30, None)
    assert lib.kk_hier_select_pool(*args(4, 1000, 128, 64, 8, (0, 200, 100), 16)) == kk.KK_ERR_INVALID
    assert lib.kk_hier_select_pool(*args(4, 1000, 128, 64, 8, (500, 200, 1001), 16)) == kk.KK_ERR_INVALID
    assert lib.kk_hier_select_pool(*args(4, 1000, 128, 64, 8, (500, 200, 100), 0)) == kk.KK_ERR_INVALID
    assert lib.kk_hier_select_pool(*args(4, 1000, 128, 64, 8, (500, 200, 100), 257)) == kk.KK_ERR_INVALID
    assert lib.kk_hier_select_pool(*args(4, 1000, 128, 0, 8, (500, 200, 100), 16)) == kk.KK_ERR_INVALID
    assert lib.kk_hier_select_pool(*args(4, 1000, 96, 64, 8, (500, 200, 100), 16)) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_hier_select_pool(*args(4, 1 << 20, 128, 16, 8, (500, 200, 100), 16)) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_hier_select_pool(*args(0, 1000, 128, 64, 8, (500, 200, 100), 16)) == kk.KK_OK
    assert lib.kk_hier_pool_reps(16, 1000, 64, 64, 8, None) == kk.KK_ERR_UNSUPPORTED
    assert lib.kk_hier_pool_reps(16, 1000, 128, 0, 8, None) == kk.KK_ERR_INVALID
    assert lib.kk_hier_pool_reps(None, 0, 128, 64, 8, None) == kk.KK_OK
