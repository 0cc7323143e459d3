"""Python binding of the C ABI in include/kk.h (ctypes; argument marshalling only).

Every function has the name of its C entry point and takes torch CUDA tensors
where the C function takes device pointers. Calls are enqueued on the current
torch stream unless ``stream`` (a torch.cuda.Stream) is given. A non-zero
status raises :class:`KKError`. Nothing here computes any part of the method:
each call goes straight to the CUDA library, which must be built
(``python -m kv_cache_block_gb300.build``); importing this module without it
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkk.so")

KK_OK, KK_ERR_INVALID, KK_ERR_UNSUPPORTED, KK_ERR_CUDA, KK_ERR_BAD_INDEX, KK_ERR_TIMEOUT = range(6)
KK_F32, KK_BF16 = 0, 1


class KKError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: status {status} ({status_str(status)})")
        self.status = status


class kk_kcache_desc(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("stride_layer", ctypes.c_int64),
        ("stride_page", ctypes.c_int64),
        ("stride_head", ctypes.c_int64),
        ("stride_token", ctypes.c_int64),
    ]


class kk_block_table(ctypes.Structure):
    _fields_ = [
        ("pages", ctypes.c_void_p),
        ("offsets", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("num_requests", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
    ]


class kk_anchor_ring(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("slots", ctypes.c_int32)]


class kk_step_options(ctypes.Structure):
    _fields_ = [("ring", ctypes.POINTER(kk_anchor_ring)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("k_new", ctypes.c_void_p), ("block_sum", ctypes.c_void_p),
                ("sel_pages", ctypes.c_void_p), ("sel_logical", ctypes.c_void_p), ("sel_count", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m kv_cache_block_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    KC, BT = ctypes.POINTER(kk_kcache_desc), ctypes.POINTER(kk_block_table)
    RG, OP = ctypes.POINTER(kk_anchor_ring), ctypes.POINTER(kk_step_options)
    sig = {
        "kk_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "kk_debug_set_wait_limit": (ctypes.c_int, [ctypes.c_uint64]),
        "kk_debug_skip_pool_copy": (ctypes.c_int, [I64]),
        "kk_device_error": (ctypes.c_int, [P, ctypes.POINTER(I32)]),
        "kk_pool_blocks": (ctypes.c_int, [KC, P, P, I32, P, I32, P, P, P]),
        "kk_head_variance_workspace_bytes": (SZ, [KC, I32, I32]),
        "kk_head_variance": (ctypes.c_int, [KC, BT, I32, P, P, SZ, P]),
        "kk_pool_blocks_weighted": (ctypes.c_int, [KC, BT, I32, P, P, P, SZ, P]),
        "kk_pool_blocks_weighted_static": (ctypes.c_int, [KC, BT, I32, P, P, P]),
        "kk_anchor": (ctypes.c_int, [KC, BT, I32, P, P, P]),
        "kk_score": (ctypes.c_int, [P, I32, I32, BT, P, P, P]),
        "kk_topk": (ctypes.c_int, [P, P, I32, I32, I32, P, P, OP, P]),
        "kk_score_topk": (ctypes.c_int, [P, I32, I32, BT, P, I32, P, P, P, OP, P]),
        "kk_select_step": (ctypes.c_int, [KC, BT, I32, P, P, I32, P, P, P, P, OP, P]),
        "kk_score_topk_stable": (ctypes.c_int, [P, I32, I32, BT, P, I32, I32, F, P, P, P, P, P, OP, P]),
        "kk_select_step_stable": (ctypes.c_int, [KC, BT, I32, P, P, I32, I32, F, P, P, P, P, P, P, OP, P]),
        "kk_compact_table": (ctypes.c_int, [P, I32, BT, P, P, P, P]),
        "kk_hier_reps": (ctypes.c_int, [P, I32, I32, BT, I32, I32, P, P, P]),
        "kk_hier_select": (ctypes.c_int, [P, I32, I32, BT, P, P, P, I32, I32, I32, I32, I32, I32, P, P, P, OP, P]),
        "kk_append_tokens": (ctypes.c_int, [KC, BT, P, P, P, P, RG, P]),
        "kk_anchor_ring_fill": (ctypes.c_int, [KC, BT, P, RG, P]),
        "kk_select_step_workspace_bytes": (SZ, [I32, I32, I32]),
        "kk_score_pool_batched_workspace_bytes": (SZ, [I32, I32, I32]),
        "kk_score_pool_batched": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, P, P, P, SZ, P]),
        "kk_coarse_means": (ctypes.c_int, [P, I32, I32, BT, I32, P, P]),
        "kk_hier_pool_coarse_rows": (I32, [I32, I32, I32]),
        "kk_hier_pool_reps": (ctypes.c_int, [P, I32, I32, I32, I32, P]),
        "kk_hier_select_pool_workspace_bytes": (SZ, [I32, I32, I32, I32]),
        "kk_hier_select_pool": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, I32, I32, I32, I32, I32, P, P, P, P,
                                               SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    del F
    return lib


_lib = _load()

#: the C entry points declared in include/kk.h
EXPORTS = (
    "kk_status_str", "kk_device_error", "kk_debug_set_wait_limit", "kk_debug_skip_pool_copy", "kk_pool_blocks", "kk_head_variance_workspace_bytes",
    "kk_head_variance", "kk_pool_blocks_weighted", "kk_pool_blocks_weighted_static", "kk_anchor", "kk_score", "kk_topk",
    "kk_score_topk", "kk_select_step", "kk_score_topk_stable", "kk_select_step_stable",
    "kk_compact_table", "kk_append_tokens", "kk_anchor_ring_fill", "kk_select_step_workspace_bytes",
    "kk_hier_reps", "kk_hier_select",
    "kk_score_pool_batched_workspace_bytes",
    "kk_score_pool_batched", "kk_coarse_means", "kk_hier_pool_coarse_rows", "kk_hier_pool_reps",
    "kk_hier_select_pool_workspace_bytes", "kk_hier_select_pool",
)


def status_str(status: int) -> str:
    return _lib.kk_status_str(status).decode()


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != KK_OK:
        raise KKError(fn, status)


# ---- descriptors ---------------------------------------------------------


def kcache_desc(storage: torch.Tensor, dtype: int, num_layers: int, num_kv_heads: int, head_dim: int,
                block_size: int, num_pages: int, strides) -> kk_kcache_desc:
    """Describe a paged K cache held in ``storage`` (element strides: layer, page, head, token)."""
    if not storage.is_cuda:
        raise ValueError("storage must live on a CUDA device")
    sL, sP, sH, sT = (int(s) for s in strides)
    return kk_kcache_desc(storage.data_ptr(), dtype, num_layers, num_kv_heads, head_dim, block_size,
                          num_pages, sL, sP, sH, sT)


class BlockTable:
    """Per-request block tables (CSR) on the device; keeps its tensors alive."""

    def __init__(self, pages: torch.Tensor, offsets: torch.Tensor, seq_lens, max_blocks: int):
        self.pages, self.offsets, self.seq_lens = pages, offsets, seq_lens
        self.c = kk_block_table(
            _ptr(pages, torch.int32, "pages") if pages.numel() else None,
            _ptr(offsets, torch.int32, "offsets"),
            _ptr(seq_lens, torch.int32, "seq_lens") if seq_lens is not None else None,
            offsets.numel() - 1,
            int(max_blocks),
        )

    @property
    def num_requests(self) -> int:
        return self.c.num_requests


class AnchorRing:
    """A caller-owned anchor ring on the device: ``rows`` float32 [R][slots][D]
    and ``pos`` int32 [R][slots] (see kk_anchor_ring in include/kk.h)."""

    def __init__(self, R: int, slots: int, D: int, device="cuda"):
        self.rows = torch.zeros((R, slots, D), dtype=torch.float32, device=device)
        self.pos = torch.full((R, slots), -1, dtype=torch.int32, device=device)
        self.c = kk_anchor_ring(self.rows.data_ptr(), self.pos.data_ptr(), slots)

    @property
    def slots(self) -> int:
        return self.c.slots


def _options(ring=None, workspace=None, append=None, compact=None):
    """kk_step_options for a call (None when nothing is given); the returned
    objects must stay alive until the call returns. ``append``: (k_new,
    block_sum) of the fused write side; ``compact``: (sel_pages, sel_logical,
    sel_count) of the fused table (the last two may be None)."""
    if ring is None and workspace is None and append is None and compact is None:
        return None
    o = kk_step_options()
    if ring is not None:
        o.ring = ctypes.pointer(ring.c)
    if workspace is not None:
        o.workspace = _ptr(workspace, name="workspace")
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    if append is not None:
        k_new, block_sum = append
        if not k_new.is_cuda or not k_new.is_contiguous():
            raise ValueError("k_new must be a contiguous CUDA tensor")
        o.k_new = k_new.data_ptr()
        o.block_sum = _ptr(block_sum, torch.float32, "block_sum")
    if compact is not None:
        sp, sl, sc = compact
        o.sel_pages = _ptr(sp, torch.int32, "sel_pages")
        o.sel_logical = _ptr(sl, torch.int32, "sel_logical")
        o.sel_count = _ptr(sc, torch.int32, "sel_count")
    return ctypes.byref(o), o


def _opt(o):
    return None if o is None else o[0]


# ---- entry points --------------------------------------------------------


def kk_debug_set_wait_limit(ns: int):
    """Limit (ns) of every bounded wait of the launches that follow; 0 restores 1 s."""
    _check("kk_debug_set_wait_limit", _lib.kk_debug_set_wait_limit(int(ns)))


def kk_debug_skip_pool_copy(box: int):
    """The next persistent pool launch leaves TMA box ``box`` of its first CTA uncopied (-1 cancels)."""
    _check("kk_debug_skip_pool_copy", _lib.kk_debug_skip_pool_copy(int(box)))


def kk_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check("kk_device_error", _lib.kk_device_error(_stream(stream), ctypes.byref(code)))
    return code.value


def kk_pool_blocks(kc: kk_kcache_desc, pages, n_valid, vb, head_w=None, w_set=None, stream=None):
    n_sets = 0 if head_w is None else head_w.shape[0]
    _check("kk_pool_blocks", _lib.kk_pool_blocks(
        ctypes.byref(kc), _ptr(pages, torch.int32, "pages"), _ptr(n_valid, torch.int32, "n_valid"),
        pages.numel(), _ptr(head_w, torch.float32, "head_w"), n_sets, _ptr(w_set, torch.int32, "w_set"),
        _ptr(vb, torch.float32, "vb"), _stream(stream)))


def kk_head_variance_workspace_bytes(kc: kk_kcache_desc, total_blocks: int, num_requests: int) -> int:
    return _lib.kk_head_variance_workspace_bytes(ctypes.byref(kc), total_blocks, num_requests)


def kk_head_variance(kc, bt: BlockTable, total_blocks: int, head_w_out, workspace, stream=None):
    _check("kk_head_variance", _lib.kk_head_variance(
        ctypes.byref(kc), ctypes.byref(bt.c), total_blocks, _ptr(head_w_out, torch.float32, "head_w_out"),
        _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))


def kk_pool_blocks_weighted(kc, bt: BlockTable, total_blocks: int, head_w_out, vb, workspace, stream=None):
    _check("kk_pool_blocks_weighted", _lib.kk_pool_blocks_weighted(
        ctypes.byref(kc), ctypes.byref(bt.c), total_blocks, _ptr(head_w_out, torch.float32, "head_w_out"),
        _ptr(vb, torch.float32, "vb"), _ptr(workspace, name="workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kk_pool_blocks_weighted_static(kc, bt: BlockTable, total_blocks: int, head_w_out, vb, stream=None):
    """kk_pool_blocks_weighted without a workspace argument: for callers that
    cannot allocate device memory (scratch is a 32 MiB array the library owns)."""
    _check("kk_pool_blocks_weighted_static", _lib.kk_pool_blocks_weighted_static(
        ctypes.byref(kc), ctypes.byref(bt.c), total_blocks, _ptr(head_w_out, torch.float32, "head_w_out"),
        _ptr(vb, torch.float32, "vb"), _stream(stream)))


def kk_anchor(kc, bt: BlockTable, W: int, va, head_w=None, stream=None):
    _check("kk_anchor", _lib.kk_anchor(ctypes.byref(kc), ctypes.byref(bt.c), W,
                                       _ptr(head_w, torch.float32, "head_w"), _ptr(va, torch.float32, "va"),
                                       _stream(stream)))


def kk_score(vb, bt: BlockTable, va, scores, stream=None):
    _check("kk_score", _lib.kk_score(_ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c),
                                     _ptr(va, torch.float32, "va"), _ptr(scores, torch.float32, "scores"),
                                     _stream(stream)))


def kk_select_step_workspace_bytes(R: int, max_blocks: int, K: int) -> int:
    return _lib.kk_select_step_workspace_bytes(R, max_blocks, K)


def kk_topk(scores, offsets, max_n: int, K: int, idx, top_scores=None, workspace=None, stream=None):
    o = _options(workspace=workspace)
    _check("kk_topk", _lib.kk_topk(_ptr(scores, torch.float32, "scores"), _ptr(offsets, torch.int32, "offsets"),
                                   offsets.numel() - 1, max_n, K, _ptr(idx, torch.int32, "idx"),
                                   _ptr(top_scores, torch.float32, "top_scores"), _opt(o), _stream(stream)))


def kk_score_topk(vb, bt: BlockTable, va, K: int, idx, top_scores=None, scores=None, workspace=None, compact=None,
                  stream=None):
    o = _options(workspace=workspace, compact=compact)
    _check("kk_score_topk", _lib.kk_score_topk(
        _ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c), _ptr(va, torch.float32, "va"),
        K, _ptr(idx, torch.int32, "idx"), _ptr(top_scores, torch.float32, "top_scores"),
        _ptr(scores, torch.float32, "scores"), _opt(o), _stream(stream)))


def kk_select_step(kc, bt: BlockTable, W: int, vb, K: int, idx, top_scores=None, va=None, scores=None,
                   head_w=None, ring=None, workspace=None, append=None, compact=None, stream=None):
    """``ring``: an :class:`AnchorRing` to take the anchor from (else the K cache);
    ``append`` / ``compact``: the fused write side and table (see kk_step_options)."""
    o = _options(ring, workspace, append, compact)
    _check("kk_select_step", _lib.kk_select_step(
        ctypes.byref(kc), ctypes.byref(bt.c), W, _ptr(head_w, torch.float32, "head_w"),
        _ptr(vb, torch.float32, "vb"), K, _ptr(va, torch.float32, "va"), _ptr(idx, torch.int32, "idx"),
        _ptr(top_scores, torch.float32, "top_scores"), _ptr(scores, torch.float32, "scores"), _opt(o),
        _stream(stream)))


def kk_score_topk_stable(vb, bt: BlockTable, va, K: int, stab_window: int, theta: float, hist, idx,
                         stab=None, top_scores=None, scores=None, workspace=None, stream=None):
    """``hist``: int32 tensor [offsets[R]] holding the uint32 history words (updated in place)."""
    o = _options(workspace=workspace)
    _check("kk_score_topk_stable", _lib.kk_score_topk_stable(
        _ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c), _ptr(va, torch.float32, "va"),
        K, stab_window, float(theta), _ptr(hist, torch.int32, "hist"), _ptr(stab, torch.float32, "stab"),
        _ptr(idx, torch.int32, "idx"), _ptr(top_scores, torch.float32, "top_scores"),
        _ptr(scores, torch.float32, "scores"), _opt(o), _stream(stream)))


def kk_select_step_stable(kc, bt: BlockTable, W: int, vb, K: int, stab_window: int, theta: float, hist, idx,
                          stab=None, top_scores=None, va=None, scores=None, head_w=None, ring=None, workspace=None,
                          append=None, compact=None, stream=None):
    """``hist``: int32 tensor [offsets[R]] holding the uint32 history words (updated in place)."""
    o = _options(ring, workspace, append, compact)
    _check("kk_select_step_stable", _lib.kk_select_step_stable(
        ctypes.byref(kc), ctypes.byref(bt.c), W, _ptr(head_w, torch.float32, "head_w"),
        _ptr(vb, torch.float32, "vb"), K, stab_window, float(theta), _ptr(hist, torch.int32, "hist"),
        _ptr(stab, torch.float32, "stab"), _ptr(va, torch.float32, "va"), _ptr(idx, torch.int32, "idx"),
        _ptr(top_scores, torch.float32, "top_scores"), _ptr(scores, torch.float32, "scores"), _opt(o),
        _stream(stream)))


def kk_compact_table(idx, bt: BlockTable, sel_pages, sel_logical=None, sel_count=None, stream=None):
    _check("kk_compact_table", _lib.kk_compact_table(
        _ptr(idx, torch.int32, "idx"), idx.shape[1], ctypes.byref(bt.c), _ptr(sel_pages, torch.int32, "sel_pages"),
        _ptr(sel_logical, torch.int32, "sel_logical"), _ptr(sel_count, torch.int32, "sel_count"), _stream(stream)))


def kk_append_tokens(kc, bt: BlockTable, k_new, block_sum, vb, head_w=None, ring=None, stream=None):
    """``k_new``: [R][L][H][D] tensor of the cache's element type (int16 bf16 bits or float32);
    ``ring``: an :class:`AnchorRing` that also receives each token's pooled Keys."""
    if not k_new.is_cuda or not k_new.is_contiguous():
        raise ValueError("k_new must be a contiguous CUDA tensor")
    _check("kk_append_tokens", _lib.kk_append_tokens(
        ctypes.byref(kc), ctypes.byref(bt.c), ctypes.c_void_p(k_new.data_ptr()), _ptr(head_w, torch.float32, "head_w"),
        _ptr(block_sum, torch.float32, "block_sum"), _ptr(vb, torch.float32, "vb"),
        None if ring is None else ctypes.byref(ring.c), _stream(stream)))


def kk_anchor_ring_fill(kc, bt: BlockTable, ring: AnchorRing, head_w=None, stream=None):
    _check("kk_anchor_ring_fill", _lib.kk_anchor_ring_fill(
        ctypes.byref(kc), ctypes.byref(bt.c), _ptr(head_w, torch.float32, "head_w"), ctypes.byref(ring.c),
        _stream(stream)))


def kk_hier_reps(vb, bt: BlockTable, chunk_pages: int, grid_chunks: int, chunk_reps, grid_reps, stream=None):
    _check("kk_hier_reps", _lib.kk_hier_reps(
        _ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c), chunk_pages, grid_chunks,
        _ptr(chunk_reps, torch.float32, "chunk_reps"), _ptr(grid_reps, torch.float32, "grid_reps"), _stream(stream)))


def kk_hier_select(vb, bt: BlockTable, chunk_reps, grid_reps, va, chunk_pages: int, grid_chunks: int, permille,
                   idx, top_scores=None, kept=None, workspace=None, stream=None):
    pg, pc, pp = (int(x) for x in permille)
    o = _options(workspace=workspace)
    _check("kk_hier_select", _lib.kk_hier_select(
        _ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c),
        _ptr(chunk_reps, torch.float32, "chunk_reps"), _ptr(grid_reps, torch.float32, "grid_reps"),
        _ptr(va, torch.float32, "va"), chunk_pages, grid_chunks, pg, pc, pp, idx.shape[1],
        _ptr(idx, torch.int32, "idx"), _ptr(top_scores, torch.float32, "top_scores"), _ptr(kept, torch.int32, "kept"),
        _opt(o), _stream(stream)))


def kk_score_pool_batched_workspace_bytes(R: int, N: int, K: int) -> int:
    return _lib.kk_score_pool_batched_workspace_bytes(R, N, K)


def kk_score_pool_batched(A, V, mask, K: int, idx, top_scores=None, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kk_score_pool_batched", _lib.kk_score_pool_batched(
        _ptr(A, (torch.int16, torch.bfloat16), "A"), _ptr(V, (torch.int16, torch.bfloat16), "V"),
        _ptr(mask, torch.int32, "mask"), A.shape[0], V.shape[0], A.shape[1], K, _ptr(idx, torch.int32, "idx"),
        _ptr(top_scores, torch.float32, "top_scores"), _ptr(workspace, name="workspace"), ws_bytes,
        _stream(stream)))


def kk_hier_pool_coarse_rows(N: int, chunk_pages: int, grid_chunks: int) -> int:
    return _lib.kk_hier_pool_coarse_rows(N, chunk_pages, grid_chunks)


def _pool_matrix(M, N: int, chunk_pages: int, grid_chunks: int):
    H = kk_hier_pool_coarse_rows(N, chunk_pages, grid_chunks)
    if M is not None and H >= 0 and M.shape[0] != H + N:
        raise ValueError(f"M has {M.shape[0]} rows, expected {H} coarse rows + {N} blocks")
    return _ptr(M, (torch.int16, torch.bfloat16), "M")


def kk_hier_pool_reps(M, N: int, chunk_pages: int, grid_chunks: int, stream=None):
    _check("kk_hier_pool_reps", _lib.kk_hier_pool_reps(
        _pool_matrix(M, N, chunk_pages, grid_chunks), N, M.shape[1], chunk_pages, grid_chunks, _stream(stream)))


def kk_hier_select_pool_workspace_bytes(R: int, N: int, chunk_pages: int, grid_chunks: int) -> int:
    return _lib.kk_hier_select_pool_workspace_bytes(R, N, chunk_pages, grid_chunks)


def kk_hier_select_pool(A, M, mask, N: int, chunk_pages: int, grid_chunks: int, permille, idx, top_scores=None,
                        kept=None, workspace=None, stream=None):
    pg, pc, pp = (int(x) for x in permille)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kk_hier_select_pool", _lib.kk_hier_select_pool(
        _ptr(A, (torch.int16, torch.bfloat16), "A"), _pool_matrix(M, N, chunk_pages, grid_chunks),
        _ptr(mask, torch.int32, "mask"), A.shape[0], N, A.shape[1], chunk_pages, grid_chunks, pg, pc, pp,
        idx.shape[1], _ptr(idx, torch.int32, "idx"), _ptr(top_scores, torch.float32, "top_scores"),
        _ptr(kept, torch.int32, "kept"), _ptr(workspace, name="workspace"), ws_bytes, _stream(stream)))


def kk_coarse_means(vb, bt: BlockTable, group: int, out, stream=None):
    _check("kk_coarse_means", _lib.kk_coarse_means(
        _ptr(vb, torch.float32, "vb"), vb.shape[1], vb.shape[0], ctypes.byref(bt.c), group,
        _ptr(out, torch.float32, "out"), _stream(stream)))
