"""The allocation-free weighted pool (kk_pool_blocks_weighted_static), for
callers that cannot allocate device memory, must give what the workspace form
(kk_pool_blocks_weighted) gives. Called through the C ABI, twice in a row on
different caches, so a second call cannot lean on what the first left in the
shared scratch array. This file sorts last so a stop-at-first-failure run
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests.helpers import DeviceCache, assert_vec_close

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 << 20


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _with_workspace(kk, dev):
    sp = dev.spec
    LH = sp.L * sp.H
    ws = torch.empty(kk.kk_head_variance_workspace_bytes(dev.desc, sp.total_blocks, sp.R), dtype=torch.uint8,
                     device="cuda")
    w = torch.zeros((sp.R, LH), device="cuda")
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks_weighted(dev.desc, dev.bt, sp.total_blocks, w, vb, ws)
    return w, vb


def _static_through_c_abi(kk, dev):
    sp = dev.spec
    w = torch.full((sp.R, sp.L * sp.H), -1.0, device="cuda")
    vb = torch.full((sp.num_pages, sp.D), -1.0, device="cuda")
    lib = ctypes.CDLL(kk.LIB_PATH)
    fn = lib.kk_pool_blocks_weighted_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kk.kk_kcache_desc), ctypes.POINTER(kk.kk_block_table), ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    status = fn(ctypes.byref(dev.desc), ctypes.byref(dev.bt.c), sp.total_blocks, w.data_ptr(), vb.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
    return status, w, vb


def test_static_scratch_matches_workspace_form_twice(kk):
    specs = [
        synth.qwen7b(L=6, H=4, bs=32, seq_lens=[32 * 20 + 7, 32 * 9], num_topics=4, sigma_range=(0.5, 3.0),
                     shuffle_pages=True, extra_pages=3, seed=41),
        synth.tiny_05b(L=4, seq_lens=[16 * 30 + 1, 16 * 3, 5], num_topics=3, sigma_range=(0.5, 2.0), seed=42),
    ]
    for spec in specs:  # two calls in a row, different shapes and contents
        dev = DeviceCache(spec)
        sp = dev.spec
        need = kk.kk_head_variance_workspace_bytes(dev.desc, sp.total_blocks, sp.R)
        assert need <= SCRATCH_LIMIT
        w_ref, vb_ref = _with_workspace(kk, dev)
        status, w, vb = _static_through_c_abi(kk, dev)
        assert status == kk.KK_OK
        assert kk.kk_device_error() == 0
        assert_vec_close(w.cpu().numpy(), w_ref.cpu().numpy(), "head weights")
        assert_vec_close(vb.cpu().numpy()[sp.pages], vb_ref.cpu().numpy()[sp.pages], "weighted vb")
        untouched = np.setdiff1d(np.arange(sp.num_pages), sp.pages)
        assert np.all(vb.cpu().numpy()[untouched] == -1.0)


def test_static_scratch_rejects_oversized_workloads(kk):
    # 7B geometry: 28 * 4 slices * 128 dims * 4 B = 57 KB of scratch per block,
    # so 600 blocks need more than the 32 MiB array
    spec = synth.qwen7b(L=28, H=4, bs=16, seq_lens=[16 * 600], num_topics=4, seed=43)
    dev = DeviceCache(spec)
    assert kk.kk_head_variance_workspace_bytes(dev.desc, spec.total_blocks, spec.R) > SCRATCH_LIMIT
    status, w, vb = _static_through_c_abi(kk, dev)
    assert status == kk.KK_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(vb == -1.0)  # nothing was launched


def test_static_scratch_bounds_and_bad_pages(kk):
    """A block table that reaches past total_blocks is reported and skipped
    (nothing is indexed past the array), and a block with an out-of-range page
    counts as zero in its request's variance instead of whatever an earlier
    call left in the array: the static form then equals the workspace form."""
    # 300 blocks: more than one per SM, so the persistent slice kernel runs
    spec = synth.qwen7b(L=6, H=4, bs=32, seq_lens=[32 * 200 + 3, 32 * 100], num_topics=4, sigma_range=(0.5, 3.0),
                        shuffle_pages=True, seed=44)
    dev = DeviceCache(spec)
    sp = dev.spec
    # fill the array with this cache's sums first
    status, _, _ = _static_through_c_abi(kk, dev)
    assert status == kk.KK_OK and kk.kk_device_error() == 0
    # total_blocks short of offsets[R]: both requests reported, no output written
    lib = ctypes.CDLL(kk.LIB_PATH)
    fn = lib.kk_pool_blocks_weighted_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kk.kk_kcache_desc), ctypes.POINTER(kk.kk_block_table), ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    w = torch.full((sp.R, sp.L * sp.H), -1.0, device="cuda")
    vb = torch.full((sp.num_pages, sp.D), -1.0, device="cuda")
    status = fn(ctypes.byref(dev.desc), ctypes.byref(dev.bt.c), sp.nb[0] - 1, w.data_ptr(), vb.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
    assert status == kk.KK_OK
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    assert torch.all(w == -1.0) and torch.all(vb == -1.0)
    # one page id out of range in request 1
    pages = dev.pages.clone()
    pages[sp.offsets[1] + 7] = sp.num_pages + 5
    bad = DeviceCache.__new__(DeviceCache)
    bad.__dict__.update(dev.__dict__)
    bad.pages = pages
    bad.bt = kk.BlockTable(pages, dev.offsets, dev.seq_lens, max(sp.nb))
    w_ref, vb_ref = _with_workspace(kk, bad)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    status, w, vb = _static_through_c_abi(kk, bad)
    assert status == kk.KK_OK
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    assert_vec_close(w.cpu().numpy(), w_ref.cpu().numpy(), "head weights with a bad page")
    good = np.setdiff1d(sp.pages, [sp.pages[sp.offsets[1] + 7]])
    assert_vec_close(vb.cpu().numpy()[good], vb_ref.cpu().numpy()[good], "weighted vb with a bad page")
