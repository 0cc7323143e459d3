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
