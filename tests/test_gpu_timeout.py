"""Failure detection without a GPU fault. Every spin of a kernel on an
mbarrier is bounded; past the limit the kernel records KK_ERR_TIMEOUT in the
device error word, waits (bounded) for the copies it still has in flight and
returns, so the context stays usable. Here the persistent pool kernel's first
CTA is told to issue no copy for one of its TMA boxes (nothing is in flight
for it, so nothing can complete its wait), with the wait limit cut to 200 us:
the call must report the timeout and return, and the next ordinary call must
be correct."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import DeviceCache, assert_vec_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def test_pool_wait_runs_out_and_is_reported(kk):
    # 608 one-box blocks: four per CTA of the persistent pool on 152 SMs
    spec = synth.qwen7b(L=2, H=2, D=128, bs=16, seq_lens=[16 * 608], num_topics=4, W=4, K=4, seed=17)
    dev = DeviceCache(spec)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert spec.total_blocks >= 2 * sms, "the first CTA must own at least two blocks"
    first_cta = spec.total_blocks // sms  # blocks of CTA 0: [0, first_cta)
    assert kk.kk_device_error() == 0
    vb = torch.full((spec.num_pages, spec.D), -1.0, device="cuda")
    try:
        kk.kk_debug_set_wait_limit(200_000)
        kk.kk_debug_skip_pool_copy(1)  # CTA 0's second box (its second block) is never copied
        kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
        code = kk.kk_device_error()
    finally:
        kk.kk_debug_set_wait_limit(0)
        kk.kk_debug_skip_pool_copy(-1)
    assert code == kk.KK_ERR_TIMEOUT
    got = vb.cpu().numpy()
    # CTA 0 stopped at the box that never came: its later blocks were not written
    assert np.all(got[spec.pages[1:first_cta]] == -1.0)
    # the other CTAs pooled their blocks
    host = dev.host_view()
    rest = spec.pages[first_cta:]
    assert_vec_close(got[rest], ko.pool_blocks(host, rest, spec.n_valid[first_cta:]), "other CTAs' vb")
    # the context is usable and the next ordinary call is right
    vb2 = torch.zeros_like(vb)
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb2)
    assert kk.kk_device_error() == 0
    assert_vec_close(vb2.cpu().numpy()[spec.pages], ko.pool_blocks(host, spec.pages, spec.n_valid), "after timeout")


def test_skip_request_is_used_up(kk):
    """The skip request applies to one launch only; a cancelled one to none."""
    spec = synth.qwen7b(L=2, H=2, D=128, bs=16, seq_lens=[16 * 400], num_topics=4, W=4, K=4, seed=18)
    dev = DeviceCache(spec)
    host = dev.host_view()
    want = ko.pool_blocks(host, spec.pages, spec.n_valid)
    kk.kk_debug_skip_pool_copy(0)
    kk.kk_debug_skip_pool_copy(-1)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0
    assert_vec_close(vb.cpu().numpy()[spec.pages], want, "cancelled skip")
    with pytest.raises(kk.KKError):
        kk.kk_debug_skip_pool_copy(-2)
