"""The anchor ring, through the C ABI, against the fp64 oracle: the anchor of
a decode step ("Key-Key Semantic Affinity" page, §5.2 step 1: the mean of the
last W tokens' Keys) formed from per-token pooled rows that the write path
keeps (kk_anchor_ring_fill after a prefill, kk_append_tokens token by token)
equals the oracle's anchor over the cache, for every W up to the ring's
size, including requests with fewer than W tokens."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import DeviceCache, assert_topk_valid, assert_vec_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32).cuda()


def _weights(spec, weighted, seed):
    if not weighted:
        return None, None
    w = np.random.default_rng(seed).uniform(0.1, 1.0, size=(spec.R, spec.L * spec.H)).astype(np.float32)
    return w, torch.from_numpy(w).cuda()


def _check_positions(ring, lens):
    pos = ring.pos.cpu().numpy()
    for r, T in enumerate(lens):
        want = np.full(ring.slots, -1)
        for t in range(max(0, T - ring.slots), T):
            want[t % ring.slots] = t
        np.testing.assert_array_equal(pos[r], want, err_msg=f"ring positions of request {r}")


def _select_with_ring(kk, dev, bt, vb, W, K, ring, w_dev, R, D):
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    va = torch.zeros((R, D), device="cuda")
    kk.kk_select_step(dev.desc, bt, W, vb, K, idx, top, va=va, head_w=w_dev, ring=ring)
    return idx.cpu().numpy(), top.cpu().numpy(), va.cpu().numpy()


SPECS = {
    "bf16": lambda: synth.qwen7b(L=4, H=2, D=128, bs=16, seq_lens=[16 * 5 + 3, 5, 1, 0, 16 * 2], num_topics=4,
                                 W=8, K=6, shuffle_pages=True, extra_pages=3, sigma_range=(0.5, 2.0)),
    "f32": lambda: synth.tiny_05b(L=3, H=2, D=64, bs=8, seq_lens=[8 * 6 + 1, 7, 8 * 3], num_topics=3, W=8, K=5),
    "d32": lambda: synth.qwen7b(L=2, H=2, D=32, bs=4, seq_lens=[4 * 9 + 2, 3], num_topics=2, W=4, K=3),
    "d256": lambda: synth.qwen7b(L=2, H=1, D=256, bs=4, seq_lens=[4 * 7, 6], num_topics=2, W=4, K=3,
                                 layout="PLHTD"),
    "token-major": lambda: synth.qwen7b(L=3, H=4, D=64, bs=8, seq_lens=[8 * 4 + 5, 8 * 2], num_topics=3, W=8,
                                        K=4, layout="LPTHD"),
}


@pytest.mark.parametrize("name", sorted(SPECS))
@pytest.mark.parametrize("weighted", [False, True])
def test_ring_fill_then_select(kk, name, weighted):
    spec = SPECS[name]()
    dev = DeviceCache(spec)
    host = dev.host_view()
    w, w_dev = _weights(spec, weighted, 7)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    vb_o = ko.pool_blocks(host, spec.pages, spec.n_valid)
    for slots in (spec.W, 2 * spec.W + 3):
        ring = kk.AnchorRing(spec.R, slots, spec.D)
        ring.rows.fill_(float("nan"))  # every slot the fill uses must be written
        kk.kk_anchor_ring_fill(dev.desc, dev.bt, ring, head_w=w_dev)
        assert kk.kk_device_error() == 0
        _check_positions(ring, spec.seq_lens)
        for W in sorted({1, 3, spec.W, slots}):
            idx, top, va = _select_with_ring(kk, dev, dev.bt, vb, W, spec.K, ring, w_dev, spec.R, spec.D)
            assert kk.kk_device_error() == 0
            for r in range(spec.R):
                pr = spec.pages_of(r)
                va_o = ko.anchor(host, pr, spec.seq_lens[r], spec.bs, W, None if w is None else w[r])
                assert_vec_close(va[r][None], va_o[None], f"{name} slots={slots} W={W} r={r} anchor")
                s_o = ko.affinity(vb_o[spec.offsets[r]:spec.offsets[r + 1]], va_o)
                assert_topk_valid(idx[r], top[r], s_o, spec.K, f"{name} W={W} r={r}")


def test_ring_matches_the_cache_gather(kk):
    """The ring path and the K-cache path of kk_select_step give the same
    anchor within float32 rounding and the same selection."""
    spec = synth.qwen7b(L=28, H=4, D=128, bs=128, seq_lens=[128 * 6 + 17, 128 * 3, 40], num_topics=8, W=32, K=16,
                        sigma_range=(0.5, 3.0), shuffle_pages=True)
    dev = DeviceCache(spec)
    w, w_dev = _weights(spec, True, 9)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    ring = kk.AnchorRing(spec.R, 64, spec.D)
    kk.kk_anchor_ring_fill(dev.desc, dev.bt, ring, head_w=w_dev)
    i1, t1, va1 = _select_with_ring(kk, dev, dev.bt, vb, spec.W, spec.K, ring, w_dev, spec.R, spec.D)
    i2, t2, va2 = _select_with_ring(kk, dev, dev.bt, vb, spec.W, spec.K, None, w_dev, spec.R, spec.D)
    assert kk.kk_device_error() == 0
    assert_vec_close(va1, va2, "ring vs cache anchor")
    np.testing.assert_array_equal(i1, i2)


@pytest.mark.parametrize("weighted", [False, True])
def test_ring_follows_appended_tokens(kk, weighted):
    """A ring filled after the prefill and then kept by kk_append_tokens: at
    every decode step the anchor formed from it is the oracle's anchor over
    the cache as written so far (requests start with 3, 16 and 37 tokens, so
    the first steps have fewer than W tokens)."""
    spec = synth.qwen7b(L=3, H=2, D=128, bs=16, seq_lens=[3, 16, 37], num_topics=4, W=8, K=4, extra_pages=12,
                        shuffle_pages=True)
    dev = DeviceCache(spec)
    host = dev.host_view().copy()
    rng = np.random.default_rng(11 + weighted)
    L, H, D, bs = spec.L, spec.H, spec.D, spec.bs
    w, w_dev = _weights(spec, weighted, 13)
    spare = list(np.setdiff1d(np.arange(spec.num_pages), spec.pages))
    tables = [list(spec.pages_of(r)) for r in range(spec.R)]
    lens = list(spec.seq_lens)
    block_sum = torch.zeros((spec.num_pages, D), device="cuda")
    vb = torch.zeros((spec.num_pages, D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb, head_w=w_dev,
                      w_set=_i32(np.repeat(np.arange(spec.R), spec.nb)) if weighted else None)
    # the running sums of the blocks being filled, as the write path keeps them
    for r in range(spec.R):
        if lens[r] % bs:
            p = tables[r][-1]
            n = lens[r] % bs
            keys = ko.block_keys(host, p, n)
            ww = np.ones((L, H)) if w is None else w[r].reshape(L, H).astype(np.float64)
            block_sum[p] = torch.from_numpy(np.einsum("lh,lhtd->d", ww, keys).astype(np.float32)).cuda()
    ring = kk.AnchorRing(spec.R, 12, D)
    kk.kk_anchor_ring_fill(dev.desc, dev.bt, ring, head_w=w_dev)
    for step in range(21):
        for r in range(spec.R):
            if lens[r] % bs == 0:
                tables[r].append(spare.pop(0))
            lens[r] += 1
        offsets = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
        pages = np.concatenate(tables).astype(np.int32)
        bt = kk.BlockTable(_i32(pages), _i32(offsets), _i32(lens), max(len(t) for t in tables))
        kn = (1.5 * spec.cs[rng.integers(0, spec.num_topics, size=spec.R)][:, None, None, :]
              + rng.standard_normal((spec.R, L, H, D))).astype(np.float32)
        kn_store = synth.bf16_rne(kn)
        kk.kk_append_tokens(dev.desc, bt, torch.from_numpy(kn_store.view(np.int16)).cuda(), block_sum, vb,
                            head_w=w_dev, ring=ring)
        for r in range(spec.R):
            ko.append_token(host, tables[r], lens[r], bs, kn_store[r], None if w is None else w[r])
        for W in (1, 5, spec.W, 12):
            _, _, va = _select_with_ring(kk, dev, bt, vb, W, spec.K, ring, w_dev, spec.R, D)
            assert kk.kk_device_error() == 0
            for r in range(spec.R):
                va_o = ko.anchor(host, tables[r], lens[r], bs, W, None if w is None else w[r])
                assert_vec_close(va[r][None], va_o[None], f"step {step} W={W} r={r} anchor")
        _check_positions(ring, lens)


def test_stale_ring_slot_is_reported(kk):
    spec = SPECS["bf16"]()
    dev = DeviceCache(spec)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    ring = kk.AnchorRing(spec.R, spec.W, spec.D)
    kk.kk_anchor_ring_fill(dev.desc, dev.bt, ring)
    assert kk.kk_device_error() == 0
    _, _, good = _select_with_ring(kk, dev, dev.bt, vb, spec.W, spec.K, ring, None, spec.R, spec.D)
    T0 = spec.seq_lens[0]
    ring.pos[0, (T0 - 1) % spec.W] = T0 - 1 - spec.W  # the slot holds an older token
    _, _, va = _select_with_ring(kk, dev, dev.bt, vb, spec.W, spec.K, ring, None, spec.R, spec.D)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    # the stale row counts as zero; the other requests are untouched
    assert not np.allclose(va[0], good[0])
    np.testing.assert_array_equal(va[1:], good[1:])
