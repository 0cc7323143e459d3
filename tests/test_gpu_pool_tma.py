"""kk_pool_blocks with more blocks than SMs, the regime served by the
persistent TMA pipeline: parity with the fp64 oracle on every layout (layer-,
token- and page-major), boxes of several tokens, heads or layers, token
boxes smaller than a block, block sizes that are not powers of two, partial
and empty blocks, explicit weights, and bad entries mixed into a long list."""
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


def _lens(bs, blocks, ragged):
    """Three requests totalling `blocks` blocks, each with a partial last block."""
    per = [blocks // 3, blocks // 3, blocks - 2 * (blocks // 3)]
    return [bs * (b - 1) + max(1, (r * bs) // 4) for b, r in zip(per, ragged)]


def tma_specs():
    return [
        # 16-token blocks: a box holds every head of two layers
        synth.qwen7b(L=4, H=4, D=128, bs=16, seq_lens=_lens(16, 420, [1, 2, 3]), num_topics=6, W=8, K=8,
                     shuffle_pages=True, extra_pages=9),
        # L not divisible by the layers a box could hold
        synth.qwen7b(L=3, H=4, D=128, bs=16, seq_lens=_lens(16, 330, [3, 1, 2]), num_topics=4, W=8, K=8),
        # token-major pages: the head axis is the innermost strided axis
        synth.tiny_05b(L=2, H=3, D=64, bs=32, seq_lens=_lens(32, 360, [2, 3, 1]), num_topics=4, W=8, K=8,
                       layout="LPTHD", shuffle_pages=True),
        # page-major pool, D=256: two 64-token boxes per 128-token block
        synth.qwen7b(L=2, H=2, D=256, bs=128, seq_lens=_lens(128, 320, [1, 3, 2]), num_topics=3, W=8, K=8,
                     layout="PLHTD", shuffle_pages=True, extra_pages=5),
        # a block size that is not a power of two, D=32 (many layers per box)
        synth.qwen7b(L=6, H=2, D=32, bs=24, seq_lens=_lens(24, 400, [2, 1, 3]), num_topics=5, W=8, K=8),
        # fp32 rows of 512 bytes
        synth.tiny_05b(L=3, H=4, D=128, bs=8, seq_lens=_lens(8, 500, [3, 2, 1]), num_topics=4, W=8, K=8,
                       layout="PLHTD"),
    ]


SPECS = tma_specs()
IDS = [f"{s.dtype}-D{s.D}-bs{s.bs}-L{s.L}H{s.H}-{s.layout}" for s in SPECS]


@pytest.fixture(scope="module", params=range(len(SPECS)), ids=IDS)
def dev(request, kk):
    d = DeviceCache(SPECS[request.param])
    assert d.spec.total_blocks >= 2 * torch.cuda.get_device_properties(0).multi_processor_count
    return d


def test_generator_bits_match_numpy(dev):
    if dev.spec.layout != "PLHTD":
        pytest.skip("the other layouts are checked with the small parity specs")
    want = synth.gen_paged_numpy(dev.spec)
    got = dev.storage.cpu().numpy()
    if dev.spec.dtype == "bf16":
        got = got.view(np.uint16)
    np.testing.assert_array_equal(got.view(np.uint8), want.view(np.uint8))


def test_pool_many_blocks(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    vb = torch.full((sp.num_pages, sp.D), 7.0, device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0
    got = vb.cpu().numpy()
    assert_vec_close(got[sp.pages], ko.pool_blocks(kc, sp.pages, sp.n_valid), "vb")
    untouched = np.setdiff1d(np.arange(sp.num_pages), sp.pages)
    assert np.all(got[untouched] == 7.0)


def test_pool_many_blocks_weighted(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    rng = np.random.default_rng(11)
    w = rng.uniform(0.1, 2.0, size=(4, sp.L * sp.H)).astype(np.float32)
    w_set = rng.integers(0, 4, size=sp.total_blocks).astype(np.int32)
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb, head_w=torch.from_numpy(w).cuda(),
                      w_set=torch.from_numpy(w_set).cuda())
    assert kk.kk_device_error() == 0
    want = ko.pool_blocks(kc, sp.pages, sp.n_valid, w.astype(np.float64), w_set)
    assert_vec_close(vb.cpu().numpy()[sp.pages], want, "weighted vb")


def test_pool_many_blocks_shorter_counts(kk, dev):
    """n_valid below the table's (empty blocks, a few tokens, one token box
    short), and the same page listed twice."""
    sp = dev.spec
    kc = dev.host_view()
    rng = np.random.default_rng(3)
    n = sp.total_blocks
    nv = np.minimum(rng.integers(0, sp.bs + 1, size=n), sp.n_valid).astype(np.int32)  # tails hold NaN
    nv[:7] = 0
    nv[7:15] = 1
    pages = sp.pages.copy()
    pages[-1] = pages[0]
    nv[-1] = nv[0]
    vb = torch.full((sp.num_pages, sp.D), 3.0, device="cuda")
    kk.kk_pool_blocks(dev.desc, torch.from_numpy(pages).cuda(), torch.from_numpy(nv).cuda(), vb)
    assert kk.kk_device_error() == 0
    got = vb.cpu().numpy()
    want = ko.pool_blocks(kc, pages, nv)
    assert_vec_close(got[pages], want, "vb")
    assert np.all(got[pages[:7]] == 0.0)


def test_bad_entries_in_a_long_list(kk):
    sp = synth.qwen7b(L=2, H=2, D=64, bs=16, seq_lens=[16 * 400], num_topics=3, W=4, K=3)
    dev = DeviceCache(sp)
    kc = dev.host_view()
    n = sp.total_blocks
    pages = sp.pages.copy()
    nv = sp.n_valid.copy()
    bad = np.zeros(n, bool)
    bad[[5, 200, 399]] = True
    pages[5] = sp.num_pages  # out of range
    pages[200] = -1
    nv[399] = sp.bs + 1  # more tokens than a block holds
    vb = torch.full((sp.num_pages, sp.D), 9.0, device="cuda")
    assert kk.kk_device_error() == 0
    kk.kk_pool_blocks(dev.desc, torch.from_numpy(pages).cuda(), torch.from_numpy(nv).cuda(), vb)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    got = vb.cpu().numpy()
    ok = ~bad
    assert_vec_close(got[pages[ok]], ko.pool_blocks(kc, pages[ok], nv[ok]), "valid rows")
    assert np.all(got[sp.pages[399]] == 9.0)  # the skipped entry wrote nothing
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0


def test_both_regimes_agree(kk):
    """The same blocks pooled as one long list and in lists shorter than the
    SM count (the cluster kernel) give the same rows up to rounding."""
    sp = synth.qwen7b(L=3, H=2, D=128, bs=32, seq_lens=[32 * 320 + 5], num_topics=3, W=4, K=3)
    dev = DeviceCache(sp)
    vb_long = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb_long)
    vb_short = torch.zeros_like(vb_long)
    for s in range(0, sp.total_blocks, 100):
        kk.kk_pool_blocks(dev.desc, dev.pages[s:s + 100], dev.n_valid[s:s + 100], vb_short)
    assert kk.kk_device_error() == 0
    a, b = vb_long.cpu().numpy(), vb_short.cpu().numpy()
    assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max()


def test_weighted_pool_many_blocks(kk, dev):
    """kk_pool_blocks_weighted on more blocks than SMs: the per-(layer, head)
    token sums and squares come from the TMA ring (token-innermost layouts),
    then the head-variance weights and the weighted v_b."""
    sp = dev.spec
    kc = dev.host_view()
    LH = sp.L * sp.H
    ws = torch.empty(kk.kk_head_variance_workspace_bytes(dev.desc, sp.total_blocks, sp.R), dtype=torch.uint8,
                     device="cuda")
    w_out = torch.zeros((sp.R, LH), device="cuda")
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks_weighted(dev.desc, dev.bt, sp.total_blocks, w_out, vb, ws)
    assert kk.kk_device_error() == 0
    want_w = np.stack([ko.head_variance_weights(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs) for r in range(sp.R)])
    assert_vec_close(w_out.cpu().numpy(), want_w, "head weights")
    got = vb.cpu().numpy()
    for r in range(sp.R):
        blk = slice(sp.offsets[r], sp.offsets[r + 1])
        want = ko.pool_blocks(kc, sp.pages[blk], sp.n_valid[blk], [want_w[r]], [0] * (blk.stop - blk.start))
        assert_vec_close(got[sp.pages[blk]], want, f"weighted vb r={r}")
