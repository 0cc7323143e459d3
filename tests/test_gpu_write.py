"""The write side around a decode step, through the C ABI, against the fp64
oracle: the compact table of selected blocks ("Key-Key Semantic Affinity"
page, §5.2 step 4) and incremental pooling fused with the write of each
decode token's Keys (§5.2 step 2)."""
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


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32).cuda()


@pytest.mark.parametrize("K", [1, 7, 64, 256])
def test_compact_table(kk, K):
    rng = np.random.default_rng(K)
    nb = [300, 5, 0, 90, 1]
    offsets = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
    pages = rng.permutation(2000)[: offsets[-1]].astype(np.int32)
    idx = np.full((len(nb), K), -1, dtype=np.int32)
    for r, n in enumerate(nb):
        take = min(n, K)
        chosen = rng.permutation(n)[:take]
        slots = rng.permutation(K)[:take]  # gaps anywhere, as -1
        idx[r, slots] = chosen
    bt = kk.BlockTable(_i32(pages), _i32(offsets), None, max(nb))
    sel_pages = torch.full((len(nb), K), 7, dtype=torch.int32, device="cuda")
    sel_logical = torch.full_like(sel_pages, 7)
    sel_count = torch.full((len(nb),), 7, dtype=torch.int32, device="cuda")
    kk.kk_compact_table(_i32(idx), bt, sel_pages, sel_logical, sel_count)
    assert kk.kk_device_error() == 0
    gp, gl, gc = sel_pages.cpu().numpy(), sel_logical.cpu().numpy(), sel_count.cpu().numpy()
    for r in range(len(nb)):
        want_p, want_l, n = ko.compact_table(pages[offsets[r]:offsets[r + 1]], idx[r])
        np.testing.assert_array_equal(gp[r], want_p)
        np.testing.assert_array_equal(gl[r], want_l)
        assert gc[r] == n


def test_compact_table_reports_bad_indices(kk):
    pages = np.arange(10, dtype=np.int32)
    offsets = np.array([0, 4, 10], dtype=np.int32)
    idx = np.array([[3, 4, -1, 0], [5, -2, 1, 9]], dtype=np.int32)  # 4 is past request 0's table; -2 is invalid
    bt = kk.BlockTable(_i32(pages), _i32(offsets), None, 6)
    sel = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    kk.kk_compact_table(_i32(idx), bt, sel, sel_count=cnt)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    np.testing.assert_array_equal(sel.cpu().numpy(), [[0, 3, -1, -1], [5, 9, -1, -1]])
    np.testing.assert_array_equal(cnt.cpu().numpy(), [2, 2])


def _decode_run(kk, spec, steps, weighted, seed):
    """Append `steps` tokens to every request (requests start at a block
    boundary; spare pages take the new blocks) and check v_b after each token
    and the cache bytes at the end."""
    dev = DeviceCache(spec)
    host = dev.host_view().copy()  # the oracle's own copy of the cache, written by ko.append_token
    rng = np.random.default_rng(seed)
    L, H, D, bs = spec.L, spec.H, spec.D, spec.bs
    spare = list(np.setdiff1d(np.arange(spec.num_pages), spec.pages))
    tables = [list(spec.pages_of(r)) for r in range(spec.R)]
    lens = list(spec.seq_lens)
    w = rng.uniform(0.2, 1.0, size=(spec.R, L * H)).astype(np.float32) if weighted else None
    w_dev = torch.from_numpy(w).cuda() if weighted else None
    block_sum = torch.zeros((spec.num_pages, D), device="cuda")
    vb = torch.full((spec.num_pages, D), 5.0, device="cuda")
    for step in range(steps):
        for r in range(spec.R):
            if lens[r] % bs == 0:
                tables[r].append(spare.pop(0))
            lens[r] += 1
        offsets = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
        pages = np.concatenate(tables).astype(np.int32)
        bt = kk.BlockTable(_i32(pages), _i32(offsets), _i32(lens), max(len(t) for t in tables))
        kn = (1.5 * spec.cs[rng.integers(0, spec.num_topics, size=spec.R)][:, None, None, :]
              + rng.standard_normal((spec.R, L, H, D))).astype(np.float32)
        if spec.dtype == "bf16":
            kn_store = synth.bf16_rne(kn)  # uint16 bits
            k_dev = torch.from_numpy(kn_store.view(np.int16)).cuda()
        else:
            kn_store = kn
            k_dev = torch.from_numpy(kn).cuda()
        kk.kk_append_tokens(dev.desc, bt, k_dev, block_sum, vb, head_w=w_dev)
        assert kk.kk_device_error() == 0
        got = vb.cpu().numpy()
        for r in range(spec.R):
            page, want = ko.append_token(host, tables[r], lens[r], bs, kn_store[r], None if w is None else w[r])
            assert_vec_close(got[page][None, :], want[None, :], f"step {step} r={r} vb")
    # every byte of the cache equals the oracle's copy (appended slots included)
    g = dev.storage.cpu().numpy()
    if spec.dtype == "bf16":
        g = g.view(np.uint16)
    want = np.empty_like(g)
    synth.view_paged(want, spec)[...] = host
    np.testing.assert_array_equal(g.view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("weighted", [False, True])
def test_append_tokens_bf16(kk, weighted):
    spec = synth.qwen7b(L=3, H=2, D=128, bs=16, seq_lens=[16 * 4, 16 * 2, 16], num_topics=4, W=8, K=8,
                        extra_pages=12, shuffle_pages=True)
    _decode_run(kk, spec, steps=35, weighted=weighted, seed=1 + weighted)


def test_append_tokens_fp32_token_major(kk):
    spec = synth.tiny_05b(L=2, H=3, D=64, bs=8, seq_lens=[8 * 3, 8], num_topics=3, W=4, K=4, extra_pages=8,
                          layout="LPTHD")
    _decode_run(kk, spec, steps=19, weighted=False, seed=3)


def test_append_tokens_d32_and_d256(kk):
    for spec in (synth.qwen7b(L=2, H=2, D=32, bs=4, seq_lens=[8, 4], num_topics=2, W=2, K=2, extra_pages=6),
                 synth.qwen7b(L=2, H=1, D=256, bs=4, seq_lens=[4], num_topics=2, W=2, K=2, extra_pages=3,
                              layout="PLHTD")):
        _decode_run(kk, spec, steps=9, weighted=False, seed=4)


def test_append_tokens_reports_a_bad_table(kk):
    spec = synth.qwen7b(L=2, H=2, D=64, bs=8, seq_lens=[16, 8], num_topics=2, W=2, K=2, extra_pages=2)
    dev = DeviceCache(spec)
    before = dev.storage.clone()
    lens = np.array([17, 9], dtype=np.int32)  # the tables were not grown: both requests are skipped
    bt = kk.BlockTable(dev.pages, dev.offsets, _i32(lens), max(spec.nb))
    k_new = torch.zeros((2, 2, 2, 64), dtype=torch.int16, device="cuda")
    block_sum = torch.zeros((spec.num_pages, 64), device="cuda")
    vb = torch.zeros((spec.num_pages, 64), device="cuda")
    kk.kk_append_tokens(dev.desc, bt, k_new, block_sum, vb)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    assert torch.equal(dev.storage, before) and not vb.any()
