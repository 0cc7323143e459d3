"""GPU parity through the C ABI against the fp64 CPU oracle, on sizes the
oracle finishes in seconds: several CTA tiles, ragged tails, partial blocks,
shuffled pages, both dtypes, every supported head_dim, both layouts, and the
degenerate cases (empty blocks, empty requests, K beyond the candidates,
ties, bad indices)."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import (DeviceCache, assert_scores_close, assert_topk_valid, assert_vec_close)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def small_specs():
    return [
        # fp32, D=64, partial last block, two requests
        synth.tiny_05b(L=5, seq_lens=[16 * 40 + 7, 16 * 9], num_topics=4, W=8, K=16),
        # bf16, D=128, token-major pages, shuffled pages and spare pages
        synth.qwen7b(L=3, H=4, bs=32, seq_lens=[32 * 70 + 31, 5, 32 * 3], num_topics=8, W=40, K=24,
                     shuffle_pages=True, extra_pages=11, layout="LPTHD"),
        # bf16, D=256 and D=32 geometries
        synth.qwen7b(L=2, H=2, D=256, bs=16, seq_lens=[16 * 33 + 1], num_topics=3, W=20, K=8),
        synth.qwen7b(L=4, H=3, D=32, bs=8, seq_lens=[8 * 100, 8 * 64 + 3], num_topics=5, W=3, K=40),
        # fp32 D=32 and D=128, block size 1 and 64
        synth.tiny_05b(L=2, H=1, D=32, bs=1, seq_lens=[300], num_topics=3, W=5, K=7),
        synth.tiny_05b(L=2, H=2, D=128, bs=64, seq_lens=[64 * 11 + 60], num_topics=4, W=70, K=5),
    ]


SPECS = small_specs()
IDS = [f"{s.dtype}-D{s.D}-bs{s.bs}-{s.layout}" for s in SPECS]


@pytest.fixture(scope="module", params=range(len(SPECS)), ids=IDS)
def dev(request, kk):
    return DeviceCache(SPECS[request.param])


def oracle_vb_table(dev, kc):
    sp = dev.spec
    vb = np.zeros((sp.num_pages, sp.D))
    vb[sp.pages] = ko.pool_blocks(kc, sp.pages, sp.n_valid)
    return vb


def test_generator_bits_match_numpy(dev):
    want = synth.gen_paged_numpy(dev.spec)
    got = dev.storage.cpu().numpy()
    if dev.spec.dtype == "bf16":
        got = got.view(np.uint16)
    np.testing.assert_array_equal(got.view(np.uint8), want.view(np.uint8))


def test_pool_blocks_unweighted(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    vb = torch.full((sp.num_pages, sp.D), 7.0, device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0
    got = vb.cpu().numpy()
    assert_vec_close(got[sp.pages], ko.pool_blocks(kc, sp.pages, sp.n_valid), "vb")
    untouched = np.setdiff1d(np.arange(sp.num_pages), sp.pages)
    assert np.all(got[untouched] == 7.0)


def test_pool_blocks_explicit_weights(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    rng = np.random.default_rng(5)
    LH = sp.L * sp.H
    w = rng.uniform(0.1, 2.0, size=(3, LH)).astype(np.float32)
    w_set = rng.integers(0, 3, size=sp.total_blocks).astype(np.int32)
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb, head_w=torch.from_numpy(w).cuda(),
                      w_set=torch.from_numpy(w_set).cuda())
    assert kk.kk_device_error() == 0
    want = ko.pool_blocks(kc, sp.pages, sp.n_valid, w.astype(np.float64), w_set)
    assert_vec_close(vb.cpu().numpy()[sp.pages], want, "weighted vb")


def test_anchor(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    for W in (1, sp.W, sp.bs + 3, 1024):
        va = torch.zeros((sp.R, sp.D), device="cuda")
        kk.kk_anchor(dev.desc, dev.bt, W, va)
        assert kk.kk_device_error() == 0
        want = np.stack([ko.anchor(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs, W) for r in range(sp.R)])
        assert_vec_close(va.cpu().numpy(), want, f"va W={W}")


def test_head_variance_and_weighted_pool(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    LH = sp.L * sp.H
    ws = torch.empty(kk.kk_head_variance_workspace_bytes(dev.desc, sp.total_blocks, sp.R), dtype=torch.uint8,
                     device="cuda")
    w_only = torch.zeros((sp.R, LH), device="cuda")
    kk.kk_head_variance(dev.desc, dev.bt, sp.total_blocks, w_only, ws)
    w_out = torch.zeros((sp.R, LH), device="cuda")
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks_weighted(dev.desc, dev.bt, sp.total_blocks, w_out, vb, ws)
    assert kk.kk_device_error() == 0
    want_w = np.stack([ko.head_variance_weights(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs) for r in range(sp.R)])
    assert_vec_close(w_only.cpu().numpy(), want_w, "head weights")
    assert torch.equal(w_only, w_out)
    got = vb.cpu().numpy()
    for r in range(sp.R):
        blk = slice(sp.offsets[r], sp.offsets[r + 1])
        want = ko.pool_blocks(kc, sp.pages[blk], sp.n_valid[blk], [want_w[r]], [0] * (blk.stop - blk.start))
        assert_vec_close(got[sp.pages[blk]], want, f"weighted vb r={r}")
    # the anchor with the same weights
    va = torch.zeros((sp.R, sp.D), device="cuda")
    kk.kk_anchor(dev.desc, dev.bt, sp.W, va, head_w=w_out)
    want_va = np.stack([ko.anchor(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs, sp.W, want_w[r]) for r in range(sp.R)])
    assert_vec_close(va.cpu().numpy(), want_va, "weighted va")


def test_select_step_matches_oracle(kk, dev):
    sp = dev.spec
    kc = dev.host_view()
    vb_o = oracle_vb_table(dev, kc)
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    for K in (1, sp.K, 256):
        idx = torch.zeros((sp.R, K), dtype=torch.int32, device="cuda")
        top = torch.zeros((sp.R, K), device="cuda")
        va = torch.zeros((sp.R, sp.D), device="cuda")
        scores = torch.zeros(sp.total_blocks, device="cuda")
        kk.kk_select_step(dev.desc, dev.bt, sp.W, vb, K, idx, top, va=va, scores=scores)
        assert kk.kk_device_error() == 0
        for r in range(sp.R):
            va_o = ko.anchor(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs, sp.W)
            assert_vec_close(va.cpu().numpy()[r], va_o, "step va")
            s_o = ko.affinity(vb_o[sp.pages_of(r)], va_o)
            assert_scores_close(scores.cpu().numpy()[sp.offsets[r]:sp.offsets[r + 1]], s_o, f"step scores r={r}")
            assert_topk_valid(idx.cpu().numpy()[r], top.cpu().numpy()[r], s_o, K, f"step top-K r={r} K={K}")


def test_score_and_topk_on_given_vectors(kk, dev):
    """kk_score / kk_topk / kk_score_topk on a v_b table and anchors drawn by
    the generator (so both sides read identical float32 inputs)."""
    sp = dev.spec
    rows = synth.RowsSpec(N=sp.num_pages, D=sp.D, num_topics=4, scale=1.0, sigma=0.3, seed=9, stream=4)
    vb_np = synth.gen_rows_numpy(rows)
    vb_np[sp.pages[::7]] = 0.0  # some zero vectors: score 0.5
    anc = synth.RowsSpec(N=sp.R, D=sp.D, num_topics=4, scale=1.0, sigma=0.3, seed=9, stream=5, centroid_seed=9)
    va_np = synth.gen_rows_numpy(anc)
    vb, va = torch.from_numpy(vb_np).cuda(), torch.from_numpy(va_np).cuda()
    scores = torch.zeros(sp.total_blocks, device="cuda")
    kk.kk_score(vb, dev.bt, va, scores)
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top = torch.zeros((sp.R, sp.K), device="cuda")
    kk.kk_score_topk(vb, dev.bt, va, sp.K, idx, top)
    idx2 = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top2 = torch.zeros((sp.R, sp.K), device="cuda")
    kk.kk_topk(scores, dev.offsets, max(sp.nb), sp.K, idx2, top2)
    assert kk.kk_device_error() == 0
    s_gpu = scores.cpu().numpy()
    for r in range(sp.R):
        s_o = ko.affinity(vb_np[sp.pages_of(r)], va_np[r])
        assert_scores_close(s_gpu[sp.offsets[r]:sp.offsets[r + 1]], s_o, f"scores r={r}")
        assert_topk_valid(idx.cpu().numpy()[r], top.cpu().numpy()[r], s_o, sp.K, f"score_topk r={r}")
        # kk_topk on the GPU's own scores is exact: compare with the oracle's top-K of those floats
        want_idx, want_val = ko.topk(s_gpu[sp.offsets[r]:sp.offsets[r + 1]], sp.K)
        np.testing.assert_array_equal(idx2.cpu().numpy()[r], want_idx)
        np.testing.assert_array_equal(top2.cpu().numpy()[r], want_val.astype(np.float32))


def test_topk_exact_with_ties_and_many_tiles(kk):
    rng = np.random.default_rng(3)
    sizes = [0, 1, 5, 255, 256, 257, 1000, 4097, 20000]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    scores = rng.integers(0, 50, size=offsets[-1]).astype(np.float32) / 50  # many exact ties
    scores[offsets[6]:offsets[7]] = 0.25  # a request of all-equal scores
    for K in (1, 3, 64, 256):
        idx = torch.zeros((len(sizes), K), dtype=torch.int32, device="cuda")
        top = torch.zeros((len(sizes), K), device="cuda")
        kk.kk_topk(torch.from_numpy(scores).cuda(), torch.from_numpy(offsets).cuda(), max(sizes), K, idx, top)
        assert kk.kk_device_error() == 0
        for r in range(len(sizes)):
            want_idx, want_val = ko.topk(scores[offsets[r]:offsets[r + 1]], K)
            np.testing.assert_array_equal(idx.cpu().numpy()[r], want_idx, err_msg=f"r={r} K={K}")
            np.testing.assert_array_equal(top.cpu().numpy()[r], want_val.astype(np.float32))


@pytest.mark.parametrize("sizes", [[65536], [100003, 0, 70001], [40000, 30000, 1], [9000] * 5 + [300000]])
def test_topk_split_long_requests(kk, sizes):
    """Requests long enough that their candidates are split over several
    clusters (each ranks its share; the last to finish merges the lists):
    exact against the oracle with many ties, an empty and a one-candidate
    request among them, K up to 256, and repeated calls (the per-request
    arrival counters must be back at zero after every call)."""
    rng = np.random.default_rng(len(sizes) * 7 + sizes[0])
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    scores = rng.integers(0, 4000, size=offsets[-1]).astype(np.float32) / 4000
    s_gpu = torch.from_numpy(scores).cuda()
    off_gpu = torch.from_numpy(offsets).cuda()
    for K in (1, 100, 256):
        want = [ko.topk(scores[offsets[r]:offsets[r + 1]], K) for r in range(len(sizes))]
        nws = kk.kk_select_step_workspace_bytes(len(sizes), max(sizes), K)
        assert nws > 0
        ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
        for rep in range(4):
            idx = torch.full((len(sizes), K), 7, dtype=torch.int32, device="cuda")
            top = torch.zeros((len(sizes), K), device="cuda")
            # the last call without a workspace: every request on one cluster
            kk.kk_topk(s_gpu, off_gpu, max(sizes), K, idx, top, workspace=ws if rep < 3 else None)
            assert kk.kk_device_error() == 0
            for r in range(len(sizes)):
                np.testing.assert_array_equal(idx.cpu().numpy()[r], want[r][0], err_msg=f"r={r} K={K} call {rep}")
                np.testing.assert_array_equal(top.cpu().numpy()[r], want[r][1].astype(np.float32))


def test_coarse_means(kk, dev):
    sp = dev.spec
    rows = synth.RowsSpec(N=sp.num_pages, D=sp.D, num_topics=3, scale=1.0, sigma=0.5, seed=12, stream=6)
    vb_np = synth.gen_rows_numpy(rows)
    vb = torch.from_numpy(vb_np).cuda()
    for group in (1, 3, 8, 64):
        ng = (max(sp.nb) + group - 1) // group
        out = torch.full((sp.R, ng, sp.D), 5.0, device="cuda")
        kk.kk_coarse_means(vb, dev.bt, group, out)
        assert kk.kk_device_error() == 0
        got = out.cpu().numpy()
        for r in range(sp.R):
            want = ko.coarse_means(vb_np[sp.pages_of(r)], group)
            assert_vec_close(got[r, :len(want)], want, f"coarse g={group} r={r}")
            assert np.all(got[r, len(want):] == 0.0)


def test_empty_blocks_and_requests(kk):
    sp = synth.qwen7b(L=2, H=2, D=64, bs=8, seq_lens=[0, 20, 0, 8], num_topics=2, W=4, K=5, extra_pages=2)
    dev = DeviceCache(sp)
    kc = dev.host_view()
    # a block pooled with zero valid tokens is the zero vector
    vb = torch.full((sp.num_pages, sp.D), 3.0, device="cuda")
    pages = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")
    nv = torch.tensor([0, 8, 5], dtype=torch.int32, device="cuda")
    kk.kk_pool_blocks(dev.desc, pages, nv, vb)
    assert kk.kk_device_error() == 0
    got = vb.cpu().numpy()
    assert np.all(got[0] == 0.0)
    assert_vec_close(got[[1, 3]], ko.pool_blocks(kc, [1, 3], [8, 5]), "vb")
    # empty requests: zero anchor, all slots -1 / -inf
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top = torch.zeros((sp.R, sp.K), device="cuda")
    va = torch.ones((sp.R, sp.D), device="cuda")
    kk.kk_select_step(dev.desc, dev.bt, sp.W, vb, sp.K, idx, top, va=va)
    assert kk.kk_device_error() == 0
    for r in (0, 2):
        assert np.all(va.cpu().numpy()[r] == 0)
        assert np.all(idx.cpu().numpy()[r] == -1)
        assert np.all(np.isneginf(top.cpu().numpy()[r]))
    assert list(idx.cpu().numpy()[3][:1]) == [0] and np.all(idx.cpu().numpy()[3][1:] == -1)


def test_bad_indices_are_reported_not_faulted(kk):
    sp = synth.qwen7b(L=2, H=2, D=64, bs=8, seq_lens=[40, 16], num_topics=2, W=4, K=3)
    dev = DeviceCache(sp)
    assert kk.kk_device_error() == 0
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    # page id out of range, n_valid above block size: recorded, skipped
    kk.kk_pool_blocks(dev.desc, torch.tensor([0, 99], dtype=torch.int32, device="cuda"),
                      torch.tensor([8, 8], dtype=torch.int32, device="cuda"), vb)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    assert kk.kk_device_error() == 0  # cleared by the read
    kk.kk_pool_blocks(dev.desc, torch.tensor([0], dtype=torch.int32, device="cuda"),
                      torch.tensor([9], dtype=torch.int32, device="cuda"), vb)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    # a block table that disagrees with seq_lens: the request is skipped
    bad_lens = torch.tensor([40, 17], dtype=torch.int32, device="cuda")
    bt = kk.BlockTable(dev.pages, dev.offsets, bad_lens, max(sp.nb))
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    kk.kk_select_step(dev.desc, bt, sp.W, vb, sp.K, idx)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    assert np.all(idx.cpu().numpy()[1] == -1)
    # a page id beyond the table in the block table
    pages = dev.pages.clone()
    pages[2] = 1000
    bt2 = kk.BlockTable(pages, dev.offsets, dev.seq_lens, max(sp.nb))
    scores = torch.zeros(sp.total_blocks, device="cuda")
    va = torch.ones((sp.R, sp.D), device="cuda")
    kk.kk_score(vb, bt2, va, scores)
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    # and the library stays usable
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0


def _pool_inputs(R, N, owned, seed):
    v = synth.RowsSpec(N=N, D=128, num_topics=8, scale=1.5, sigma=0.05, seed=seed, stream=2, dtype="bf16")
    a = synth.RowsSpec(N=R, D=128, num_topics=8, scale=1.5, sigma=0.15, seed=seed, stream=3, dtype="bf16",
                       centroid_seed=seed)
    return synth.gen_rows_numpy(a), synth.gen_rows_numpy(v), synth.owned_mask(R, N, owned, seed + 1)


def check_batched_against_oracle(A, V, mask, K, idx, top, rows=None):
    R, N = A.shape[0], V.shape[0]
    j = np.arange(N)
    for r in (range(R) if rows is None else rows):
        owned = np.flatnonzero((mask[r, j // 32] >> (j % 32).astype(np.uint32)) & 1)
        s_o = ko.affinity(V[owned], A[r])
        pos = {int(b): p for p, b in enumerate(owned)}
        g = idx[r]
        assert all(int(b) in pos for b in g if b >= 0), f"row {r}: picked a block it does not own"
        g_pos = np.array([pos[int(b)] if b >= 0 else -1 for b in g])
        assert_topk_valid(g_pos, top[r], s_o, K, f"batched row {r}")


@pytest.mark.parametrize("R,N,K,owned", [(5, 300, 7, 40), (130, 1000, 16, 300), (3, 129, 256, 129),
                                         (1, 64, 1, 0), (200, 4096, 128, 1024), (129, 257, 33, 250)])
def test_score_pool_batched_small(kk, R, N, K, owned):
    A, V, mask = _pool_inputs(R, N, owned, seed=R + N)
    At = torch.from_numpy(A.view(np.int16)).cuda()
    Vt = torch.from_numpy(V.view(np.int16)).cuda()
    Mt = torch.from_numpy(mask.view(np.int32)).cuda()
    ws = torch.empty(kk.kk_score_pool_batched_workspace_bytes(R, N, K), dtype=torch.uint8, device="cuda")
    results = []
    for _ in range(2):  # a second call must not see the first call's candidate lists
        idx = torch.full((R, K), 7, dtype=torch.int32, device="cuda")
        top = torch.zeros((R, K), device="cuda")
        kk.kk_score_pool_batched(At, Vt, Mt, K, idx, top, ws)
        assert kk.kk_device_error() == 0
        results.append((idx.cpu().numpy(), top.cpu().numpy()))
    np.testing.assert_array_equal(results[0][0], results[1][0])
    np.testing.assert_array_equal(results[0][1], results[1][1])
    check_batched_against_oracle(A, V, mask, K, *results[0])


@pytest.mark.parametrize("K", [1, 5, 128, 256])
def test_score_pool_batched_exact_ties(kk, K):
    """Pools of repeated rows, so whole groups of candidates score exactly
    alike and the order falls to the lower pool index. (a) Every row is the
    anchor's own vector: one score for all, so the select goes straight to
    the radix digits of the 64-bit keys; the top K are the K lowest owned
    indices. (b) Rows 0..31 mod 256 point away from the anchor, the rest are
    the anchor's vector: two scores, the boundary bucket holds more ties than
    are ranked exactly, and the radix select finishes; the top K are the K
    lowest high rows."""
    rng = np.random.default_rng(K)
    R, N = 3, 2048
    a = rng.standard_normal(128).astype(np.float32)
    a_bits = (torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    A = np.tile(a_bits, (R, 1))
    neg = a_bits ^ np.uint16(0x8000)
    full = np.full((R, N // 32), 0xFFFFFFFF, dtype=np.uint32)
    cases = []
    # (a) all rows alike, a random ownership per anchor
    mask_a = synth.owned_mask(R, N, 700, 17)
    cases.append((np.tile(a_bits, (N, 1)), mask_a,
                  [np.flatnonzero((mask_a[r, np.arange(N) // 32] >> (np.arange(N) % 32).astype(np.uint32)) & 1)[:K]
                   for r in range(R)]))
    # (b) the low rows are the negated anchor, every block owned
    low = (np.arange(N) % 256) < 32
    Vb = np.where(low[:, None], neg[None, :], a_bits[None, :]).astype(np.uint16)
    cases.append((Vb, full, [np.flatnonzero(~low)[:K]] * R))
    for V, mask, want in cases:
        At = torch.from_numpy(A.view(np.int16)).cuda()
        Vt = torch.from_numpy(V.view(np.int16)).cuda()
        Mt = torch.from_numpy(mask.view(np.int32)).cuda()
        ws = torch.empty(kk.kk_score_pool_batched_workspace_bytes(R, N, K), dtype=torch.uint8, device="cuda")
        idx = torch.full((R, K), 7, dtype=torch.int32, device="cuda")
        top = torch.zeros((R, K), device="cuda")
        kk.kk_score_pool_batched(At, Vt, Mt, K, idx, top, ws)
        assert kk.kk_device_error() == 0
        g_idx, g_top = idx.cpu().numpy(), top.cpu().numpy()
        for r in range(R):
            np.testing.assert_array_equal(g_idx[r], want[r], err_msg=f"row {r}")
            assert np.all(g_top[r] == g_top[r][0]) and abs(g_top[r][0] - 1.0) < 1e-5
