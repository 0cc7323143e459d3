"""Hierarchical Grid -> Chunk -> Page selection ("Key-Key Semantic Affinity"
page, §5.1) through the C ABI against the fp64 oracle: the coarse levels'
representations, and the level-by-level selection with masked children,
for several fan-outs, retention shares and request lengths."""
import numpy as np
import pytest
import torch

from oracle import kk_oracle as ko
from tests.helpers import assert_scores_close, assert_topk_valid, assert_vec_close

pytestmark = pytest.mark.gpu

GAP = 1e-5  # every cut between kept and dropped members is wider than this (fp32 scores agree)


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32).cuda()


def _case(nb, D, seed, topics=12):
    """A v_b table with planted topics (fp32), shuffled pages, and one anchor per request."""
    rng = np.random.default_rng(seed)
    R = len(nb)
    offsets = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
    P = int(offsets[-1]) + 7
    pages = rng.permutation(P)[: offsets[-1]].astype(np.int32)
    cent = rng.standard_normal((topics, D))
    cent /= np.linalg.norm(cent, axis=1, keepdims=True)
    vb = (0.3 * rng.standard_normal((P, D))).astype(np.float32)
    for r in range(R):
        seg = rng.integers(0, topics, size=(nb[r] + 31) // 32)  # topic runs of 32 blocks
        for j in range(nb[r]):
            vb[pages[offsets[r] + j]] += (1.5 * cent[seg[j // 32]]).astype(np.float32)
    va = np.stack([1.5 * cent[rng.integers(0, topics)] + 0.2 * rng.standard_normal(D) for _ in range(R)])
    return offsets, pages, vb, va.astype(np.float32)


def _cuts_are_clear(vb_l, va, cp, gc, pm):
    """Every level's boundary between kept and dropped members is wider than GAP."""
    chunks, grids = ko.hier_reps(vb_l, cp, gc)
    _, _, _, gk, ck = ko.hier_select(vb_l, va, 1, cp, gc, pm)
    def clear(scores, members, kept):
        drop = np.setdiff1d(members, kept)
        return len(drop) == 0 or len(kept) == 0 or scores[kept].min() - scores[drop].max() > GAP
    G, C, nb = len(grids), len(chunks), len(vb_l)
    ca = np.array([c for c in range(C) if c // gc in set(gk.tolist())], dtype=np.int64)
    pa = np.array([j for j in range(nb) if j // cp in set(ck.tolist())], dtype=np.int64)
    s = ko.affinity(vb_l, va)
    pk = ko._keep(s, pa, pm[2])
    return (clear(ko.affinity(grids, va), np.arange(G), gk) and clear(ko.affinity(chunks, va), ca, ck)
            and clear(s, pa, pk))


@pytest.mark.parametrize("cp,gc,pm,K", [
    (64, 8, (500, 200, 100), 64),
    (4, 3, (500, 200, 100), 16),
    (8, 2, (700, 400, 250), 256),
    (64, 8, (1000, 1000, 100), 128),
    (16, 4, (300, 300, 500), 5),
])
def test_hier_select(kk, cp, gc, pm, K):
    _check_hier(kk, [1024, 300, 77, 1, 2048, 0], 128, cp, gc, pm, K, seed=cp * 100 + gc)


@pytest.mark.parametrize("cp,gc,pm,K,seed", [
    (16, 4, (500, 400, 300), 32, 46),
    (16, 4, (500, 400, 300), 10, 46),
    (16, 4, (500, 400, 5), 32, 41),
    (64, 8, (500, 200, 100), 40, 41),
])
def test_hier_select_long_requests(kk, cp, gc, pm, K, seed):
    """Two long requests, so each is scored by a cluster of CTAs, each CTA
    taking every CL-th kept Chunk: K 32, K 10, a block level that keeps fewer
    blocks than K, and K 40."""
    _check_hier(kk, [20000, 16000], 128, cp, gc, pm, K, seed)


@pytest.mark.parametrize("D", [32, 64, 256])
def test_hier_select_head_dims(kk, D):
    """Other head dims, with requests whose Grids and Chunks are scored in
    one round of row loads, in two, and through the Chunk list (700, 1200
    and 3000 blocks at 8 blocks a Chunk, 4 Chunks a Grid; at D 256 a warp
    takes 8 rows a round, so the 1200-block request takes the list)."""
    _check_hier(kk, [700, 1200, 3000, 1, 150], D, 8, 4, (500, 300, 200), 24, seed=1)


def _check_hier(kk, nb, D, cp, gc, pm, K, seed):
    offsets, pages, vb, va = _case(nb, D, seed=seed)
    R = len(nb)
    bt = kk.BlockTable(_i32(pages), _i32(offsets), None, max(nb))
    C_max = -(-max(nb) // cp)
    G_max = -(-C_max // gc)
    vb_d = torch.from_numpy(vb).cuda()
    chunk = torch.full((R, C_max, D), 3.0, device="cuda")
    grid = torch.full((R, G_max, D), 3.0, device="cuda")
    kk.kk_hier_reps(vb_d, bt, cp, gc, chunk, grid)
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    kept = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    kk.kk_hier_select(vb_d, bt, chunk, grid, torch.from_numpy(va).cuda(), cp, gc, pm, idx, top, kept)
    assert kk.kk_device_error() == 0
    g_chunk, g_grid = chunk.cpu().numpy(), grid.cpu().numpy()
    g_idx, g_top, g_kept = idx.cpu().numpy(), top.cpu().numpy(), kept.cpu().numpy()
    vb64 = vb.astype(np.float64)
    for r in range(R):
        vb_l = vb64[pages[offsets[r]:offsets[r + 1]]]
        ch, gr = ko.hier_reps(vb_l, cp, gc) if nb[r] else (np.zeros((0, D)), np.zeros((0, D)))
        if len(ch):
            assert_vec_close(g_chunk[r, :len(ch)], ch, f"r={r} chunks")
            assert_vec_close(g_grid[r, :len(gr)], gr, f"r={r} grids")
        assert np.all(g_chunk[r, len(ch):] == 0) and np.all(g_grid[r, len(gr):] == 0)
        want_idx, want_val, want_kept, _, _ = ko.hier_select(vb_l, va[r].astype(np.float64), max(1, nb[r]), cp, gc,
                                                             pm)
        assert g_kept[r] == want_kept, (r, g_kept[r], want_kept)
        if nb[r]:
            assert _cuts_are_clear(vb_l, va[r].astype(np.float64), cp, gc, pm), f"r={r}: a cut is a near-tie"
        kept_set = want_idx[:want_kept]
        m = min(K, want_kept)
        assert np.all(g_idx[r, m:] == -1) and np.all(np.isneginf(g_top[r, m:]))
        if m == 0:
            continue
        s = ko.affinity(vb_l, va[r].astype(np.float64))
        sel = g_idx[r, :m].astype(np.int64)
        assert len(set(sel.tolist())) == m and set(sel.tolist()) <= set(kept_set.tolist()), f"r={r}"
        rest = np.setdiff1d(kept_set, sel)
        if len(rest):
            assert s[sel].min() >= s[rest].max() - 1e-6, f"r={r}: not the best {m} of the kept blocks"
        assert np.all(np.diff(g_top[r, :m]) <= 0)
        assert_scores_close(g_top[r, :m].astype(np.float64), s[sel], f"r={r} top")


def test_hier_everything_kept_is_plain_topk(kk):
    """permille 1000/1000/1000: every block is kept, in kk_score_topk order."""
    nb = [500, 130]
    D = 64
    offsets, pages, vb, va = _case(nb, D, seed=9)
    bt = kk.BlockTable(_i32(pages), _i32(offsets), None, max(nb))
    vb_d, va_d = torch.from_numpy(vb).cuda(), torch.from_numpy(va).cuda()
    C_max, G_max = -(-max(nb) // 64), -(-(-(-max(nb) // 64)) // 8)
    chunk = torch.zeros((2, C_max, D), device="cuda")
    grid = torch.zeros((2, G_max, D), device="cuda")
    kk.kk_hier_reps(vb_d, bt, 64, 8, chunk, grid)
    K = 256
    i1 = torch.zeros((2, K), dtype=torch.int32, device="cuda")
    i2 = torch.zeros_like(i1)
    t1 = torch.zeros((2, K), device="cuda")
    t2 = torch.zeros_like(t1)
    kk.kk_hier_select(vb_d, bt, chunk, grid, va_d, 64, 8, (1000, 1000, 1000), i1, t1)
    kk.kk_score_topk(vb_d, bt, va_d, K, i2, top_scores=t2)
    assert kk.kk_device_error() == 0
    assert torch.equal(i1, i2) and torch.equal(t1, t2)


def test_hier_select_split_request(kk):
    """One request of 70000 blocks whose kept Chunks hold ~35000 blocks: with
    a workspace, their blocks are scored by several clusters, which meet in
    the workspace. The Grid and Chunk cuts are clear, so the active blocks
    are the oracle's; the output is the best K of them (ties within 1e-6 may
    swap) and the kept count is exact."""
    nb, D, cp, gc, pm, K = [70000], 128, 64, 8, (1000, 500, 100), 64
    offsets, pages, vb, va = _case(nb, D, seed=71)
    bt = kk.BlockTable(_i32(pages), _i32(offsets), None, nb[0])
    C_max = -(-nb[0] // cp)
    G_max = -(-C_max // gc)
    vb_d = torch.from_numpy(vb).cuda()
    chunk = torch.zeros((1, C_max, D), device="cuda")
    grid = torch.zeros((1, G_max, D), device="cuda")
    kk.kk_hier_reps(vb_d, bt, cp, gc, chunk, grid)
    ws = torch.zeros(kk.kk_select_step_workspace_bytes(1, nb[0], K), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    vb_l = vb.astype(np.float64)[pages]
    va0 = va[0].astype(np.float64)
    chunks, grids = ko.hier_reps(vb_l, cp, gc)
    _, _, want_kept, gk, ck = ko.hier_select(vb_l, va0, 1, cp, gc, pm)
    ca = np.array([c for c in range(len(chunks)) if c // gc in set(gk.tolist())], dtype=np.int64)
    sc = ko.affinity(chunks, va0)
    drop = np.setdiff1d(ca, ck)
    assert sc[ck].min() - sc[drop].max() > GAP, "the Chunk cut is a near-tie"
    active = np.array([j for j in range(nb[0]) if j // cp in set(ck.tolist())], dtype=np.int64)
    s = np.full(nb[0], -np.inf)  # blocks outside the kept Chunks are never candidates
    s[active] = ko.affinity(vb_l, va0)[active]
    for rep in range(3):
        idx = torch.zeros((1, K), dtype=torch.int32, device="cuda")
        top = torch.zeros((1, K), device="cuda")
        kept = torch.zeros(1, dtype=torch.int32, device="cuda")
        kk.kk_hier_select(vb_d, bt, chunk, grid, torch.from_numpy(va).cuda(), cp, gc, pm, idx, top, kept,
                          workspace=ws)
        assert kk.kk_device_error() == 0
        assert int(kept.item()) == want_kept
        assert_topk_valid(idx.cpu().numpy()[0], top.cpu().numpy()[0], s, K, f"call {rep}")
        # the indices are logical blocks of the active set
        sel = idx.cpu().numpy()[0]
        assert set(sel.tolist()) <= set(active.tolist())
        assert ws[:8].cpu().numpy().view(np.uint64)[0] == 0
