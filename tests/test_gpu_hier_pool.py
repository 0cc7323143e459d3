"""Hierarchical selection over a shared pool ("Key-Key Semantic Affinity"
page, §5.1: the Grid, Chunk and block representations scored against the
anchors in one product, then parent -> child masks) through the C ABI
against the fp64 oracle: the coarse rows of the pool matrix, and the
level-by-level selection per anchor for several fan-outs, masks and
retention shares, ragged sizes, and both the listed and the streamed block
paths."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import assert_scores_close

pytestmark = pytest.mark.gpu

GAP = 1e-5  # a level's cut is compared exactly when it is wider than this (fp32 vs fp64 scores)


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _rows(N, R, seed, run=32, topics=12):
    """bf16 pool rows with a topic per run of blocks, and anchors near the topics."""
    v = synth.RowsSpec(N=N, D=128, num_topics=topics, scale=1.5, sigma=0.3, seed=seed, stream=2, dtype="bf16",
                       topics=synth.topic_runs(N, topics, run, seed + 11))
    a = synth.RowsSpec(N=R, D=128, num_topics=topics, scale=1.5, sigma=0.3, seed=seed, stream=3, dtype="bf16",
                       centroid_seed=seed)
    return synth.gen_rows_numpy(a), synth.gen_rows_numpy(v)


def _mask(kind, R, N, seed):
    rng = np.random.default_rng(seed)
    if kind.startswith("runs"):
        run = int(kind[4:])
        m = synth.owned_runs_mask(R, N, run, max(1, N // run // 4), seed)
    else:
        bits = rng.random((R, N)) < float(kind)
        m = np.zeros((R, (N + 31) // 32), dtype=np.uint32)
        for r in range(R):
            j = np.flatnonzero(bits[r])
            np.bitwise_or.at(m[r], j // 32, np.uint32(1) << (j % 32).astype(np.uint32))
    m[0] = 0  # an anchor that owns nothing
    if R > 1:
        m[1] = 0xFFFFFFFF  # and one that owns everything (bits past N are ignored)
    return m


def _matrix(kk, V, cp, gc):
    """M = [Grids | Chunks | zeros | blocks] as bf16 bits; the coarse rows are
    the oracle's means rounded to bf16 on the host."""
    N = V.shape[0]
    H = kk.kk_hier_pool_coarse_rows(N, cp, gc)
    chunks, grids = ko.hier_reps(ko.decode(V), cp, gc)
    G, C = len(grids), len(chunks)
    M = np.zeros((H + N, 128), dtype=np.uint16)
    M[:G] = synth.bf16_rne(grids.astype(np.float32))
    M[G:G + C] = synth.bf16_rne(chunks.astype(np.float32))
    M[H:] = V
    return M, G, C, H


def _allowed(mask, r, N):
    j = np.arange(N)
    return ((mask[r, j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)


def _levels(A_r, M, G, C, H, allowed, cp, gc, pm):
    """The oracle's view of one anchor: whether the Grid and Chunk cuts are
    wider than GAP (then both sides see the same active blocks), the active
    blocks in selection order, how many the block level keeps, the block scores."""
    N = len(allowed)
    s_g, s_c, s_p = (ko.affinity(M[a:b], A_r) for a, b in ((0, G), (G, G + C), (H, H + N)))
    c_ok = np.zeros(C, bool)
    c_ok[np.flatnonzero(allowed) // cp] = True
    g_ok = np.zeros(G, bool)
    g_ok[np.flatnonzero(c_ok) // gc] = True
    clear = True

    def keep(s, members, q):
        nonlocal clear
        order = sorted(members, key=lambda i: (-s[i], i))
        m = -(-len(order) * q // 1000)
        if 0 < m < len(order) and s[order[m - 1]] - s[order[m]] <= GAP:
            clear = False
        return set(order[:m])

    gk = keep(s_g, np.flatnonzero(g_ok).tolist(), pm[0])
    ck = keep(s_c, [c for c in np.flatnonzero(c_ok).tolist() if c // gc in gk], pm[1])
    active = [b for b in np.flatnonzero(allowed).tolist() if b // cp in ck]
    order = sorted(active, key=lambda i: (-s_p[i], i))
    return clear, order, -(-len(order) * pm[2] // 1000), s_p


def _run(kk, A, M, mask, N, cp, gc, pm, K):
    R = A.shape[0]
    At = torch.from_numpy(A.view(np.int16)).cuda()
    Mt = torch.from_numpy(M.view(np.int16)).cuda()
    mt = torch.from_numpy(mask.view(np.int32)).cuda()
    ws = torch.empty(max(1, kk.kk_hier_select_pool_workspace_bytes(R, N, cp, gc)), dtype=torch.uint8, device="cuda")
    out = []
    for _ in range(2):  # a second call must not see the first call's candidates
        idx = torch.full((R, K), 7, dtype=torch.int32, device="cuda")
        top = torch.zeros((R, K), device="cuda")
        kept = torch.full((R,), -3, dtype=torch.int32, device="cuda")
        kk.kk_hier_select_pool(At, Mt, mt, N, cp, gc, pm, idx, top, kept, ws)
        assert kk.kk_device_error() == 0
        out.append((idx.cpu().numpy(), top.cpu().numpy(), kept.cpu().numpy()))
    for a, b in zip(*out):
        np.testing.assert_array_equal(a, b)
    return out[0]


def check_against_oracle(A, M, G, C, H, mask, N, cp, gc, pm, K, g_idx, g_top, g_kept, rows=None, min_clear=0.8):
    """Every anchor: the picks are allowed, distinct, ordered, -1 padded and
    scored right. Anchors whose Grid and Chunk cuts are clear (at least
    min_clear of them): the kept count is the oracle's, and the picks are the
    best min(K, kept) active blocks (up to GAP), the oracle's own set where
    that last cut is clear as well."""
    rows = range(A.shape[0]) if rows is None else rows
    grids, chunks, V = M[:G], M[G:G + C], M[H:]
    n_clear = 0
    for r in rows:
        allowed = _allowed(mask, r, N)
        w_idx, w_val, w_kept = ko.hier_select_pool(A[r:r + 1], grids, chunks, V, mask[r:r + 1], K, cp, gc, pm)
        coarse_clear, order, m_keep, s_p = _levels(ko.decode(A[r]), M, G, C, H, allowed, cp, gc, pm)
        m = min(K, int(g_kept[r]))
        sel = g_idx[r, :m].astype(np.int64)
        assert np.all(g_idx[r, m:] == -1) and np.all(np.isneginf(g_top[r, m:])), f"r={r} padding"
        assert len(set(sel.tolist())) == m and np.all(allowed[sel]), f"r={r}: picked a block it does not own"
        assert np.all(np.diff(g_top[r, :m]) <= 0), f"r={r} order"
        assert_scores_close(g_top[r, :m].astype(np.float64), s_p[sel], f"r={r} scores")
        if not coarse_clear:
            continue
        n_clear += 1
        assert g_kept[r] == m_keep == w_kept[0], (r, g_kept[r], m_keep, w_kept[0])
        assert w_idx[0, :m].tolist() == order[:m]
        picked = set(sel.tolist())
        assert picked <= set(order), f"r={r}: a pick outside the kept Chunks"
        rest = [b for b in order if b not in picked]
        if m and rest:
            assert s_p[sel].min() >= s_p[rest].max() - GAP, f"r={r}: not the best {m} active blocks"
        if m == len(order) or s_p[order[m - 1]] - s_p[order[m]] > GAP:
            assert picked == set(order[:m]), f"r={r}: kept blocks differ"
    assert n_clear >= min_clear * len(rows), f"only {n_clear} of {len(rows)} anchors have clear coarse cuts"


@pytest.mark.parametrize("R,N,cp,gc,pm,K,kind", [
    (5, 300, 8, 3, (500, 200, 100), 7, "0.3"),
    (130, 3000, 16, 4, (500, 200, 100), 64, "runs64"),
    (64, 4097, 64, 8, (500, 500, 500), 256, "runs512"),
    (33, 2000, 4, 3, (700, 400, 250), 100, "0.5"),
    (9, 777, 32, 1, (300, 1000, 600), 33, "0.05"),
])
def test_hier_select_pool(kk, R, N, cp, gc, pm, K, kind):
    A, V = _rows(N, R, seed=N + cp)
    M, G, C, H = _matrix(kk, V, cp, gc)
    mask = _mask(kind, R, N, seed=R + N)
    g_idx, g_top, g_kept = _run(kk, A, M, mask, N, cp, gc, pm, K)
    assert g_kept[0] == 0 and np.all(g_idx[0] == -1)
    check_against_oracle(A, M, G, C, H, mask, N, cp, gc, pm, K, g_idx, g_top, g_kept)


def test_everything_kept_is_the_flat_batched_topk(kk):
    """permille 1000/1000/1000: the allowed blocks' top K, as kk_score_pool_batched gives them."""
    R, N, cp, gc, K = 70, 2500, 16, 4, 200
    A, V = _rows(N, R, seed=3)
    M, G, C, H = _matrix(kk, V, cp, gc)
    mask = _mask("0.2", R, N, seed=4)
    g_idx, g_top, g_kept = _run(kk, A, M, mask, N, cp, gc, (1000, 1000, 1000), K)
    At, Vt = torch.from_numpy(A.view(np.int16)).cuda(), torch.from_numpy(V.view(np.int16)).cuda()
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    ws = torch.empty(kk.kk_score_pool_batched_workspace_bytes(R, N, K), dtype=torch.uint8, device="cuda")
    kk.kk_score_pool_batched(At, Vt, torch.from_numpy(mask.view(np.int32)).cuda(), K, idx, top, ws)
    assert kk.kk_device_error() == 0
    np.testing.assert_array_equal(g_idx, idx.cpu().numpy())
    np.testing.assert_array_equal(g_top, top.cpu().numpy())
    want = [int(_allowed(mask, r, N).sum()) for r in range(R)]
    assert g_kept.tolist() == want


@pytest.mark.parametrize("pm", [(1000, 1000, 1000), (1000, 1000, 500)])
def test_streamed_block_level(kk, pm):
    """More active blocks than the shared-memory list holds: the block level
    is selected straight from the candidate segments."""
    R, N, cp, gc, K = 3, 20000, 16, 8, 64
    A, V = _rows(N, R, seed=17)
    M, G, C, H = _matrix(kk, V, cp, gc)
    mask = np.full((R, (N + 31) // 32), 0xFFFFFFFF, dtype=np.uint32)
    mask[2, ::3] = 0
    g_idx, g_top, g_kept = _run(kk, A, M, mask, N, cp, gc, pm, K)
    assert g_kept[0] > 4096  # more active blocks than the shared-memory list holds (4096)
    check_against_oracle(A, M, G, C, H, mask, N, cp, gc, pm, K, g_idx, g_top, g_kept)


@pytest.mark.parametrize("N,cp,gc", [(300, 8, 3), (4097, 64, 8), (129, 128, 1), (1, 64, 8), (5000, 5, 7)])
def test_hier_pool_reps(kk, N, cp, gc):
    _, V = _rows(N, 1, seed=N)
    H = kk.kk_hier_pool_coarse_rows(N, cp, gc)
    M = np.full((H + N, 128), 0x7777, dtype=np.uint16)
    M[H:] = V
    Mt = torch.from_numpy(M.view(np.int16)).cuda()
    kk.kk_hier_pool_reps(Mt, N, cp, gc)
    torch.cuda.synchronize()
    got = Mt.cpu().numpy().view(np.uint16)
    chunks, grids = ko.hier_reps(ko.decode(V), cp, gc)
    G, C = len(grids), len(chunks)
    np.testing.assert_array_equal(got[H:], V)
    assert np.all(got[G + C:H] == 0)
    for name, rows, ref in (("grids", got[:G], grids), ("chunks", got[G:G + C], chunks)):
        g = ko.decode(rows)
        # float32 sums rounded once to bf16: within one bf16 ulp of the exact mean
        np.testing.assert_array_less(np.abs(g - ref), 2.0**-7 * np.abs(ref) + 1e-6, err_msg=name)
        exact = np.mean(rows == synth.bf16_rne(ref.astype(np.float32)))
        assert exact >= 0.99, f"{name}: only {exact:.4f} of the values round like the exact mean"


def test_empty_pool_and_large_k(kk):
    """N = 0: nothing is kept and every slot is padding; K larger than the
    blocks kept: the kept blocks, then padding."""
    R, K = 3, 256
    A, _ = _rows(1, R, seed=2)
    mask = np.zeros((R, 1), dtype=np.uint32)
    M = np.zeros((0, 128), dtype=np.uint16)
    At = torch.from_numpy(A.view(np.int16)).cuda()
    Mt = torch.zeros((0, 128), dtype=torch.int16, device="cuda")
    mt = torch.from_numpy(mask.view(np.int32)).cuda()
    ws = torch.empty(max(1, kk.kk_hier_select_pool_workspace_bytes(R, 0, 64, 8)), dtype=torch.uint8, device="cuda")
    idx = torch.full((R, K), 7, dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    kept = torch.full((R,), -3, dtype=torch.int32, device="cuda")
    kk.kk_hier_select_pool(At, Mt, mt, 0, 64, 8, (500, 200, 100), idx, top, kept, ws)
    assert kk.kk_device_error() == 0
    assert np.all(idx.cpu().numpy() == -1) and np.all(np.isneginf(top.cpu().numpy()))
    assert np.all(kept.cpu().numpy() == 0)
    # a small pool where every level is kept whole: K exceeds the allowed blocks
    N, cp, gc = 150, 16, 2
    A, V = _rows(N, R, seed=5)
    M, G, C, H = _matrix(kk, V, cp, gc)
    mask = _mask("0.4", R, N, seed=6)
    g_idx, g_top, g_kept = _run(kk, A, M, mask, N, cp, gc, (1000, 1000, 1000), K)
    allowed = [int(_allowed(mask, r, N).sum()) for r in range(R)]
    assert g_kept.tolist() == allowed and max(allowed) < K
    check_against_oracle(A, M, G, C, H, mask, N, cp, gc, (1000, 1000, 1000), K, g_idx, g_top, g_kept)


def test_single_anchor(kk):
    """One anchor: the GEMM's anchor tile holds one real row of 128."""
    N, cp, gc, K = 1000, 8, 4, 20
    A, V = _rows(N, 1, seed=8)
    M, G, C, H = _matrix(kk, V, cp, gc)
    mask = _mask("0.5", 1, N, seed=9)
    mask[0] = np.random.default_rng(3).integers(0, 2**32, size=mask.shape[1], dtype=np.uint64).astype(np.uint32)
    g_idx, g_top, g_kept = _run(kk, A, M, mask, N, cp, gc, (500, 300, 200), K)
    check_against_oracle(A, M, G, C, H, mask, N, cp, gc, (500, 300, 200), K, g_idx, g_top, g_kept)
