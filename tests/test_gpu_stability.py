"""The stability filter ("Key-Key Semantic Affinity" page, §5.3) fused into
scoring, over many decode steps through the C ABI, against the fp64 oracle:
the per-block history words persist across calls, the stability is the
fraction of the last W steps above the threshold, and the top K is ranked by
stability, then by the current score, then by the lower index."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import DeviceCache, assert_scores_close, assert_topk_valid

pytestmark = pytest.mark.gpu

GAP = 1e-5  # no oracle score lies this close to the threshold (fp32 scores decide the same bits)


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _pick_theta(all_scores):
    """A threshold in [0.45, 0.55] as far as possible from every score."""
    s = np.sort(np.concatenate([np.ravel(x) for x in all_scores]))
    best, gap = 0.5, -1.0
    for th in np.linspace(0.45, 0.55, 2001):
        i = np.searchsorted(s, th)
        d = min(abs(s[i] - th) if i < len(s) else 1.0, abs(s[i - 1] - th) if i > 0 else 1.0)
        if d > gap:
            best, gap = float(np.float32(th)), d
    assert gap > GAP, "no threshold far enough from every score"
    return best


def _check_step(kk_idx, kk_top, kk_stab, scores_hist, W, theta, K, what):
    stab = ko.stability(scores_hist, W, theta)
    count = np.rint(stab * W).astype(np.int64)
    np.testing.assert_array_equal(kk_stab, (count / np.float64(W)).astype(np.float32), err_msg=what + " stability")
    s = np.asarray(scores_hist[-1], dtype=np.float64)
    composite = count * 10.0 + s  # ranks exactly like (stability, score); scores are in [0, 1]
    assert_topk_valid(kk_idx, None, composite, K, what)
    k = min(K, len(s))
    assert_scores_close(np.asarray(kk_top[:k], dtype=np.float64), s[np.asarray(kk_idx[:k])], what + " top scores")
    want_idx, _ = ko.stable_topk(stab, s, K)
    # away from near-ties the order is the oracle's
    if k and np.all(np.abs(np.diff(np.sort(composite)[::-1][: k + 1])) > 1e-6):
        np.testing.assert_array_equal(kk_idx[:k], want_idx[:k], err_msg=what)


@pytest.mark.parametrize("W", [20, 5, 1, 32])
def test_score_topk_stable_over_steps(kk, W):
    sp = synth.qwen7b(L=2, H=2, D=64, bs=8, seq_lens=[8 * 60 + 3, 8 * 17, 8 * 230], num_topics=6, W=8, K=24,
                      shuffle_pages=True, extra_pages=5)
    dev = DeviceCache(sp)
    kc = dev.host_view()
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    vb_o = np.zeros((sp.num_pages, sp.D))
    vb_o[sp.pages] = ko.pool_blocks(kc, sp.pages, sp.n_valid)
    steps = 27
    rng = np.random.default_rng(100 + W)
    # anchors drift between topics from step to step, so blocks go in and out of the high set
    vas = []
    for t in range(steps):
        mix = rng.dirichlet(np.full(sp.num_topics, 0.3), size=sp.R)
        vas.append((mix @ sp.cs + 0.05 * rng.standard_normal((sp.R, sp.D))).astype(np.float32))
    oracle_scores = [[ko.affinity(vb_o[sp.pages_of(r)], vas[t][r].astype(np.float64)) for r in range(sp.R)]
                     for t in range(steps)]
    theta = _pick_theta([x for step in oracle_scores for x in step])
    hist = torch.zeros(sp.total_blocks, dtype=torch.int32, device="cuda")
    stab = torch.zeros(sp.total_blocks, device="cuda")
    scores = torch.zeros(sp.total_blocks, device="cuda")
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top = torch.zeros((sp.R, sp.K), device="cuda")
    for t in range(steps):
        va = torch.from_numpy(vas[t]).cuda()
        kk.kk_score_topk_stable(vb, dev.bt, va, sp.K, W, theta, hist, idx, stab=stab, top_scores=top, scores=scores)
        assert kk.kk_device_error() == 0
        g_idx, g_top, g_stab, g_sc = idx.cpu().numpy(), top.cpu().numpy(), stab.cpu().numpy(), scores.cpu().numpy()
        for r in range(sp.R):
            blk = slice(sp.offsets[r], sp.offsets[r + 1])
            hist_r = [oracle_scores[u][r] for u in range(t + 1)]
            assert_scores_close(g_sc[blk], hist_r[-1], f"W={W} step {t} r={r} scores")
            _check_step(g_idx[r], g_top[r], g_stab[blk], hist_r, W, theta, sp.K, f"W={W} step {t} r={r}")
    # the history words hold the last W bits, newest in bit 0
    h = hist.cpu().numpy().view(np.uint32)
    for r in range(sp.R):
        for j in range(sp.nb[r]):
            bits = [(oracle_scores[steps - 1 - b][r][j] > theta) for b in range(min(W, steps))]
            assert h[sp.offsets[r] + j] == sum(int(x) << b for b, x in enumerate(bits))


def test_select_step_stable_accumulates(kk):
    """kk_select_step_stable: the anchor comes from the cache, so every step
    has the same scores; a block above the threshold climbs by 1/W a step up
    to 1, the others stay at 0, and the ranking follows."""
    sp = synth.qwen7b(L=3, H=2, D=128, bs=16, seq_lens=[16 * 90 + 5, 16 * 33], num_topics=4, W=12, K=16)
    dev = DeviceCache(sp)
    kc = dev.host_view()
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    vb_o = np.zeros((sp.num_pages, sp.D))
    vb_o[sp.pages] = ko.pool_blocks(kc, sp.pages, sp.n_valid)
    s_o = [ko.affinity(vb_o[sp.pages_of(r)], ko.anchor(kc, sp.pages_of(r), sp.seq_lens[r], sp.bs, sp.W))
           for r in range(sp.R)]
    theta = _pick_theta(s_o)
    W = 6
    hist = torch.zeros(sp.total_blocks, dtype=torch.int32, device="cuda")
    stab = torch.zeros(sp.total_blocks, device="cuda")
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top = torch.zeros((sp.R, sp.K), device="cuda")
    for t in range(W + 3):
        kk.kk_select_step_stable(dev.desc, dev.bt, sp.W, vb, sp.K, W, theta, hist, idx, stab=stab, top_scores=top)
        assert kk.kk_device_error() == 0
        g_idx, g_top, g_stab = idx.cpu().numpy(), top.cpu().numpy(), stab.cpu().numpy()
        for r in range(sp.R):
            blk = slice(sp.offsets[r], sp.offsets[r + 1])
            _check_step(g_idx[r], g_top[r], g_stab[blk], [s_o[r]] * (t + 1), W, theta, sp.K, f"step {t} r={r}")
            hi = s_o[r] > theta
            np.testing.assert_array_equal(g_stab[blk][hi], np.float32(min(t + 1, W) / W))
            assert np.all(g_stab[blk][~hi] == 0)


def test_stable_matches_plain_when_every_block_is_equally_stable(kk):
    """With theta below every score all blocks have the same stability, so
    the stable ranking is the plain score ranking."""
    sp = synth.qwen7b(L=2, H=2, D=64, bs=8, seq_lens=[8 * 120], num_topics=5, W=8, K=32)
    dev = DeviceCache(sp)
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    va = torch.from_numpy(sp.cs[:1].astype(np.float32)).cuda()
    hist = torch.zeros(sp.total_blocks, dtype=torch.int32, device="cuda")
    i1 = torch.zeros((1, sp.K), dtype=torch.int32, device="cuda")
    i2 = torch.zeros_like(i1)
    t1 = torch.zeros((1, sp.K), device="cuda")
    t2 = torch.zeros_like(t1)
    kk.kk_score_topk_stable(vb, dev.bt, va, sp.K, 20, -1.0, hist, i1, top_scores=t1)
    kk.kk_score_topk(vb, dev.bt, va, sp.K, i2, top_scores=t2)
    assert kk.kk_device_error() == 0
    assert torch.equal(i1, i2) and torch.equal(t1, t2)
    assert np.all(hist.cpu().numpy() == 1)


def test_score_topk_stable_long_request_split(kk):
    """A request of 70000 blocks (split over several clusters of CTAs, the
    last of which merges their lists) beside a short one, over several steps:
    sampled scores against the oracle, and the ranking exactly the oracle's
    (stability, score, index) order of the returned scores, whose threshold
    decisions both sides take in float32."""
    sizes = [70000, 300]
    R, D, K, W, steps = len(sizes), 64, 64, 4, 6
    n = sum(sizes)
    rows = synth.RowsSpec(N=n, D=D, num_topics=6, scale=1.0, sigma=0.4, seed=21, stream=7)
    vb_np = synth.gen_rows_numpy(rows)
    rng = np.random.default_rng(21)
    pages = rng.permutation(n).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    vb = torch.from_numpy(vb_np).cuda()
    bt = kk.BlockTable(torch.from_numpy(pages).cuda(), torch.from_numpy(offsets).cuda(),
                       torch.tensor(sizes, dtype=torch.int32, device="cuda"), max(sizes))
    theta = float(np.float32(0.5))
    hist = torch.zeros(n, dtype=torch.int32, device="cuda")
    stab = torch.zeros(n, device="cuda")
    scores = torch.zeros(n, device="cuda")
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    ws = torch.zeros(kk.kk_select_step_workspace_bytes(R, max(sizes), K), dtype=torch.uint8, device="cuda")
    g_hist = []
    for t in range(steps):
        va_np = (rng.standard_normal((R, D)) + 2.0 * rows.cs[rng.integers(0, 6, R)]).astype(np.float32)
        kk.kk_score_topk_stable(vb, bt, torch.from_numpy(va_np).cuda(), K, W, theta, hist, idx, stab=stab,
                                top_scores=top, scores=scores, workspace=ws)
        assert kk.kk_device_error() == 0
        g_sc, g_idx, g_top, g_stab = scores.cpu().numpy(), idx.cpu().numpy(), top.cpu().numpy(), stab.cpu().numpy()
        g_hist.append(g_sc)
        for r in range(R):
            blk = slice(offsets[r], offsets[r + 1])
            sample = rng.choice(sizes[r], min(200, sizes[r]), replace=False)
            s_o = ko.affinity(vb_np[pages[blk][sample]], va_np[r].astype(np.float64))
            assert_scores_close(g_sc[blk][sample], s_o, f"step {t} r={r} sampled scores")
            st = ko.stability([h[blk] for h in g_hist], W, theta)
            np.testing.assert_array_equal(g_stab[blk], st.astype(np.float32), err_msg=f"step {t} r={r} stability")
            want_idx, want_val = ko.stable_topk(st, g_sc[blk], K)
            np.testing.assert_array_equal(g_idx[r], want_idx, err_msg=f"step {t} r={r}")
            np.testing.assert_array_equal(g_top[r], want_val.astype(np.float32))
