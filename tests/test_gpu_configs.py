"""The five workloads at full size, called exactly as bench.py calls them.
The oracle checks sampled outputs it can compute one by one (sampled blocks,
sampled requests, sampled coarse groups); properties that hold at any size
(planted-topic ranking, reblocking) cover the rest."""
import dataclasses
import gc

import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import DeviceCache, assert_scores_close, assert_topk_valid, assert_vec_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _pool_all(kk, dev):
    sp = dev.spec
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    assert kk.kk_device_error() == 0
    return vb


def _check_sampled_blocks(dev, vb, blocks, head_w=None):
    sp = dev.spec
    pages = sp.pages[blocks]
    kc = dev.host_pages(pages)
    want = ko.pool_blocks(kc, np.arange(len(pages)), sp.n_valid[blocks],
                          None if head_w is None else [head_w], None if head_w is None else [0] * len(pages))
    assert_vec_close(vb.cpu().numpy()[pages], want, f"{sp.name} sampled vb")


def _check_request_step(dev, r, va_gpu, scores_gpu, idx_gpu, top_gpu, K, head_w=None):
    sp = dev.spec
    kc_r, local = dev.host_request(r)
    T = sp.seq_lens[r]
    va_o = ko.anchor(kc_r, local, T, sp.bs, sp.W, head_w)
    assert_vec_close(va_gpu, va_o, f"{sp.name} va r={r}")
    nb = len(local)
    w = None if head_w is None else [head_w]
    vb_o = ko.pool_blocks(kc_r, local, sp.n_valid[sp.offsets[r]:sp.offsets[r + 1]], w,
                          None if w is None else [0] * nb)
    s_o = ko.affinity(vb_o, va_o)
    assert_scores_close(scores_gpu, s_o, f"{sp.name} scores r={r}")
    assert_topk_valid(idx_gpu, top_gpu, s_o, K, f"{sp.name} top-K r={r}")


def _check_planted(dev, idx):
    sp = dev.spec
    for r in range(sp.R):
        topic = sp.block_topic[sp.offsets[r]:sp.offsets[r + 1]]
        same = set(np.flatnonzero(topic == sp.query_topic[r]).tolist())
        m = min(sp.K, len(same))
        assert set(idx[r][:m].tolist()) <= same, f"{sp.name} r={r}: planted topic not ranked first"


def _step(kk, dev, vb, head_w=None):
    """One select step, with the workspace that lets long requests split."""
    sp = dev.spec
    idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device="cuda")
    top = torch.zeros((sp.R, sp.K), device="cuda")
    va = torch.zeros((sp.R, sp.D), device="cuda")
    scores = torch.zeros(sp.total_blocks, device="cuda")
    nws = kk.kk_select_step_workspace_bytes(sp.R, max(sp.nb), sp.K)
    ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device="cuda")
    kk.kk_select_step(dev.desc, dev.bt, sp.W, vb, sp.K, idx, top, va=va, scores=scores, head_w=head_w, workspace=ws)
    assert kk.kk_device_error() == 0
    return idx.cpu().numpy(), top.cpu().numpy(), va.cpu().numpy(), scores.cpu().numpy()


def test_tiny_05b_whole_path(kk):
    dev = DeviceCache(synth.tiny_05b())
    sp = dev.spec
    vb = _pool_all(kk, dev)
    kc = dev.host_view()
    assert_vec_close(vb.cpu().numpy()[sp.pages], ko.pool_blocks(kc, sp.pages, sp.n_valid), "vb")
    idx, top, va, scores = _step(kk, dev, vb)
    _check_request_step(dev, 0, va[0], scores, idx[0], top[0], sp.K)
    _check_planted(dev, idx)


def test_qwen7b_full(kk):
    dev = DeviceCache(synth.qwen7b())
    sp = dev.spec
    vb = _pool_all(kk, dev)
    rng = np.random.default_rng(1)
    _check_sampled_blocks(dev, vb, np.unique(np.concatenate([[0, sp.total_blocks - 1],
                                                              rng.choice(sp.total_blocks, 30, replace=False)])))
    idx, top, va, scores = _step(kk, dev, vb)
    for r in (0, sp.R - 1):
        _check_request_step(dev, r, va[r], scores[sp.offsets[r]:sp.offsets[r + 1]], idx[r], top[r], sp.K)
    _check_planted(dev, idx)
    del dev, vb
    _free()


def test_qwen7b_long_weighted_full(kk):
    dev = DeviceCache(synth.qwen7b_long())
    sp = dev.spec
    LH = sp.L * sp.H
    ws = torch.empty(kk.kk_head_variance_workspace_bytes(dev.desc, sp.total_blocks, sp.R), dtype=torch.uint8,
                     device="cuda")
    w_out = torch.zeros((sp.R, LH), device="cuda")
    vb = torch.zeros((sp.num_pages, sp.D), device="cuda")
    kk.kk_pool_blocks_weighted(dev.desc, dev.bt, sp.total_blocks, w_out, vb, ws)
    assert kk.kk_device_error() == 0
    del ws
    _free()
    idx, top, va, scores = _step(kk, dev, vb, head_w=w_out)
    r = 5
    kc_r, local = dev.host_request(r)
    w_o = ko.head_variance_weights(kc_r, local, sp.seq_lens[r], sp.bs)
    assert_vec_close(w_out.cpu().numpy()[r], w_o, "head weights")
    del kc_r
    _check_request_step(dev, r, va[r], scores[sp.offsets[r]:sp.offsets[r + 1]], idx[r], top[r], sp.K, w_o)
    _check_planted(dev, idx)
    del dev, vb
    _free()


@pytest.mark.parametrize("bs", [16, 128])
def test_write_stress_pool_and_coarse(kk, bs):
    dev = DeviceCache(synth.write_stress(bs))
    sp = dev.spec
    vb = _pool_all(kk, dev)
    rng = np.random.default_rng(bs)
    _check_sampled_blocks(dev, vb, np.unique(np.concatenate([[0, sp.total_blocks - 1],
                                                              rng.choice(sp.total_blocks, 24, replace=False)])))
    for group in (64, 512):
        ng = (sp.nb[0] + group - 1) // group
        out = torch.zeros((1, ng, sp.D), device="cuda")
        kk.kk_coarse_means(vb, dev.bt, group, out)
        assert kk.kk_device_error() == 0
        g = int(rng.integers(0, ng))
        blocks = np.arange(g * group, min((g + 1) * group, sp.nb[0]))
        kc = dev.host_pages(sp.pages[blocks])
        vb_o = ko.pool_blocks(kc, np.arange(len(blocks)), sp.n_valid[blocks])
        assert_vec_close(out.cpu().numpy()[0, g], ko.coarse_means(vb_o, group)[0], f"coarse {group} g={g}")
    if bs == 16:
        # reblocking: eight 16-token blocks average to the 128-token block over the same tokens
        test_write_stress_pool_and_coarse.vb16 = vb.cpu().numpy()
    else:
        vb16 = getattr(test_write_stress_pool_and_coarse, "vb16", None)
        if vb16 is not None:
            fine = vb16.reshape(-1, 8, sp.D).mean(axis=1)
            assert_vec_close(fine, vb.cpu().numpy(), "reblocking 16 -> 128")
    del dev, vb
    _free()


def test_write_stress_select_step(kk):
    """One request of 65536 blocks (2^20 tokens at block size 16): long
    enough that its blocks are split over several clusters, the last of
    which merges their lists. The anchor against the oracle's over the last
    W tokens, sampled scores against the oracle's, and the top-K exactly the
    ranking of the returned scores, the same on repeated calls."""
    dev = DeviceCache(synth.write_stress(16))
    sp = dev.spec
    vb = _pool_all(kk, dev)
    idx, top, va, scores = _step(kk, dev, vb)
    T, nb = sp.seq_lens[0], sp.nb[0]
    last = np.arange((T - min(sp.W, T)) // sp.bs, nb)
    local = np.zeros(nb, dtype=np.int64)
    local[last] = np.arange(len(last))
    va_o = ko.anchor(dev.host_pages(sp.pages[last]), local, T, sp.bs, sp.W)
    assert_vec_close(va[0], va_o, "write16 va")
    rng = np.random.default_rng(16)
    blocks = np.unique(np.concatenate([[0, nb - 1], rng.choice(nb, 40, replace=False), idx[0][:8]]))
    vb_o = ko.pool_blocks(dev.host_pages(sp.pages[blocks]), np.arange(len(blocks)), sp.n_valid[blocks])
    assert_scores_close(scores[blocks], ko.affinity(vb_o, va_o), "write16 sampled scores")
    want_idx, want_val = ko.topk(scores[:nb], sp.K)
    np.testing.assert_array_equal(idx[0], want_idx)
    np.testing.assert_array_equal(top[0], want_val.astype(np.float32))
    _check_planted(dev, idx)
    for _ in range(3):
        idx2, top2, _, _ = _step(kk, dev, vb)
        np.testing.assert_array_equal(idx2, idx)
        np.testing.assert_array_equal(top2, top)
    del dev, vb
    _free()


def test_shared_pool_full(kk):
    from tests.test_gpu_parity import check_batched_against_oracle

    v_spec, a_spec, mask, K = synth.shared_pool()
    V = synth.gen_rows_cuda(v_spec)
    A = synth.gen_rows_cuda(a_spec)
    R, N = A.shape[0], V.shape[0]
    Mt = torch.from_numpy(mask.view(np.int32)).cuda()
    ws = torch.empty(kk.kk_score_pool_batched_workspace_bytes(R, N, K), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    kk.kk_score_pool_batched(A, V, Mt, K, idx, top, ws)
    assert kk.kk_device_error() == 0
    A_h = A.cpu().numpy().view(np.uint16)
    V_h = V.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(A_h, synth.gen_rows_numpy(a_spec))  # generator bits, GPU == numpy
    idx_h, top_h = idx.cpu().numpy(), top.cpu().numpy()
    check_batched_against_oracle(A_h, V_h, mask, K, idx_h, top_h)
    # planted topics: the owned blocks of the anchor's topic come first
    j = np.arange(N)
    for r in range(R):
        owned = np.flatnonzero((mask[r, j // 32] >> (j % 32).astype(np.uint32)) & 1)
        same = set(owned[v_spec.topics[owned] == a_spec.topics[r]].tolist())
        m = min(K, len(same))
        assert set(idx_h[r][:m].tolist()) <= same, f"row {r}"


def test_shared_pool_hier_full(kk):
    """The shared pool as documents, three levels in one product (256 anchors x
    65536 blocks, Chunks of 64, Grids of 8 Chunks, 50 / 20 / 10 %), as bench.py
    calls it: every coarse row against the oracle's means, sampled anchors
    against the oracle's selection."""
    from tests.test_gpu_hier_pool import check_against_oracle

    v_spec, a_spec, mask, K = synth.shared_pool_hier()
    R, N, cp, gc_, pm = a_spec.N, v_spec.N, 64, 8, (500, 200, 100)
    H = kk.kk_hier_pool_coarse_rows(N, cp, gc_)
    M = torch.zeros((H + N, 128), dtype=torch.int16, device="cuda")
    M[H:] = synth.gen_rows_cuda(v_spec)
    A = synth.gen_rows_cuda(a_spec)
    kk.kk_hier_pool_reps(M, N, cp, gc_)
    mt = torch.from_numpy(mask.view(np.int32)).cuda()
    ws = torch.empty(kk.kk_hier_select_pool_workspace_bytes(R, N, cp, gc_), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    top = torch.zeros((R, K), device="cuda")
    kept = torch.zeros(R, dtype=torch.int32, device="cuda")
    kk.kk_hier_select_pool(A, M, mt, N, cp, gc_, pm, idx, top, kept, ws)
    assert kk.kk_device_error() == 0
    M_h = M.cpu().numpy().view(np.uint16)
    A_h = A.cpu().numpy().view(np.uint16)
    V_h = M_h[H:]
    head = dataclasses.replace(v_spec, N=4096, topics=v_spec.topics[:4096])
    np.testing.assert_array_equal(V_h[:4096], synth.gen_rows_numpy(head))  # generator bits, GPU == numpy
    chunks, grids = ko.hier_reps(ko.decode(V_h), cp, gc_)
    G, C = len(grids), len(chunks)
    for rows, ref in ((M_h[:G], grids), (M_h[G:G + C], chunks)):
        np.testing.assert_array_less(np.abs(ko.decode(rows) - ref), 2.0**-7 * np.abs(ref) + 1e-6)
    rows = np.random.default_rng(5).choice(R, size=8, replace=False)
    check_against_oracle(A_h, M_h, G, C, H, mask, N, cp, gc_, pm, K, idx.cpu().numpy(), top.cpu().numpy(),
                         kept.cpu().numpy(), rows=rows.tolist(), min_clear=0.5)
    _free()
