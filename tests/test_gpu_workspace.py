"""Decode-step calls with caller-owned split workspaces, through the C ABI,
against the fp64 oracle ("Key-Key Semantic Affinity" page, §5.2 steps 3-4):
very long requests are split over several clusters of CTAs that meet in the
caller's workspace. Two such calls run at once on two streams, each with its
own workspace, and both select exactly what the oracle's scores say; a
workspace is left ready for the next call, and one that was never zeroed is
reported."""
import numpy as np
import pytest
import torch

import synth
from oracle import kk_oracle as ko
from tests.helpers import assert_scores_close, assert_topk_valid

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kk(cuda):
    from kv_cache_block_gb300 import kk as mod

    return mod


N, D, K = 60000, 128, 32


@pytest.fixture(scope="module")
def pool_rows():
    rows = synth.RowsSpec(N=N, D=D, num_topics=8, scale=1.0, sigma=0.5, seed=31, stream=9)
    return rows, synth.gen_rows_numpy(rows)


def _case(kk, rows, c, rng):
    pages = rng.permutation(N).astype(np.int32)
    va = (2.0 * rows.cs[c % rows.num_topics] + rng.standard_normal(D)).astype(np.float32)[None]
    bt = kk.BlockTable(torch.from_numpy(pages).cuda(), torch.tensor([0, N], dtype=torch.int32, device="cuda"), None,
                       N)
    ws = torch.zeros(kk.kk_select_step_workspace_bytes(1, N, K), dtype=torch.uint8, device="cuda")
    out = dict(pages=pages, va=va, bt=bt, va_dev=torch.from_numpy(va).cuda(), ws=ws,
               idx=torch.zeros((1, K), dtype=torch.int32, device="cuda"), top=torch.zeros((1, K), device="cuda"),
               scores=torch.zeros(N, device="cuda"))
    return out


def _check(vb_np, c, what):
    s_o = ko.affinity(vb_np[c["pages"]], c["va"][0].astype(np.float64))
    g_sc = c["scores"].cpu().numpy()
    assert_scores_close(g_sc, s_o, what + " scores")
    idx, top = c["idx"].cpu().numpy()[0], c["top"].cpu().numpy()[0]
    assert_topk_valid(idx, top, s_o, K, what)
    # exactly the ranking of the returned scores (ties to the lower index)
    want_idx, want_val = ko.topk(g_sc, K)
    np.testing.assert_array_equal(idx, want_idx, err_msg=what)
    np.testing.assert_array_equal(top, want_val.astype(np.float32), err_msg=what)


def test_two_streams_with_separate_workspaces(kk, pool_rows):
    rows, vb_np = pool_rows
    vb = torch.from_numpy(vb_np).cuda()
    rng = np.random.default_rng(3)
    cases = [_case(kk, rows, c, rng) for c in range(2)]
    assert cases[0]["ws"].numel() > 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(6):
        for c, s in zip(cases, streams):
            with torch.cuda.stream(s):
                kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], scores=c["scores"],
                                 workspace=c["ws"], stream=s)
        torch.cuda.synchronize()
        assert kk.kk_device_error() == 0
        for i, c in enumerate(cases):
            _check(vb_np, c, f"stream {i} call {rep}")
    for c in cases:
        w = c["ws"].cpu().numpy()
        # the request was split (its clusters left their lists) and its
        # counter is back at zero
        assert w[:8].view(np.uint64)[0] == 0
        assert np.any(w[256:] != 0)


def test_workspace_contents_between_calls(kk, pool_rows):
    """The lists region may hold anything before a call (each cluster rewrites
    its list); the counters must be zero, as a zeroed workspace leaves them
    after every call. A counter found past its bound (a workspace never
    zeroed) is reported, and a zeroed workspace works again."""
    rows, vb_np = pool_rows
    vb = torch.from_numpy(vb_np).cuda()
    c = _case(kk, rows, 5, np.random.default_rng(5))
    for rep in range(3):
        c["ws"][256:].fill_(0x5A + rep)
        kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], scores=c["scores"],
                         workspace=c["ws"])
        assert kk.kk_device_error() == 0
        _check(vb_np, c, f"lists filled before call {rep}")
        assert c["ws"][:8].cpu().numpy().view(np.uint64)[0] == 0  # back at zero
    c["ws"].fill_(0x77)
    kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], workspace=c["ws"])
    assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX
    c["ws"].zero_()
    kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], scores=c["scores"],
                     workspace=c["ws"])
    assert kk.kk_device_error() == 0
    _check(vb_np, c, "zeroed again")


def test_without_workspace_the_result_is_the_same(kk, pool_rows):
    rows, vb_np = pool_rows
    vb = torch.from_numpy(vb_np).cuda()
    c = _case(kk, rows, 2, np.random.default_rng(8))
    kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], scores=c["scores"],
                     workspace=c["ws"])
    i1, t1 = c["idx"].clone(), c["top"].clone()
    kk.kk_score_topk(vb, c["bt"], c["va_dev"], K, c["idx"], top_scores=c["top"], scores=c["scores"])
    assert kk.kk_device_error() == 0
    assert torch.equal(i1, c["idx"]) and torch.equal(t1, c["top"])
    _check(vb_np, c, "no workspace")
