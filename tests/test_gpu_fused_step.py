"""The fused decode step, through the C ABI: one kk_select_step(_stable) call
that first writes every request's decode token (kk_step_options.k_new: the
cache slot, the block's running sum, v_b and the anchor-ring slot; "Key-Key
Semantic Affinity" page, §5.2 step 2, v_b kept as the block is written), then
selects on the updated v_b and ring (§5.2 steps 1, 3-4), and writes the table
of the selected blocks (§5.2 step 4, only the selected blocks are loaded),
leaves every byte of its outputs as the three separate calls leave them
(kk_append_tokens, the step with the ring, kk_compact_table), and both agree
with the fp64 oracle step by step while the requests grow past block
boundaries."""
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


def _compact_expected(idx, pages_r):
    """The selected logical blocks in ascending order, their pages, their
    number (slots past it -1)."""
    K = idx.shape[0]
    v = np.sort(idx[idx >= 0])
    lg = np.full(K, -1, dtype=np.int32)
    pg = np.full(K, -1, dtype=np.int32)
    lg[:v.size] = v
    pg[:v.size] = np.asarray(pages_r)[v]
    return pg, lg, v.size


class _State:
    """One copy of the mutable decode state: cache, running sums, v_b, ring."""

    def __init__(self, kk, spec, w_dev, slots):
        self.dev = DeviceCache(spec)
        self.block_sum = torch.zeros((spec.num_pages, spec.D), device="cuda")
        self.vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
        self.ring = kk.AnchorRing(spec.R, slots, spec.D)


def _prefill(kk, st, spec, w, w_dev):
    host = st.dev.host_view()
    kk.kk_pool_blocks(st.dev.desc, st.dev.pages, st.dev.n_valid, st.vb, head_w=w_dev,
                      w_set=_i32(np.repeat(np.arange(spec.R), spec.nb)) if w is not None else None)
    for r in range(spec.R):
        n = spec.seq_lens[r] % spec.bs
        if n:
            p = spec.pages_of(r)[-1]
            ww = np.ones((spec.L, spec.H)) if w is None else w[r].reshape(spec.L, spec.H).astype(np.float64)
            s = np.einsum("lh,lhtd->d", ww, ko.block_keys(host, p, n))
            st.block_sum[p] = torch.from_numpy(s.astype(np.float32)).cuda()
    kk.kk_anchor_ring_fill(st.dev.desc, st.dev.bt, st.ring, head_w=w_dev)


SPECS = {
    # short requests: one CTA a request
    "short": lambda: synth.qwen7b(L=3, H=2, D=128, bs=16, seq_lens=[3, 16, 37, 1], num_topics=4, W=8, K=4,
                                  extra_pages=16, shuffle_pages=True),
    # a long request among short ones: clusters of several CTAs
    "cluster": lambda: synth.qwen7b(L=2, H=2, D=128, bs=16, seq_lens=[16 * 300 - 2, 40, 16 * 64], num_topics=6,
                                    W=16, K=32, extra_pages=16, shuffle_pages=True),
    "f32-d64": lambda: synth.tiny_05b(L=3, H=2, D=64, bs=8, seq_lens=[8 * 6 + 1, 7, 8 * 3], num_topics=3, W=8,
                                      K=5, extra_pages=8),
    "d256": lambda: synth.qwen7b(L=2, H=1, D=256, bs=4, seq_lens=[4 * 7, 6], num_topics=2, W=4, K=3,
                                 layout="PLHTD", extra_pages=8),
    "token-major": lambda: synth.qwen7b(L=3, H=4, D=64, bs=8, seq_lens=[8 * 4 + 5, 8 * 2], num_topics=3, W=8,
                                        K=4, layout="LPTHD", extra_pages=8),
}


@pytest.mark.parametrize("name", sorted(SPECS))
@pytest.mark.parametrize("stable", [False, True])
@pytest.mark.parametrize("weighted", [False, True])
def test_fused_equals_separate_and_oracle(kk, name, stable, weighted):
    spec = SPECS[name]()
    R, L, H, D, bs, K, W = spec.R, spec.L, spec.H, spec.D, spec.bs, spec.K, spec.W
    rng = np.random.default_rng(101 + 2 * stable + weighted)
    w = rng.uniform(0.1, 1.0, size=(R, L * H)).astype(np.float32) if weighted else None
    w_dev = None if w is None else torch.from_numpy(w).cuda()
    slots = W + 3
    sep, fus = _State(kk, spec, w_dev, slots), _State(kk, spec, w_dev, slots)
    for st in (sep, fus):
        _prefill(kk, st, spec, w, w_dev)
    host = sep.dev.host_view().copy()
    f32 = spec.dtype == "f32"
    spare = list(np.setdiff1d(np.arange(spec.num_pages), spec.pages))
    tables = [list(spec.pages_of(r)) for r in range(R)]
    lens = list(spec.seq_lens)
    for step in range(2 * bs + 3):
        for r in range(R):
            if lens[r] % bs == 0:
                tables[r].append(spare.pop(0))
            lens[r] += 1
        offsets = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
        pages = np.concatenate(tables).astype(np.int32)
        bt = kk.BlockTable(_i32(pages), _i32(offsets), _i32(lens), max(len(t) for t in tables))
        kn = (1.5 * spec.cs[rng.integers(0, spec.num_topics, size=R)][:, None, None, :]
              + rng.standard_normal((R, L, H, D))).astype(np.float32)
        kn_store = kn if f32 else synth.bf16_rne(kn)
        kn_dev = torch.from_numpy(kn_store if f32 else kn_store.view(np.int16)).cuda()
        hist0 = torch.from_numpy(rng.integers(0, 2 ** 31, size=int(offsets[-1]), dtype=np.int64)
                                 .astype(np.int32)).cuda()
        outs = {}
        for tag, st in (("sep", sep), ("fus", fus)):
            o = dict(idx=torch.zeros((R, K), dtype=torch.int32, device="cuda"), top=torch.zeros((R, K), device="cuda"),
                     va=torch.zeros((R, D), device="cuda"),
                     sp=torch.full((R, K), 7, dtype=torch.int32, device="cuda"),
                     sl=torch.full((R, K), 7, dtype=torch.int32, device="cuda"),
                     sc=torch.full((R,), 7, dtype=torch.int32, device="cuda"), hist=hist0.clone())
            args = dict(top_scores=o["top"], va=o["va"], head_w=w_dev, ring=st.ring)
            if tag == "sep":
                kk.kk_append_tokens(st.dev.desc, bt, kn_dev, st.block_sum, st.vb, head_w=w_dev, ring=st.ring)
            else:
                args.update(append=(kn_dev, st.block_sum), compact=(o["sp"], o["sl"], o["sc"]))
            if stable:
                kk.kk_select_step_stable(st.dev.desc, bt, W, st.vb, K, 4, 0.55, o["hist"], o["idx"], **args)
            else:
                kk.kk_select_step(st.dev.desc, bt, W, st.vb, K, o["idx"], **args)
            if tag == "sep":
                kk.kk_compact_table(o["idx"], bt, o["sp"], o["sl"], o["sc"])
            assert kk.kk_device_error() == 0, f"{tag} step {step}"
            outs[tag] = {k: v.cpu().numpy() for k, v in o.items()}
        what = f"{name} stable={stable} weighted={weighted} step {step}"
        # every output and every piece of state, byte for byte
        for k in outs["sep"]:
            np.testing.assert_array_equal(outs["fus"][k], outs["sep"][k], err_msg=f"{what} {k}")
        for a, b, n in ((fus.block_sum, sep.block_sum, "block_sum"), (fus.vb, sep.vb, "vb"),
                        (fus.ring.rows, sep.ring.rows, "ring rows"), (fus.ring.pos, sep.ring.pos, "ring pos"),
                        (fus.dev.storage, sep.dev.storage, "cache")):
            # bytes, not values: unwritten cache slots hold NaN
            assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), f"{what} {n}"
        # and the oracle's decode step over the cache as written so far
        for r in range(R):
            ko.append_token(host, tables[r], lens[r], bs, kn_store[r], None if w is None else w[r])
        vb_now = fus.vb.cpu().numpy()
        for r in range(R):
            wr = None if w is None else w[r]
            va_o = ko.anchor(host, tables[r], lens[r], bs, W, wr)
            assert_vec_close(outs["fus"]["va"][r][None], va_o[None], f"{what} r={r} anchor")
            nvalid = [min(bs, lens[r] - j * bs) for j in range(len(tables[r]))]
            vb_o = ko.pool_blocks(host, tables[r], nvalid, None if wr is None else wr[None],
                                  np.zeros(len(tables[r]), dtype=np.int64))
            assert_vec_close(vb_now[tables[r]], vb_o, f"{what} r={r} v_b")
            if not stable:
                s_o = ko.affinity(vb_o, va_o)
                assert_topk_valid(outs["fus"]["idx"][r], outs["fus"]["top"][r], s_o, min(K, len(tables[r])),
                                  f"{what} r={r}")
            pg, lg, n = _compact_expected(outs["fus"]["idx"][r], tables[r])
            np.testing.assert_array_equal(outs["fus"]["sp"][r], pg, err_msg=f"{what} r={r} sel_pages")
            np.testing.assert_array_equal(outs["fus"]["sl"][r], lg, err_msg=f"{what} r={r} sel_logical")
            assert outs["fus"]["sc"][r] == n


def test_score_topk_compact_table(kk):
    """kk_score_topk with the compact-table option writes what
    kk_compact_table writes from its output."""
    spec = SPECS["cluster"]()
    dev = DeviceCache(spec)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    va = torch.randn((spec.R, spec.D), device="cuda")
    R, K = spec.R, spec.K
    res = []
    for fused in (False, True):
        idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
        sp, sl, sc = (torch.full((R, K), 9, dtype=torch.int32, device="cuda"),
                      torch.full((R, K), 9, dtype=torch.int32, device="cuda"),
                      torch.full((R,), 9, dtype=torch.int32, device="cuda"))
        if fused:
            kk.kk_score_topk(vb, dev.bt, va, K, idx, compact=(sp, sl, sc))
        else:
            kk.kk_score_topk(vb, dev.bt, va, K, idx)
            kk.kk_compact_table(idx, dev.bt, sp, sl, sc)
        assert kk.kk_device_error() == 0
        res.append([t.cpu().numpy() for t in (idx, sp, sl, sc)])
    for a, b in zip(*res):
        np.testing.assert_array_equal(a, b)
    for r in range(R):
        pg, lg, n = _compact_expected(res[1][0][r], spec.pages_of(r))
        np.testing.assert_array_equal(res[1][1][r], pg)
        assert res[1][3][r] == n


def test_fused_options_are_checked(kk):
    spec = SPECS["short"]()
    st = _State(kk, spec, None, spec.W)
    _prefill(kk, st, spec, None, None)
    kn = torch.zeros((spec.R, spec.L, spec.H, spec.D), dtype=torch.int16, device="cuda")
    idx = torch.zeros((spec.R, spec.K), dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):  # the fused write side needs the ring
        kk.kk_select_step(st.dev.desc, st.dev.bt, spec.W, st.vb, spec.K, idx, append=(kn, st.block_sum))
    with pytest.raises(RuntimeError):  # k_new off its 16-byte boundary
        kk.kk_select_step(st.dev.desc, st.dev.bt, spec.W, st.vb, spec.K, idx, ring=st.ring,
                          append=(kn.view(-1)[1:1 + kn.numel() - 8], st.block_sum))


@pytest.mark.parametrize("K", [32, 64])
@pytest.mark.parametrize("stable", [False, True])
def test_fused_split_request(kk, K, stable):
    """A request long enough to be split over several clusters (a caller
    workspace): the fused call's token write, output and compact table
    (written by the cluster that merges the splits' lists) are those of the
    separate calls, byte for byte, over steps that cross a block boundary;
    the selection is the oracle's top-K of the returned scores."""
    spec = synth.qwen7b(L=1, H=2, D=128, bs=16, seq_lens=[16 * 12000 - 2, 37], num_topics=8, W=16, K=K,
                        extra_pages=4, shuffle_pages=True)
    R, D, W = spec.R, spec.D, spec.W
    rng = np.random.default_rng(7 + stable)
    sep, fus = _State(kk, spec, None, W), _State(kk, spec, None, W)
    for st in (sep, fus):
        _prefill(kk, st, spec, None, None)
    nws = kk.kk_select_step_workspace_bytes(R, max(spec.nb) + 1, K)
    assert nws > 0
    spare = list(np.setdiff1d(np.arange(spec.num_pages), spec.pages))
    tables = [list(spec.pages_of(r)) for r in range(R)]
    lens = list(spec.seq_lens)
    for step in range(4):
        for r in range(R):
            if lens[r] % spec.bs == 0:
                tables[r].append(spare.pop(0))
            lens[r] += 1
        offsets = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
        pages = np.concatenate(tables).astype(np.int32)
        bt = kk.BlockTable(_i32(pages), _i32(offsets), _i32(lens), max(len(t) for t in tables))
        kn = synth.bf16_rne((1.5 * spec.cs[rng.integers(0, spec.num_topics, size=R)][:, None, None, :]
                             + rng.standard_normal((R, spec.L, spec.H, D))).astype(np.float32))
        kn_dev = torch.from_numpy(kn.view(np.int16)).cuda()
        hist0 = torch.from_numpy(rng.integers(0, 2 ** 31, size=int(offsets[-1]), dtype=np.int64).astype(np.int32)).cuda()
        outs = {}
        for tag, st in (("sep", sep), ("fus", fus)):
            ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
            o = dict(idx=torch.zeros((R, K), dtype=torch.int32, device="cuda"), top=torch.zeros((R, K), device="cuda"),
                     va=torch.zeros((R, D), device="cuda"), scores=torch.zeros(int(offsets[-1]), device="cuda"),
                     sp=torch.full((R, K), 7, dtype=torch.int32, device="cuda"),
                     sl=torch.full((R, K), 7, dtype=torch.int32, device="cuda"),
                     sc=torch.full((R,), 7, dtype=torch.int32, device="cuda"), hist=hist0.clone())
            args = dict(top_scores=o["top"], va=o["va"], scores=o["scores"], ring=st.ring, workspace=ws)
            if tag == "sep":
                kk.kk_append_tokens(st.dev.desc, bt, kn_dev, st.block_sum, st.vb, ring=st.ring)
            else:
                args.update(append=(kn_dev, st.block_sum), compact=(o["sp"], o["sl"], o["sc"]))
            if stable:
                kk.kk_select_step_stable(st.dev.desc, bt, W, st.vb, K, 4, 0.55, o["hist"], o["idx"], **args)
            else:
                kk.kk_select_step(st.dev.desc, bt, W, st.vb, K, o["idx"], **args)
            if tag == "sep":
                kk.kk_compact_table(o["idx"], bt, o["sp"], o["sl"], o["sc"])
            assert kk.kk_device_error() == 0, f"{tag} step {step}"
            w = ws.cpu().numpy()
            assert np.all(w[:8 * R].view(np.uint64) == 0) and np.any(w[256:] != 0), "the request was split"
            outs[tag] = {k: v.cpu().numpy() for k, v in o.items()}
        what = f"split K={K} stable={stable} step {step}"
        for k in outs["sep"]:
            np.testing.assert_array_equal(outs["fus"][k], outs["sep"][k], err_msg=f"{what} {k}")
        for a, b, n in ((fus.block_sum, sep.block_sum, "block_sum"), (fus.vb, sep.vb, "vb"),
                        (fus.ring.rows, sep.ring.rows, "ring rows"), (fus.ring.pos, sep.ring.pos, "ring pos"),
                        (fus.dev.storage, sep.dev.storage, "cache")):
            assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), f"{what} {n}"
        for r in range(R):
            sc = outs["fus"]["scores"][offsets[r]:offsets[r + 1]]
            if not stable:
                want_idx, _ = ko.topk(sc, K)
                np.testing.assert_array_equal(outs["fus"]["idx"][r], want_idx, err_msg=f"{what} r={r}")
            pg, lg, n = _compact_expected(outs["fus"]["idx"][r], tables[r])
            np.testing.assert_array_equal(outs["fus"]["sp"][r], pg, err_msg=f"{what} r={r} sel_pages")
            np.testing.assert_array_equal(outs["fus"]["sl"][r], lg, err_msg=f"{what} r={r} sel_logical")


def test_split_score_topk_compact_table(kk):
    """kk_score_topk with a workspace on a request long enough to split over
    clusters: the table the merging cluster writes is kk_compact_table's."""
    spec = synth.qwen7b(L=1, H=2, D=128, bs=16, seq_lens=[16 * 12000, 16 * 40], num_topics=8, W=16, K=64,
                        shuffle_pages=True)
    dev = DeviceCache(spec)
    vb = torch.zeros((spec.num_pages, spec.D), device="cuda")
    kk.kk_pool_blocks(dev.desc, dev.pages, dev.n_valid, vb)
    va = torch.randn((spec.R, spec.D), device="cuda")
    R, K = spec.R, spec.K
    res = []
    for fused in (False, True):
        ws = torch.zeros(kk.kk_select_step_workspace_bytes(R, max(spec.nb), K), dtype=torch.uint8, device="cuda")
        idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
        sp, sl, sc = (torch.full((R, K), 9, dtype=torch.int32, device="cuda"),
                      torch.full((R, K), 9, dtype=torch.int32, device="cuda"),
                      torch.full((R,), 9, dtype=torch.int32, device="cuda"))
        if fused:
            kk.kk_score_topk(vb, dev.bt, va, K, idx, workspace=ws, compact=(sp, sl, sc))
        else:
            kk.kk_score_topk(vb, dev.bt, va, K, idx, workspace=ws)
            kk.kk_compact_table(idx, dev.bt, sp, sl, sc)
        assert kk.kk_device_error() == 0
        assert np.any(ws.cpu().numpy()[256:] != 0), "the request was split"
        res.append([t.cpu().numpy() for t in (idx, sp, sl, sc)])
    for a, b in zip(*res):
        np.testing.assert_array_equal(a, b)


def test_fused_bad_token_page_is_reported(kk):
    """A request whose token block holds an out-of-range page: the fused call
    reports it on the device error word and leaves the other requests'
    outputs and state as the separate calls leave them."""
    spec = SPECS["short"]()
    R, D, K, W = spec.R, spec.D, spec.K, spec.W
    sep, fus = _State(kk, spec, None, W + 3), _State(kk, spec, None, W + 3)
    for st in (sep, fus):
        _prefill(kk, st, spec, None, None)
    # requests whose next token fits in their last block take one; the others
    # take none this step (their table and length stay as they are)
    grow = [r for r in range(R) if spec.seq_lens[r] % spec.bs]
    lens = [spec.seq_lens[r] + (1 if r in grow else 0) for r in range(R)]
    pages = np.array(spec.pages, dtype=np.int32)
    bad_r = grow[0]
    pages[spec.offsets[bad_r + 1] - 1] = spec.num_pages + 7  # the token's block
    bt = kk.BlockTable(_i32(pages), _i32(spec.offsets), _i32(lens), max(spec.nb))
    kn = torch.from_numpy(synth.bf16_rne(np.random.default_rng(3).standard_normal((R, spec.L, spec.H, D))
                                         .astype(np.float32)).view(np.int16)).cuda()
    outs = {}
    for tag, st in (("sep", sep), ("fus", fus)):
        idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
        va = torch.zeros((R, D), device="cuda")
        if tag == "sep":
            kk.kk_append_tokens(st.dev.desc, bt, kn, st.block_sum, st.vb, ring=st.ring)
            kk.kk_select_step(st.dev.desc, bt, W, st.vb, K, idx, va=va, ring=st.ring)
        else:
            kk.kk_select_step(st.dev.desc, bt, W, st.vb, K, idx, va=va, ring=st.ring, append=(kn, st.block_sum))
        assert kk.kk_device_error() == kk.KK_ERR_BAD_INDEX, tag
        outs[tag] = (idx.cpu().numpy(), va.cpu().numpy())
    ok = [r for r in range(R) if r != bad_r]
    np.testing.assert_array_equal(outs["fus"][0][ok], outs["sep"][0][ok])
    np.testing.assert_array_equal(outs["fus"][1][ok], outs["sep"][1][ok])
    for a, b in ((fus.vb, sep.vb), (fus.block_sum, sep.block_sum), (fus.dev.storage, sep.dev.storage)):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    assert kk.kk_device_error() == 0  # the word was cleared by the read


def _long_state(kk, seed):
    spec = synth.qwen7b(L=1, H=2, D=128, bs=16, seq_lens=[16 * 9000 - 3, 16 * 20 + 1], num_topics=8, W=16, K=32,
                        shuffle_pages=True, seed=seed)
    st = _State(kk, spec, None, spec.W)
    _prefill(kk, st, spec, None, None)
    lens = [t + 1 for t in spec.seq_lens]  # both tokens fit in their last blocks
    bt = kk.BlockTable(_i32(spec.pages), _i32(spec.offsets), _i32(lens), max(spec.nb))
    kn = torch.from_numpy(synth.bf16_rne(np.random.default_rng(seed).standard_normal(
        (spec.R, spec.L, spec.H, spec.D)).astype(np.float32)).view(np.int16)).cuda()
    ws = torch.zeros(kk.kk_select_step_workspace_bytes(spec.R, max(spec.nb), spec.K), dtype=torch.uint8,
                     device="cuda")
    out = dict(idx=torch.zeros((spec.R, spec.K), dtype=torch.int32, device="cuda"),
               sp=torch.zeros((spec.R, spec.K), dtype=torch.int32, device="cuda"),
               sc=torch.zeros(spec.R, dtype=torch.int32, device="cuda"))
    return spec, st, bt, kn, ws, out


def _fused_call(kk, spec, st, bt, kn, ws, out, stream=None):
    kk.kk_select_step(st.dev.desc, bt, spec.W, st.vb, spec.K, out["idx"], ring=st.ring, workspace=ws,
                      append=(kn, st.block_sum), compact=(out["sp"], None, out["sc"]), stream=stream)


def _snapshot(st, out):
    return [t.clone() for t in (st.vb, st.block_sum, st.ring.rows, st.ring.pos, out["idx"], out["sp"], out["sc"])]


def test_fused_two_streams_and_graph_replay(kk):
    """Two fused decode steps on split requests run at once on two streams,
    each with its own workspace, and as CUDA-graph replays: each leaves the
    bytes its eager call on a fresh copy of the same state leaves (the token
    is rewritten with the same Keys, so repeated calls are idempotent but for
    the running sums, which the eager reference repeats the same number of
    times)."""
    cases = [_long_state(kk, s) for s in (21, 22)]
    refs = [_long_state(kk, s) for s in (21, 22)]
    # eager references, one call each on the default stream
    for c in refs:
        _fused_call(kk, *c)
    torch.cuda.synchronize()
    assert kk.kk_device_error() == 0
    want = [_snapshot(c[1], c[5]) for c in refs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for c, s in zip(cases, streams):
        with torch.cuda.stream(s):
            _fused_call(kk, *c, stream=s)
    torch.cuda.synchronize()
    assert kk.kk_device_error() == 0
    for i, c in enumerate(cases):
        got = _snapshot(c[1], c[5])
        for a, b in zip(got, want[i]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"stream {i}"
    # the same call captured in a graph and replayed once more: a second
    # eager call on the references gives the state to compare with
    for c in refs:
        _fused_call(kk, *c)
    torch.cuda.synchronize()
    want2 = [_snapshot(c[1], c[5]) for c in refs]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c in cases:
                _fused_call(kk, *c, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert kk.kk_device_error() == 0
    for i, c in enumerate(cases):
        got = _snapshot(c[1], c[5])
        for a, b in zip(got, want2[i]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"graph {i}"
