"""Pins of the CPU oracle to things other than itself: hand-computed values
(tests/golden), closed forms, brute force written as plain loops, and
invariants that follow from the definitions. Each check is written as a
function of an oracle namespace so that test_oracle_mutants.py can show a
plausible mistake planted in the oracle fails at least one of them."""
import json
import math
import os
import random

import numpy as np
import pytest

import synth
from oracle import kk_oracle as ko

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _f(x):
    return float("-inf") if x == "-inf" else float(x)


# --------------------------------------------------------------------------
# checks parameterised by the oracle namespace
# --------------------------------------------------------------------------


def check_pool_golden(o):
    g = gold("pool_tiny.json")
    K = np.array(g["K"], dtype=np.float64)  # [L][H][n][D]
    np.testing.assert_allclose(o.pool_block(K), g["vb_uniform"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o.pool_block(K, g["head_w"]), g["vb_weighted"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o.pool_block(K[:, :, :1, :]), g["vb_uniform_n1"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(o.pool_block(K[:, :, :0, :]), [0.0, 0.0])


def check_decode_golden(o):
    # bf16 bit patterns and their exact values, worked out from the format's bit fields
    for c in gold("bf16_decode.json")["cases"]:
        got = float(o.decode(np.array([int(c["bits"], 16)], dtype=np.uint16))[0])
        want = float(c["value"]) if c["value"] in ("inf", "-inf") else float.fromhex(c["value"])
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (c, got)
    # float32 and float64 inputs are taken as they are
    np.testing.assert_array_equal(o.decode(np.array([1.5, -2.25], dtype=np.float32)), [1.5, -2.25])


def check_affinity_golden(o):
    for c in gold("affinity.json")["cases"]:
        s = o.affinity(np.array([c["vb"]], float), np.array(c["va"], float))[0]
        assert abs(s - c["score"]) < 1e-15, c


def check_topk_golden(o):
    g = gold("topk.json")
    for c in g["cases"]:
        idx, val = o.topk(g["scores"], c["K"])
        assert list(idx) == c["idx"]
        assert [float(v) for v in val] == [_f(v) for v in c["score"]]


def _anchor_cache(g):
    # [L=1][P=2][H=1][bs=2][D=2], invalid slot = NaN
    kc = np.full((1, 2, 1, 2, 2), np.nan)
    for p, page in enumerate(g["K"]):
        for t, row in enumerate(page):
            if row is not None:
                kc[0, p, 0, t] = row
    return kc


def check_anchor_golden(o):
    g = gold("anchor.json")
    kc = _anchor_cache(g)
    for c in g["cases"]:
        va = o.anchor(kc, g["pages_r"], g["seq_len"], 2, c["W"])
        np.testing.assert_allclose(va, c["va"], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(o.anchor(kc, g["pages_r"], 0, 2, 4), [0.0, 0.0])


def check_variance_golden(o):
    for c in gold("variance.json")["cases"]:
        k = np.array(c["K_h_t_d"], float)  # [H][T][D]
        H, T, D = k.shape
        kc = k[None, None, :, :, :]  # [L=1][P=1][H][bs=T][D]
        w = o.head_variance_weights(kc, [0], T, T)
        np.testing.assert_allclose(w, c["weights"], rtol=1e-14, atol=1e-15)


def check_coarse_golden(o):
    g = gold("coarse.json")
    np.testing.assert_allclose(o.coarse_means(np.array(g["vb"], float), g["group"]), g["out"], atol=0)


def check_batched_golden(o):
    g = gold("batched.json")
    idx, val = o.score_pool_batched(np.array(g["A"], float), np.array(g["V"], float),
                                    np.array(g["mask_words"], np.uint32), g["K"])
    assert idx.tolist() == g["idx"]
    np.testing.assert_allclose(val, g["score"], rtol=1e-15)


# ---- brute force: plain loops, written independently of the oracle ------


def bf_pool(K, n, w=None):
    L, H, _, D = K.shape
    out = [0.0] * D
    for d in range(D):
        acc = 0.0
        for l in range(L):
            for h in range(H):
                s = 0.0
                for t in range(n):
                    s += float(K[l][h][t][d])
                wl = (1.0 / (L * H)) if w is None else float(w[l * H + h])
                acc += wl * (s / n if n else 0.0)
        out[d] = acc
    return out


def bf_cos_score(a, b):
    dot = sum(float(x) * float(y) for x, y in zip(a, b))
    na = math.sqrt(sum(float(x) ** 2 for x in a))
    nb = math.sqrt(sum(float(y) ** 2 for y in b))
    c = 0.0 if na == 0 or nb == 0 else dot / (na * nb)
    return (1.0 + c) / 2.0


def bf_topk(s, K):
    order = sorted(range(len(s)), key=lambda j: (-s[j], j))[:K]
    return order + [-1] * (K - len(order))


def check_bruteforce(o, seed=0):
    rng = random.Random(seed)
    for _ in range(20):
        L, H, bs, D = rng.randint(1, 3), rng.randint(1, 3), rng.randint(1, 4), rng.randint(2, 4)
        P = rng.randint(2, 5)
        kc = np.array([[[[[rng.randint(-4, 4) for _ in range(D)] for _ in range(bs)] for _ in range(H)]
                        for _ in range(P)] for _ in range(L)], dtype=np.float64)
        p, n = rng.randrange(P), rng.randint(0, bs)
        w = [rng.random() for _ in range(L * H)]
        blk = kc[:, p, :, :, :]
        np.testing.assert_allclose(o.pool_blocks(kc, [p], [n])[0], bf_pool(blk, n), atol=1e-12)
        np.testing.assert_allclose(o.pool_blocks(kc, [p], [n], [w], [0])[0], bf_pool(blk, n, w), atol=1e-12)
        # anchor through a random block table
        nbk = rng.randint(1, P)
        pages_r = rng.sample(range(P), nbk)
        T = rng.randint((nbk - 1) * bs + 1, nbk * bs)
        W = rng.randint(1, T + 2)
        we = min(W, T)
        want = [0.0] * D
        for d in range(D):
            for l in range(L):
                for h in range(H):
                    s = 0.0
                    for q in range(T - we, T):
                        s += kc[l][pages_r[q // bs]][h][q % bs][d]
                    want[d] += s / we / (L * H)
        np.testing.assert_allclose(o.anchor(kc, pages_r, T, bs, W), want, atol=1e-12)
        # affinity + top-K on random vectors (some zero)
        vb = [[rng.randint(-3, 3) for _ in range(D)] for _ in range(rng.randint(1, 9))]
        va = [rng.randint(-3, 3) for _ in range(D)]
        s_bf = [bf_cos_score(v, va) for v in vb]
        s_o = o.affinity(np.array(vb, float), np.array(va, float))
        np.testing.assert_allclose(s_o, s_bf, atol=1e-14)
        K = rng.randint(1, len(vb) + 2)
        assert list(o.topk(s_bf, K)[0]) == bf_topk(s_bf, K)


def check_batched_bruteforce(o, seed=1):
    rng = np.random.default_rng(seed)
    R, N, D, K = 3, 70, 4, 5
    A = rng.integers(-3, 4, size=(R, D)).astype(float)
    V = rng.integers(-3, 4, size=(N, D)).astype(float)
    mask = np.zeros((R, 3), np.uint32)
    owned = [sorted(rng.choice(N, size=rng.integers(0, 12), replace=False).tolist()) for _ in range(R)]
    for r, js in enumerate(owned):
        for j in js:
            mask[r, j // 32] |= np.uint32(1 << (j % 32))
    idx, val = o.score_pool_batched(A, V, mask, K)
    for r in range(R):
        s = {j: bf_cos_score(V[j], A[r]) for j in owned[r]}
        order = sorted(s, key=lambda j: (-s[j], j))[:K]
        assert idx[r].tolist() == order + [-1] * (K - len(order))


# ---- invariants ----------------------------------------------------------


def small_specs():
    return [
        synth.tiny_05b(L=3, seq_lens=[16 * 12 + 5, 16 * 3], num_topics=4),
        synth.qwen7b(L=2, H=2, D=32, bs=8, seq_lens=[64, 40, 8], num_topics=4, W=5, K=6),
    ]


def check_reblocking(o):
    # same tokens cut at block size 8 and 32 (topics change every 32 tokens)
    a = synth.qwen7b(L=2, H=2, D=16, bs=8, seq_lens=[128], span=32, num_topics=4, seed=11)
    b = synth.qwen7b(L=2, H=2, D=16, bs=32, seq_lens=[128], span=32, num_topics=4, seed=11)
    ka = synth.view_paged(synth.gen_paged_numpy(a), a)
    kb = synth.view_paged(synth.gen_paged_numpy(b), b)
    va = o.pool_blocks(ka, a.pages, a.n_valid)
    vb = o.pool_blocks(kb, b.pages, b.n_valid)
    np.testing.assert_allclose(va.reshape(4, 4, -1).mean(axis=1), vb, rtol=1e-12, atol=1e-12)
    # coarse means of the fine level reproduce the coarse blocks
    np.testing.assert_allclose(o.coarse_means(va, 4), vb, rtol=1e-12, atol=1e-12)
    # and the mean over all blocks is the same at both block sizes
    np.testing.assert_allclose(o.coarse_means(va, 16), o.coarse_means(vb, 4), rtol=1e-12, atol=1e-12)


def check_linearity_and_symmetry(o, seed=2):
    rng = np.random.default_rng(seed)
    L, H, n, D = 3, 2, 5, 4
    k1, k2 = rng.standard_normal((2, L, H, n, D))
    np.testing.assert_allclose(o.pool_block(2.0 * k1 - 3.0 * k2), 2.0 * o.pool_block(k1) - 3.0 * o.pool_block(k2),
                               rtol=1e-12, atol=1e-12)
    perm_l, perm_h = rng.permutation(L), rng.permutation(H)
    np.testing.assert_allclose(o.pool_block(k1[perm_l][:, perm_h]), o.pool_block(k1), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o.pool_block(k1, [0.7] * (L * H)) / (0.7 * L * H), o.pool_block(k1), rtol=1e-12)
    # scaling either vector leaves the score unchanged
    vb, va = rng.standard_normal((5, D)), rng.standard_normal(D)
    np.testing.assert_allclose(o.affinity(3.5 * vb, 0.25 * va), o.affinity(vb, va), rtol=1e-13)
    # an equal set of weights is the unweighted mean: scale-free variance weights
    kc = rng.standard_normal((L, 1, H, n, D))
    w = o.head_variance_weights(kc, [0], n, n)
    w2 = o.head_variance_weights(3.0 * kc + 1.0, [0], n, n)
    np.testing.assert_allclose(w, w2, rtol=1e-12)
    assert abs(w.sum() - 1.0) < 1e-12


def check_page_shuffle(o):
    a = synth.qwen7b(L=2, H=2, D=16, bs=4, seq_lens=[30, 17], num_topics=3, seed=21)
    b = synth.qwen7b(L=2, H=2, D=16, bs=4, seq_lens=[30, 17], num_topics=3, seed=21, shuffle_pages=True, extra_pages=5)
    assert not np.array_equal(a.pages, b.pages[: a.total_blocks])
    ka = synth.view_paged(synth.gen_paged_numpy(a), a)
    kb = synth.view_paged(synth.gen_paged_numpy(b), b)
    for r in range(a.R):
        T = a.seq_lens[r]
        la = o.pool_blocks(ka, a.pages_of(r), a.n_valid[a.offsets[r]:a.offsets[r + 1]])
        lb = o.pool_blocks(kb, b.pages_of(r), b.n_valid[b.offsets[r]:b.offsets[r + 1]])
        np.testing.assert_array_equal(la, lb)
        np.testing.assert_array_equal(o.anchor(ka, a.pages_of(r), T, 4, 6), o.anchor(kb, b.pages_of(r), T, 4, 6))
        np.testing.assert_array_equal(o.head_variance_weights(ka, a.pages_of(r), T, 4),
                                      o.head_variance_weights(kb, b.pages_of(r), T, 4))


def check_planted_topics(o):
    for spec in small_specs() + [synth.tiny_05b()]:
        kc = synth.view_paged(synth.gen_paged_numpy(spec), spec)
        vb_table = np.zeros((spec.num_pages, spec.D))
        vb_table[spec.pages] = o.pool_blocks(kc, spec.pages, spec.n_valid)
        for r in range(spec.R):
            pr = spec.pages_of(r)
            va = o.anchor(kc, pr, spec.seq_lens[r], spec.bs, spec.W)
            s, idx, _ = o.score_topk(vb_table, pr, va, spec.K)
            topic = spec.block_topic[spec.offsets[r]:spec.offsets[r + 1]]
            same = np.flatnonzero(topic == spec.query_topic[r])
            m = min(spec.K, len(same))
            assert set(idx[:m].tolist()) <= set(same.tolist()), (spec.name, r)
            off = np.flatnonzero(topic != spec.query_topic[r])
            if len(off):
                assert s[same].min() > s[off].max()


def check_stability_golden(o):
    g = gold("stability.json")
    for c in g["cases"]:
        hist = np.array(c["history"], dtype=np.float64)[:, None]  # [steps][1 block]
        got = o.stability(hist, g["W"], g["theta"])
        assert abs(got[0] - c["stability"]) < 1e-15, c


def check_stability_window(o):
    # the threshold is strict, the fraction is over W, and the window slides
    W, th = 4, 0.5
    hist = np.array([[0.9, 0.5, 0.51, 0.0],
                     [0.9, 0.5, 0.49, 0.0],
                     [0.1, 0.5, 0.51, 0.0]])
    np.testing.assert_array_equal(o.stability(hist, W, th), [2 / 4, 0.0, 2 / 4, 0.0])  # 3 steps, still over W
    more = np.vstack([hist, [[0.1, 0.6, 0.1, 0.7]] * 2])  # 5 steps: the first drops out
    np.testing.assert_array_equal(o.stability(more, W, th), [1 / 4, 2 / 4, 1 / 4, 2 / 4])
    # W = 1: the indicator of the last step
    np.testing.assert_array_equal(o.stability(more, 1, th), [0.0, 1.0, 0.0, 1.0])


def check_stable_topk(o):
    stab = [0.05, 1.0, 1.0, 0.5, 1.0]
    scores = [0.9, 0.3, 0.7, 0.8, 0.7]
    idx, val = o.stable_topk(stab, scores, 6)
    assert list(idx) == [2, 4, 1, 3, 0, -1]  # stability, then affinity, then the lower index
    assert [float(v) for v in val] == [0.7, 0.7, 0.3, 0.8, 0.9, float("-inf")]


def check_compact_table_golden(o):
    g = gold("compact_table.json")
    for c in g["cases"]:
        pages, logical, n = o.compact_table(g["pages"], c["idx"])
        assert list(pages) == c["pages"] and list(logical) == c["logical"] and n == c["count"], c


def check_append_token(o):
    # one layer, one head, D = 2, block size 3: hand-computed running means
    kc = np.full((1, 3, 1, 3, 2), np.nan)
    pages_r = [2, 0]
    toks = [[2.0, 4.0], [4.0, 0.0], [0.0, 8.0], [6.0, -2.0]]
    want = [(2, [2.0, 4.0]), (2, [3.0, 2.0]), (2, [2.0, 4.0]), (0, [6.0, -2.0])]
    for t, (k, (pg, vb)) in enumerate(zip(toks, want)):
        page, got = o.append_token(kc, pages_r, t + 1, 3, np.array(k).reshape(1, 1, 2))
        assert page == pg and np.array_equal(got, vb), (t, page, got)
    assert np.array_equal(kc[0, 2, 0], [[2, 4], [4, 0], [0, 8]]) and np.array_equal(kc[0, 0, 0, 0], [6, -2])
    assert np.isnan(kc[0, 0, 0, 1:]).all() and np.isnan(kc[0, 1]).all()  # nothing else written
    # a block filled token by token equals the block pooled at once (weighted too)
    spec = synth.tiny_05b(L=2, H=3, D=4, bs=5, seq_lens=[5 * 3], num_topics=2, W=2, K=2)
    full = synth.view_paged(synth.gen_paged_numpy(spec), spec)
    kc = np.full_like(full, np.nan)
    w = np.arange(1.0, 7.0) / 21.0
    pr = spec.pages_of(0)
    for t in range(spec.seq_lens[0]):
        j, slot = divmod(t, spec.bs)
        page, got = o.append_token(kc, pr, t + 1, spec.bs, full[:, pr[j], :, slot, :], w)
        want = o.pool_blocks(full, [pr[j]], [slot + 1], [w], [0])[0]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def check_hier_golden(o):
    g = gold("hier.json")
    vb = np.array(g["vb"], dtype=np.float64)
    chunks, grids = o.hier_reps(vb, g["chunk_pages"], g["grid_chunks"])
    np.testing.assert_array_equal(chunks, g["chunks"])
    np.testing.assert_array_equal(grids, g["grids"])
    for c in g["cases"]:
        idx, val, kept, gk, ck = o.hier_select(vb, np.array(g["va"]), c["K"], g["chunk_pages"], g["grid_chunks"],
                                               c["permille"])
        assert list(idx) == c["idx"] and kept == c["kept"], c
        assert list(gk) == c["grids_kept"] and list(ck) == c["chunks_kept"], c


def check_hier_invariants(o):
    rng = np.random.default_rng(21)
    for nb, cp, gc in ((1000, 64, 8), (77, 4, 3), (5, 64, 8), (130, 8, 2)):
        vb = rng.standard_normal((nb, 6))
        va = rng.standard_normal(6)
        s = o.affinity(vb, va)
        # keeping every grid and chunk reduces to the plain top-k of all pages
        for q in (100, 333, 1000):
            k = -(-nb * q // 1000)
            idx, val, kept, _, _ = o.hier_select(vb, va, nb, cp, gc, (1000, 1000, q))
            want, _ = o.topk(s, k)
            assert kept == k and list(idx[:k]) == list(want)
        # the kept sets nest, and each level keeps its share of the active members
        idx, val, kept, gk, ck = o.hier_select(vb, va, nb, cp, gc)
        C = -(-nb // cp)
        G = -(-C // gc)
        assert len(gk) == -(-G * 500 // 1000)
        active_c = [c for c in range(C) if c // gc in set(gk.tolist())]
        assert set(ck.tolist()) <= set(active_c) and len(ck) == -(-len(active_c) * 200 // 1000)
        active_p = [j for j in range(nb) if j // cp in set(ck.tolist())]
        assert set(idx[:kept].tolist()) <= set(active_p) and kept == -(-len(active_p) * 100 // 1000)
        np.testing.assert_array_equal(val[:kept], s[idx[:kept]])
    # a Grid is the mean of its Chunks, not of its pages (partial last chunk)
    vb = np.array([[1.0, 0.0]] * 4 + [[0.0, 1.0]])
    chunks, grids = o.hier_reps(vb, 2, 4)
    np.testing.assert_allclose(grids[0], [2.0 / 3.0, 1.0 / 3.0], rtol=0, atol=1e-15)


def check_hier_pool_golden(o):
    g = gold("hier_pool.json")
    vb = np.array(g["vb"], dtype=np.float64)
    for c in g["cases"]:
        idx, val, kept = o.hier_select_pool(np.array([c["va"]]), np.array(g["grids"]), np.array(g["chunks"]), vb,
                                            np.array([[c["mask"]]], dtype=np.uint32), c["K"], g["chunk_pages"],
                                            g["grid_chunks"], c["permille"])
        assert list(idx[0]) == c["idx"] and kept[0] == c["kept"], c


def _zeroed_levels(sg, sc, sp, allowed, cp, gc, pm):
    """The page's formulation, as plain loops: scores of members whose parent
    was not kept (or that cover no allowed block) are set to zero, and each
    level takes its share of the active count from the whole zeroed level."""
    N, C, G = len(sp), len(sc), len(sg)
    c_ok = [any(allowed[b] for b in range(c * cp, min(N, (c + 1) * cp))) for c in range(C)]
    g_ok = [any(c_ok[c] for c in range(g * gc, min(C, (g + 1) * gc))) for g in range(G)]

    def take(scores, active, q):
        n = sum(active)
        m = (n * q + 999) // 1000
        z = [scores[i] if active[i] else 0.0 for i in range(len(scores))]
        return sorted(range(len(z)), key=lambda i: (-z[i], i))[:m]

    gk = set(take(sg, g_ok, pm[0]))
    ck = set(take(sc, [c_ok[c] and c // gc in gk for c in range(C)], pm[1]))
    return take(sp, [bool(allowed[b]) and b // cp in ck for b in range(N)], pm[2])


def check_hier_pool_bruteforce(o):
    rng = np.random.default_rng(33)
    for N, cp, gc, pm, density in ((300, 8, 3, (500, 200, 100), 0.3), (64, 4, 2, (700, 500, 400), 0.05),
                                   (257, 16, 4, (300, 1000, 250), 0.9), (40, 64, 8, (500, 500, 500), 0.5)):
        D, R = 5, 6
        V = rng.standard_normal((N, D))
        A = rng.standard_normal((R, D))
        chunks, grids = o.hier_reps(V, cp, gc)
        bits = rng.random((R, N)) < density
        bits[0, :] = False
        mw = np.zeros((R, (N + 31) // 32), dtype=np.uint32)
        for r in range(R):
            for j in np.nonzero(bits[r])[0]:
                mw[r, j // 32] |= np.uint32(1 << (j % 32))
        idx, val, kept = o.hier_select_pool(A, grids, chunks, V, mw, N, cp, gc, pm)
        for r in range(R):
            want = _zeroed_levels(o.affinity(grids, A[r]), o.affinity(chunks, A[r]), o.affinity(V, A[r]),
                                  bits[r], cp, gc, pm)
            assert kept[r] == len(want) and list(idx[r, :kept[r]]) == want, (N, r)
            assert np.all(idx[r, kept[r]:] == -1)
    # one request's blocks at the start of the pool, on a Grid boundary: the per-request hierarchy
    V = rng.standard_normal((700, 4))
    A = rng.standard_normal((1, 4))
    chunks, grids = o.hier_reps(V, 8, 4)
    nb = 8 * 4 * 15
    mw = np.zeros((1, (700 + 31) // 32), dtype=np.uint32)
    mw[0, :nb // 32] = 0xFFFFFFFF
    idx, val, kept = o.hier_select_pool(A, grids, chunks, V, mw, 50, 8, 4, (400, 300, 200))
    w_idx, w_val, w_kept, _, _ = o.hier_select(V[:nb], A[0], 50, 8, 4, (400, 300, 200))
    assert kept[0] == w_kept and list(idx[0]) == list(w_idx)
    # every level kept whole: the batched scorer's top-K of the allowed blocks
    mw = rng.integers(0, 2**32, size=(3, (700 + 31) // 32), dtype=np.uint64).astype(np.uint32)
    A = rng.standard_normal((3, 4))
    idx, val, kept = o.hier_select_pool(A, grids, chunks, V, mw, 90, 8, 4, (1000, 1000, 1000))
    w_idx, w_val = o.score_pool_batched(A, V, mw, 90)
    assert np.array_equal(idx, w_idx) and np.array_equal(val, w_val)
    allowed = [sum(bin(int(w)).count("1") for w in mw[r, :700 // 32]) +
               bin(int(mw[r, 700 // 32]) & ((1 << (700 % 32)) - 1)).count("1") for r in range(3)]
    assert list(kept) == allowed


ALL_CHECKS = [
    check_decode_golden,
    check_pool_golden, check_affinity_golden, check_topk_golden, check_anchor_golden,
    check_variance_golden, check_coarse_golden, check_batched_golden, check_bruteforce,
    check_batched_bruteforce, check_reblocking, check_linearity_and_symmetry, check_page_shuffle,
    check_planted_topics, check_stability_golden, check_stability_window, check_stable_topk,
    check_compact_table_golden, check_append_token, check_hier_golden, check_hier_invariants,
    check_hier_pool_golden, check_hier_pool_bruteforce,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ko)


# --------------------------------------------------------------------------
# the generator itself
# --------------------------------------------------------------------------


def test_splitmix64_published_vector():
    # SplitMix64 seeded with 0: the first three outputs of the reference
    # generator (Steele, Lea & Flood 2014).
    z = [synth._mix64_int(k * synth.GOLDEN) for k in (1, 2, 3)]
    assert z == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    arr = synth.mix64(np.array([k * synth.GOLDEN & synth.MASK64 for k in (1, 2, 3)], dtype=np.uint64))
    assert arr.tolist() == z


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = (np.random.default_rng(0).standard_normal(200000) * 37).astype(np.float32)
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 0.0]  # exact halfway cases: ties to even
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.bf16_rne(x), want)


def test_noise_moments_and_exactness():
    n = synth.noise(synth.stream_key(9, 1), np.arange(400000, dtype=np.uint64))
    assert abs(float(n.mean())) < 0.01 and abs(float(n.var()) - 1.0) < 0.01
    assert np.all(np.abs(n) <= 6.0)
    # every value is an exact multiple of 2^-16 (integer numerator, exact scale)
    scaled = n.astype(np.float64) * 2.0**17
    assert np.array_equal(scaled, np.round(scaled))


def test_generator_layouts_hold_same_keys():
    a = synth.qwen7b(L=2, H=3, D=8, bs=4, seq_lens=[9, 4], num_topics=3, seed=5)
    b = synth.qwen7b(L=2, H=3, D=8, bs=4, seq_lens=[9, 4], num_topics=3, seed=5, layout="LPTHD")
    ka = synth.view_paged(synth.gen_paged_numpy(a), a)
    kb = synth.view_paged(synth.gen_paged_numpy(b), b)
    np.testing.assert_array_equal(ka, kb)
    # tails of partial blocks are NaN sentinels
    tail = ka[:, a.pages[2], :, 1:, :]
    assert np.all(tail == synth.BF16_NAN_BITS)
