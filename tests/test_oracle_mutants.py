"""Plausible mistakes planted in a copy of the CPU oracle must each fail at
least one pin of tests/test_oracle_pins.py (the mistakes live only here, on
the CPU, in a namespace copy; the real oracle is untouched)."""
import types

import numpy as np
import pytest

from oracle import kk_oracle as ko
from tests.test_oracle_pins import ALL_CHECKS


def _copy():
    return types.SimpleNamespace(**{k: getattr(ko, k) for k in dir(ko) if not k.startswith("__")})


def m_pool_divides_by_heads_only(o):
    def pool_block(keys, head_w=None):
        L, H, n, D = keys.shape
        if n == 0:
            return np.zeros(D)
        w = o._weights(L, H, head_w)
        return np.einsum("lh,lhd->d", w * L, keys.sum(axis=2) / n)
    o.pool_block = pool_block


def m_pool_weights_transposed(o):
    def _weights(L, H, head_w):
        if head_w is None:
            return np.full((L, H), 1.0 / (L * H))
        return np.asarray(head_w, dtype=np.float64).reshape(H, L).T

    def pool_block(keys, head_w=None):
        L, H, n, D = keys.shape
        if n == 0:
            return np.zeros(D)
        return np.einsum("lh,lhd->d", _weights(L, H, head_w), keys.sum(axis=2) / n)
    o.pool_block = pool_block


def m_pool_sum_not_mean(o):
    def pool_block(keys, head_w=None):
        L, H, n, D = keys.shape
        if n == 0:
            return np.zeros(D)
        return np.einsum("lh,lhd->d", o._weights(L, H, head_w), keys.sum(axis=2))
    o.pool_block = pool_block


def m_decode_shift_15(o):
    def decode(x):
        x = np.asarray(x)
        if x.dtype == np.uint16:
            return (x.astype(np.uint32) << 15).view(np.float32).astype(np.float64)
        return x.astype(np.float64)
    o.decode = decode


def m_decode_reads_fp16(o):
    def decode(x):
        x = np.asarray(x)
        if x.dtype == np.uint16:
            return x.view(np.float16).astype(np.float64)
        return x.astype(np.float64)
    o.decode = decode


def m_decode_drops_sign(o):
    def decode(x):
        x = np.asarray(x)
        if x.dtype == np.uint16:
            return ((x.astype(np.uint32) & 0x7FFF) << 16).view(np.float32).astype(np.float64)
        return x.astype(np.float64)
    o.decode = decode


def m_affinity_not_halved(o):
    base = ko.affinity
    o.affinity = lambda vb, va: 2.0 * base(vb, va)


def m_affinity_raw_dot(o):
    def affinity(vb, va):
        vb = np.atleast_2d(ko.decode(vb))
        return (1.0 + vb @ ko.decode(va)) / 2.0
    o.affinity = affinity


def m_affinity_zero_vector_scores_zero(o):
    def affinity(vb, va):
        vb = np.atleast_2d(ko.decode(vb))
        va = ko.decode(va)
        denom = np.sqrt((vb * vb).sum(axis=1)) * np.sqrt((va * va).sum())
        return np.where(denom > 0, (1.0 + (vb @ va) / np.where(denom > 0, denom, 1)) / 2.0, 0.0)
    o.affinity = affinity


def m_topk_ties_to_higher_index(o):
    def topk(scores, K):
        s = np.asarray(scores, dtype=np.float64)
        order = np.lexsort((-np.arange(len(s)), -s))[:K]
        idx = np.full(K, -1, dtype=np.int64)
        val = np.full(K, -np.inf)
        idx[: len(order)] = order
        val[: len(order)] = s[order]
        return idx, val
    o.topk = topk


def m_topk_ascending(o):
    base = ko.topk
    o.topk = lambda scores, K: base(-np.asarray(scores, dtype=np.float64), K)


def m_anchor_first_tokens(o):
    def anchor(kc, pages_r, seq_len, bs, W, head_w=None):
        L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
        w_eff = min(W, seq_len)
        if w_eff == 0:
            return np.zeros(D)
        rows = np.stack([ko.decode(kc[:, int(pages_r[p // bs]), :, p % bs, :]) for p in range(w_eff)])
        return np.einsum("lh,lhd->d", o._weights(L, H, head_w), rows.mean(axis=0))
    o.anchor = anchor


def m_anchor_ignores_block_table(o):
    def anchor(kc, pages_r, seq_len, bs, W, head_w=None):
        L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
        w_eff = min(W, seq_len)
        if w_eff == 0:
            return np.zeros(D)
        rows = np.stack([ko.decode(kc[:, p // bs, :, p % bs, :]) for p in range(seq_len - w_eff, seq_len)])
        return np.einsum("lh,lhd->d", o._weights(L, H, head_w), rows.mean(axis=0))
    o.anchor = anchor


def m_variance_one_mean_for_all_dims(o):
    # (a sample variance, ddof=1, is not a mistake here: the factor T/(T-1)
    # is shared by every head of a request and cancels in the normalisation)
    def head_variance_weights(kc, pages_r, seq_len, bs):
        L, H = kc.shape[0], kc.shape[2]
        var = np.zeros((L, H))
        for layer in range(L):
            k = ko.request_tokens_of_layer(kc, layer, pages_r, seq_len, bs)
            var[layer] = k.reshape(H, -1).var(axis=1) if k.shape[1] else 0.0
        return (var / var.sum()).reshape(L * H) if var.sum() else np.full(L * H, 1.0 / (L * H))
    o.head_variance_weights = head_variance_weights


def m_variance_std_not_var(o):
    def head_variance_weights(kc, pages_r, seq_len, bs):
        L, H = kc.shape[0], kc.shape[2]
        var = np.zeros((L, H))
        for layer in range(L):
            k = ko.request_tokens_of_layer(kc, layer, pages_r, seq_len, bs)
            var[layer] = np.sqrt(k.var(axis=1).mean(axis=1))
        return (var / var.sum()).reshape(L * H) if var.sum() else np.full(L * H, 1.0 / (L * H))
    o.head_variance_weights = head_variance_weights


def m_coarse_last_group_divided_by_group(o):
    def coarse_means(vb_logical, group):
        vb_logical = ko.decode(vb_logical)
        nb = vb_logical.shape[0]
        ng = (nb + group - 1) // group
        return np.stack([vb_logical[g * group:(g + 1) * group].sum(axis=0) / group for g in range(ng)])
    o.coarse_means = coarse_means


def m_batched_ignores_mask(o):
    def score_pool_batched(A, V, mask_words, K):
        full = np.full_like(np.asarray(mask_words, dtype=np.uint32), 0xFFFFFFFF)
        return ko.score_pool_batched(A, V, full, K)
    o.score_pool_batched = score_pool_batched


def m_stability_counts_equal_theta(o):
    def stability(score_history, W=20, theta=0.5):
        h = np.asarray(score_history, dtype=np.float64)
        return (h[max(0, h.shape[0] - W):] >= theta).sum(axis=0) / float(W)
    o.stability = stability


def m_stability_divides_by_steps_seen(o):
    def stability(score_history, W=20, theta=0.5):
        h = np.asarray(score_history, dtype=np.float64)
        recent = h[max(0, h.shape[0] - W):]
        return (recent > theta).sum(axis=0) / float(recent.shape[0])
    o.stability = stability


def m_stability_window_one_too_long(o):
    def stability(score_history, W=20, theta=0.5):
        h = np.asarray(score_history, dtype=np.float64)
        return (h[max(0, h.shape[0] - W - 1):] > theta).sum(axis=0) / float(W)
    o.stability = stability


def m_stable_topk_ignores_stability(o):
    o.stable_topk = lambda stab, scores, K: ko.topk(scores, K)


def m_compact_table_keeps_topk_order(o):
    def compact_table(pages_r, idx_r):
        pages_r = np.asarray(pages_r, dtype=np.int64)
        idx_r = np.asarray(idx_r, dtype=np.int64)
        chosen = idx_r[idx_r >= 0]
        logical = np.full(len(idx_r), -1, dtype=np.int64)
        pages = np.full(len(idx_r), -1, dtype=np.int64)
        logical[:len(chosen)] = chosen
        pages[:len(chosen)] = pages_r[chosen]
        return pages, logical, len(chosen)
    o.compact_table = compact_table


def m_append_token_divides_by_block_size(o):
    def append_token(kc, pages_r, seq_len, bs, k_new, head_w=None):
        t = seq_len - 1
        page = int(np.asarray(pages_r)[t // bs])
        kc[:, page, :, t % bs, :] = k_new
        v = ko.pool_block(ko.block_keys(kc, page, t % bs + 1), head_w)
        return page, v * (t % bs + 1) / bs
    o.append_token = append_token


def m_append_token_slot_off_by_one(o):
    def append_token(kc, pages_r, seq_len, bs, k_new, head_w=None):
        page = int(np.asarray(pages_r)[(seq_len - 1) // bs])
        slot = seq_len % bs
        kc[:, page, :, slot, :] = k_new
        return page, ko.pool_block(ko.block_keys(kc, page, slot + 1), head_w)
    o.append_token = append_token


def m_hier_grid_is_mean_of_pages(o):
    def hier_reps(vb_logical, chunk_pages=64, grid_chunks=8):
        chunks = ko.coarse_means(vb_logical, chunk_pages)
        return chunks, ko.coarse_means(vb_logical, chunk_pages * grid_chunks)
    o.hier_reps = hier_reps


def m_hier_no_mask(o):
    def hier_select(vb_logical, va, K, chunk_pages=64, grid_chunks=8, permille=(500, 200, 100)):
        vb_logical = ko.decode(vb_logical)
        nb = vb_logical.shape[0]
        chunks, grids = o.hier_reps(vb_logical, chunk_pages, grid_chunks)
        gk = ko._keep(ko.affinity(grids, va), np.arange(len(grids)), permille[0])
        n_active_c = sum(1 for c in range(len(chunks)) if c // grid_chunks in set(gk.tolist()))
        ck = ko._keep(ko.affinity(chunks, va), np.arange(len(chunks)), permille[1] * n_active_c / max(1, len(chunks)))
        pk = ko._keep(ko.affinity(vb_logical, va), np.arange(nb), permille[2])
        s = ko.affinity(vb_logical, va)
        idx = np.full(K, -1, dtype=np.int64)
        val = np.full(K, -np.inf)
        m = min(K, len(pk))
        idx[:m], val[:m] = pk[:m], s[pk[:m]]
        return idx, val, len(pk), np.sort(gk), np.sort(ck)
    o.hier_select = hier_select


def m_hier_rates_of_all_members(o):
    def hier_select(vb_logical, va, K, chunk_pages=64, grid_chunks=8, permille=(500, 200, 100)):
        vb_logical = ko.decode(vb_logical)
        nb = vb_logical.shape[0]
        chunks, grids = o.hier_reps(vb_logical, chunk_pages, grid_chunks)
        gk = ko._keep(ko.affinity(grids, va), np.arange(len(grids)), permille[0])
        ca = np.array([c for c in range(len(chunks)) if c // grid_chunks in set(gk.tolist())], dtype=np.int64)
        k = -(-len(chunks) * permille[1] // 1000)
        order = np.lexsort((ca, -ko.affinity(chunks, va)[ca]))
        ck = ca[order[:k]]
        pa = np.array([j for j in range(nb) if j // chunk_pages in set(ck.tolist())], dtype=np.int64)
        k = -(-nb * permille[2] // 1000)
        s = ko.affinity(vb_logical, va)
        order = np.lexsort((pa, -s[pa]))
        pk = pa[order[:k]]
        idx = np.full(K, -1, dtype=np.int64)
        val = np.full(K, -np.inf)
        m = min(K, len(pk))
        idx[:m], val[:m] = pk[:m], s[pk[:m]]
        return idx, val, len(pk), np.sort(gk), np.sort(ck)
    o.hier_select = hier_select


def _hier_pool_variant(o, coarse_mask=True, page_mask=True, share_of_active=True):
    """The shared-pool hierarchy with one of its rules changed."""
    def hier_select_pool(A, grids, chunks, V, mask_words, K, chunk_pages=64, grid_chunks=8,
                         permille=(500, 200, 100)):
        A, grids, chunks, V = (np.atleast_2d(ko.decode(x)) for x in (A, grids, chunks, V))
        R, N, C, G = A.shape[0], V.shape[0], chunks.shape[0], grids.shape[0]
        mw = np.asarray(mask_words, dtype=np.uint32)
        idx = np.full((R, K), -1, dtype=np.int64)
        val = np.full((R, K), -np.inf)
        kept = np.zeros(R, dtype=np.int64)

        def keep(scores, members, pool, q):
            members = np.asarray(members, dtype=np.int64)
            k = -(-(len(members) if share_of_active else pool) * int(q) // 1000)
            order = np.lexsort((members, -np.asarray(scores)[members]))
            return members[order[:k]]

        for r in range(R):
            j = np.arange(N)
            allowed = ((mw[r, j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)
            c_ok = np.zeros(C, bool)
            c_ok[j[allowed] // chunk_pages] = True
            g_ok = np.zeros(G, bool)
            g_ok[np.arange(C)[c_ok] // grid_chunks] = True
            if not coarse_mask:
                c_ok[:] = True
                g_ok[:] = True
            s_g, s_c, s_p = ko.affinity(grids, A[r]), ko.affinity(chunks, A[r]), ko.affinity(V, A[r])
            gk = set(keep(s_g, np.nonzero(g_ok)[0], G, permille[0]).tolist())
            ca = [c for c in range(C) if c_ok[c] and c // grid_chunks in gk]
            ck = set(keep(s_c, ca, int(c_ok.sum()), permille[1]).tolist())
            pa = [b for b in range(N) if (allowed[b] or not page_mask) and b // chunk_pages in ck]
            pk = keep(s_p, pa, int(allowed.sum()), permille[2])
            m = min(K, len(pk))
            idx[r, :m] = pk[:m]
            val[r, :m] = s_p[pk[:m]]
            kept[r] = len(pk)
        return idx, val, kept
    o.hier_select_pool = hier_select_pool


def m_hier_pool_coarse_ignores_mask(o):
    _hier_pool_variant(o, coarse_mask=False)


def m_hier_pool_blocks_ignore_mask(o):
    _hier_pool_variant(o, page_mask=False)


def m_hier_pool_share_of_allowed(o):
    _hier_pool_variant(o, share_of_active=False)


MUTANTS = [
    m_decode_shift_15, m_decode_reads_fp16, m_decode_drops_sign,
    m_pool_divides_by_heads_only, m_pool_weights_transposed, m_pool_sum_not_mean,
    m_affinity_not_halved, m_affinity_raw_dot, m_affinity_zero_vector_scores_zero,
    m_topk_ties_to_higher_index, m_topk_ascending, m_anchor_first_tokens,
    m_anchor_ignores_block_table, m_variance_one_mean_for_all_dims, m_variance_std_not_var,
    m_coarse_last_group_divided_by_group, m_batched_ignores_mask, m_stability_counts_equal_theta,
    m_stability_divides_by_steps_seen, m_stability_window_one_too_long, m_stable_topk_ignores_stability,
    m_compact_table_keeps_topk_order, m_append_token_divides_by_block_size, m_append_token_slot_off_by_one,
    m_hier_grid_is_mean_of_pages, m_hier_no_mask, m_hier_rates_of_all_members,
    m_hier_pool_coarse_ignores_mask, m_hier_pool_blocks_ignore_mask, m_hier_pool_share_of_allowed,
]


def _bind(o):
    """Re-bind the oracle's composite functions to the mutated namespace."""
    def pool_blocks(kc, pages, n_valid, head_w=None, w_set=None):
        L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
        out = np.zeros((len(pages), D))
        for i, (p, n) in enumerate(zip(pages, n_valid)):
            w = None if head_w is None else np.asarray(head_w, float).reshape(-1, L * H)[w_set[i]]
            out[i] = o.pool_block(ko.block_keys(kc, int(p), int(n)), w)
        return out

    def score_topk(vb_table, pages_r, va, K):
        s = o.affinity(np.asarray(vb_table)[np.asarray(pages_r, dtype=np.int64)], va)
        idx, val = o.topk(s, K)
        return s, idx, val

    o.pool_blocks = pool_blocks
    o.score_topk = score_topk
    return o


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    o = _copy()
    mutant(o)
    _bind(o)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"no pin catches {mutant.__name__}"
