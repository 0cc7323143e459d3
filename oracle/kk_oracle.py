"""fp64 CPU oracle for Key-Key Semantic Affinity block scoring.

TEST INFRASTRUCTURE. This module is the slow, plain statement of what the
hot path computes. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The library's own code path
never calls it, and it shares no code with the CUDA sources.

Source: the page "Key-Key Semantic Affinity: 用 Key 向量替代注意力分数的 KV
Cache 重要性评估" (cited below as [KK §n]):

* [KK §2.2 step 1], [KK §5.2 step 2-3]: a block's representation v_b is the
  mean of its Key vectors over all tokens of the block, all KV heads and all
  layers; it is computed once, when the block is written.
* [KK §2.2 step 2], [KK §5.2 step 1]: the query anchor v_anchor is the mean of
  the Keys of the most recent W_local tokens.
* [KK §2.2 step 3], [KK §3.2]: the affinity of a block is the similarity of
  v_b and v_anchor, normalised. The formula itself is lost from the page; the
  reading used here is score = (1 + cos(v_b, v_anchor)) / 2, so orthogonal
  vectors score 0.5, identical directions 1 and opposite directions 0.
* [KK §5.2 step 4], [KK §5.1]: the K blocks with the highest affinity are
  selected.
* [KK §3.3 finding 2], [KK §6.1]: optional weighting of each head by its
  variance.  Read here as the Key variance of each (layer, KV head):
  the mean over d of the population variance over the request's tokens,
  normalised so the weights sum to one.
* [KK §5.1]: a coarse (Grid / Chunk) representation is the mean of its
  children's representations.
* [KK §5.2 step 4]: only the selected blocks are loaded for attention. The
  compact table lists the physical pages of the selected blocks in logical
  order (the order a paged-attention kernel walks them), -1 padded.
* [KK §5.2 step 2], [KK §2.2 step 1]: v_b is computed when the block is
  written. Maintained incrementally, after each appended token the block's
  v_b equals the pooled mean of the tokens it holds so far.
* [KK §5.1]: hierarchical selection Grid -> Chunk -> Page. Readings used
  here: a Chunk is 64 consecutive pages and a Grid 8 consecutive Chunks of a
  request (the page fixes neither); a Chunk's representation is the mean of
  its pages' v_b and a Grid's the mean of its Chunks' representations; every
  level is scored with the same affinity; a level keeps ceil(rate * n) of
  its n active members (rates 50 %, 20 %, 10 %: of the active children, which
  gives the page's 1 % of the cache), the children of unselected parents are
  excluded (their scores "set to zero" on the page, read as masked out), and
  ties go to the lower index.
* [KK §5.3]: the stability score of a block is the fraction of the last W
  decode steps (W = 20 by default) in which its affinity exceeded the
  threshold theta (0.5 by default); the page's example: one step at 0.9 and
  nineteen at 0.2 give 1/20 = 0.05, twenty steps above 0.6 give 1.0. Reading
  used here: "exceeded" is strict (a score equal to theta does not count),
  the fraction is always over W (before W steps exist the missing steps count
  as not high), and the loading decision ranks blocks by stability, then by
  the current affinity, then by the lower index.
* [KK §5.1], the three levels in one product: the representations of all
  levels are rows of one matrix scored against the anchors at once, and
  boolean parent -> child masks do the filtering. Reading used here for a
  pool shared by many anchors (the batched scorer's pool): Chunks are
  consecutive pool ids and Grids consecutive Chunks, with the pool's own
  coarse representations (the same for every anchor); for one anchor a
  coarse member is active only if it covers at least one block the anchor's
  mask allows (below the Grid level also only if its parent was kept), and a
  block is active if the mask allows it and its Chunk was kept. With a mask
  that allows exactly one request's blocks, in order and starting on a Grid
  boundary, this is the per-request hierarchy above.

Every function accumulates in float64. bf16 inputs are decoded exactly
(bits << 16). Parity of the variance weighting and of the (1+cos)/2 formula
with the published method is unpinned (the page does not print either);
everything else here is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "decode",
    "block_keys",
    "pool_block",
    "pool_blocks",
    "head_variance_weights",
    "anchor",
    "affinity",
    "topk",
    "score_topk",
    "score_pool_batched",
    "coarse_means",
    "stability",
    "stable_topk",
    "compact_table",
    "append_token",
    "hier_reps",
    "hier_select",
    "hier_select_pool",
]


def decode(x) -> np.ndarray:
    """Return ``x`` as float64. uint16 arrays are bf16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def block_keys(kc, page: int, n: int) -> np.ndarray:
    """Keys of the first ``n`` tokens of physical page ``page``.

    ``kc`` is the paged K cache viewed as [L][P][H][bs][D] (any strides).
    Returns float64 [L][H][n][D].
    """
    return decode(kc[:, page, :, :n, :])


def _weights(L: int, H: int, head_w) -> np.ndarray:
    """Per-(layer, head) weights: uniform 1/(L*H) unless given [KK §5.2 step 3]."""
    if head_w is None:
        return np.full((L, H), 1.0 / (L * H))
    return np.asarray(head_w, dtype=np.float64).reshape(L, H)


def pool_block(keys: np.ndarray, head_w=None) -> np.ndarray:
    """v_b of one block [KK §2.2 step 1], [KK §5.2 step 3].

    keys: float64 [L][H][n][D]. Each (layer, head) contributes the mean of its
    n token Keys; those means are combined with weights w[l,h] (uniform
    1/(L*H) when ``head_w`` is None, which is the plain mean over tokens,
    heads and layers). A block with no valid token pools to the zero vector.
    """
    L, H, n, D = keys.shape
    if n == 0:
        return np.zeros(D)
    token_mean = keys.sum(axis=2) / n  # [L][H][D]
    w = _weights(L, H, head_w)
    return np.einsum("lh,lhd->d", w, token_mean)


def pool_blocks(kc, pages, n_valid, head_w=None, w_set=None) -> np.ndarray:
    """v_b rows for a list of physical pages; row i belongs to pages[i].

    head_w: None, or [n_sets][L*H] weights; w_set[i] picks the set for row i.
    """
    L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
    out = np.zeros((len(pages), D))
    for i, (p, n) in enumerate(zip(pages, n_valid)):
        w = None
        if head_w is not None:
            w = np.asarray(head_w, dtype=np.float64).reshape(-1, L * H)[w_set[i]]
        out[i] = pool_block(block_keys(kc, int(p), int(n)), w)
    return out


def request_tokens_of_layer(kc, layer: int, pages_r, seq_len: int, bs: int) -> np.ndarray:
    """float64 [H][T][D]: every Key of one layer of one request, in token order."""
    pages_r = np.asarray(pages_r, dtype=np.int64)
    nb = len(pages_r)
    if nb == 0 or seq_len == 0:
        return np.zeros((kc.shape[2], 0, kc.shape[4]))
    k = decode(kc[layer, pages_r])  # [nb][H][bs][D]
    k = np.transpose(k, (1, 0, 2, 3)).reshape(k.shape[1], nb * bs, k.shape[3])
    return k[:, :seq_len, :]


def head_variance_weights(kc, pages_r, seq_len: int, bs: int) -> np.ndarray:
    """Head-variance weights of one request [KK §3.3 finding 2], [KK §6.1].

    For each (layer, KV head): mu_d = mean over the request's T tokens of K_d;
    Var = (1/D) * sum_d (1/T) * sum_t (K_d - mu_d)^2 (two passes, float64).
    Weights are Var / sum(Var) over all (layer, head), returned as [L*H];
    when every Var is 0 (no tokens, or constant Keys) the weights are uniform.
    """
    L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
    var = np.zeros((L, H))
    for layer in range(L):
        k = request_tokens_of_layer(kc, layer, pages_r, seq_len, bs)  # [H][T][D]
        if k.shape[1]:
            mu = k.mean(axis=1, keepdims=True)
            var[layer] = ((k - mu) ** 2).mean(axis=1).mean(axis=1)
    if var.sum() == 0:
        return np.full(L * H, 1.0 / (L * H))
    return (var / var.sum()).reshape(L * H)


def anchor(kc, pages_r, seq_len: int, bs: int, W: int, head_w=None) -> np.ndarray:
    """v_anchor of one request [KK §2.2 step 2], [KK §5.2 step 1].

    The mean of the Keys of the last min(W, T) tokens, taken per (layer, head)
    over those tokens and combined with the same per-(layer, head) weights as
    the block pooling. The tokens are read from the paged cache through the
    request's block table. A request with no token gives the zero vector.
    """
    L, H, D = kc.shape[0], kc.shape[2], kc.shape[4]
    w_eff = min(W, seq_len)
    if w_eff == 0:
        return np.zeros(D)
    rows = np.stack(
        [decode(kc[:, int(pages_r[p // bs]), :, p % bs, :]) for p in range(seq_len - w_eff, seq_len)]
    )  # [W][L][H][D]
    token_mean = rows.mean(axis=0)  # [L][H][D]
    w = _weights(L, H, head_w)
    return np.einsum("lh,lhd->d", w, token_mean)


def affinity(vb: np.ndarray, va: np.ndarray) -> np.ndarray:
    """score = (1 + cos(v_b, v_anchor)) / 2 per row of ``vb`` [KK §2.2 step 3], [KK §3.2].

    cos is taken as 0 when either vector is zero, so such a block scores 0.5.
    """
    vb = np.atleast_2d(decode(vb))
    va = decode(va)
    dot = vb @ va
    nb = np.sqrt((vb * vb).sum(axis=1))
    na = np.sqrt((va * va).sum())
    denom = nb * na
    cos = np.where(denom > 0, dot / np.where(denom > 0, denom, 1.0), 0.0)
    return (1.0 + cos) / 2.0


def topk(scores, K: int):
    """The K highest scores [KK §5.2 step 4]: order by score descending, ties
    to the lower index. Slots beyond the number of candidates hold -1 / -inf.

    Returns (idx int64 [K], score float64 [K]).
    """
    s = np.asarray(scores, dtype=np.float64)
    order = np.lexsort((np.arange(len(s)), -s))[:K]
    idx = np.full(K, -1, dtype=np.int64)
    val = np.full(K, -np.inf)
    idx[: len(order)] = order
    val[: len(order)] = s[order]
    return idx, val


def score_topk(vb_table, pages_r, va, K: int):
    """Affinity of every block in a request's table, then its top-K.

    vb_table is indexed by physical page; the returned indices are logical
    (positions in the request's block table).
    """
    s = affinity(np.asarray(vb_table)[np.asarray(pages_r, dtype=np.int64)], va)
    idx, val = topk(s, K)
    return s, idx, val


def score_pool_batched(A, V, mask_words, K: int):
    """Scores of R anchors against a shared pool of N block vectors, each
    anchor restricted to the blocks its mask marks, then top-K per anchor
    [KK §5.1] (all representations against the anchor in one product).

    A: [R][D], V: [N][D] (bf16 bits or floats); mask_words: uint32
    [R][ceil(N/32)], bit (j % 32) of word j // 32 marks block j.
    Returns (idx int64 [R][K] pool ids, score float64 [R][K]).
    """
    A = decode(A)
    V = decode(V)
    R, N = A.shape[0], V.shape[0]
    mw = np.asarray(mask_words, dtype=np.uint32)
    idx = np.full((R, K), -1, dtype=np.int64)
    val = np.full((R, K), -np.inf)
    for r in range(R):
        j = np.arange(N)
        owned = ((mw[r, j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)
        cand = j[owned]
        s = affinity(V[cand], A[r])
        i_loc, v = topk(s, K)
        keep = i_loc >= 0
        idx[r, keep] = cand[i_loc[keep]]
        val[r] = v
    return idx, val


def coarse_means(vb_logical, group: int) -> np.ndarray:
    """Coarse representations [KK §5.1]: the mean of ``group`` consecutive
    block representations; the last group averages whatever blocks remain.
    """
    vb_logical = decode(vb_logical)
    nb = vb_logical.shape[0]
    ng = (nb + group - 1) // group
    out = np.zeros((ng, vb_logical.shape[1]))
    for g in range(ng):
        out[g] = vb_logical[g * group : min((g + 1) * group, nb)].mean(axis=0)
    return out


def stability(score_history, W: int = 20, theta: float = 0.5) -> np.ndarray:
    """Stability score of every block [KK §5.3]: over the last W decode steps
    (``score_history`` oldest first, one score array per step), the number of
    steps whose affinity was strictly above ``theta``, divided by W.
    """
    hist = np.asarray(score_history, dtype=np.float64)
    if hist.ndim != 2:
        raise ValueError("score_history must be [steps][blocks]")
    recent = hist[max(0, hist.shape[0] - W):]
    return (recent > theta).sum(axis=0) / float(W)


def stable_topk(stab, scores, K: int):
    """The K blocks to load under the stability filter [KK §5.3]: order by
    stability descending, then by the current affinity descending, then by
    the lower index. Slots beyond the candidates hold -1 / -inf.

    Returns (idx int64 [K], current affinity float64 [K]).
    """
    stab = np.asarray(stab, dtype=np.float64)
    s = np.asarray(scores, dtype=np.float64)
    order = np.lexsort((np.arange(len(s)), -s, -stab))[:K]
    idx = np.full(K, -1, dtype=np.int64)
    val = np.full(K, -np.inf)
    idx[: len(order)] = order
    val[: len(order)] = s[order]
    return idx, val


def compact_table(pages_r, idx_r):
    """The selected blocks of one request as a table for attention
    [KK §5.2 step 4]: their logical indices in ascending order, the physical
    pages in that order, and their number. Entries of ``idx_r`` that are -1
    (empty top-K slots) are skipped; slots past the count hold -1.

    Returns (pages int64 [len(idx_r)], logical int64 [len(idx_r)], count).
    """
    pages_r = np.asarray(pages_r, dtype=np.int64)
    idx_r = np.asarray(idx_r, dtype=np.int64)
    chosen = np.sort(idx_r[idx_r >= 0])
    n = len(chosen)
    logical = np.full(len(idx_r), -1, dtype=np.int64)
    pages = np.full(len(idx_r), -1, dtype=np.int64)
    logical[:n] = chosen
    pages[:n] = pages_r[chosen]
    return pages, logical, n


def append_token(kc, pages_r, seq_len: int, bs: int, k_new, head_w=None):
    """Write one decode token's Keys into the paged cache and return the new
    v_b of the block that holds it [KK §5.2 step 2].

    kc: the cache view [L][P][H][bs][D] (float32 or bf16 bits), modified in
    place; seq_len: the request's length after the append (the token sits at
    position seq_len - 1); k_new: [L][H][D] in the cache's storage type.
    Returns (physical page, v_b float64 [D]): the pooled mean of the block's
    tokens so far, i.e. pool_block over its first (seq_len - 1) % bs + 1 tokens.
    """
    t = seq_len - 1
    page = int(np.asarray(pages_r)[t // bs])
    slot = t % bs
    kc[:, page, :, slot, :] = k_new
    return page, pool_block(block_keys(kc, page, slot + 1), head_w)


def hier_reps(vb_logical, chunk_pages: int = 64, grid_chunks: int = 8):
    """Chunk and Grid representations of one request [KK §5.1]: a Chunk is
    the mean of its pages' v_b, a Grid the mean of its Chunks'
    representations (the last of each may be partial).

    vb_logical: [nb][D] in logical order. Returns (chunks [C][D], grids [G][D]).
    """
    chunks = coarse_means(vb_logical, chunk_pages)
    grids = coarse_means(chunks, grid_chunks) if len(chunks) else np.zeros((0, chunks.shape[1]))
    return chunks, grids


def _keep(scores, members, permille: int):
    """The ceil(n * permille / 1000) members with the highest scores (ties:
    lower index); integer arithmetic, so the count is exact."""
    members = np.asarray(members, dtype=np.int64)
    n = len(members)
    k = -(-n * int(permille) // 1000)
    order = np.lexsort((members, -np.asarray(scores, dtype=np.float64)[members]))
    return members[order[:k]]


def hier_select(vb_logical, va, K: int, chunk_pages: int = 64, grid_chunks: int = 8,
                permille=(500, 200, 100)):
    """Hierarchical selection of one request's pages [KK §5.1]: score the
    Grids and keep the best share of them, then score only the Chunks of the
    kept Grids and keep the best share of those, then the pages of the kept
    Chunks likewise. The kept pages are returned in the order of kk_topk
    (score descending, ties to the lower index), the first K of them.

    Returns (idx int64 [K] logical pages, score float64 [K], number of pages
    the last level keeps, kept grids, kept chunks).
    """
    vb_logical = decode(vb_logical)
    nb = vb_logical.shape[0]
    chunks, grids = hier_reps(vb_logical, chunk_pages, grid_chunks)
    g_keep = _keep(affinity(grids, va) if len(grids) else [], np.arange(len(grids)), permille[0])
    c_active = np.array([c for c in range(len(chunks)) if c // grid_chunks in set(g_keep.tolist())],
                        dtype=np.int64)
    c_keep = _keep(affinity(chunks, va) if len(chunks) else [], c_active, permille[1])
    p_active = np.array([j for j in range(nb) if j // chunk_pages in set(c_keep.tolist())], dtype=np.int64)
    p_keep = _keep(affinity(vb_logical, va) if nb else [], p_active, permille[2])
    s = affinity(vb_logical, va) if nb else np.zeros(0)
    idx = np.full(K, -1, dtype=np.int64)
    val = np.full(K, -np.inf)
    m = min(K, len(p_keep))
    idx[:m] = p_keep[:m]
    val[:m] = s[p_keep[:m]]
    return idx, val, len(p_keep), np.sort(g_keep), np.sort(c_keep)


def hier_select_pool(A, grids, chunks, V, mask_words, K: int, chunk_pages: int = 64, grid_chunks: int = 8,
                     permille=(500, 200, 100)):
    """Hierarchical selection over a shared pool for R anchors [KK §5.1]:
    every Grid, Chunk and block representation is scored against every anchor
    (one product), then per anchor the levels are filtered top down. A level
    keeps ceil(n * permille / 1000) of its n active members (ties to the
    lower index). Active Grids: those covering an allowed block. Active
    Chunks: those of kept Grids covering an allowed block. Active blocks:
    allowed blocks of kept Chunks.

    A: [R][D] anchors; grids [G][D], chunks [C][D], V [N][D] (bf16 bits or
    floats), Chunk c = blocks [c*chunk_pages, (c+1)*chunk_pages) of the pool,
    Grid g = Chunks [g*grid_chunks, (g+1)*grid_chunks); mask_words uint32
    [R][ceil(N/32)], bit (j % 32) of word j // 32 allows block j.
    Returns (idx int64 [R][K] pool ids in kk_topk order, score float64
    [R][K], kept int64 [R] blocks the last level keeps).
    """
    A = decode(A)
    grids = np.atleast_2d(decode(grids))
    chunks = np.atleast_2d(decode(chunks))
    V = decode(V)
    R, N = A.shape[0], V.shape[0]
    C = -(-N // chunk_pages) if N else 0
    G = -(-C // grid_chunks) if C else 0
    assert chunks.shape[0] == C and grids.shape[0] == G
    mw = np.asarray(mask_words, dtype=np.uint32)
    idx = np.full((R, K), -1, dtype=np.int64)
    val = np.full((R, K), -np.inf)
    kept = np.zeros(R, dtype=np.int64)
    for r in range(R):
        j = np.arange(N)
        allowed = ((mw[r, j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool) if N else np.zeros(0, bool)
        chunk_allowed = np.zeros(C, dtype=bool)
        chunk_allowed[j[allowed] // chunk_pages] = True
        grid_allowed = np.zeros(G, dtype=bool)
        grid_allowed[np.arange(C)[chunk_allowed] // grid_chunks] = True
        s_g = affinity(grids, A[r]) if G else np.zeros(0)
        s_c = affinity(chunks, A[r]) if C else np.zeros(0)
        s_p = affinity(V, A[r]) if N else np.zeros(0)
        g_keep = set(_keep(s_g, np.arange(G)[grid_allowed], permille[0]).tolist())
        c_active = [c for c in range(C) if chunk_allowed[c] and c // grid_chunks in g_keep]
        c_keep = set(_keep(s_c, c_active, permille[1]).tolist())
        p_active = [b for b in range(N) if allowed[b] and b // chunk_pages in c_keep]
        p_keep = _keep(s_p, p_active, permille[2])
        m = min(K, len(p_keep))
        idx[r, :m] = p_keep[:m]
        val[r, :m] = s_p[p_keep[:m]]
        kept[r] = len(p_keep)
    return idx, val, kept
