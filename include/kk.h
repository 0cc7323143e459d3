/*
 * kk.h - C ABI of the Key-Key Semantic Affinity block selector (sm_103a).
 *
 * The method: the page "Key-Key Semantic Affinity: 用 Key 向量替代注意力分数的
 * KV Cache 重要性评估" (cited as [KK §n]). A paged K cache is summarised per
 * block by a mean-pooled Key vector v_b, written once ([KK §2.2 step 1],
 * [KK §5.2 step 2]); each decode step pools the last W tokens' Keys into
 * v_anchor ([KK §2.2 step 2], [KK §5.2 step 1]), scores every candidate block by
 * (1 + cos(v_b, v_anchor)) / 2 ([KK §2.2 step 3], [KK §3.2]; the page's own
 * formula was lost, this is the reading used) and keeps the top K blocks
 * ([KK §5.2 step 4]).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are device memory owned by the caller; nothing
 *    here allocates or frees memory. Scratch comes from a caller-provided
 *    workspace whose size a *_workspace_bytes() function reports.
 *  - Every call is asynchronous on `stream` and returns a kk_status. Argument
 *    errors found on the host are returned before anything is launched.
 *    Errors that depend on device data (a page id out of range, a block table
 *    whose length disagrees with seq_lens) are recorded in a device error
 *    word; the offending item is skipped and kk_device_error() reports the
 *    first such error. No kernel traps.
 *  - Key caches are bf16 or float32; pooled vectors, anchors and scores are
 *    float32, accumulated in float32.
 *  - The first call on a device looks up the device error word's address;
 *    make that first call outside CUDA stream capture.
 *  - The decode-step calls (kk_select_step, kk_score_topk, kk_topk and their
 *    stable forms) keep no state in the library: calls on different streams
 *    may run at once as long as they do not share a workspace (see
 *    kk_step_options).
 */
#ifndef KK_H_
#define KK_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kk_status {
  KK_OK = 0,
  KK_ERR_INVALID = 1,     /* bad argument (null pointer, negative size, K or W out of range) */
  KK_ERR_UNSUPPORTED = 2, /* valid but not handled: head_dim, alignment, strides */
  KK_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  KK_ERR_BAD_INDEX = 4,   /* (device) a page id, weight-set id or block table entry out of range */
  KK_ERR_TIMEOUT = 5      /* (device) a bounded wait gave up */
} kk_status;

typedef enum kk_dtype { KK_F32 = 0, KK_BF16 = 1 } kk_dtype;

/*
 * Paged K cache layout [KK §1] (fixed-size token blocks managed as pages).
 * Element (layer l, page p, head h, token t, dim d) is at
 *   base + l*stride_layer + p*stride_page + h*stride_head + t*stride_token + d
 * (strides in elements; the dim stride is 1). base and every stride times the
 * element size must be multiples of 16 bytes, else KK_ERR_UNSUPPORTED.
 * head_dim must be 32, 64, 128 or 256 (float32: 32, 64 or 128).
 */
typedef struct kk_kcache_desc {
  const void* base; /* device */
  int32_t dtype;    /* kk_dtype */
  int32_t num_layers;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_pages;
  int64_t stride_layer;
  int64_t stride_page;
  int64_t stride_head;
  int64_t stride_token;
} kk_kcache_desc;

/*
 * Per-request block tables, CSR style. Request r owns logical blocks
 * j = 0 .. nb_r-1 with nb_r = offsets[r+1] - offsets[r], which must equal
 * ceil(seq_lens[r] / block_size); its block j lives in physical page
 * pages[offsets[r] + j] and holds min(block_size, seq_lens[r] - j*block_size)
 * valid tokens. max_blocks (host value) bounds every nb_r.
 */
typedef struct kk_block_table {
  const int32_t* pages;    /* device [offsets[R]] */
  const int32_t* offsets;  /* device [R+1], non-decreasing, offsets[0] = 0 */
  const int32_t* seq_lens; /* device [R] */
  int32_t num_requests;    /* R */
  int32_t max_blocks;      /* host bound of nb_r */
} kk_block_table;

/*
 * Diagnostics for failure-detection tests (no part of the method). Every spin
 * of a kernel on an mbarrier is bounded: past the limit it records
 * KK_ERR_TIMEOUT in the device error word, waits (again bounded) for the
 * copies it has in flight, frees what it holds and returns, so the context
 * stays usable.
 * kk_debug_set_wait_limit: the limit, in ns, of every wait of the launches
 *   that follow (0 restores the default of 1 s). Launches already captured in
 *   a CUDA graph keep the limit they were captured with.
 * kk_debug_skip_pool_copy: the next launch of the persistent pool kernel
 *   (kk_pool_blocks on at least one block per SM) issues no copy for TMA box
 *   `box` of its first CTA (counted from 0 in that CTA's issue order), so the
 *   wait for that box runs out; -1 cancels. The request is used up by that
 *   launch. KK_ERR_INVALID for box < -1.
 */
kk_status kk_debug_set_wait_limit(uint64_t ns);
kk_status kk_debug_skip_pool_copy(int64_t box);

/* Name of a status code (static string). */
const char* kk_status_str(kk_status s);

/* Synchronises `stream`, returns the first device-side error recorded since
 * the last call in *code (KK_OK if none) and clears it. */
kk_status kk_device_error(cudaStream_t stream, int32_t* code);

/*
 * kk_pool_blocks - block representation v_b [KK §2.2 step 1], [KK §5.2 step 2-3].
 * For i < n, with p = pages[i] and m = n_valid[i] (0..block_size):
 *   vb[p][d] = sum_{l,h} w[l,h] * (1/m) * sum_{t<m} K[l,p,h,t,d]
 * where w = 1/(L*H) when head_w is NULL, else w = head_w[w_set[i]][l*H+h]
 * (head_w: device [n_sets][L*H]; w_set: device [n], values < n_sets).
 * m = 0 writes the zero vector. vb: device [num_pages][head_dim], rows not
 * named in `pages` are left untouched. Tokens t >= m are never read.
 */
kk_status kk_pool_blocks(const kk_kcache_desc* kc, const int32_t* pages, const int32_t* n_valid,
                         int32_t n, const float* head_w, int32_t n_sets, const int32_t* w_set,
                         float* vb, cudaStream_t stream);

/*
 * Head-variance weights [KK §3.3 finding 2], [KK §6.1]: for request r and
 * each (layer, head), Var = (1/D) sum_d (mean_t K^2 - (mean_t K)^2) over the
 * request's seq_lens[r] tokens, and head_w_out[r][l*H+h] = Var / sum Var
 * (uniform 1/(L*H) if every Var is 0). head_w_out: device [R][L*H].
 * Needs kk_head_variance_workspace_bytes() bytes of device workspace.
 * total_blocks must be offsets[R]; a request whose table reaches past it is
 * skipped (its weights and blocks are not written) and reported through the
 * device error word, as is a block with a page id out of range (its Keys
 * count as zero in the request's variance).
 */
size_t kk_head_variance_workspace_bytes(const kk_kcache_desc* kc, int32_t total_blocks,
                                        int32_t num_requests);
kk_status kk_head_variance(const kk_kcache_desc* kc, const kk_block_table* bt,
                           int32_t total_blocks, float* head_w_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Weighted pooling of every block of every request in one pass over K:
 * the head-variance weights of each request (as kk_head_variance, written to
 * head_w_out [R][L*H]) and vb[pages[offsets[r]+j]] pooled with them (as
 * kk_pool_blocks). total_blocks = offsets[R]. Same workspace size as
 * kk_head_variance.
 */
kk_status kk_pool_blocks_weighted(const kk_kcache_desc* kc, const kk_block_table* bt,
                                  int32_t total_blocks, float* head_w_out, float* vb,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Allocation-free form of kk_pool_blocks_weighted (the page describes no such
 * variant; it exists for callers). Some callers cannot call cudaMalloc: a
 * serving engine that reserves nearly all device memory for its paged KV cache
 * at start-up and hands none out afterwards, or a plugin running inside such
 * an engine's write path, where an allocation would fail or stall the device.
 * This entry point takes only the inputs and outputs of
 * kk_pool_blocks_weighted and keeps its scratch in a 32 MiB array that the
 * library owns on each GPU that loads it (held until the process exits).
 * - The scratch needed is kk_head_variance_workspace_bytes(kc, total_blocks,
 *   R); above 32 MiB the call returns KK_ERR_UNSUPPORTED and launches nothing.
 * - It allocates nothing: no cudaMalloc or cudaFree, no allocating library
 *   call. The first call on a device looks up the array's device address (and
 *   the error word's) and keeps it for the life of the process; make that
 *   first call before any stream capture, and do not reset the device
 *   (cudaDeviceReset) after it: the kept address would then be stale.
 * - Every call shares the one array. Calls that overlap on the GPU (on two
 *   streams, or from two threads) race on it and give wrong results; order
 *   them on one stream. Nothing needs clearing between calls: each call
 *   writes every scratch byte before reading it (a block whose page id is out
 *   of range has its sums written as zero, and the call reports
 *   KK_ERR_BAD_INDEX). A table that reaches past total_blocks is reported and
 *   its requests are skipped; the kernels never index past the array.
 * Results are the same as kk_pool_blocks_weighted's.
 */
kk_status kk_pool_blocks_weighted_static(const kk_kcache_desc* kc, const kk_block_table* bt,
                                         int32_t total_blocks, float* head_w_out, float* vb,
                                         cudaStream_t stream);

/*
 * kk_anchor - query anchor [KK §2.2 step 2], [KK §5.2 step 1]:
 *   va[r][d] = sum_{l,h} w[l,h] * (1/W') * sum_{T-W' <= p < T} K[l, page(p), h, p % bs, d]
 * with T = seq_lens[r], W' = min(W, T), page(p) = pages[offsets[r] + p / bs],
 * w uniform 1/(L*H) or head_w[r][l*H+h] (device [R][L*H]). T = 0 gives the
 * zero vector. 1 <= W <= 1024. va: device [R][head_dim].
 */
kk_status kk_anchor(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                    const float* head_w, float* va, cudaStream_t stream);

/*
 * kk_score - affinity [KK §2.2 step 3], [KK §3.2], [KK §5.2 step 3]:
 *   scores[offsets[r]+j] = (1 + cos(vb[pages[offsets[r]+j]], va[r])) / 2
 * cos = 0 when either vector is zero. vb: device [num_pages][D] float32
 * (num_pages bounds the page ids), va: device [R][D], scores: device
 * [offsets[R]]. D in {32, 64, 128, 256}.
 */
kk_status kk_score(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                   const float* va, float* scores, cudaStream_t stream);

/*
 * Anchor ring: the per-token pooled Keys of each request's most recent
 * tokens, kept as the tokens are written, so that a decode step forms
 * v_anchor from W rows of head_dim floats instead of re-reading W tokens'
 * Keys of every layer and head from the cache. The anchor is a mean over
 * tokens of a weighted sum over (layer, head) [KK §5.2 step 1], so it can
 * be summed token by token:
 *   rows[r][t % slots][d] = sum_{l,h} w[l,h] * K[l, page(t), h, t % bs, d]
 *   pos[r][t % slots]     = t      (-1: the slot holds no token)
 * with w = head_w[r][l*H+h] when the ring is written with head weights, else
 * 1. kk_anchor_ring_fill writes it from the cache (for example after a
 * prefill); kk_append_tokens keeps it current token by token. A ring written
 * with head weights must be read with the same head weights.
 * rows: device float [R][slots][head_dim], 16-byte aligned (else
 * KK_ERR_UNSUPPORTED); pos: device int32 [R][slots]; 1 <= slots <= 1024. The
 * ring belongs to the caller.
 */
typedef struct kk_anchor_ring {
  float* rows;
  int32_t* pos;
  int32_t slots;
} kk_anchor_ring;

/*
 * Writes the anchor ring of every request from the K cache: for request r
 * with T = seq_lens[r], the tokens t in [T - min(slots, T), T) (slot
 * t % slots), and pos = -1 in every other slot. head_w: nullable device
 * [R][L*H] (the weights the ring carries).
 */
kk_status kk_anchor_ring_fill(const kk_kcache_desc* kc, const kk_block_table* bt, const float* head_w,
                              const kk_anchor_ring* ring, cudaStream_t stream);

/*
 * Options of the decode-step calls (the whole struct may be NULL):
 *  - ring (kk_select_step and kk_select_step_stable only; nullable): take
 *    v_anchor from this ring instead of from the K cache:
 *      va[r] = (1/W') * sum_{T-W' <= t < T} rows[r][t % slots]   (/ (L*H) when head_w is NULL)
 *    The result is kk_anchor's, summed in another order. W <= slots. A slot
 *    whose pos is not the token expected there counts as zero and is
 *    reported through the device error word (KK_ERR_BAD_INDEX).
 *  - workspace, workspace_bytes (nullable): device memory, 16-byte aligned,
 *    of at least kk_select_step_workspace_bytes(R, max_blocks, K) bytes. With
 *    it, a few very long requests are each split over several clusters of
 *    CTAs (more SMs per request); the clusters of a request meet at a counter
 *    in the workspace, which the last of them sets back to zero. Zero the
 *    workspace once before its first use (cudaMemsetAsync), and again after a
 *    call that did not run to completion (a CUDA error); a counter found past
 *    its bound is reported as KK_ERR_BAD_INDEX. Without a workspace, every
 *    request is served by one cluster. Calls that may run at once need
 *    separate workspaces.
 *  - k_new, block_sum (kk_select_step and kk_select_step_stable only, with a
 *    ring; nullable together): the decode token of every request is first
 *    written as kk_append_tokens(kc, bt, k_new, head_w, block_sum, vb, ring)
 *    would write it (cache slot, running sum, v_b, ring slot), in the same
 *    launch, and the step then selects on the updated v_b and ring; vb is
 *    written, with the same bits as the two calls write. The page that
 *    receives a request's token must be in no other request's table (that
 *    request would read its v_b row while it is written). k_new: device,
 *    16-byte aligned, [R][L][H][D] of the cache's element type; fp32 caches
 *    with D = 256 are not supported (KK_ERR_UNSUPPORTED).
 *  - sel_pages, sel_logical, sel_count (not kk_topk; sel_pages nullable, the
 *    other two nullable): the step also writes the table of the selected
 *    blocks as kk_compact_table(idx, K, bt, ...) would, in the same launch.
 */
typedef struct kk_step_options {
  const kk_anchor_ring* ring;
  void* workspace;
  size_t workspace_bytes;
  const void* k_new;
  float* block_sum;
  int32_t* sel_pages;
  int32_t* sel_logical;
  int32_t* sel_count;
} kk_step_options;

/* Workspace bytes that let the decode-step calls split long requests (0:
 * tables of at most max_blocks blocks per request are never split). */
size_t kk_select_step_workspace_bytes(int32_t R, int32_t max_blocks, int32_t K);

/*
 * kk_topk - top-K selection [KK §5.2 step 4]. For each request r, among
 * scores[offsets[r] .. offsets[r+1]) the K largest, ordered by score
 * descending, equal scores by lower index. idx[r][k] is the logical index
 * (position within the request's range), top_scores[r][k] (nullable) its
 * score; slots past the request's count hold -1 and -inf.
 * offsets: device [R+1]; max_n bounds every range; 1 <= K <= 256.
 */
kk_status kk_topk(const float* scores, const int32_t* offsets, int32_t R, int32_t max_n, int32_t K,
                  int32_t* idx, float* top_scores, const kk_step_options* opt, cudaStream_t stream);

/* kk_score followed by kk_topk in one launch; `scores` (nullable) receives
 * the full score vector as kk_score would. */
kk_status kk_score_topk(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                        const float* va, int32_t K, int32_t* idx, float* top_scores, float* scores,
                        const kk_step_options* opt, cudaStream_t stream);

/*
 * One decode step of the selector in one launch: kk_anchor, kk_score and
 * kk_topk [KK §5.2 steps 1-4]. vb: device [num_pages][head_dim] (the
 * table kk_pool_blocks wrote). va, scores and top_scores are nullable outputs.
 */
kk_status kk_select_step(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                         const float* head_w, const float* vb, int32_t K, float* va, int32_t* idx,
                         float* top_scores, float* scores, const kk_step_options* opt, cudaStream_t stream);

/*
 * Stability filter [KK §5.3] fused into scoring: kk_score_topk and
 * kk_select_step that also keep, per block, the last stab_window (1..32)
 * steps' "score > theta" bits and rank the top K by their count (the
 * block's stability is count / stab_window), then by the current score,
 * then by the lower index.
 * hist: device uint32 [offsets[R]], one word per logical block of the
 *   table, caller-owned state that persists across steps: bit 0 is the
 *   newest step. A block with no history starts at 0 (append a 0 word when
 *   a request's table grows). Updated in place by every call.
 * stab: nullable device float [offsets[R]]: count / stab_window after this
 *   step's update.
 * top_scores hold the current step's scores of the selected blocks.
 * Requires max_blocks < 2^27 - 1 (KK_ERR_UNSUPPORTED otherwise); theta
 * must be finite. Other arguments as in kk_score_topk / kk_select_step.
 */
kk_status kk_score_topk_stable(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                               const float* va, int32_t K, int32_t stab_window, float theta,
                               uint32_t* hist, float* stab, int32_t* idx, float* top_scores, float* scores,
                               const kk_step_options* opt, cudaStream_t stream);
kk_status kk_select_step_stable(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                                const float* head_w, const float* vb, int32_t K, int32_t stab_window,
                                float theta, uint32_t* hist, float* stab, float* va, int32_t* idx,
                                float* top_scores, float* scores, const kk_step_options* opt,
                                cudaStream_t stream);

/*
 * The selected blocks as a table for the attention kernel [KK §5.2 step 4]
 * (only they are loaded): for request r, the valid entries of
 * idx[r][0..K) (logical block indices as kk_topk writes them; -1 slots are
 * skipped) sorted ascending, their physical pages
 *   sel_pages[r][i] = pages[offsets[r] + logical_i]      (device int32 [R][K])
 * and optionally the logical indices sel_logical[r][i] (device int32 [R][K])
 * and their number sel_count[r] (device int32 [R]); slots past the count
 * are -1. An index outside [-1, nb_r) is skipped and reported through the
 * device error word. 1 <= K <= 256.
 */
kk_status kk_compact_table(const int32_t* idx, int32_t K, const kk_block_table* bt, int32_t* sel_pages,
                           int32_t* sel_logical, int32_t* sel_count, cudaStream_t stream);

/*
 * Incremental write-path pooling [KK §5.2 step 2] (v_b computed as the
 * block is written), fused with the write of the Keys: for every request r,
 * the decode token at position seq_lens[r] - 1 (seq_lens counts it; the
 * table already holds its block) has its Keys k_new[r] (device, the cache's
 * element type, [R][L][H][D], 16-byte aligned) written into slot
 * (seq_lens[r] - 1) % block_size of its page in the cache at kc->base
 * (which this call writes), and
 *   block_sum[p][d] = sum over the block's tokens so far and (l, h) of
 *                     w_lh * K[l][p][h][t][d]   (restarted at slot 0)
 *   vb[p][d]        = block_sum[p][d] / n_p      (/ (L*H) when head_w is NULL)
 * with w = head_w[r] (device float [R][L*H]) or 1. block_sum: device float
 * [num_pages][D], caller-owned state carried from token to token; vb: the
 * v_b table of kk_pool_blocks. A request whose table disagrees with seq_lens
 * or holds a bad page is skipped and reported through the device error word.
 * Blocks must not be shared between the requests of one call. ring
 * (nullable): the token's pooled Keys also go to its anchor ring slot
 * ((seq_lens[r] - 1) % slots, with its position), weighted as block_sum is.
 */
kk_status kk_append_tokens(const kk_kcache_desc* kc, const kk_block_table* bt, const void* k_new,
                           const float* head_w, float* block_sum, float* vb, const kk_anchor_ring* ring,
                           cudaStream_t stream);

/*
 * Hierarchical selection Grid -> Chunk -> Page [KK §5.1]. A Chunk is
 * chunk_pages consecutive blocks of a request's table and a Grid grid_chunks
 * consecutive Chunks (the page names the levels but not their sizes; 64 and
 * 8 are the usual choice).
 *
 * kk_hier_reps builds the two coarse levels from the v_b table (device float
 * [num_pages][D], as kk_pool_blocks writes it):
 *   chunk_reps[r][c] = mean of vb[pages[offsets[r] + j]], j in Chunk c
 *                      (device float [R][C_max][D], C_max = ceil(max_blocks / chunk_pages))
 *   grid_reps[r][g]  = mean of chunk_reps[r][c], c in Grid g
 *                      (device float [R][G_max][D], G_max = ceil(C_max / grid_chunks))
 * Levels past a request's end are zero. Call it when blocks change (write
 * time). vb must be 16-byte aligned (else KK_ERR_UNSUPPORTED).
 *
 * kk_hier_select scores the levels against the anchor va (device float
 * [R][D]) with the affinity of kk_score and keeps, level by level,
 * ceil(n * permille / 1000) of its n active members (permille in 1..1000;
 * 500 / 200 / 100 keep 1 % of the blocks), where only the Chunks of kept
 * Grids and the blocks of kept Chunks are active (ties to the lower index).
 * The kept blocks of request r are written to idx[r][0..K) in kk_topk order
 * (logical indices, -1 / -inf padding; at most K of them: the best min(K,
 * kept) blocks of the block level) and their number to kept[r] (nullable,
 * device int32 [R]; may exceed K). 1 <= K <= 256. Returns
 * KK_ERR_UNSUPPORTED when the Grid level, or the Chunks of the kept Grids, of
 * the table's longest request could hold more than 32 * D members, or more
 * than 2048 Chunks could be kept. D in {32, 64, 128, 256}; vb, chunk_reps and
 * grid_reps 16-byte aligned. opt (nullable): the workspace of
 * kk_step_options lets the blocks of a few very long requests' kept Chunks be
 * scored by several clusters (no ring: the anchor is given).
 */
kk_status kk_hier_reps(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                       int32_t chunk_pages, int32_t grid_chunks, float* chunk_reps, float* grid_reps,
                       cudaStream_t stream);
kk_status kk_hier_select(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                         const float* chunk_reps, const float* grid_reps, const float* va, int32_t chunk_pages,
                         int32_t grid_chunks, int32_t permille_grid, int32_t permille_chunk, int32_t permille_page,
                         int32_t K, int32_t* idx, float* top_scores, int32_t* kept, const kk_step_options* opt,
                         cudaStream_t stream);

/*
 * Shared-pool scoring [KK §5.1] (every representation against the anchors
 * in one matrix product, then a mask): R anchors A (device bf16 bits [R][D])
 * against N pooled block vectors V (device bf16 bits [N][D]); anchor r may
 * only pick blocks j whose bit (j % 32) of mask[r][j / 32] is set (device
 * uint32 [R][ceil(N/32)]). Scores are (1 + cos)/2 from float32 dot products
 * of the bf16 values; per anchor the top K pool ids (ordered as kk_topk) go
 * to idx [R][K] and top_scores [R][K] (nullable). D = 128, 1 <= K <= 256.
 * workspace: caller-owned device memory, 256-byte aligned, of at least
 * kk_score_pool_batched_workspace_bytes(R, N, K) bytes (8 * R * N bytes of
 * candidate keys plus R * (ceil(N/128) + 1) int32 offsets). Concurrent calls
 * need separate workspaces.
 */
size_t kk_score_pool_batched_workspace_bytes(int32_t R, int32_t N, int32_t K);
kk_status kk_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask,
                                int32_t R, int32_t N, int32_t D, int32_t K, int32_t* idx,
                                float* top_scores, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * Hierarchical selection over the shared pool [KK §5.1]: the representations
 * of all three levels are rows of one matrix, scored against every anchor in
 * one product, and parent -> child masks filter the levels. A Chunk is
 * chunk_pages consecutive pool blocks (C = ceil(N / chunk_pages)), a Grid
 * grid_chunks consecutive Chunks (G = ceil(C / grid_chunks)).
 *
 * M: device bf16 bits [H + N][128], H = kk_hier_pool_coarse_rows(N,
 * chunk_pages, grid_chunks) (G + C rounded up to a multiple of 128): rows
 * [0, G) the Grids, [G, G + C) the Chunks, [G + C, H) zero, [H, H + N) the
 * pool's blocks (the V of kk_score_pool_batched, which the caller writes).
 *
 * kk_hier_pool_reps writes rows [0, H) of M from its block rows: a Chunk's
 * row is the mean of its blocks' rows, a Grid's the mean of its Chunks' (the
 * last of each may be partial), summed in float32 and rounded once to bf16.
 * Call it whenever the pool's blocks change.
 *
 * kk_hier_select_pool scores A (device bf16 bits [R][128]) against all H + N
 * rows in one tcgen05 pass (float32 dot products of the bf16 values, (1 +
 * cos)/2), then for each anchor keeps, level by level, ceil(n * permille /
 * 1000) of the level's n active members (ties to the lower index), where a
 * Grid is active if it covers a block the anchor's mask allows (mask as in
 * kk_score_pool_batched), a Chunk if it covers an allowed block and its Grid
 * was kept, and a block if it is allowed and its Chunk was kept. The kept
 * blocks go to idx [R][K] (pool ids, kk_topk order, -1 / -inf padding, at
 * most K) and top_scores (nullable); their number to kept [R] (nullable; may
 * exceed K). 1 <= K <= 256, permille in 1..1000, D = 128, G + C <= 4096.
 * workspace: device memory, 256-byte aligned, of at least
 * kk_hier_select_pool_workspace_bytes(R, N, chunk_pages, grid_chunks) bytes
 * (the flat call's plus 4 * R * H for the coarse scores); concurrent calls
 * need separate workspaces. Returns KK_ERR_UNSUPPORTED beyond the limits above.
 */
int32_t kk_hier_pool_coarse_rows(int32_t N, int32_t chunk_pages, int32_t grid_chunks);
kk_status kk_hier_pool_reps(uint16_t* M, int32_t N, int32_t D, int32_t chunk_pages, int32_t grid_chunks,
                            cudaStream_t stream);
size_t kk_hier_select_pool_workspace_bytes(int32_t R, int32_t N, int32_t chunk_pages, int32_t grid_chunks);
kk_status kk_hier_select_pool(const uint16_t* A, const uint16_t* M, const uint32_t* mask, int32_t R, int32_t N,
                              int32_t D, int32_t chunk_pages, int32_t grid_chunks, int32_t permille_grid,
                              int32_t permille_chunk, int32_t permille_page, int32_t K, int32_t* idx,
                              float* top_scores, int32_t* kept, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * Coarse representations [KK §5.1] (a coarser level's representation is the
 * mean of its children's): for request r and group g,
 *   out[r][g][d] = mean over j in [g*group, min((g+1)*group, nb_r)) of vb[pages[offsets[r]+j]][d]
 * out: device [R][ceil(max_blocks/group)][D]; groups past a request's last
 * block are written as zero. D in {32, 64, 128, 256}, group >= 1; vb
 * 16-byte aligned (else KK_ERR_UNSUPPORTED).
 */
kk_status kk_coarse_means(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                          int32_t group, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KK_H_ */
