// C ABI of the selector (include/kk.h): argument checks on the host, then
// launches. Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/kk.h"

#include "kk_device.cuh"
#include "kk_internal.h"

namespace {

__device__ int g_kk_error = 0;  // first device-side error since the last kk_device_error()

// Device address of g_kk_error for the current device (looked up once per device).
int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::mutex mu;
  static int* ptr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kk_error) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int*>(p);
  }
  return ptr[dev];
}

kk_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KK_OK : KK_ERR_CUDA; }

// Limit of every bounded wait, and the one-shot request to leave a pool copy
// out (failure-detection tests), both set by the diagnostic calls below.
std::atomic<unsigned long long> g_wait_ns{kk::kDefaultWaitNs};
std::atomic<long long> g_skip_box{-1};

bool dim_supported(int dtype, int D) {
  if (D != 32 && D != 64 && D != 128 && D != 256) return false;
  return !(dtype == KK_F32 && D == 256);
}

kk_status check_kcache(const kk_kcache_desc* kc, kk::KCache* out) {
  if (!kc || !kc->base) return KK_ERR_INVALID;
  if (kc->dtype != KK_F32 && kc->dtype != KK_BF16) return KK_ERR_INVALID;
  if (kc->num_layers <= 0 || kc->num_kv_heads <= 0 || kc->head_dim <= 0 || kc->block_size <= 0 ||
      kc->num_pages <= 0)
    return KK_ERR_INVALID;
  if ((long long)kc->num_layers * kc->num_kv_heads > kk::kMaxLH) return KK_ERR_UNSUPPORTED;
  if (!dim_supported(kc->dtype, kc->head_dim)) return KK_ERR_UNSUPPORTED;
  const long long es = kc->dtype == KK_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(kc->base) % 16) return KK_ERR_UNSUPPORTED;
  const int64_t st[4] = {kc->stride_layer, kc->stride_page, kc->stride_head, kc->stride_token};
  for (int i = 0; i < 4; ++i)
    if (st[i] < 0 || (st[i] * es) % 16) return KK_ERR_UNSUPPORTED;
  *out = kk::KCache{kc->base,       kc->dtype,          kc->num_layers,  kc->num_kv_heads,
                    kc->head_dim,   kc->block_size,     kc->num_pages,   kc->stride_layer,
                    kc->stride_page, kc->stride_head,   kc->stride_token};
  return KK_OK;
}

kk_status check_table(const kk_block_table* bt, bool need_seq, kk::Table* out) {
  if (!bt || bt->num_requests < 0 || bt->num_requests > 65535 || bt->max_blocks < 0)
    return KK_ERR_INVALID;
  if (bt->num_requests > 0 && (!bt->offsets || !bt->pages || (need_seq && !bt->seq_lens)))
    return KK_ERR_INVALID;
  *out = kk::Table{bt->pages, bt->offsets, bt->seq_lens, bt->num_requests, bt->max_blocks};
  return KK_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct VarWorkspace {
  float* S;
  float* Q;
  double* var;
};

size_t var_workspace_bytes(int LH, int D, long long total_blocks, int R) {
  return align256(sizeof(float) * (size_t)total_blocks * LH * D) +
         align256(sizeof(float) * (size_t)total_blocks * LH) + align256(sizeof(double) * (size_t)R * LH);
}

VarWorkspace carve(void* ws, int LH, int D, long long total_blocks) {
  char* p = static_cast<char*>(ws);
  VarWorkspace w;
  w.S = reinterpret_cast<float*>(p);
  p += align256(sizeof(float) * (size_t)total_blocks * LH * D);
  w.Q = reinterpret_cast<float*>(p);
  p += align256(sizeof(float) * (size_t)total_blocks * LH);
  w.var = reinterpret_cast<double*>(p);
  return w;
}

}  // namespace

extern "C" {

kk_status kk_debug_set_wait_limit(uint64_t ns) {
  g_wait_ns = ns ? (unsigned long long)ns : kk::kDefaultWaitNs;
  return KK_OK;
}

kk_status kk_debug_skip_pool_copy(int64_t box) {
  if (box < -1) return KK_ERR_INVALID;
  g_skip_box = (long long)box;
  return KK_OK;
}

const char* kk_status_str(kk_status s) {
  switch (s) {
    case KK_OK: return "ok";
    case KK_ERR_INVALID: return "invalid argument";
    case KK_ERR_UNSUPPORTED: return "unsupported layout or size";
    case KK_ERR_CUDA: return "CUDA error";
    case KK_ERR_BAD_INDEX: return "index out of range in device data";
    case KK_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

kk_status kk_device_error(cudaStream_t stream, int32_t* code) {
  if (!code) return KK_ERR_INVALID;
  if (!error_word()) return KK_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_kk_error, sizeof(int)) != cudaSuccess) return KK_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_kk_error, &zero, sizeof(int)) != cudaSuccess) return KK_ERR_CUDA;
  *code = v;
  return KK_OK;
}

kk_status kk_pool_blocks(const kk_kcache_desc* kc, const int32_t* pages, const int32_t* n_valid,
                         int32_t n, const float* head_w, int32_t n_sets, const int32_t* w_set,
                         float* vb, cudaStream_t stream) {
  kk::KCache c;
  kk_status st = check_kcache(kc, &c);
  if (st != KK_OK) return st;
  if (n < 0) return KK_ERR_INVALID;
  if (n == 0) return KK_OK;
  if (!pages || !n_valid || !vb) return KK_ERR_INVALID;
  if (head_w && (!w_set || n_sets <= 0)) return KK_ERR_INVALID;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_pool_direct(c, pages, n_valid, n, head_w, n_sets, w_set, vb, err, stream));
}

size_t kk_head_variance_workspace_bytes(const kk_kcache_desc* kc, int32_t total_blocks,
                                        int32_t num_requests) {
  if (!kc || total_blocks < 0 || num_requests < 0) return 0;
  return var_workspace_bytes(kc->num_layers * kc->num_kv_heads, kc->head_dim, total_blocks,
                             num_requests);
}

static kk_status variance_common(const kk_kcache_desc* kc, const kk_block_table* bt,
                                 int32_t total_blocks, float* head_w_out, float* vb, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  kk::KCache c;
  kk::Table t;
  kk_status st = check_kcache(kc, &c);
  if (st != KK_OK) return st;
  if ((st = check_table(bt, true, &t)) != KK_OK) return st;
  if (total_blocks < 0 || !head_w_out) return KK_ERR_INVALID;
  if (t.R == 0) return KK_OK;
  const int LH = c.L * c.H;
  if (!ws || ws_bytes < var_workspace_bytes(LH, c.D, total_blocks, t.R)) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return KK_ERR_UNSUPPORTED;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  VarWorkspace w = carve(ws, LH, c.D, total_blocks);
  cudaError_t e = kk::launch_pool_slices(c, t, total_blocks, w.S, w.Q, err, stream);
  if (e == cudaSuccess) e = kk::launch_head_var(c, t, total_blocks, w.S, w.Q, w.var, err, stream);
  if (e == cudaSuccess) e = kk::launch_finalize_weights(c, t, total_blocks, w.var, head_w_out, stream);
  if (e == cudaSuccess && vb) e = kk::launch_combine(c, t, total_blocks, w.S, head_w_out, vb, err, stream);
  return from_cuda(e);
}

kk_status kk_head_variance(const kk_kcache_desc* kc, const kk_block_table* bt,
                           int32_t total_blocks, float* head_w_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  return variance_common(kc, bt, total_blocks, head_w_out, nullptr, workspace, workspace_bytes,
                         stream);
}

kk_status kk_pool_blocks_weighted(const kk_kcache_desc* kc, const kk_block_table* bt,
                                  int32_t total_blocks, float* head_w_out, float* vb,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!vb) return KK_ERR_INVALID;
  return variance_common(kc, bt, total_blocks, head_w_out, vb, workspace, workspace_bytes, stream);
}

// Decode-step options: the anchor ring (select steps only) and the split
// workspace.
static kk_status step_options(const kk_step_options* opt, bool allow_ring, kk::StepParams* p) {
  if (!opt) return KK_OK;
  if ((opt->k_new == nullptr) != (opt->block_sum == nullptr)) return KK_ERR_INVALID;
  if (opt->k_new) {
    // the fused write side: select steps with an anchor ring only
    if (!allow_ring || !opt->ring) return KK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(opt->k_new) % 16) return KK_ERR_UNSUPPORTED;
    if (p->kc.dtype != 1 && p->kc.D > 128) return KK_ERR_UNSUPPORTED;  // as kk_append_tokens
    p->k_new = opt->k_new;
    p->block_sum = opt->block_sum;
  }
  if (opt->sel_pages) {
    if (!p->bt.pages) return KK_ERR_INVALID;  // kk_topk has no block table
    p->sel_pages = opt->sel_pages;
    p->sel_logical = opt->sel_logical;
    p->sel_count = opt->sel_count;
  }
  if (opt->ring) {
    const kk_anchor_ring* g = opt->ring;
    if (!allow_ring || !g->rows || !g->pos || g->slots < 1 || g->slots > kk::kMaxW || p->W > g->slots)
      return KK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(g->rows) % 16 || reinterpret_cast<uintptr_t>(g->pos) % 4)
      return KK_ERR_UNSUPPORTED;
    p->ring_rows = g->rows;
    p->ring_pos = g->pos;
    p->ring_slots = g->slots;
  }
  if (opt->workspace) {
    const size_t need = kk::step_workspace_bytes(p->bt.R, p->bt.max_blocks, p->K);
    if (opt->workspace_bytes < need) return KK_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(opt->workspace) % 16) return KK_ERR_UNSUPPORTED;
    const int cap = kk::step_split_cap(p->bt.max_blocks, p->K);
    if (need > 0 && cap >= 2) {
      char* w = static_cast<char*>(opt->workspace);
      p->split_ctr = reinterpret_cast<unsigned long long*>(w);
      p->split_keys = reinterpret_cast<uint64_t*>(w + (((size_t)p->bt.R * sizeof(unsigned long long) + 255) &
                                                        ~size_t(255)));
      p->split_cap = cap;
    }
  }
  return KK_OK;
}

static kk_status step_common(kk::StepParams& p, cudaStream_t stream) {
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  p.err = err;
  return from_cuda(kk::launch_step(p, stream));
}

kk_status kk_anchor(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                    const float* head_w, float* va, cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = check_kcache(kc, &p.kc);
  if (st != KK_OK) return st;
  if ((st = check_table(bt, true, &p.bt)) != KK_OK) return st;
  if (W < 1 || W > kk::kMaxW || !va) return KK_ERR_INVALID;
  p.W = W;
  p.head_w = head_w;
  p.va_out = va;
  p.D = p.kc.D;
  p.flags = kk::kStepAnchor;
  return step_common(p, stream);
}

static kk_status score_args(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                            const float* va, kk::StepParams* p) {
  kk_status st = check_table(bt, false, &p->bt);
  if (st != KK_OK) return st;
  if (!vb || !va || num_pages <= 0) return KK_ERR_INVALID;
  if (!dim_supported(KK_BF16, D)) return KK_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(vb) % 16) return KK_ERR_UNSUPPORTED;
  p->vb = vb;
  p->vb_rows = num_pages;
  p->D = D;
  p->va_in = va;
  return KK_OK;
}

kk_status kk_score(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                   const float* va, float* scores, cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = score_args(vb, D, num_pages, bt, va, &p);
  if (st != KK_OK) return st;
  if (!scores) return KK_ERR_INVALID;
  p.scores_out = scores;
  p.flags = kk::kStepScore;
  return step_common(p, stream);
}

size_t kk_select_step_workspace_bytes(int32_t R, int32_t max_blocks, int32_t K) {
  if (R < 0 || max_blocks < 0 || K < 1 || K > kk::kMaxK) return 0;
  return kk::step_workspace_bytes(R, max_blocks, K);
}

kk_status kk_topk(const float* scores, const int32_t* offsets, int32_t R, int32_t max_n, int32_t K,
                  int32_t* idx, float* top_scores, const kk_step_options* opt, cudaStream_t stream) {
  if (R < 0 || R > 65535 || max_n < 0 || K < 1 || K > kk::kMaxK) return KK_ERR_INVALID;
  if (R == 0) return KK_OK;
  if (!scores || !offsets || !idx) return KK_ERR_INVALID;
  kk::StepParams p = {};
  p.bt = kk::Table{nullptr, offsets, nullptr, R, max_n};
  p.D = 128;
  p.scores_in = scores;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top_scores;
  p.flags = kk::kStepTopK | kk::kStepTopKFromScores;
  kk_status st = step_options(opt, false, &p);
  if (st != KK_OK) return st;
  return step_common(p, stream);
}

kk_status kk_score_topk(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                        const float* va, int32_t K, int32_t* idx, float* top_scores, float* scores,
                        const kk_step_options* opt, cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = score_args(vb, D, num_pages, bt, va, &p);
  if (st != KK_OK) return st;
  if (K < 1 || K > kk::kMaxK || !idx) return KK_ERR_INVALID;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top_scores;
  p.scores_out = scores;
  p.flags = kk::kStepScore | kk::kStepTopK;
  if ((st = step_options(opt, false, &p)) != KK_OK) return st;
  return step_common(p, stream);
}

kk_status kk_select_step(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                         const float* head_w, const float* vb, int32_t K, float* va, int32_t* idx,
                         float* top_scores, float* scores, const kk_step_options* opt, cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = check_kcache(kc, &p.kc);
  if (st != KK_OK) return st;
  if ((st = check_table(bt, true, &p.bt)) != KK_OK) return st;
  if (W < 1 || W > kk::kMaxW || K < 1 || K > kk::kMaxK || !vb || !idx) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(vb) % 16) return KK_ERR_UNSUPPORTED;
  p.W = W;
  p.head_w = head_w;
  p.va_out = va;
  p.vb = vb;
  p.vb_rows = p.kc.num_pages;
  p.D = p.kc.D;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top_scores;
  p.scores_out = scores;
  p.flags = kk::kStepAnchor | kk::kStepScore | kk::kStepTopK;
  if ((st = step_options(opt, true, &p)) != KK_OK) return st;
  return step_common(p, stream);
}

// Stability-filter arguments shared by the two *_stable entry points.
static kk_status stability_args(int32_t stab_window, float theta, uint32_t* hist, float* stab,
                                kk::StepParams* p) {
  if (stab_window < 1 || stab_window > 32 || !hist || !std::isfinite(theta)) return KK_ERR_INVALID;
  if (p->bt.max_blocks > (int32_t)kk::kStabIdxMask - 1) return KK_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(hist) % 4 || reinterpret_cast<uintptr_t>(stab) % 4) return KK_ERR_INVALID;
  p->hist = hist;
  p->stab_out = stab;
  p->stab_w = stab_window;
  p->stab_theta = theta;
  return KK_OK;
}

kk_status kk_score_topk_stable(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                               const float* va, int32_t K, int32_t stab_window, float theta,
                               uint32_t* hist, float* stab, int32_t* idx, float* top_scores, float* scores,
                               const kk_step_options* opt, cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = score_args(vb, D, num_pages, bt, va, &p);
  if (st != KK_OK) return st;
  if (K < 1 || K > kk::kMaxK || !idx) return KK_ERR_INVALID;
  if ((st = stability_args(stab_window, theta, hist, stab, &p)) != KK_OK) return st;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top_scores;
  p.scores_out = scores;
  p.flags = kk::kStepScore | kk::kStepTopK;
  if ((st = step_options(opt, false, &p)) != KK_OK) return st;
  return step_common(p, stream);
}

kk_status kk_select_step_stable(const kk_kcache_desc* kc, const kk_block_table* bt, int32_t W,
                                const float* head_w, const float* vb, int32_t K, int32_t stab_window,
                                float theta, uint32_t* hist, float* stab, float* va, int32_t* idx,
                                float* top_scores, float* scores, const kk_step_options* opt,
                                cudaStream_t stream) {
  kk::StepParams p = {};
  kk_status st = check_kcache(kc, &p.kc);
  if (st != KK_OK) return st;
  if ((st = check_table(bt, true, &p.bt)) != KK_OK) return st;
  if (W < 1 || W > kk::kMaxW || K < 1 || K > kk::kMaxK || !vb || !idx) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(vb) % 16) return KK_ERR_UNSUPPORTED;
  if ((st = stability_args(stab_window, theta, hist, stab, &p)) != KK_OK) return st;
  p.W = W;
  p.head_w = head_w;
  p.va_out = va;
  p.vb = vb;
  p.vb_rows = p.kc.num_pages;
  p.D = p.kc.D;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top_scores;
  p.scores_out = scores;
  p.flags = kk::kStepAnchor | kk::kStepScore | kk::kStepTopK;
  if ((st = step_options(opt, true, &p)) != KK_OK) return st;
  return step_common(p, stream);
}

kk_status kk_compact_table(const int32_t* idx, int32_t K, const kk_block_table* bt, int32_t* sel_pages,
                           int32_t* sel_logical, int32_t* sel_count, cudaStream_t stream) {
  kk::Table t;
  kk_status st = check_table(bt, false, &t);
  if (st != KK_OK) return st;
  if (K < 1 || K > kk::kMaxK || (t.R > 0 && (!idx || !sel_pages))) return KK_ERR_INVALID;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_compact_table(idx, K, t, sel_pages, sel_logical, sel_count, err, stream));
}

// The anchor ring's pointers and size, checked on the host.
static kk_status ring_args(const kk_anchor_ring* ring, kk::Ring* out) {
  if (!ring || !ring->rows || !ring->pos || ring->slots < 1 || ring->slots > kk::kMaxW) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(ring->rows) % 16 || reinterpret_cast<uintptr_t>(ring->pos) % 4)
    return KK_ERR_UNSUPPORTED;
  *out = kk::Ring{ring->rows, ring->pos, ring->slots};
  return KK_OK;
}

kk_status kk_append_tokens(const kk_kcache_desc* kc, const kk_block_table* bt, const void* k_new,
                           const float* head_w, float* block_sum, float* vb, const kk_anchor_ring* ring,
                           cudaStream_t stream) {
  kk::KCache c;
  kk_status st = check_kcache(kc, &c);
  if (st != KK_OK) return st;
  kk::Table t;
  if ((st = check_table(bt, true, &t)) != KK_OK) return st;
  if (t.R > 0 && (!k_new || !block_sum || !vb)) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(k_new) % 16) return KK_ERR_UNSUPPORTED;
  kk::Ring g = {};
  if (ring && (st = ring_args(ring, &g)) != KK_OK) return st;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_append(c, t, k_new, head_w, block_sum, vb, ring ? &g : nullptr, err, stream));
}

kk_status kk_anchor_ring_fill(const kk_kcache_desc* kc, const kk_block_table* bt, const float* head_w,
                              const kk_anchor_ring* ring, cudaStream_t stream) {
  kk::KCache c;
  kk_status st = check_kcache(kc, &c);
  if (st != KK_OK) return st;
  kk::Table t;
  if ((st = check_table(bt, true, &t)) != KK_OK) return st;
  kk::Ring g;
  if ((st = ring_args(ring, &g)) != KK_OK) return st;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_ring_fill(c, t, head_w, g, err, stream));
}

// Sizes of the hierarchical levels for a table whose longest request has
// max_blocks blocks, and whether the worst case fits the step kernel's
// hierarchical mode (Grids and active Chunks held in shared memory at once,
// kept Chunks listed per request).
static bool hier_dims(int32_t max_blocks, int32_t D, int32_t chunk_pages, int32_t grid_chunks,
                      const int32_t* permille, int* c_max, int* g_max) {
  const long long C = ((long long)max_blocks + chunk_pages - 1) / chunk_pages;
  const long long G = (C + grid_chunks - 1) / grid_chunks;
  *c_max = (int)C;
  *g_max = (int)G;
  const long long kg = (G * permille[0] + 999) / 1000;
  const long long ac = std::min(C, kg * grid_chunks);
  const long long kc = (ac * permille[1] + 999) / 1000;
  const long long cap = kk::step_hier_level_cap(D);
  return G <= cap && ac <= cap && kc <= kk::kHierKeptChunks && C < (1ll << 31);
}

kk_status kk_hier_reps(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                       int32_t chunk_pages, int32_t grid_chunks, float* chunk_reps, float* grid_reps,
                       cudaStream_t stream) {
  kk::Table t;
  kk_status st = check_table(bt, false, &t);
  if (st != KK_OK) return st;
  if (!vb || !chunk_reps || !grid_reps || chunk_pages < 1 || grid_chunks < 1 || num_pages <= 0)
    return KK_ERR_INVALID;
  if (!dim_supported(KK_BF16, D) || reinterpret_cast<uintptr_t>(vb) % 16) return KK_ERR_UNSUPPORTED;
  const long long C = ((long long)t.max_blocks + chunk_pages - 1) / chunk_pages;
  const long long G = (C + grid_chunks - 1) / grid_chunks;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  cudaError_t e = kk::launch_coarse(vb, D, num_pages, t, chunk_pages, chunk_reps, err, stream);
  if (e == cudaSuccess)
    e = kk::launch_grid_reps(chunk_reps, D, (int)C, (int)G, t, chunk_pages, grid_chunks, grid_reps, stream);
  return from_cuda(e);
}

kk_status kk_hier_select(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                         const float* chunk_reps, const float* grid_reps, const float* va, int32_t chunk_pages,
                         int32_t grid_chunks, int32_t permille_grid, int32_t permille_chunk, int32_t permille_page,
                         int32_t K, int32_t* idx, float* top_scores, int32_t* kept, const kk_step_options* opt,
                         cudaStream_t stream) {
  kk::Table t;
  kk_status st = check_table(bt, false, &t);
  if (st != KK_OK) return st;
  const int32_t pm[3] = {permille_grid, permille_chunk, permille_page};
  if (!vb || !chunk_reps || !grid_reps || !va || !idx || chunk_pages < 1 || grid_chunks < 1 || num_pages <= 0 ||
      K < 1 || K > kk::kMaxK)
    return KK_ERR_INVALID;
  for (int32_t q : pm)
    if (q < 1 || q > 1000) return KK_ERR_INVALID;
  if (!dim_supported(KK_BF16, D)) return KK_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(vb) % 16 || reinterpret_cast<uintptr_t>(chunk_reps) % 16 ||
      reinterpret_cast<uintptr_t>(grid_reps) % 16)
    return KK_ERR_UNSUPPORTED;
  int c_max = 0, g_max = 0;
  if (!hier_dims(t.max_blocks, D, chunk_pages, grid_chunks, pm, &c_max, &g_max)) return KK_ERR_UNSUPPORTED;
  kk::StepParams sp = {};  // only the split workspace is taken from the options
  sp.bt = t;
  sp.K = K;
  if ((st = step_options(opt, false, &sp)) != KK_OK) return st;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_hier_select(vb, D, num_pages, t, chunk_reps, grid_reps, c_max, g_max, va,
                                          chunk_pages, grid_chunks, pm, K, idx, top_scores, kept, sp.split_ctr,
                                          sp.split_keys, sp.split_cap, err, stream));
}

size_t kk_score_pool_batched_workspace_bytes(int32_t R, int32_t N, int32_t K) {
  (void)K;
  if (R < 0 || N < 0) return 0;
  return kk::batched_workspace_bytes(R, N, N);
}

kk_status kk_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask,
                                int32_t R, int32_t N, int32_t D, int32_t K, int32_t* idx,
                                float* top_scores, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  if (R < 0 || N < 0 || K < 1 || K > kk::kMaxK) return KK_ERR_INVALID;
  if (R == 0) return KK_OK;
  if (D != 128) return KK_ERR_UNSUPPORTED;
  if (!idx || !workspace || (N > 0 && (!A || !V || !mask))) return KK_ERR_INVALID;
  if (workspace_bytes < kk::batched_workspace_bytes(R, N, N)) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(V) % 16 ||
      reinterpret_cast<uintptr_t>(workspace) % 256)
    return KK_ERR_UNSUPPORTED;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_score_pool_batched(A, V, mask, R, N, K, idx, top_scores, workspace,
                                                 err, stream));
}

static bool hier_pool_dims(int32_t N, int32_t chunk_pages, int32_t grid_chunks) {
  if (N < 0 || chunk_pages < 1 || grid_chunks < 1) return false;
  const long long C = N > 0 ? ((long long)N + chunk_pages - 1) / chunk_pages : 0;
  const long long G = C > 0 ? (C + grid_chunks - 1) / grid_chunks : 0;
  return G + C <= kk::kHierPoolCoarseMax;
}

int32_t kk_hier_pool_coarse_rows(int32_t N, int32_t chunk_pages, int32_t grid_chunks) {
  if (!hier_pool_dims(N, chunk_pages, grid_chunks)) return -1;
  return kk::hier_pool_coarse_rows(N, chunk_pages, grid_chunks);
}

kk_status kk_hier_pool_reps(uint16_t* M, int32_t N, int32_t D, int32_t chunk_pages, int32_t grid_chunks,
                            cudaStream_t stream) {
  if (N < 0 || chunk_pages < 1 || grid_chunks < 1) return KK_ERR_INVALID;
  if (D != 128 || !hier_pool_dims(N, chunk_pages, grid_chunks)) return KK_ERR_UNSUPPORTED;
  if (N == 0) return KK_OK;
  if (!M) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(M) % 16) return KK_ERR_UNSUPPORTED;
  return from_cuda(kk::launch_hier_pool_reps(M, N, chunk_pages, grid_chunks, stream));
}

size_t kk_hier_select_pool_workspace_bytes(int32_t R, int32_t N, int32_t chunk_pages, int32_t grid_chunks) {
  if (R < 0 || !hier_pool_dims(N, chunk_pages, grid_chunks)) return 0;
  return kk::hier_pool_workspace_bytes(R, N, chunk_pages, grid_chunks);
}

kk_status kk_hier_select_pool(const uint16_t* A, const uint16_t* M, const uint32_t* mask, int32_t R, int32_t N,
                              int32_t D, int32_t chunk_pages, int32_t grid_chunks, int32_t permille_grid,
                              int32_t permille_chunk, int32_t permille_page, int32_t K, int32_t* idx,
                              float* top_scores, int32_t* kept, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  const int32_t permille[3] = {permille_grid, permille_chunk, permille_page};
  if (R < 0 || N < 0 || K < 1 || K > kk::kMaxK || chunk_pages < 1 || grid_chunks < 1) return KK_ERR_INVALID;
  for (int32_t q : permille)
    if (q < 1 || q > 1000) return KK_ERR_INVALID;
  if (R == 0) return KK_OK;
  if (D != 128 || !hier_pool_dims(N, chunk_pages, grid_chunks)) return KK_ERR_UNSUPPORTED;
  if (!idx || !workspace || (N > 0 && (!A || !M || !mask))) return KK_ERR_INVALID;
  if (workspace_bytes < kk_hier_select_pool_workspace_bytes(R, N, chunk_pages, grid_chunks)) return KK_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(M) % 16 ||
      reinterpret_cast<uintptr_t>(workspace) % 256)
    return KK_ERR_UNSUPPORTED;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_hier_select_pool(A, M, mask, R, N, chunk_pages, grid_chunks, permille, K, idx,
                                               top_scores, kept, workspace, err, stream));
}

kk_status kk_coarse_means(const float* vb, int32_t D, int32_t num_pages, const kk_block_table* bt,
                          int32_t group, float* out, cudaStream_t stream) {
  kk::Table t;
  kk_status st = check_table(bt, false, &t);
  if (st != KK_OK) return st;
  if (!vb || !out || group < 1 || num_pages <= 0) return KK_ERR_INVALID;
  if (!dim_supported(KK_BF16, D) || reinterpret_cast<uintptr_t>(vb) % 16) return KK_ERR_UNSUPPORTED;
  int* err = error_word();
  if (!err) return KK_ERR_CUDA;
  return from_cuda(kk::launch_coarse(vb, D, num_pages, t, group, out, err, stream));
}

}  // extern "C"

// Internal helpers for the allocation-free weighted pool (kk_static.cu): the
// same argument checks as kk_pool_blocks_weighted, and the device error word.
namespace kk {

kk_status check_weighted_args(const kk_kcache_desc* kc, const kk_block_table* bt,
                              int32_t total_blocks, const float* head_w_out, const float* vb,
                              KCache* c, Table* t) {
  kk_status st = check_kcache(kc, c);
  if (st != KK_OK) return st;
  if ((st = check_table(bt, true, t)) != KK_OK) return st;
  if (total_blocks < 0 || !head_w_out || !vb) return KK_ERR_INVALID;
  return KK_OK;
}

int* device_error_word() { return error_word(); }

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }

long long take_skip_box() { return g_skip_box.exchange(-1); }

}  // namespace kk
