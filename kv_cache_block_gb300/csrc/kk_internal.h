// Host-side launch interface between the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kk {

constexpr int kMaxLH = 1024;       // layers * KV heads
constexpr int kMaxW = 1024;        // anchor tokens
constexpr int kMaxK = 256;         // top-K
constexpr int kMaxCluster = 16;    // CTAs per request in the step kernel
constexpr int kMergeSlots = 2048;  // cluster size * K

enum ErrorCode { kErrBadIndex = 4, kErrTimeout = 5 };

// Stability-ranked keys keep a block index in 27 bits (see make_stab_key).
constexpr int kStabIdxBits = 27;
constexpr uint32_t kStabIdxMask = (1u << kStabIdxBits) - 1u;

struct KCache {
  const void* base;
  int dtype;  // 0 f32, 1 bf16
  int L, H, D, bs, num_pages;
  long long sL, sP, sH, sT;  // element strides
};

struct Table {
  const int* pages;
  const int* offsets;
  const int* seq_lens;
  int R, max_blocks;
};

// kk_pool.cu
cudaError_t launch_pool_direct(const KCache& kc, const int* pages, const int* n_valid, int n,
                               const float* head_w, int n_sets, const int* w_set, float* vb,
                               int* err, cudaStream_t s);
cudaError_t launch_pool_slices(const KCache& kc, const Table& bt, long long total_blocks, float* S, float* Q,
                               int* err, cudaStream_t s);
// total_blocks: rows of the S / Q scratch; a request whose table reaches
// past it is skipped and reported (the kernels never index past the scratch)
cudaError_t launch_head_var(const KCache& kc, const Table& bt, long long total_blocks, const float* S,
                            const float* Q, double* var, int* err, cudaStream_t s);
cudaError_t launch_finalize_weights(const KCache& kc, const Table& bt, long long total_blocks, const double* var,
                                    float* head_w_out, cudaStream_t s);
cudaError_t launch_combine(const KCache& kc, const Table& bt, long long total_blocks, const float* S,
                           const float* head_w, float* vb, int* err, cudaStream_t s);

// kk_step.cu
enum StepFlags {
  kStepAnchor = 1,           // pool the anchor from the K cache
  kStepScore = 2,            // score blocks against the anchor
  kStepTopK = 4,             // select the top K
  kStepTopKFromScores = 8,   // keys come from a score array
};

struct StepParams {
  KCache kc;
  Table bt;
  int W;
  const float* head_w;  // [R][L*H] or null
  const float* va_in;   // [R][D] or null
  float* va_out;        // [R][D] or null
  const float* vb;      // [vb_rows][D]
  int vb_rows;
  int D;
  const float* scores_in;  // [offsets[R]] (top-K only mode)
  float* scores_out;       // [offsets[R]] or null
  int K;
  int* idx_out;      // [R][K]
  float* top_out;    // [R][K] or null
  int flags;
  // stability filter (nullable): per logical block, the last stab_w steps'
  // "score > stab_theta" bits (newest in bit 0); ranks by their count first
  uint32_t* hist;
  float* stab_out;
  int stab_w;
  float stab_theta;
  // anchor ring (nullable rows): the anchor is the mean of the W' newest
  // rows[r][t % ring_slots], checked against pos
  const float* ring_rows;
  const int* ring_pos;
  int ring_slots;
  // split scratch (nullable): per-request counters of the clusters done
  // (zero between calls) and each cluster's sorted list, split_cap lists a
  // request
  unsigned long long* split_ctr;
  uint64_t* split_keys;
  int split_cap;
  // fused write side (nullable k_new): the decode token of every request is
  // appended (kk_append_tokens, with head_w and the ring) before the step;
  // fused compact table (nullable sel_pages): kk_compact_table of the output
  const void* k_new;
  float* block_sum;
  int* sel_pages;
  int* sel_logical;
  int* sel_count;
  // hierarchical selection (nullable hier_grid): the Grid and Chunk levels
  // pick the Chunks whose blocks are scored; kept[r] (nullable) receives the
  // number of blocks the block level keeps, and at most that many are output
  const float* hier_grid;   // [R][g_max][D]
  const float* hier_chunk;  // [R][c_max][D]
  int g_max, c_max, chunk_pages, grid_chunks;
  int permille[3];
  int* kept;
  unsigned long long wait_ns;  // limit of every bounded wait
  int* err;
  int splits;  // clusters per request (set by the launcher; > 1 for very long requests)
};
cudaError_t launch_step(const StepParams& p, cudaStream_t s);
// launch_step's instantiations with the decode token's append fused in (k_new)
cudaError_t launch_step_fused(const StepParams& p, cudaStream_t s);
// Lists a request may be split into (a power of two), and the workspace that
// holds them for R requests of at most max_blocks blocks (0: never split).
int step_split_cap(int max_blocks, int K);
size_t step_workspace_bytes(int R, int max_blocks, int K);
// Members of a coarse level the step kernel's hierarchical mode holds at once
// (Grids, or the active Chunks), and kept Chunks of a request.
int step_hier_level_cap(int D);
constexpr int kHierKeptChunks = 2048;

// kk_batched.cu
// Shared-pool GEMM (kk_batched.cu): each anchor's candidate keys (score,
// row), contiguous in pool order, up to `cap` = N of them; offsets[r][mtiles]
// is the count (offsets[r][t] the keys before block tile t). V has `rows`
// rows: `rows - N` coarse rows (a multiple of 128, scored for every anchor
// into `coarse`, float [R][rows - N], dense, no keys), then the N pool
// blocks, which the mask (uint32 [R][ceil(N/32)]) filters; `coarse_rows` of
// the coarse rows are real.
struct PoolLists {
  const uint64_t* keys;  // [R][cap]
  const int* offsets;    // [R][mtiles + 1]
  int mtiles;            // 128-block tiles of the pool
  long long cap;
};
size_t batched_workspace_bytes(int R, int rows, int N);
cudaError_t launch_pool_gemm(const uint16_t* A, const uint16_t* V, int rows, const uint32_t* mask, int R, int N,
                             int coarse_rows, float* coarse, void* ws, int* err, cudaStream_t s, PoolLists* out);
// Shared-pool hierarchy (kk_hier_pool.cu): coarse rows in front of the pool
// (Grids, Chunks, zero padding to a multiple of 128), at most
// kHierPoolCoarseMax Grids + Chunks.
constexpr int kHierPoolCoarseMax = 4096;
int hier_pool_coarse_rows(int N, int cp, int gc);
size_t hier_pool_workspace_bytes(int R, int N, int cp, int gc);
cudaError_t launch_hier_pool_reps(uint16_t* M, int N, int cp, int gc, cudaStream_t s);
cudaError_t launch_hier_select_pool(const uint16_t* A, const uint16_t* M, const uint32_t* mask, int R, int N,
                                    int cp, int gc, const int* permille, int K, int* idx, float* top, int* kept,
                                    void* ws, int* err, cudaStream_t s);
cudaError_t launch_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask, int R,
                                      int N, int K, int* idx, float* top, void* ws, int* err,
                                      cudaStream_t s);

// kk_write.cu
cudaError_t launch_compact_table(const int* idx, int K, const Table& bt, int* out_pages, int* out_logical,
                                 int* out_count, int* err, cudaStream_t s);
struct Ring {
  float* rows;  // [R][slots][D]
  int* pos;     // [R][slots]
  int slots;
};
cudaError_t launch_append(const KCache& kc, const Table& bt, const void* k_new, const float* head_w,
                          float* block_sum, float* vb, const Ring* ring, int* err, cudaStream_t s);
cudaError_t launch_ring_fill(const KCache& kc, const Table& bt, const float* head_w, const Ring& ring, int* err,
                             cudaStream_t s);

// kk_hier.cu: the Grid level from the Chunk level, and the hierarchical
// selection (a mode of the step kernel, see StepParams)
cudaError_t launch_grid_reps(const float* chunk, int D, int c_max, int g_max, const Table& bt, int chunk_pages,
                             int grid_chunks, float* grid, cudaStream_t s);
cudaError_t launch_hier_select(const float* vb, int D, int vb_rows, const Table& bt, const float* chunk,
                               const float* grid, int c_max, int g_max, const float* va, int chunk_pages,
                               int grid_chunks, const int* permille, int K, int* idx, float* top, int* kept,
                               unsigned long long* split_ctr, uint64_t* split_keys, int split_cap, int* err,
                               cudaStream_t s);

// kk_host.cu
void* tensor_map_encoder();  // cuTensorMapEncodeTiled (driver ABI 12.0), or null
int sm_count();              // SMs of the current device

// kk_pool_tma.cu: the persistent TMA pool for many blocks; returns
// cudaErrorNotSupported (nothing launched) when the cache layout or the block
// count does not suit it, and the caller falls back to launch_pool_direct.
cudaError_t launch_pool_tma(const KCache& kc, const int* pages, const int* n_valid, int n,
                            const float* head_w, int n_sets, const int* w_set, float* vb, int* err,
                            cudaStream_t s);
// the per-(layer, head) token sums and squares of every block of a table
// (inputs of the head-variance weights) on the same TMA ring
cudaError_t launch_pool_tma_slices(const KCache& kc, const Table& bt, long long total_blocks, float* S, float* Q,
                                   int* err, cudaStream_t s);

// kk_api.cu (used by kk_static.cu)
int* device_error_word();
// kk_api.cu: the limit of every bounded wait (kDefaultWaitNs unless a
// diagnostic call set another), and a one-shot request, for failure-detection
// tests, that the next persistent pool launch leave TMA box `box` of its first
// CTA uncopied (-1: none; taking it clears it).
unsigned long long wait_limit_ns();
long long take_skip_box();

// kk_coarse.cu
cudaError_t launch_coarse(const float* vb, int D, int num_pages, const Table& bt, int group,
                          float* out, int* err, cudaStream_t s);

}  // namespace kk
