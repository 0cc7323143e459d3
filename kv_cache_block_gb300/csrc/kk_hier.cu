// Hierarchical Grid -> Chunk -> Page selection ("Key-Key Semantic Affinity"
// page, §5.1). The Chunk level's representations are kk_coarse_means over the
// blocks; grid_reps_kernel builds the Grid level from them. The selection
// itself is a mode of the decode-step kernel (kk_step.cuh): every CTA of a
// request's cluster runs the Grid and Chunk levels itself, then the blocks of
// the kept Chunks are scored and ranked like a request's table.
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;

// grid[r][g][d] = mean over chunks c in [g*gc, min((g+1)*gc, C_r)) of
// chunk[r][c][d] (float64 sum), zero past the request's last Grid.
__global__ void __launch_bounds__(kThreads) grid_reps_kernel(const float* chunk, int D, int c_max, int g_max,
                                                             Table bt, int chunk_pages, int grid_chunks,
                                                             float* grid) {
  const int g = blockIdx.x, r = blockIdx.y;
  const int nb = bt.offsets[r + 1] - bt.offsets[r];
  const int C = nb > 0 ? (nb + chunk_pages - 1) / chunk_pages : 0;
  const int c0 = g * grid_chunks, c1 = min(C, c0 + grid_chunks);
  float* out = grid + ((long long)r * g_max + g) * D;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    double acc = 0.0;
    for (int c = c0; c < c1; ++c) acc += (double)chunk[((long long)r * c_max + c) * D + d];
    out[d] = c1 > c0 ? (float)(acc / (double)(c1 - c0)) : 0.f;
  }
}

}  // namespace

cudaError_t launch_grid_reps(const float* chunk, int D, int c_max, int g_max, const Table& bt, int chunk_pages,
                             int grid_chunks, float* grid, cudaStream_t s) {
  if (bt.R == 0 || g_max == 0) return cudaSuccess;
  grid_reps_kernel<<<dim3(g_max, bt.R), kThreads, 0, s>>>(chunk, D, c_max, g_max, bt, chunk_pages, grid_chunks,
                                                          grid);
  return cudaGetLastError();
}

cudaError_t launch_hier_select(const float* vb, int D, int vb_rows, const Table& bt, const float* chunk,
                               const float* grid, int c_max, int g_max, const float* va, int chunk_pages,
                               int grid_chunks, const int* permille, int K, int* idx, float* top, int* kept,
                               unsigned long long* split_ctr, uint64_t* split_keys, int split_cap, int* err,
                               cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  StepParams p = {};
  p.bt = bt;
  p.vb = vb;
  p.vb_rows = vb_rows;
  p.D = D;
  p.va_in = va;
  p.K = K;
  p.idx_out = idx;
  p.top_out = top;
  p.flags = kStepScore | kStepTopK;
  p.hier_grid = grid;
  p.hier_chunk = chunk;
  p.g_max = g_max;
  p.c_max = c_max;
  p.chunk_pages = chunk_pages;
  p.grid_chunks = grid_chunks;
  for (int i = 0; i < 3; ++i) p.permille[i] = permille[i];
  p.kept = kept;
  p.split_ctr = split_ctr;
  p.split_keys = split_keys;
  p.split_cap = split_cap;
  p.err = err;
  return launch_step(p, s);
}

}  // namespace kk
