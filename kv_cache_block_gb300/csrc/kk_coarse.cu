// Coarse block representations ("Key-Key Semantic Affinity" page, §5.1): a
// coarser level's representation is the mean of its children's, here the mean
// of `group` consecutive logical blocks of a request. One CTA per (group,
// request): thread (k, c4) sums the 16-byte column c4 of rows k, k + RL, ...
// of the group, loading the page ids of a batch of rows, then their rows,
// together (two round trips per batch instead of two per row), in
// compensated (Kahan) float32: a group may hold hundreds of rows, and float64
// arithmetic runs at a small fraction of the float32 rate on this GPU. The RL
// partial rows are added the same way (measured: adding them and dividing in
// float64 made the kernel 4 times slower than its HBM time). Groups of 256
// rows or more take 1024 threads (measured, groups of 512 rows: loading in
// two rounds of 8 rows a thread instead of four of 4 took 14.3 -> 12.4 us
// over 65536 blocks).
#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

template <int D, int kThreads, int kBatch>  // kBatch: rows a thread has in flight
__global__ void __launch_bounds__(kThreads) coarse_kernel(const float* vb, int num_pages, const int* pages,
                                                          const int* offsets, int max_blocks, int group, int ng_max,
                                                          float* out, int* err) {
  constexpr int V4 = D / 4;            // 16-byte columns of a row
  constexpr int RL = kThreads / V4;    // rows summed side by side
  static_assert(kThreads % V4 == 0, "whole rows per pass");
  __shared__ float s_acc[RL][D];
  const int g = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const int off = offsets[r];
  int nb = offsets[r + 1] - off;
  if (nb < 0 || nb > max_blocks) {
    if (tid == 0 && g == 0) flag_error(err, kErrBadIndex);
    nb = 0;
  }
  const int j0 = g * group;
  const int j1 = min(nb, j0 + group);
  const int c4 = tid % V4, k = tid / V4;
  const float4* rows = reinterpret_cast<const float4*>(vb);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, cmp[4] = {0.f, 0.f, 0.f, 0.f};
  auto add = [&](int e, float x) {
    const float y = x - cmp[e];
    const float t = acc[e] + y;
    cmp[e] = (t - acc[e]) - y;
    acc[e] = t;
  };
  for (int jb = j0 + k; jb < j1; jb += RL * kBatch) {
    int pg[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = jb + u * RL;
      pg[u] = j < j1 ? __ldg(pages + off + j) : -1;
    }
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const bool ok = pg[u] >= 0 && pg[u] < num_pages;
      if (!ok && jb + u * RL < j1) flag_error(err, kErrBadIndex);
      v[u] = ok ? __ldg(rows + (long long)pg[u] * V4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      add(0, v[u].x);
      add(1, v[u].y);
      add(2, v[u].z);
      add(3, v[u].w);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) s_acc[k][c4 * 4 + e] = acc[e] - cmp[e];
  __syncthreads();
  const int cnt = j1 - j0;
  for (int d = tid; d < D; d += kThreads) {
    float s = 0.f, c = 0.f;
    for (int q = 0; q < RL; ++q) {
      const float y = s_acc[q][d] - c;
      const float t = s + y;
      c = (t - s) - y;
      s = t;
    }
    out[((long long)r * ng_max + g) * D + d] = cnt > 0 ? (s - c) / (float)cnt : 0.f;
  }
}

template <int D>
cudaError_t launch_d(const float* vb, int num_pages, const Table& bt, int group, int ng_max, float* out, int* err,
                     cudaStream_t s) {
  const dim3 grid(ng_max, bt.R);
  if (group >= 256)  // 32 rows side by side, 8 in flight a thread: a group of 512 in two rounds of loads
    coarse_kernel<D, 1024, 8><<<grid, 1024, 0, s>>>(vb, num_pages, bt.pages, bt.offsets, bt.max_blocks, group, ng_max,
                                                 out, err);
  else
    coarse_kernel<D, 256, 8><<<grid, 256, 0, s>>>(vb, num_pages, bt.pages, bt.offsets, bt.max_blocks, group, ng_max,
                                               out, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_coarse(const float* vb, int D, int num_pages, const Table& bt, int group,
                          float* out, int* err, cudaStream_t s) {
  const int ng_max = (bt.max_blocks + group - 1) / group;
  if (bt.R == 0 || ng_max == 0) return cudaSuccess;
  switch (D) {
    case 32: return launch_d<32>(vb, num_pages, bt, group, ng_max, out, err, s);
    case 64: return launch_d<64>(vb, num_pages, bt, group, ng_max, out, err, s);
    case 128: return launch_d<128>(vb, num_pages, bt, group, ng_max, out, err, s);
    case 256: return launch_d<256>(vb, num_pages, bt, group, ng_max, out, err, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kk
