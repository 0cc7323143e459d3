// Coarse block representations ("Key-Key Semantic Affinity" page, §5.1): a
// coarser level's representation is the mean of its children's, here the mean
// of `group` consecutive logical blocks of a request. Accumulated in float64
// (a group may hold hundreds of rows); one CTA per (group, request).
#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) coarse_kernel(const float* vb, int D, int num_pages,
                                                          const int* pages, const int* offsets,
                                                          int max_blocks, int group, int ng_max,
                                                          float* out, int* err) {
  __shared__ double s_acc[kThreads];
  const int g = blockIdx.x, r = blockIdx.y;
  const int off = offsets[r];
  int nb = offsets[r + 1] - off;
  if (nb < 0 || nb > max_blocks) {
    if (threadIdx.x == 0 && g == 0) flag_error(err, kErrBadIndex);
    nb = 0;
  }
  const int j0 = g * group;
  const int j1 = min(nb, j0 + group);
  const int KS = kThreads / D;
  const int d = threadIdx.x % D, k = threadIdx.x / D;
  double acc = 0.0;
  for (int j = j0 + k; j < j1; j += KS) {
    const int pg = pages[off + j];
    if (pg < 0 || pg >= num_pages) {
      flag_error(err, kErrBadIndex);
      continue;
    }
    acc += (double)vb[(long long)pg * D + d];
  }
  s_acc[threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.x < D) {
    double s = 0.0;
    for (int q = 0; q < KS; ++q) s += s_acc[q * D + threadIdx.x];
    const int cnt = j1 - j0;
    out[((long long)r * ng_max + g) * D + threadIdx.x] = cnt > 0 ? (float)(s / cnt) : 0.f;
  }
}

}  // namespace

cudaError_t launch_coarse(const float* vb, int D, int num_pages, const Table& bt, int group,
                          float* out, int* err, cudaStream_t s) {
  const int ng_max = (bt.max_blocks + group - 1) / group;
  if (bt.R == 0 || ng_max == 0) return cudaSuccess;
  coarse_kernel<<<dim3(ng_max, bt.R), kThreads, 0, s>>>(vb, D, num_pages, bt.pages, bt.offsets,
                                                        bt.max_blocks, group, ng_max, out, err);
  return cudaGetLastError();
}

}  // namespace kk
