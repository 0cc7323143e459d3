// Block pooling on the write path: v_b is the mean of a block's Keys over its
// tokens, KV heads and layers ("Key-Key Semantic Affinity" page, §2.2 step 1
// and §5.2 steps 2-3), optionally weighted per (layer, head) by the head's
// Key variance (same page, §3.3 finding 2 and §6.1).
//
// The pool streams bf16/fp32 Keys from HBM exactly once. Each CTA owns one
// block; each warp owns whole (layer, head) slices of it, so a slice's token
// sum needs no cross-warp traffic. A lane reads one 16-byte vector of a token
// row per load and keeps 8 loads in flight; lanes that share a dim range are
// combined with shuffles, warps through shared memory.
#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;

struct PoolArgs {
  const char* base;
  int L, H, bs, num_pages;
  long long sL, sP, sH, sT;
  // direct mode: a list of pages
  const int* pages;
  const int* n_valid;
  const float* head_w;
  int n_sets;
  const int* w_set;
  float* vb;
  // slice mode: every block of a block table
  const int* bt_pages;
  const int* offsets;
  const int* seq_lens;
  int max_blocks;
  long long total;  // rows of S / Q (blocks of the whole table)
  float* S;  // [total_blocks][L*H][D] token sums per (layer, head)
  float* Q;  // [total_blocks][L*H] sums of squares over tokens and dims
  int* err;
};

// Token sum of one (layer, head) slice for this lane's dims, plus (optionally)
// the lane's sum of squares. Rows are tokens t < n at stride sT.
template <typename T, int D, bool kSquares>
__device__ __forceinline__ void slice_sum(const char* rowp, long long tok_bytes, int n, int tl,
                                          float (&ps)[Vec16<T>::kElems], float& q) {
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int RPW = 32 / (D / EPV);
#pragma unroll
  for (int e = 0; e < EPV; ++e) ps[e] = 0.f;
  q = 0.f;
  for (int t0 = 0; t0 < n; t0 += kUnroll * RPW) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = t0 + u * RPW + tl;
      v[u] = ld_stream16(rowp + (long long)(t0 + u * RPW) * tok_bytes, t < n);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[EPV];
      Vec16<T>::unpack(v[u], f);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        ps[e] += f[e];
        if (kSquares) q = fmaf(f[e], f[e], q);
      }
    }
  }
}

// One CTA per block, or (direct mode) a cluster of S CTAs per block that
// split the block's (layer, head) slices and sum their partial vectors in the
// leader CTA through distributed shared memory; S > 1 only when there are too
// few blocks to fill the GPU evenly.
template <typename T, int D, bool kSlices>
__global__ void __launch_bounds__(kThreads) pool_kernel(PoolArgs a) {
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int V16 = D / EPV;
  static_assert(V16 >= 1 && V16 <= 32 && (32 % V16) == 0, "row must be 16..512 bytes");
  constexpr int ES = elem_bytes<T>();
  constexpr int kMaxSplit = 8;
  __shared__ float s_w[kSlices ? 1 : kMaxLH];
  __shared__ float s_red[kWarps][D];
  __shared__ float s_part[kSlices ? 1 : kMaxSplit][D];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int vec = lane % V16, tl = lane / V16;
  const int LH = a.L * a.H;
  const int S = kSlices ? 1 : (int)cluster_size();
  const int crank = S > 1 ? (int)cluster_rank() : 0;
  if (S > 1) cluster_arrive_relaxed();

  int page = 0, n = 0, g = 0, wsel = 0;
  bool valid = true;
  if (kSlices) {
    const int r = blockIdx.y, j = blockIdx.x;
    const int off = a.offsets[r];
    const int nb = a.offsets[r + 1] - off;
    if (j >= nb) return;
    const int T_r = a.seq_lens[r];
    if (off < 0 || nb > a.max_blocks || (long long)off + nb > a.total || T_r < 0 || nb != (T_r + a.bs - 1) / a.bs) {
      if (threadIdx.x == 0 && j == 0) flag_error(a.err, kErrBadIndex);
      return;
    }
    g = off + j;
    page = a.bt_pages[g];
    n = min(a.bs, T_r - j * a.bs);
    if (page < 0 || page >= a.num_pages) {
      // the block's sums read as zero: the request's variance sums never see
      // what an earlier call left in the scratch
      if (threadIdx.x == 0) flag_error(a.err, kErrBadIndex);
      for (int i = threadIdx.x; i < LH * D; i += kThreads) a.S[(long long)g * LH * D + i] = 0.f;
      for (int i = threadIdx.x; i < LH; i += kThreads) a.Q[(long long)g * LH + i] = 0.f;
      return;
    }
  } else {
    const int i = blockIdx.x / S;
    page = a.pages[i];
    n = a.n_valid[i];
    if (a.head_w && a.w_set) wsel = a.w_set[i];
    valid = !(n < 0 || n > a.bs || page < 0 || page >= a.num_pages ||
              (a.head_w && (wsel < 0 || wsel >= a.n_sets)));
    if (!valid) {
      if (threadIdx.x == 0 && crank == 0) flag_error(a.err, kErrBadIndex);
      n = 0;
      page = 0;
    }
    for (int s = threadIdx.x; s < LH; s += kThreads)
      s_w[s] = a.head_w ? a.head_w[(long long)wsel * LH + s] : 1.f;
    __syncthreads();
  }

  const long long tok_bytes = a.sT * ES;
  const char* page_base = a.base + ((long long)page * a.sP + (long long)tl * a.sT) * ES + vec * 16;
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.f;

  for (int s = crank + S * warp; s < LH; s += S * kWarps) {
    const int l = s / a.H, h = s - l * a.H;
    const char* rowp = page_base + ((long long)l * a.sL + (long long)h * a.sH) * ES;
    float ps[EPV], q;
    slice_sum<T, D, kSlices>(rowp, tok_bytes, n, tl, ps, q);
    if (kSlices) {
#pragma unroll
      for (int e = 0; e < EPV; ++e)
#pragma unroll
        for (int o = V16; o < 32; o <<= 1) ps[e] += __shfl_xor_sync(kFull, ps[e], o);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(kFull, q, o);
      float* dst = a.S + ((long long)g * LH + s) * D + vec * EPV;
      if (tl == 0) {
#pragma unroll
        for (int e = 0; e < EPV; e += 4)
          *reinterpret_cast<float4*>(dst + e) = make_float4(ps[e], ps[e + 1], ps[e + 2], ps[e + 3]);
      }
      if (lane == 0) a.Q[(long long)g * LH + s] = q;
    } else {
      const float w = s_w[s];
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[e] = fmaf(w, ps[e], acc[e]);
    }
  }
  if (kSlices) return;

#pragma unroll
  for (int e = 0; e < EPV; ++e)
#pragma unroll
    for (int o = V16; o < 32; o <<= 1) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
  if (tl == 0) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) s_red[warp][vec * EPV + e] = acc[e];
  }
  __syncthreads();
  float part[(D + kThreads - 1) / kThreads];
#pragma unroll
  for (int k = 0; k < (D + kThreads - 1) / kThreads; ++k) {
    const int d = threadIdx.x + k * kThreads;
    float v = 0.f;
    if (d < D) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += s_red[w][d];
    }
    part[k] = v;
  }
  if (S > 1) {
    cluster_wait_acquire();  // every CTA of the cluster has started
#pragma unroll
    for (int k = 0; k < (D + kThreads - 1) / kThreads; ++k) {
      const int d = threadIdx.x + k * kThreads;
      if (d < D) st_cluster_f32(map_to_rank(smem_u32(&s_part[crank][d]), 0), part[k]);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    if (crank != 0) return;
#pragma unroll
    for (int k = 0; k < (D + kThreads - 1) / kThreads; ++k) {
      const int d = threadIdx.x + k * kThreads;
      if (d < D) {
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += s_part[q][d];
        part[k] = v;
      }
    }
  }
  if (!valid) return;
  const float scale = (n == 0) ? 0.f : (a.head_w ? 1.f / (float)n : 1.f / ((float)n * (float)LH));
#pragma unroll
  for (int k = 0; k < (D + kThreads - 1) / kThreads; ++k) {
    const int d = threadIdx.x + k * kThreads;
    if (d < D) a.vb[(long long)page * D + d] = part[k] * scale;
  }
}

// Per (request, layer-head): Var = E_t[sum_d K^2]/D - sum_d (E_t K_d)^2 / D,
// from the per-block sums, accumulated in float64 in a fixed order. A thread
// owns four dims (16-byte loads) of every kThreads/(D/4)-th block.
__global__ void __launch_bounds__(kThreads) head_var_kernel(const float* S, const float* Q,
                                                            const int* offsets, const int* seq_lens,
                                                            int bs, int LH, int D, int max_blocks,
                                                            long long total, double* var, int* err) {
  __shared__ double s_sum[kThreads * 4];  // [row group][D]: kThreads / (D/4) groups of D
  __shared__ double s_q[kThreads];
  const int s = blockIdx.x, r = blockIdx.y;
  const int off = offsets[r];
  const int nb = offsets[r + 1] - off;
  const int T_r = seq_lens[r];
  if (off < 0 || nb < 0 || nb > max_blocks || (long long)off + nb > total || T_r < 0 || nb != (T_r + bs - 1) / bs) {
    if (threadIdx.x == 0 && s == 0) flag_error(err, kErrBadIndex);
    return;
  }
  const int C4 = D / 4;            // float4 columns of a row
  const int KS = kThreads / C4;    // row groups
  const int c4 = threadIdx.x % C4, kr = threadIdx.x / C4;
  const float4* S4 = reinterpret_cast<const float4*>(S);
  // compensated (Kahan) float32 sums: float64 arithmetic is scarce on this
  // GPU, and the compensation keeps the error independent of the block count
  float a[4] = {0.f, 0.f, 0.f, 0.f}, cmp[4] = {0.f, 0.f, 0.f, 0.f};
  auto add4 = [&](const float4& v) {
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y = x[e] - cmp[e];
      const float t = a[e] + y;
      cmp[e] = (t - a[e]) - y;
      a[e] = t;
    }
  };
  int j = kr;
  for (; j + 3 * KS < nb; j += 4 * KS) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = S4[((long long)(off + j + u * KS) * LH + s) * C4 + c4];
#pragma unroll
    for (int u = 0; u < 4; ++u) add4(v[u]);
  }
  for (; j < nb; j += KS) add4(S4[((long long)(off + j) * LH + s) * C4 + c4]);
  const double a0 = (double)a[0] - (double)cmp[0], a1 = (double)a[1] - (double)cmp[1];
  const double a2 = (double)a[2] - (double)cmp[2], a3 = (double)a[3] - (double)cmp[3];
  double q = 0.0;
  for (int jj = threadIdx.x; jj < nb; jj += kThreads) q += (double)Q[(long long)(off + jj) * LH + s];
  double* row = s_sum + kr * D + c4 * 4;
  row[0] = a0;
  row[1] = a1;
  row[2] = a2;
  row[3] = a3;
  s_q[threadIdx.x] = q;
  __syncthreads();
  // per dim: the mean over the request's tokens, squared (row group 0 is
  // overwritten only after every group's value for that dim has been read)
  for (int d = threadIdx.x; d < D; d += kThreads) {
    double m = 0.0;
    for (int g = 0; g < KS; ++g) m += s_sum[g * D + d];
    const double mu = T_r > 0 ? m / (double)T_r : 0.0;
    s_sum[d] = mu * mu;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double m2 = 0.0, qt = 0.0;
    for (int i = 0; i < D; ++i) m2 += s_sum[i];
    for (int i = 0; i < kThreads; ++i) qt += s_q[i];
    double v = T_r > 0 ? (qt / ((double)T_r * D) - m2 / D) : 0.0;
    var[(long long)r * LH + s] = v > 0.0 ? v : 0.0;
  }
}

// head_w_out[r][s] = Var[r][s] / sum_s Var[r][s] (uniform if the sum is 0).
__global__ void __launch_bounds__(kThreads) finalize_weights_kernel(const double* var, int LH,
                                                                    const int* offsets,
                                                                    const int* seq_lens, int bs,
                                                                    int max_blocks, long long total,
                                                                    float* out) {
  __shared__ double s_part[kThreads];
  const int r = blockIdx.x;
  const int off = offsets[r];
  const int nb = offsets[r + 1] - off;
  const int T_r = seq_lens[r];
  if (off < 0 || nb < 0 || nb > max_blocks || (long long)off + nb > total || T_r < 0 || nb != (T_r + bs - 1) / bs)
    return;  // flagged upstream
  double acc = 0.0;
  for (int s = threadIdx.x; s < LH; s += kThreads) acc += var[(long long)r * LH + s];
  s_part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s_part[threadIdx.x] += s_part[threadIdx.x + w];
    __syncthreads();
  }
  const double tot = s_part[0];
  for (int s = threadIdx.x; s < LH; s += kThreads)
    out[(long long)r * LH + s] =
        tot > 0.0 ? (float)(var[(long long)r * LH + s] / tot) : 1.f / (float)LH;
}

// vb[page] = (1/n) * sum_s w[r][s] * S[block][s] (weights fixed per request).
// A thread owns four dims (16-byte loads) of every kThreads/(D/4)-th slice.
__global__ void __launch_bounds__(kThreads) combine_kernel(const float* S, const float* head_w,
                                                           const int* pages, const int* offsets,
                                                           const int* seq_lens, int bs, int LH,
                                                           int D, int max_blocks, long long total,
                                                           int num_pages, float* vb) {
  __shared__ float s_w[kMaxLH];
  __shared__ float4 s_part[kThreads];
  const int j = blockIdx.x, r = blockIdx.y;
  const int off = offsets[r];
  const int nb = offsets[r + 1] - off;
  const int T_r = seq_lens[r];
  if (j >= nb || off < 0 || nb > max_blocks || (long long)off + nb > total || T_r < 0 ||
      nb != (T_r + bs - 1) / bs)
    return;  // flagged upstream
  const int page = pages[off + j];
  if (page < 0 || page >= num_pages) return;  // flagged by the slice kernel
  for (int s = threadIdx.x; s < LH; s += kThreads) s_w[s] = head_w[(long long)r * LH + s];
  __syncthreads();
  const int C4 = D / 4, KS = kThreads / C4;
  const int c4 = threadIdx.x % C4, kr = threadIdx.x / C4;
  const float4* src = reinterpret_cast<const float4*>(S + (long long)(off + j) * LH * D);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = kr; s < LH; s += KS) {
    const float4 v = src[(long long)s * C4 + c4];
    const float w = s_w[s];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  s_part[threadIdx.x] = acc;
  __syncthreads();
  const int n = min(bs, T_r - j * bs);
  const float inv_n = n > 0 ? 1.f / (float)n : 0.f;
  if (threadIdx.x < C4) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < KS; ++g) {
      const float4 v = s_part[g * C4 + threadIdx.x];
      t.x += v.x;
      t.y += v.y;
      t.z += v.z;
      t.w += v.w;
    }
    float* out = vb + (long long)page * D + threadIdx.x * 4;
    if ((reinterpret_cast<uintptr_t>(out) & 15) == 0) {
      *reinterpret_cast<float4*>(out) = make_float4(t.x * inv_n, t.y * inv_n, t.z * inv_n, t.w * inv_n);
    } else {  // a v_b table not 16-byte aligned
      out[0] = t.x * inv_n;
      out[1] = t.y * inv_n;
      out[2] = t.z * inv_n;
      out[3] = t.w * inv_n;
    }
  }
}

template <typename T, int D, bool kSlices>
cudaError_t launch_pool(const PoolArgs& a, dim3 grid, int split, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pool_kernel<T, D, kSlices>, a);
}

template <bool kSlices>
cudaError_t dispatch_pool(const KCache& kc, const PoolArgs& a, dim3 grid, int split, cudaStream_t s) {
#define KK_POOL_CASE(TT, DD) \
  if (kc.D == DD) return launch_pool<TT, DD, kSlices>(a, grid, split, s);
  if (kc.dtype == 1) {
    KK_POOL_CASE(bf16_t, 32)
    KK_POOL_CASE(bf16_t, 64)
    KK_POOL_CASE(bf16_t, 128)
    KK_POOL_CASE(bf16_t, 256)
  } else {
    KK_POOL_CASE(float, 32)
    KK_POOL_CASE(float, 64)
    KK_POOL_CASE(float, 128)
  }
#undef KK_POOL_CASE
  return cudaErrorInvalidValue;
}

PoolArgs base_args(const KCache& kc, int* err) {
  PoolArgs a = {};
  a.base = reinterpret_cast<const char*>(kc.base);
  a.L = kc.L;
  a.H = kc.H;
  a.bs = kc.bs;
  a.num_pages = kc.num_pages;
  a.sL = kc.sL;
  a.sP = kc.sP;
  a.sH = kc.sH;
  a.sT = kc.sT;
  a.err = err;
  return a;
}

}  // namespace

cudaError_t launch_pool_direct(const KCache& kc, const int* pages, const int* n_valid, int n,
                               const float* head_w, int n_sets, const int* w_set, float* vb,
                               int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  // at least one block per SM: the persistent TMA pipeline (kk_pool_tma.cu)
  const cudaError_t e = launch_pool_tma(kc, pages, n_valid, n, head_w, n_sets, w_set, vb, err, s);
  if (e != cudaErrorNotSupported) return e;
  PoolArgs a = base_args(kc, err);
  a.pages = pages;
  a.n_valid = n_valid;
  a.head_w = head_w;
  a.n_sets = n_sets;
  a.w_set = w_set;
  a.vb = vb;
  // Split each block over a cluster of 2 CTAs only when there are too few
  // blocks to fill the GPU (fewer than 1024); measured on GB300, larger
  // clusters or splits of many blocks lose bandwidth to cluster scheduling.
  const int split = (n < 1024 && kc.L * kc.H >= 16) ? 2 : 1;
  return dispatch_pool<false>(kc, a, dim3((unsigned)n * split), split, s);
}

cudaError_t launch_pool_slices(const KCache& kc, const Table& bt, long long total_blocks, float* S, float* Q,
                               int* err, cudaStream_t s) {
  if (bt.R == 0 || bt.max_blocks == 0) return cudaSuccess;
  // at least one block per SM: the persistent TMA ring (kk_pool_tma.cu)
  const cudaError_t e = launch_pool_tma_slices(kc, bt, total_blocks, S, Q, err, s);
  if (e != cudaErrorNotSupported) return e;
  PoolArgs a = base_args(kc, err);
  a.bt_pages = bt.pages;
  a.offsets = bt.offsets;
  a.seq_lens = bt.seq_lens;
  a.max_blocks = bt.max_blocks;
  a.total = total_blocks;
  a.S = S;
  a.Q = Q;
  return dispatch_pool<true>(kc, a, dim3(bt.max_blocks, bt.R), 1, s);
}

cudaError_t launch_head_var(const KCache& kc, const Table& bt, long long total_blocks, const float* S,
                            const float* Q, double* var, int* err, cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  head_var_kernel<<<dim3(kc.L * kc.H, bt.R), kThreads, 0, s>>>(
      S, Q, bt.offsets, bt.seq_lens, kc.bs, kc.L * kc.H, kc.D, bt.max_blocks, total_blocks, var, err);
  return cudaGetLastError();
}

cudaError_t launch_finalize_weights(const KCache& kc, const Table& bt, long long total_blocks, const double* var,
                                    float* head_w_out, cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  finalize_weights_kernel<<<bt.R, kThreads, 0, s>>>(var, kc.L * kc.H, bt.offsets, bt.seq_lens,
                                                    kc.bs, bt.max_blocks, total_blocks, head_w_out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const KCache& kc, const Table& bt, long long total_blocks, const float* S,
                           const float* head_w, float* vb, int* err, cudaStream_t s) {
  (void)err;
  if (bt.R == 0 || bt.max_blocks == 0) return cudaSuccess;
  combine_kernel<<<dim3(bt.max_blocks, bt.R), kThreads, 0, s>>>(S, head_w, bt.pages, bt.offsets,
                                                            bt.seq_lens, kc.bs, kc.L * kc.H, kc.D,
                                                            bt.max_blocks, total_blocks, kc.num_pages, vb);
  return cudaGetLastError();
}

}  // namespace kk
