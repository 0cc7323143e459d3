// The write side around a decode step ("Key-Key Semantic Affinity" page):
//  * compact_table_kernel: the selected blocks of each request as a table for
//    the attention kernel, physical pages in logical order (§5.2 step 4: only
//    the selected blocks are loaded);
//  * append_kernel: one decode token per request written into its block of
//    the paged cache and folded into that block's running sum, so v_b is the
//    pooled mean of the block's tokens after every token (§5.2 step 2, v_b
//    computed as the block is written; §2.2 step 1); the token's pooled Keys
//    also go to the request's anchor ring;
//  * ring_fill_kernel: the anchor ring written from the cache, one token per
//    CTA (the anchor of §5.2 step 1 is a mean of these per-token rows).
#include <utility>

#include "kk_append.cuh"
#include "kk_device.cuh"
#include "kk_pdl.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;

// One CTA per request, one thread per top-K slot (K <= 256): a slot's place
// in the table is the number of valid slots with a smaller logical index
// (equal indices by slot order).
__global__ void __launch_bounds__(kThreads) compact_table_kernel(const int* idx, int K, Table bt, int* out_pages,
                                                                 int* out_logical, int* out_count, int* err) {
  __shared__ int s_v[kMaxK];
  __shared__ int s_n;
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x, t = threadIdx.x;
  const int off = bt.offsets[r];
  int nb = bt.offsets[r + 1] - off;
  if (nb < 0 || nb > bt.max_blocks) {
    if (t == 0) flag_error(err, kErrBadIndex);
    nb = 0;
  }
  if (t == 0) s_n = 0;
  int v = -1;
  if (t < K) {
    v = idx[(long long)r * K + t];
    if (v < -1 || v >= nb) {
      flag_error(err, kErrBadIndex);
      v = -1;
    }
    s_v[t] = v;
  }
  __syncthreads();
  if (v >= 0) atomicAdd(&s_n, 1);
  int rank = 0;
  if (v >= 0)
    for (int u = 0; u < K; ++u) {
      const int w = s_v[u];
      rank += (w >= 0 && (w < v || (w == v && u < t))) ? 1 : 0;
    }
  __syncthreads();
  const int n = s_n;
  int* op = out_pages + (long long)r * K;
  int* ol = out_logical ? out_logical + (long long)r * K : nullptr;
  if (v >= 0) {
    op[rank] = bt.pages[off + v];
    if (ol) ol[rank] = v;
  }
  for (int i = n + t; i < K; i += kThreads) {
    op[i] = -1;
    if (ol) ol[i] = -1;
  }
  if (t == 0 && out_count) out_count[r] = n;
}

// One CTA per request: the append of request blockIdx.x's decode token
// (kk_append.cuh).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) append_kernel(KCache kc, Table bt, const void* k_new, const float* head_w,
                                                          float* block_sum, float* vb, Ring ring, int* err) {
  __shared__ float s_red[kThreads * Vec16<T>::kElems];
  __shared__ float s_x[D];
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  int t;
  const int page = append_page(kc, bt, r, &t, err, true);
  if (page < 0) return;
  const float old = load_old_sum(block_sum, page, t, kc.bs, D);
  pool_token<T, D, kThreads>(kc, r, k_new, head_w, page, t % kc.bs, 0, 1, s_red, s_x);
  commit_token(r, page, t, kc.bs, kc.L * kc.H, head_w != nullptr, D, old, s_x, block_sum, vb, ring);
}

// CTA (i, r): slot of token t = T - 1 - i of request r when i < min(slots, T)
// (the token's Keys summed over (layer, head) with the request's weights,
// one 16-byte vector per thread, the warps' partial rows added through
// shared memory); for T < slots the CTAs i >= T mark slot i empty.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) ring_fill_kernel(KCache kc, Table bt, const float* head_w, Ring ring,
                                                             int* err) {
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int V16 = D / EPV;
  constexpr int RSTEP = kThreads / V16;
  constexpr int ES = elem_bytes<T>();
  static_assert(V16 >= 1 && V16 <= 32 && (32 % V16) == 0, "row must be 16..512 bytes");
  __shared__ float s_red[RSTEP][D];
  const int i = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const int off = bt.offsets[r];
  const int nb = bt.offsets[r + 1] - off;
  const int T_r = bt.seq_lens[r];
  const long long rbase = (long long)r * ring.slots;
  if (T_r < 0 || nb > bt.max_blocks || nb != (T_r + kc.bs - 1) / kc.bs) {
    if (tid == 0) {
      if (i == 0) flag_error(err, kErrBadIndex);
      ring.pos[rbase + i] = -1;
    }
    return;
  }
  if (i >= min(ring.slots, T_r)) {
    if (tid == 0) ring.pos[rbase + i] = -1;  // only reached for T < slots, where slot i holds no token
    return;
  }
  const int t = T_r - 1 - i, slot = t % ring.slots;
  const int page = bt.pages[off + t / kc.bs];
  if (page < 0 || page >= kc.num_pages) {
    if (tid == 0) {
      flag_error(err, kErrBadIndex);
      ring.pos[rbase + slot] = -1;
    }
    return;
  }
  const int LH = kc.L * kc.H;
  const int vec = tid % V16, s0 = tid / V16;
  const char* base = static_cast<const char*>(kc.base) +
                     ((long long)page * kc.sP + (long long)(t % kc.bs) * kc.sT + vec * EPV) * ES;
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
  for (int s = s0; s < LH; s += RSTEP) {
    const int l = s / kc.H, h = s - l * kc.H;
    const uint4 x = ld_stream16(base + ((long long)l * kc.sL + (long long)h * kc.sH) * ES, true);
    float f[EPV];
    Vec16<T>::unpack(x, f);
    const float w = head_w ? head_w[(long long)r * LH + s] : 1.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = fmaf(w, f[e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) s_red[s0][vec * EPV + e] = acc[e];
  __syncthreads();
  for (int d = tid; d < D; d += kThreads) {
    float x = 0.f;
    for (int q = 0; q < RSTEP; ++q) x += s_red[q][d];
    ring.rows[(rbase + slot) * D + d] = x;
  }
  if (tid == 0) ring.pos[rbase + slot] = t;
}

// A launch that may start behind the previous kernel of the stream (the
// kernel waits for it before touching memory: pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename T, int D>
cudaError_t launch_append_t(const KCache& kc, const Table& bt, const void* k_new, const float* head_w,
                            float* block_sum, float* vb, const Ring& ring, int* err, cudaStream_t s) {
  return launch_pdl(append_kernel<T, D>, dim3(bt.R), s, kc, bt, k_new, head_w, block_sum, vb, ring, err);
}

template <typename T, int D>
cudaError_t launch_ring_fill_t(const KCache& kc, const Table& bt, const float* head_w, const Ring& ring, int* err,
                               cudaStream_t s) {
  ring_fill_kernel<T, D><<<dim3(ring.slots, bt.R), kThreads, 0, s>>>(kc, bt, head_w, ring, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact_table(const int* idx, int K, const Table& bt, int* out_pages, int* out_logical,
                                 int* out_count, int* err, cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  return launch_pdl(compact_table_kernel, dim3(bt.R), s, idx, K, bt, out_pages, out_logical, out_count, err);
}

cudaError_t launch_append(const KCache& kc, const Table& bt, const void* k_new, const float* head_w,
                          float* block_sum, float* vb, const Ring* ring, int* err, cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  const Ring g = ring ? *ring : Ring{nullptr, nullptr, 1};
#define KK_APPEND_CASE(TT, DD) \
  case DD: return launch_append_t<TT, DD>(kc, bt, k_new, head_w, block_sum, vb, g, err, s);
  if (kc.dtype == 1) {
    switch (kc.D) { KK_APPEND_CASE(bf16_t, 32) KK_APPEND_CASE(bf16_t, 64) KK_APPEND_CASE(bf16_t, 128)
                    KK_APPEND_CASE(bf16_t, 256) }
  } else {
    switch (kc.D) { KK_APPEND_CASE(float, 32) KK_APPEND_CASE(float, 64) KK_APPEND_CASE(float, 128) }
  }
#undef KK_APPEND_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_ring_fill(const KCache& kc, const Table& bt, const float* head_w, const Ring& ring, int* err,
                             cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
#define KK_FILL_CASE(TT, DD) \
  case DD: return launch_ring_fill_t<TT, DD>(kc, bt, head_w, ring, err, s);
  if (kc.dtype == 1) {
    switch (kc.D) { KK_FILL_CASE(bf16_t, 32) KK_FILL_CASE(bf16_t, 64) KK_FILL_CASE(bf16_t, 128)
                    KK_FILL_CASE(bf16_t, 256) }
  } else {
    switch (kc.D) { KK_FILL_CASE(float, 32) KK_FILL_CASE(float, 64) KK_FILL_CASE(float, 128) }
  }
#undef KK_FILL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kk
