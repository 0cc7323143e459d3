// The write of one decode token, shared by kk_append_tokens (kk_write.cu)
// and the decode step that fuses it (kk_step.cuh). Request r's decode token
// sits at position t = T - 1 (T = seq_lens[r]; the table already holds its
// block); its Keys k_new[r] ([L][H][D], the cache's element type) go into
// slot t % bs of the block's page, their sum over (layer, head) with the
// request's weights (uniform when head_w is null) is added to the block's
// running sum (restarted at the block's first token), v_b = sum / n
// (/ (L*H) unweighted), and the token's sum goes to its anchor-ring slot with
// its position. The three pieces below are used in this order by both
// callers, so that both write the same bits.
#pragma once
#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {

// The page that receives request r's decode token, and the token's position
// in *t; -1 when the table disagrees with seq_lens or holds a bad page
// (reported when `report`). Uniform over the CTA.
__device__ __forceinline__ int append_page(const KCache& kc, const Table& bt, int r, int* t, int* err, bool report) {
  const int off = bt.offsets[r];
  const int nb = bt.offsets[r + 1] - off;
  const int T_r = bt.seq_lens[r];
  *t = T_r - 1;
  if (T_r < 1 || nb > bt.max_blocks || nb != (T_r + kc.bs - 1) / kc.bs) {
    if (report && threadIdx.x == 0) flag_error(err, kErrBadIndex);
    return -1;
  }
  const int page = bt.pages[off + (T_r - 1) / kc.bs];
  if (page < 0 || page >= kc.num_pages) {
    if (report && threadIdx.x == 0) flag_error(err, kErrBadIndex);
    return -1;
  }
  return page;
}

// xrow[d] = sum over (l, h) of w[l, h] * k_new[r][l][h][d] (shared, D floats),
// run by a whole CTA of kThreads threads. Thread (s0, vec) takes the 16-byte
// vector vec of slices s = s0 + k * RSTEP, k = 0, 1, ...; with write_page >= 0
// it also stores those with k % parts == part into slot `slot` of that page
// (several CTAs that pool the same token can share its store that way). The
// slices' cache offsets advance by additions (no division a slice), and up to
// kBatch vectors a thread are loaded before any is used, so that their
// latencies overlap (7B-like: 7 vectors a thread). red: kThreads *
// Vec16<T>::kElems floats of shared memory. Ends with xrow visible to the
// whole CTA.
template <typename T, int D, int kThreads>
__device__ __forceinline__ void pool_token(const KCache& kc, int r, const void* k_new, const float* head_w,
                                           int write_page, int slot, int part, int parts, float* red,
                                           float* xrow) {
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int V16 = D / EPV;  // 16-byte vectors per row
  constexpr int RSTEP = kThreads / V16;
  constexpr int ES = elem_bytes<T>();
  constexpr int kBatch = 8;
  static_assert(V16 >= 1 && V16 <= 32 && (32 % V16) == 0, "row must be 16..512 bytes");
  static_assert(D <= kThreads, "one dimension a thread in the final sum");
  const int tid = threadIdx.x;
  const int LH = kc.L * kc.H;
  const int vec = tid % V16, s0 = tid / V16;
  const char* src = static_cast<const char*>(k_new) + (long long)r * LH * D * ES;  // byte offsets: T is a tag
  char* dst = reinterpret_cast<char*>(const_cast<void*>(kc.base)) +
              ((long long)max(write_page, 0) * kc.sP + (long long)slot * kc.sT + vec * EPV) * ES;
  // (l, h) of slice s0 and the step to the next slice of this thread, as
  // element offsets l * sL + h * sH
  int h = s0 % kc.H;
  long long o_lh = (long long)(s0 / kc.H) * kc.sL + (long long)h * kc.sH;
  const int dh = RSTEP % kc.H;
  const long long d_lh = (long long)(RSTEP / kc.H) * kc.sL + (long long)dh * kc.sH;
  const long long wrap = (long long)kc.sL - (long long)kc.H * kc.sH;  // h passing H: next layer
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
  int k = 0;
  for (int s1 = s0; s1 < LH; s1 += RSTEP * kBatch) {
    uint4 x[kBatch];
    float w[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s1 + b * RSTEP;
      if (s < LH) {
        x[b] = *reinterpret_cast<const uint4*>(src + ((long long)s * D + vec * EPV) * ES);
        w[b] = head_w ? head_w[(long long)r * LH + s] : 1.f;
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s1 + b * RSTEP;
      if (s < LH) {
        if (write_page >= 0 && k == part) *reinterpret_cast<uint4*>(dst + o_lh * ES) = x[b];
        if (++k == parts) k = 0;
        h += dh;
        o_lh += d_lh;
        if (h >= kc.H) {
          h -= kc.H;
          o_lh += wrap;
        }
        float f[EPV];
        Vec16<T>::unpack(x[b], f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] = fmaf(w[b], f[e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) red[s0 * D + vec * EPV + e] = acc[e];
  __syncthreads();
  if (tid < D) {
    float x = 0.f;
    for (int q = 0; q < RSTEP; ++q) x += red[q * D + tid];
    xrow[tid] = x;
  }
  __syncthreads();
}

// The token's row xrow (pool_token) committed by thread d < D: the running
// sum of the block (old_sum: its value before this token, read by the caller
// ahead of time; ignored at the block's first token), v_b, and the ring slot
// with the token's position. Returns this thread's new v_b value.
__device__ __forceinline__ float commit_token(int r, int page, int t, int bs, int LH, bool weighted, int D,
                                              float old_sum, const float* xrow, float* block_sum, float* vb,
                                              const Ring& ring) {
  const int d = threadIdx.x;
  const int slot = t % bs;
  const float scale = weighted ? 1.f / (float)(slot + 1) : 1.f / ((float)(slot + 1) * (float)LH);
  const long long rslot = ring.rows ? (long long)r * ring.slots + t % ring.slots : 0;
  float v = 0.f;
  if (d < D) {
    const float x = xrow[d];
    const float total = slot == 0 ? x : old_sum + x;
    block_sum[(long long)page * D + d] = total;
    v = total * scale;
    vb[(long long)page * D + d] = v;
    if (ring.rows) ring.rows[rslot * D + d] = x;
  }
  if (ring.rows && d == 0) ring.pos[rslot] = t;
  return v;
}

// The previous running sum of the token's block for thread d < D (0 at the
// block's first token, where it is not read).
__device__ __forceinline__ float load_old_sum(const float* block_sum, int page, int t, int bs, int D) {
  const int d = threadIdx.x;
  return (d < D && t % bs != 0) ? block_sum[(long long)page * D + d] : 0.f;
}

}  // namespace kk
