// One decode step of the Key-Key selector ("Key-Key Semantic Affinity" page,
// §5.2 steps 1-4): pool the anchor from the last W tokens' Keys, score every
// block of the request's table by (1 + cos(v_b, v_anchor)) / 2 (§2.2 step 3,
// §3.2), and keep the top K (§5.2 step 4).
//
// A request is served by one thread-block cluster of CL CTAs. The CTAs split
// the anchor's (layer, head) slices and the request's blocks. A CTA starts by
// bulk-copying (TMA) the v_b rows of its blocks into shared memory, so that
// gather overlaps the anchor. Partial anchors, and each CTA's sorted top-K
// list, are exchanged through distributed shared memory; every CTA then ranks
// its own candidates in the union and writes them. A few very long requests
// are split over several clusters each: every cluster writes its sorted top-K
// list to a fixed device buffer and the last one to finish merges the lists.
// A whole step is one launch. Every stage can be switched off, which gives
// kk_anchor, kk_score, kk_topk and kk_score_topk from the same code.
//
// The kernel and its launch, included by kk_step.cu and by kk_step_fused.cu,
// which instantiates the kernel with the decode token's append fused in
// (kk_step_options.k_new): a separate instantiation, so that the plain
// step carries none of its code (measured: 1.4 us a step at 32 requests x
// 1024 blocks when it was one kernel with a run-time switch).
#pragma once
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kk_append.cuh"
#include "kk_device.cuh"
#include "kk_pdl.cuh"
#include "kk_internal.h"
#include "kk_warp.cuh"

namespace kk {
namespace {

// Very long requests are split over several clusters: each writes its sorted
// top-K list to the caller's workspace, and the last one to count itself in
// (a per-request counter in the workspace) merges the lists into the
// request's output and sets the counter back to zero.
constexpr int kSplitPerWarp = 8;     // lists each warp folds in the final merge of K <= 32
constexpr int kSplitMinBlocks = 256;  // blocks per CTA below which a request is not split further
constexpr int kHierSplitMinBlocks = 64;  // the same for the hierarchy's block level

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kThreads;  // candidates per top-K tile
constexpr int kMaxSplits = kSplitPerWarp * kThreads / 32;  // lists the final fold of K <= 32 takes
constexpr int kStage = 64;  // v_b rows staged in shared memory by bulk copies
static_assert(kMaxW * 8 >= kThreads * 16, "ring-mode partial rows fit the token-offset table");
static_assert(kMergeSlots % kThreads == 0, "the split merge holds kMergeSlots / kThreads keys a thread");
static_assert(kSplitPerWarp * 32 * kWarps <= kMergeSlots, "the final fold stages its lists in the merge buffer");

template <int D>
struct StepSmem {
  float stage[kStage][D];      // v_b rows of the CTA's first blocks (bulk copies)
  float part[kMaxCluster][D];  // anchor partial of each CTA of the cluster
  float wpart[kWarps][D];
  float va[D];
  alignas(16) long long tok[kMaxW];  // byte offset of each anchor token row (page, slot); ring mode: sums
  float w[kMaxLH];
  int pg[kTile];
  uint32_t hs[kTile];  // stability history words of the tile's blocks (loaded with their pages)
  uint64_t keys[kTile];
  uint64_t wl[kWarps][32];
  int wn[kWarps];
  uint64_t run[2][kMaxK];
  uint64_t merge[kMergeSlots];
  int mcount[kMaxCluster];
  uint64_t bar;  // completion of the staged bulk copies
};

// D floats per row: each lane holds D/32 of them (plain loads: the row may be
// in global or shared memory).
template <int D>
struct RowSlice {
  static constexpr int kPer = D / 32;
  float v[kPer];
  __device__ __forceinline__ void load(const float* row, int lane) {
    const float* q = row + lane * kPer;
    if (kPer == 8) {
      const float4 a = reinterpret_cast<const float4*>(q)[0];
      const float4 b = reinterpret_cast<const float4*>(q)[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if (kPer == 4) {
      const float4 a = reinterpret_cast<const float4*>(q)[0];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if (kPer == 2) {
      const float2 a = reinterpret_cast<const float2*>(q)[0];
      v[0] = a.x; v[1] = a.y;
    } else {
      v[0] = q[0];
    }
  }
  // the same from global memory through the read-only path
  __device__ __forceinline__ void load_global(const float* row, int lane) {
    const float* q = row + lane * kPer;
    if (kPer == 8) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(q));
      const float4 b = __ldg(reinterpret_cast<const float4*>(q) + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if (kPer == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(q));
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if (kPer == 2) {
      const float2 a = __ldg(reinterpret_cast<const float2*>(q));
      v[0] = a.x; v[1] = a.y;
    } else {
      v[0] = __ldg(q);
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[e] = 0.f;
  }
};

// Sums NV values (a power of two, <= 32) across the warp at once: afterwards
// lane L holds in v[0] the warp total of value L % NV. A butterfly that keeps
// half of the values at every step: 31 shuffles for 32 values instead of
// 5 per value.
template <int NV>
__device__ __forceinline__ void warp_sum_transpose(float (&v)[NV], int lane) {
#pragma unroll
  for (int o = 16; o >= NV; o >>= 1)
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(kFull, v[i], o);
#pragma unroll
  for (int n = NV; n > 1; n >>= 1) {
    const int o = n >> 1;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

// The smallest key T such that exactly k of keys[0..n) (distinct, in shared
// memory) are >= T, k in [1, n]. Up to one key a thread: T is the key with
// k - 1 keys above it (one counting pass). Longer lists: a radix select on
// 8-bit digits from just below the bits every key shares, stopping as soon as
// a digit's bucket holds exactly the keys still needed. hist: 256 ints of
// shared memory; scal: 2 * kWarps + 3 words of shared memory. (Ranking up to
// two keys a thread from sorted warp runs by binary search was measured
// slower here: its searches are chains of dependent loads.)
__device__ __forceinline__ uint64_t block_kth_largest(const uint64_t* keys, int n, int k, int* hist,
                                                      uint64_t* scal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t* s_lo = scal;
  uint64_t* s_hi = scal + kWarps;
  uint64_t* s_res = scal + 2 * kWarps;
  int* s_sel = reinterpret_cast<int*>(scal + 2 * kWarps + 1);
  if (n <= kThreads) {
    if (tid < n) {
      const uint64_t key = keys[tid];
      int above = 0;
#pragma unroll 8
      for (int q = 0; q < n; ++q) above += keys[q] > key ? 1 : 0;
      if (above == k - 1) *s_res = key;
    }
    __syncthreads();
    const uint64_t res = *s_res;
    __syncthreads();
    return res;
  }
  uint64_t lo = ~0ull, hi = 0ull;
  for (int i = tid; i < n; i += kThreads) {
    const uint64_t key = keys[i];
    lo = key < lo ? key : lo;
    hi = key > hi ? key : hi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t x = __shfl_xor_sync(kFull, lo, o), y = __shfl_xor_sync(kFull, hi, o);
    lo = x < lo ? x : lo;
    hi = y > hi ? y : hi;
  }
  if (lane == 0) {
    s_lo[warp] = lo;
    s_hi[warp] = hi;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    lo = s_lo[w] < lo ? s_lo[w] : lo;
    hi = s_hi[w] > hi ? s_hi[w] : hi;
  }
  __syncthreads();  // s_lo / s_hi may be rewritten by the next call
  if (lo == hi) return lo;
  const int common = __clzll(lo ^ hi);
  uint64_t pmask = common == 0 ? 0ull : ~0ull << (64 - common);
  uint64_t prefix = hi & pmask;
  int need = k;
  for (int shift = 56 - common;; shift -= 8) {
    const int sh = shift < 0 ? 0 : shift;  // the last digit may overlap bits already fixed
    for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint64_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(int)((key >> sh) & 255)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      int local = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) local += hist[lane * 8 + b];
      int sfx = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(kFull, sfx, o);
        if (lane + o < 32) sfx += y;
      }
      int above = sfx - local;
      for (int b = 7; b >= 0; --b) {
        const int hb = hist[lane * 8 + b];
        if (above < need && above + hb >= need) {
          s_sel[0] = lane * 8 + b;
          s_sel[1] = above;
        }
        above += hb;
      }
    }
    __syncthreads();
    const int b = s_sel[0];
    need -= s_sel[1];
    prefix = (prefix & ~((uint64_t)0xFF << sh)) | ((uint64_t)b << sh);
    pmask |= (uint64_t)0xFF << sh;
    const bool exact = hist[b] == need;  // every key of this bucket is needed
    __syncthreads();
    if (exact || sh == 0) break;
  }
  return prefix;
}

// Block-wide exclusive prefix sum of one count a thread; returns this
// thread's offset and writes the total to *total. wsum: kWarps ints.
__device__ __forceinline__ int block_scan(int cnt, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    before += w < warp ? wsum[w] : 0;
    tot += wsum[w];
  }
  __syncthreads();  // wsum may be rewritten by the next call
  *total = tot;
  return before + incl - cnt;
}

template <typename T, int D, bool kFused>
__global__ void __launch_bounds__(kThreads, 2) step_kernel(StepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StepSmem<D>& sm = *reinterpret_cast<StepSmem<D>*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.splits;  // clusters per request
  const int r = blockIdx.y / S, sp = blockIdx.y - r * S;
  const int CL = (int)cluster_size();
  const int crank = CL > 1 ? (int)cluster_rank() : 0;
  const bool do_anchor = p.flags & kStepAnchor;
  const bool do_score = p.flags & kStepScore;
  const bool do_topk = p.flags & kStepTopK;
  const bool from_scores = p.flags & kStepTopKFromScores;
  const bool stab = p.hist != nullptr;  // keys ranked by stability (score mode only)
  const bool hier = p.hier_grid != nullptr;  // hierarchical selection (score mode, one cluster a request)
  // the decode token appended by this launch (one cluster a request, ring
  // mode): every CTA pools the token's Keys itself for the anchor; the CTA
  // that scores the token's block writes it and scores that block from
  // shared memory, so no other CTA waits for it
  constexpr bool fused = kFused;
  const int K = p.K;
  const int Kp = K <= 1 ? 1 : 1 << (32 - __clz(K - 1));  // next power of two >= K

  // launched early behind the previous kernel of the stream (for example the
  // decode step's append): wait for it before touching global memory. The
  // next kernel is not let in early: a following step kernel's clusters,
  // parked on the SMs, would keep this one's clusters from being placed
  // (measured: 32 requests x 8 CTAs back to back, 15.8 -> 20.8 us per step).
  pdl_wait();

  // The first remote shared-memory access must follow a cluster barrier that
  // every CTA has arrived at; arrive now, wait just before that access.
  bool start_waited = true;
  if (CL > 1) {
    cluster_arrive_relaxed();
    start_waited = false;
  }

  // ---- request metadata (uniform across the cluster) ---------------------
  const int off = p.bt.offsets[r];
  int nb = p.bt.offsets[r + 1] - off;
  int T_r = 0;
  bool bad = nb < 0 || nb > p.bt.max_blocks;
  if (do_anchor) {
    T_r = p.bt.seq_lens[r];
    const int bs = p.kc.bs;
    bad = bad || T_r < 0 || nb != (T_r + bs - 1) / bs;
  }
  if (bad) {
    if (tid == 0 && crank == 0) flag_error(p.err, kErrBadIndex);
    nb = 0;
    T_r = 0;
  }
  // this cluster's blocks (split sp of S), then this CTA's share of them
  const int span = (nb + S - 1) / S;
  const int s0 = min(nb, sp * span), sn = min(nb, s0 + span) - s0;
  const int chunk = (sn + CL - 1) / CL;
  const int j0 = s0 + min(sn, crank * chunk);
  const int j1 = s0 + min(sn, crank * chunk + chunk);

  // fused append: `owner` (this CTA scores the token's block, the request's
  // last) writes the token and keeps the block's new v_b row in shared
  // memory (sm.part[1]). The token's page is loaded here and checked once the
  // bulk copies are issued, so that its latency overlaps theirs.
  const bool f_on = fused && !bad && T_r >= 1;
  const int f_t = T_r - 1;
  const bool owner = f_on && j0 <= nb - 1 && nb - 1 < j1;
  const int f_page_raw = f_on ? p.bt.pages[off + nb - 1] : -1;
  if (fused && !bad && T_r < 1 && crank == 0 && tid == 0) flag_error(p.err, kErrBadIndex);  // no token

  // ---- prefetch: one round of page-id loads for the anchor's token rows and
  // the first tile's blocks, then bulk copies of that tile's v_b rows -------
  constexpr bool kAnchorFits = D <= 32 * Vec16<T>::kElems;  // a row is at most 32 vectors
  const bool ring = p.ring_rows != nullptr;                 // anchor from the anchor ring
  const int w_eff = min(p.W, T_r);
  if (kAnchorFits && do_anchor && !ring) {
    constexpr int ES = elem_bytes<T>();
    for (int i = tid; i < w_eff; i += kThreads) {
      const int pos = T_r - w_eff + i;
      const int pgid = p.bt.pages[off + pos / p.kc.bs];
      if (pgid < 0 || pgid >= p.kc.num_pages) {
        flag_error(p.err, kErrBadIndex);
        sm.tok[i] = -1;
      } else {
        sm.tok[i] = ((long long)pgid * p.kc.sP + (long long)(pos % p.kc.bs) * p.kc.sT) * ES;
      }
    }
    if (p.head_w)
      for (int s = tid; s < p.kc.L * p.kc.H; s += kThreads)
        sm.w[s] = p.head_w[(long long)r * p.kc.L * p.kc.H + s];
  }
  const int nstage = (do_score && !hier) ? min(kStage, j1 - j0) : 0;
  const int skip = owner ? nb - 1 - j0 : -1;  // the owner's fresh row is not copied
  if (do_score) {
    const int t0count = hier ? 0 : min(kTile, j1 - j0);  // hier: the blocks are known after its levels
    int pg = -1;
    uint32_t hw = 0u;
    if (tid < t0count) {
      pg = p.bt.pages[off + j0 + tid];
      if (stab) hw = p.hist[off + j0 + tid];  // in the same round trip as the page
      if (pg < 0 || pg >= p.vb_rows) {
        flag_error(p.err, kErrBadIndex);
        pg = -1;
      }
    }
    sm.pg[tid] = pg;
    sm.hs[tid] = hw;
    if (tid == 0) {
      mbar_init(&sm.bar, 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (do_score) {
    if (warp == 0 && nstage > 0) {
      int valid = 0;
      for (int i = lane; i < nstage; i += 32) valid += (sm.pg[i] >= 0 && i != skip) ? 1 : 0;
      valid = __reduce_add_sync(kFull, valid);
      if (lane == 0) mbar_arrive_expect_tx(&sm.bar, (uint32_t)(valid * D * sizeof(float)));
      __syncwarp();
      for (int i = lane; i < nstage; i += 32)
        if (sm.pg[i] >= 0 && i != skip)
          bulk_g2s(&sm.stage[i][0], p.vb + (long long)sm.pg[i] * D, D * sizeof(float), &sm.bar);
    }
  }

  // ---- stage 1: anchor -----------------------------------------------------
  if (do_anchor && ring) {
    // Every CTA sums the W' newest ring rows itself (W' * D floats, mostly
    // from L2): thread (rr, c4) takes the 16-byte column c4 of rows rr,
    // rr + RP, ..., loading each row's slot position and values together (one
    // round trip a batch); a row whose slot does not hold the expected token
    // counts as zero and is reported. The RP partial rows are then added
    // through shared memory (the token-offset table is not used in this mode).
    // With the fused append, the newest row is the decode token's, pooled
    // by this CTA (sm.part[0]) and added in its place.
    constexpr int V4 = D / 4, RP = kThreads / V4;
    constexpr int kRowUnroll = 4;
    const int c4 = tid % V4, rr = tid / V4;
    const long long rbase = (long long)r * p.ring_slots;
    const float4* rows4 = reinterpret_cast<const float4*>(p.ring_rows);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[kRowUnroll];
    int ps[kRowUnroll], tt[kRowUnroll];
    auto load_rows = [&](int i0) {
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int i = i0 + u * RP;
        const bool valid = i < w_eff;
        const bool fresh = fused && i == 0;
        tt[u] = T_r - 1 - i;
        const long long slot = rbase + (valid ? tt[u] % p.ring_slots : 0);
        ps[u] = valid ? (fresh ? tt[u] : __ldg(p.ring_pos + slot)) : -2;
        v[u] = (valid && !fresh) ? __ldg(rows4 + slot * V4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    // fused append: the token is pooled first, while the bulk copies are in
    // flight (loading the first ring rows ahead of it as well was measured no
    // faster, and holds more registers)
    const int f_page = (fused && f_page_raw >= 0 && f_page_raw < p.kc.num_pages) ? f_page_raw : -1;
    if constexpr (D <= 32 * Vec16<T>::kElems) {  // a row of the cache is at most 32 vectors
      if (fused) {
        static_assert(sizeof(sm.tok) >= kThreads * Vec16<T>::kElems * sizeof(float), "pooling scratch");
        if (f_on && f_page < 0 && crank == 0 && tid == 0) flag_error(p.err, kErrBadIndex);
        const bool writer = owner && f_page >= 0;
        const float f_old = writer ? load_old_sum(p.block_sum, f_page, f_t, p.kc.bs, D) : 0.f;
        if (f_page >= 0) {
          // sm.part[0]: the token's pooled row (the newest row of the anchor);
          // sm.tok is local scratch here (the ring anchor reuses it after).
          // The token's Keys go into the cache slot from every CTA of the
          // cluster, 1/CL of the (layer, head) slices each (measured, 7B-like:
          // the 28 KB store adds 1.1 us to the step from one CTA, 0.8 us
          // shared; the same store into an L2-resident buffer adds 0.1 us).
          pool_token<T, D, kThreads>(p.kc, r, p.k_new, p.head_w, f_page, f_t % p.kc.bs, sp * CL + crank, S * CL,
                                     reinterpret_cast<float*>(sm.tok), &sm.part[0][0]);
          if (writer) {
            const Ring ring_w{const_cast<float*>(p.ring_rows), const_cast<int*>(p.ring_pos), p.ring_slots};
            const float vb_new = commit_token(r, f_page, f_t, p.kc.bs, p.kc.L * p.kc.H, p.head_w != nullptr, D,
                                              f_old, &sm.part[0][0], p.block_sum, const_cast<float*>(p.vb), ring_w);
            if (tid < D) sm.part[1][tid] = vb_new;  // read after the anchor's barriers
          }
        } else if (tid < D) {
          sm.part[0][tid] = 0.f;  // no token was written (reported): its row counts as zero
        }
      }
    }
    for (int i0 = rr; i0 < w_eff; i0 += RP * kRowUnroll) {
      load_rows(i0);
      if (fused && i0 == 0) v[0] = reinterpret_cast<const float4*>(&sm.part[0][0])[c4];  // the newest row
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        if (ps[u] == tt[u]) {
          acc.x += v[u].x;
          acc.y += v[u].y;
          acc.z += v[u].z;
          acc.w += v[u].w;
        } else if (ps[u] != -2 && c4 == 0) {
          flag_error(p.err, kErrBadIndex);
        }
      }
    }
    float4* red = reinterpret_cast<float4*>(sm.tok);
    red[tid] = acc;
    __syncthreads();
    const int LH = p.kc.L * p.kc.H;
    const float scale =
        w_eff > 0 ? (p.head_w ? 1.f / (float)w_eff : 1.f / ((float)w_eff * (float)LH)) : 0.f;
    if (tid < D) {
      const float* redf = reinterpret_cast<const float*>(red);
      float v = 0.f;
#pragma unroll 8
      for (int q = 0; q < RP; ++q) v += redf[(q * V4 + tid / 4) * 4 + (tid & 3)];
      v *= scale;
      sm.va[tid] = v;
      if (crank == 0 && sp == 0 && p.va_out) p.va_out[(long long)r * D + tid] = v;
    }
    __syncthreads();
  } else if (kAnchorFits && do_anchor) {
    constexpr int EPV = Vec16<T>::kElems;
    constexpr int V16 = kAnchorFits ? D / EPV : 32;
    constexpr int RPW = 32 / V16;
    constexpr int ES = elem_bytes<T>();
    const int vec = lane % V16, tl = lane / V16;
    const int LH = p.kc.L * p.kc.H;

    // Warp w of CTA crank takes the (layer, head) slices crank + CL * (w +
    // kWarps * k), two at a time: both slices' token rows are loaded before
    // either is summed, so a warp waits for memory once per pair.
    constexpr int kUnroll = 8;
    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
    const char* kbase = reinterpret_cast<const char*>(p.kc.base) + vec * 16;
    const int sstride = CL * kWarps;
    for (int s = crank + CL * warp; s < LH; s += 2 * sstride) {
      const int s2 = s + sstride;
      const bool has2 = s2 < LH;
      const int l = s / p.kc.H, h = s - l * p.kc.H;
      const int l2 = has2 ? s2 / p.kc.H : 0, h2 = has2 ? s2 - l2 * p.kc.H : 0;
      const char* sbase = kbase + ((long long)l * p.kc.sL + (long long)h * p.kc.sH) * ES;
      const char* sbase2 = kbase + ((long long)l2 * p.kc.sL + (long long)h2 * p.kc.sH) * ES;
      float ps[EPV], ps2[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        ps[e] = 0.f;
        ps2[e] = 0.f;
      }
      for (int i0 = 0; i0 < w_eff; i0 += kUnroll * RPW) {
        uint4 v[kUnroll], v2[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = i0 + u * RPW + tl;
          const long long o = (i < w_eff) ? sm.tok[i] : -1;
          v[u] = ld_stream16(sbase + (o >= 0 ? o : 0), o >= 0);
          v2[u] = ld_stream16(sbase2 + (o >= 0 ? o : 0), has2 && o >= 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          float f[EPV], f2[EPV];
          Vec16<T>::unpack(v[u], f);
          Vec16<T>::unpack(v2[u], f2);
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            ps[e] += f[e];
            ps2[e] += f2[e];
          }
        }
      }
      const float wt = p.head_w ? sm.w[s] : 1.f;
      const float wt2 = has2 ? (p.head_w ? sm.w[s2] : 1.f) : 0.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[e] = fmaf(wt2, ps2[e], fmaf(wt, ps[e], acc[e]));
    }
#pragma unroll
    for (int e = 0; e < EPV; ++e)
#pragma unroll
      for (int o = V16; o < 32; o <<= 1) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
    if (tl == 0) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) sm.wpart[warp][vec * EPV + e] = acc[e];
    }
    __syncthreads();
    float c = 0.f;
    if (tid < D) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) c += sm.wpart[w][tid];
    }
    if (CL > 1) {
      cluster_wait_acquire();  // every CTA of the cluster has started
      start_waited = true;
      if (tid < D) {
        const uint32_t a = smem_u32(&sm.part[crank][tid]);
        for (int dst = 0; dst < CL; ++dst) st_cluster_f32(map_to_rank(a, dst), c);
      }
      cluster_arrive_release();
      cluster_wait_acquire();
    } else {
      if (tid < D) sm.part[0][tid] = c;
      __syncthreads();
    }
    const float scale =
        w_eff > 0 ? (p.head_w ? 1.f / (float)w_eff : 1.f / ((float)w_eff * (float)LH)) : 0.f;
    if (tid < D) {
      float v = 0.f;
      for (int q = 0; q < CL; ++q) v += sm.part[q][tid];
      v *= scale;
      sm.va[tid] = v;
      if (crank == 0 && sp == 0 && p.va_out) p.va_out[(long long)r * D + tid] = v;
    }
    __syncthreads();
  } else if (do_score) {
    if (tid < D) sm.va[tid] = p.va_in[(long long)r * D + tid];
    __syncthreads();
  }

  // ---- hierarchical selection: the Grid and Chunk levels -----------------
  // Every CTA of the request's cluster runs both coarse levels itself (their
  // rows are few), so they need no exchange between the CTAs: score every
  // Grid, keep the best share; list the Chunks of the kept Grids, score them,
  // keep the best share. The blocks of the kept Chunks are then scored and
  // ranked below as the table of stage 2, each CTA of the request (all its
  // clusters) taking an equal run of their block positions (a few kept
  // Chunks are then spread over every CTA: measured, 32 requests x 1024
  // blocks, dealing whole Chunks left 2 of a request's 8 CTAs scoring 64
  // blocks each while the others waited). The block level keeps
  // kp = ceil(n * permille / 1000) of its n blocks; its best min(K, kp) are
  // written.
  int h_lo = 0, h_hi = 0;  // hier: this CTA's block positions in the kept Chunks (ids ascending in hchunks)
  int Kout = K;  // output slots filled with blocks
  int* hchunks = reinterpret_cast<int*>(sm.tok);
  static_assert(sizeof(sm.tok) >= kHierKeptChunks * sizeof(int), "every kept Chunk of a request is listed");
  if (hier) {
    const int NT = S * CL, gi = sp * CL + crank;  // CTAs of the request, and this one's place among them
    const int cp = p.chunk_pages, gc = p.grid_chunks;
    const int C = nb > 0 ? (nb + cp - 1) / cp : 0;
    const int G = C > 0 ? (C + gc - 1) / gc : 0;
    uint64_t* mk = reinterpret_cast<uint64_t*>(&sm.stage[0][0]);  // member list / keys of a level
    uint32_t* gbits = reinterpret_cast<uint32_t*>(&sm.wl[0][0]);  // kept Grids
    int* hist = reinterpret_cast<int*>(&sm.run[0][0]);
    uint64_t* scal = &sm.run[1][0];
    int* wsum = reinterpret_cast<int*>(&sm.run[1][64]);
    RowSlice<D> av;
    av.load(sm.va, lane);
    float t2 = 0.f;
#pragma unroll
    for (int e = 0; e < RowSlice<D>::kPer; ++e) t2 = fmaf(av.v[e], av.v[e], t2);
    const float na2 = warp_sum(t2), na = sqrtf(na2);
    // keys of members [0, n) into mk[0, n): member(i, &row, &id) names the
    // member's representation row and its id (for the Chunk list, mk[i]
    // holds the id until its key overwrites it); kR rows a warp per
    // transposed reduction
    constexpr int kR = D <= 128 ? 16 : 8;
    auto score_level = [&](int n, auto&& member) {
      for (int base = warp * kR; base < n; base += kWarps * kR) {
        RowSlice<D> b[kR];
        uint32_t id[kR];
#pragma unroll
        for (int u = 0; u < kR; ++u) {
          const int i = base + u;
          // slots past n load a fixed valid row (their result is dropped);
          // member() is asked only for real members, since a slot's id may
          // already have been overwritten by its key in the Chunk-list mode
          const float* row = p.hier_grid;
          id[u] = 0u;
          if (i < n) member(i, &row, &id[u]);
          b[u].load_global(row, lane);
        }
        float part[2 * kR];
#pragma unroll
        for (int u = 0; u < kR; ++u) {
          float dot = 0.f, n2 = 0.f;
#pragma unroll
          for (int e = 0; e < RowSlice<D>::kPer; ++e) {
            dot = fmaf(av.v[e], b[u].v[e], dot);
            n2 = fmaf(b[u].v[e], b[u].v[e], n2);
          }
          part[u] = dot;
          part[kR + u] = n2;
        }
        warp_sum_transpose<2 * kR>(part, lane);
        const float n2 = __shfl_down_sync(kFull, part[0], kR);
        uint32_t my_id = 0u;
#pragma unroll
        for (int u = 0; u < kR; ++u) my_id = lane == u ? id[u] : my_id;
        __syncwarp();  // every lane has read its ids before any key overwrites them
        if (lane < kR && base + lane < n) {
          float cosv = 0.f;
          if (na2 > 0.f && n2 > 0.f) cosv = part[0] / (na * sqrtf(n2));
          cosv = fminf(1.f, fmaxf(-1.f, cosv));
          mk[base + lane] = make_key(fmaf(0.5f, cosv, 0.5f), my_id);
        }
      }
      __syncthreads();
    };
    const float* grid_rows = p.hier_grid + (long long)r * p.g_max * D;
    const float* chunk_rows = p.hier_chunk + (long long)r * p.c_max * D;
    // Grid level. When the Grids and every Chunk fit in two rounds of row
    // loads, the Chunks are scored with the Grids (keys at mk[G + c]) and
    // those outside the kept Grids are dropped afterwards: no wait for the
    // Grid selection before the Chunks' rows are loaded, and no Chunk list.
    const bool all_chunks = G + C <= 2 * kWarps * kR;
    static_assert(2 * kWarps * 16 <= kThreads, "a thread a Chunk in the single pass below");
    if (all_chunks)
      score_level(G + C, [&](int i, const float** row, uint32_t* id) {
        *id = (uint32_t)(i < G ? i : i - G);
        *row = (i < G ? grid_rows : chunk_rows) + (long long)*id * D;
      });
    else
      score_level(G, [&](int i, const float** row, uint32_t* id) {
        *id = (uint32_t)i;
        *row = grid_rows + (long long)i * D;
      });
    const int kg = (int)(((long long)G * p.permille[0] + 999) / 1000);
    const uint64_t thr_g = G > 0 ? block_kth_largest(mk, G, kg, hist, scal) : ~0ull;
    if (!all_chunks) {  // the kept Grids as bits (the single-round path reads the Grid keys instead)
      for (int w = tid; w < (G + 31) / 32; w += kThreads) gbits[w] = 0u;
      __syncthreads();
      for (int i = tid; i < G; i += kThreads)
        if (mk[i] >= thr_g) atomicOr(&gbits[i >> 5], 1u << (i & 31));
      __syncthreads();
    }
    // Chunk level: the Chunks of the kept Grids (ids ascending), nc of them,
    // their keys ck[0, ncand)
    int nc = 0, ncand = 0;
    uint64_t* ck = mk;
    if (all_chunks) {
      ck = mk + G;
      ncand = C;
      bool in = false;
      for (int c = tid; c < C; c += kThreads) {  // C <= 2 * kWarps * kR <= kThreads: one pass
        in = mk[c / gc] >= thr_g;  // its Grid is kept
        if (!in) ck[c] = 0ull;  // below every key
      }
      nc = __syncthreads_count(in);
    } else {
      for (int g0 = 0; g0 < G; g0 += kThreads) {
        const int g = g0 + tid;
        const int cnt = (g < G && ((gbits[g >> 5] >> (g & 31)) & 1u)) ? min(gc, C - g * gc) : 0;
        int tot;
        const int at = nc + block_scan(cnt, wsum, &tot);
        for (int c = 0; c < cnt; ++c) mk[at + c] = (uint64_t)(uint32_t)(g * gc + c);
        nc += tot;
      }
      __syncthreads();
      score_level(nc, [&](int i, const float** row, uint32_t* id) {
        *id = (uint32_t)mk[i];
        *row = chunk_rows + (long long)*id * D;
      });
      ncand = nc;
    }
    const int kc = (int)(((long long)nc * p.permille[1] + 999) / 1000);
    const uint64_t thr_c = nc > 0 ? block_kth_largest(ck, ncand, kc, hist, scal) : ~0ull;
    // the kept Chunks in id order, and the blocks they hold
    int* s_nact = wsum + kWarps;
    if (tid == 0) *s_nact = 0;
    int nkept = 0;
    for (int i0 = 0; i0 < ncand; i0 += kThreads) {
      const int i = i0 + tid;
      const bool keep = i < ncand && ck[i] >= thr_c;
      const int c = keep ? (int)key_index(ck[i]) : 0;
      int tot;
      const int at = nkept + block_scan(keep ? 1 : 0, wsum, &tot);  // its syncs also order s_nact's zeroing
      if (keep) {
        hchunks[at] = c;  // at most kHierKeptChunks, checked by the caller
        atomicAdd(s_nact, min(cp, nb - c * cp));
      }
      nkept += tot;
    }
    __syncthreads();
    const int nact = *s_nact;
    const int ptot = nkept * cp;  // positions; those past the request's last block map to no block
    const int span = (ptot + NT - 1) / NT;
    h_lo = min(ptot, gi * span);
    h_hi = min(ptot, h_lo + span);
    const int kp = (int)(((long long)nact * p.permille[2] + 999) / 1000);
    Kout = min(K, kp);
    if (sp == 0 && crank == 0 && tid == 0 && p.kept) p.kept[r] = kp;
    __syncthreads();
  }
  // stage 2's table: blocks [j0, j1) of the request, or (hier) positions
  // [h_lo, h_hi) of the kept Chunks' blocks, position v -> block
  // hier_block(v) (-1 past the request's end)
  const int t_lo = hier ? h_lo : j0;
  const int t_hi = hier ? h_hi : j1;
  auto hier_block = [&](int v) {
    const int q = v / p.chunk_pages;
    const int j = hchunks[q] * p.chunk_pages + (v - q * p.chunk_pages);
    return j < nb ? j : -1;
  };

  // ---- stage 2: scores and the CTA's top-K over its share of the blocks --
  // Running top-K list: sm.run[cur][0..Kp), descending, zero-padded.
  int run_n = 0, cur = 0;
  // Few blocks per CTA: no per-CTA list; stage 3 all-gathers the raw keys
  // and every CTA ranks its own by counting.
  constexpr int kDirectMax = 64;
  const bool direct = do_topk && CL > 1 && S == 1 && chunk <= kDirectMax && !hier;
  if (do_topk)
    for (int i = tid; i < Kp; i += kThreads) sm.run[0][i] = 0ull;
  if (do_score || from_scores) {
    RowSlice<D> a;
    float na2 = 0.f;
    bool staged_ok = true;
    if (do_score) {
      a.load(sm.va, lane);
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < RowSlice<D>::kPer; ++e) t = fmaf(a.v[e], a.v[e], t);
      na2 = warp_sum(t);
      if (nstage > 0 && !mbar_wait_bounded(&sm.bar, 0, p.wait_ns)) {
        staged_ok = false;
        if (tid == 0) flag_error(p.err, kErrTimeout);
      }
    }
    const float na = sqrtf(na2);
    for (int tile0 = t_lo; tile0 < t_hi; tile0 += kTile) {
      const int tcount = min(kTile, t_hi - tile0);
      const bool first = tile0 == t_lo;
      if (do_score) {
        if (!first || hier) {
          int pg = -1;
          uint32_t hw = 0u;
          if (tid < tcount) {
            const int jt = hier ? hier_block(tile0 + tid) : tile0 + tid;
            if (jt >= 0) {
              pg = p.bt.pages[off + jt];
              if (stab) hw = p.hist[off + jt];
              if (pg < 0 || pg >= p.vb_rows) {
                flag_error(p.err, kErrBadIndex);
                pg = -1;
              }
            }
          }
          sm.pg[tid] = pg;
          sm.hs[tid] = hw;
          __syncthreads();
        }
        // warp w scores tile slots w, w + 8, w + 16, ...; kRows rows in
        // flight (4 when the tile has at most 4 rows a warp, so that small
        // tiles do not pay for a 32-value reduction)
        auto score_rows = [&](auto rows_c) {
          constexpr int kRows = decltype(rows_c)::value;
          for (int base = warp; base < tcount; base += kWarps * kRows) {
            RowSlice<D> b[kRows];
#pragma unroll
            for (int u = 0; u < kRows; ++u) {
              // always load (row 0 for empty slots, masked below): no branch, so
              // all kRows rows are in flight together
              const int slot = base + u * kWarps;
              const int pg = slot < tcount ? sm.pg[slot] : -1;
              const bool staged = first && slot < nstage;
              const bool fresh = owner && tile0 + slot == nb - 1;  // written by this launch
              if (fresh) {
                b[u].load(&sm.part[1][0], lane);
              } else if (staged) {
                b[u].load(&sm.stage[slot][0], lane);  // bulk-copied into shared memory
              } else {
                b[u].load_global(p.vb + (long long)(pg < 0 ? 0 : pg) * D, lane);
              }
              if (pg < 0 || (staged && !fresh && !staged_ok)) b[u].zero();
            }
            // per-lane partial dots and squared norms of the kRows rows, then
            // one transposed reduction: lane u ends with row u's dot, lane
            // kRows + u with its squared norm
            float part[2 * kRows];
#pragma unroll
            for (int u = 0; u < kRows; ++u) {
              float dot = 0.f, n2 = 0.f;
#pragma unroll
              for (int e = 0; e < RowSlice<D>::kPer; ++e) {
                dot = fmaf(a.v[e], b[u].v[e], dot);
                n2 = fmaf(b[u].v[e], b[u].v[e], n2);
              }
              part[u] = dot;
              part[kRows + u] = n2;
            }
            warp_sum_transpose<2 * kRows>(part, lane);
            const float n2 = __shfl_down_sync(kFull, part[0], kRows);
            const int u = lane;
            const int slot = base + u * kWarps;
            if (u < kRows && slot < tcount) {
              const float dot = part[0];
              float cosv = 0.f;
              if (na2 > 0.f && n2 > 0.f) cosv = dot / (na * sqrtf(n2));
              cosv = fminf(1.f, fmaxf(-1.f, cosv));
              const float sc = fmaf(0.5f, cosv, 0.5f);
              const int j = hier ? hier_block(tile0 + slot) : tile0 + slot;
              if (p.scores_out && j >= 0) p.scores_out[off + j] = sc;
              uint64_t key = 0ull;
              if (sm.pg[slot] >= 0) {
                if (p.hist) {
                  // stability filter: shift this step's bit into the block's window
                  const uint32_t wmask = p.stab_w >= 32 ? 0xFFFFFFFFu : ((1u << p.stab_w) - 1u);
                  const uint32_t h = ((sm.hs[slot] << 1) | (sc > p.stab_theta ? 1u : 0u)) & wmask;
                  p.hist[off + j] = h;
                  if (p.stab_out) p.stab_out[off + j] = (float)__popc(h) / (float)p.stab_w;
                  key = make_stab_key((uint32_t)__popc(h), sc, (uint32_t)j);
                } else {
                  key = make_key(sc, (uint32_t)j);
                }
              }
              sm.keys[slot] = key;
            }
          }
        };
        if (tcount <= kWarps * 4)
          score_rows(std::integral_constant<int, 4>());
        else
          score_rows(std::integral_constant<int, (D <= 128 ? 16 : 8)>());
      } else {
        const int j = tile0 + tid;
        sm.keys[tid] = (tid < tcount) ? make_key(p.scores_in[off + j], (uint32_t)j) : 0ull;
      }
      __syncthreads();
      if (!do_topk || direct) continue;
      // merge this tile into the running list
      uint64_t key = tid < tcount ? sm.keys[tid] : 0ull;
      const uint64_t thr = (run_n == K) ? sm.run[cur][K - 1] : 0ull;
      if (key <= thr) key = 0ull;
      if (!__syncthreads_or(key != 0ull)) continue;
      key = warp_sort_desc(key, lane);
      sm.wl[warp][lane] = key;
      const int cnt = __popc(__ballot_sync(kFull, key != 0ull));
      if (lane == 0) sm.wn[warp] = cnt;
      const int nxt = cur ^ 1;
      for (int i = tid; i < Kp; i += kThreads) sm.run[nxt][i] = 0ull;
      __syncthreads();
      // rank in the union = number of larger keys in every list (own list included)
      if (key != 0ull) {
        int pos[kWarps];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) pos[w] = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1)
#pragma unroll
          for (int w = 0; w < kWarps; ++w) pos[w] += (sm.wl[w][pos[w] + step] > key) ? step : 0;
        int rank = count_greater_pow2(sm.run[cur], Kp, key);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) rank += (sm.wl[w][0] > key) ? pos[w] + 1 : 0;
        if (rank < K) sm.run[nxt][rank] = key;
      }
      if (tid < run_n) {
        const uint64_t x = sm.run[cur][tid];
        int pos[kWarps];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) pos[w] = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1)
#pragma unroll
          for (int w = 0; w < kWarps; ++w) pos[w] += (sm.wl[w][pos[w] + step] > x) ? step : 0;
        int rank = tid;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) rank += (sm.wl[w][0] > x) ? pos[w] + 1 : 0;
        if (rank < K) sm.run[nxt][rank] = x;
      }
      int total = run_n;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) total += sm.wn[w];
      __syncthreads();
      run_n = min(K, total);
      cur = nxt;
    }
  }

  // ---- stage 3: merge the CTAs' lists and write the request's top-K ------
  if (do_topk) {
    int* idx_out = p.idx_out + (long long)r * K;
    float* top_out = p.top_out ? p.top_out + (long long)r * K : nullptr;
    // the place of a ranked key: the request's output, or (a split request)
    // this cluster's sorted list in the scratch
    uint64_t* slist = S > 1 ? p.split_keys + ((long long)r * p.split_cap + sp) * Kp : nullptr;
    // the compact table (sel_pages): each output's logical index also goes
    // to CTA 0 of the cluster (its sm.wl, free once every CTA has passed the
    // all-gather barrier), which orders them there
    // with its page (read by the CTA that scored the block, so mostly from
    // its L1)
    int* sel_v = reinterpret_cast<int*>(&sm.wl[0][0]);
    int* sel_p = sel_v + kMaxK;
    static_assert(sizeof(sm.wl) >= 2 * kMaxK * sizeof(int), "compact-table staging");
    auto note_sel = [&](int rank, int v) {
      if (!p.sel_pages) return;
      const int pg = p.bt.pages[off + v];
      if (CL == 1) {
        sel_v[rank] = v;
        sel_p[rank] = pg;
      } else {
        st_cluster_s32(map_to_rank(smem_u32(&sel_v[rank]), 0), v);
        st_cluster_s32(map_to_rank(smem_u32(&sel_p[rank]), 0), pg);
      }
    };
    int n_sel = 0;  // outputs filled (CTA 0)
    auto emit = [&](int rank, uint64_t k) {
      if (slist) {
        slist[rank] = k;
      } else {
        const int v = (int)(stab ? stab_key_index(k) : key_index(k));
        idx_out[rank] = v;
        if (top_out) top_out[rank] = stab ? stab_key_score(k) : key_score(k);
        note_sel(rank, v);
      }
    };
    auto pad = [&](int from) {
      if (slist) {
        for (int i = from + tid; i < Kp; i += kThreads) slist[i] = 0ull;
      } else {
        for (int i = from + tid; i < K; i += kThreads) {
          idx_out[i] = -1;
          if (top_out) top_out[i] = -__int_as_float(0x7f800000);
        }
      }
    };
    if (CL == 1) {
      const int nout = min(run_n, Kout);
      for (int i = tid; i < nout; i += kThreads) emit(i, sm.run[cur][i]);
      pad(nout);
      n_sel = nout;
    } else if (direct) {
      if (!start_waited) {
        cluster_wait_acquire();
        start_waited = true;
      }
      // all-gather of the raw keys (zero for blocks with a bad page): CTA c's
      // j1 - j0 keys at merge[c * chunk ...], its count of real keys in mcount
      const int mine = j1 - j0;
      if (mine > 0)
        for (int f = tid; f < CL * mine; f += kThreads) {
          const int dst = f / mine, i = f - dst * mine;
          st_cluster_u64(map_to_rank(smem_u32(&sm.merge[crank * chunk + i]), dst), sm.keys[i]);
        }
      const int nv = __syncthreads_count(tid < mine && sm.keys[tid] != 0ull);
      if (tid < CL) st_cluster_s32(map_to_rank(smem_u32(&sm.mcount[crank]), tid), nv);
      cluster_arrive_release();
      cluster_wait_acquire();
      // rank of each own key = the keys above it in the union; tpk threads
      // (consecutive lanes) per key split the count
      int tpk = 1;
      while (tpk < 32 && tpk * 2 * max(1, mine) <= kThreads) tpk <<= 1;
      const int ki = tid / tpk, part = tid & (tpk - 1);
      const uint64_t k = ki < mine ? sm.keys[ki] : 0ull;
      // CTA c's keys end where CTA c + 1's begin, so the union is merge[0, nb)
      int cnt = 0;
      if (k != 0ull)
        for (int j = part; j < nb; j += 8 * tpk) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int jj = j + u * tpk;
            cnt += (jj < nb && sm.merge[jj] > k) ? 1 : 0;
          }
        }
      for (int o = 1; o < tpk; o <<= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
      if (k != 0ull && part == 0 && cnt < K) emit(cnt, k);
      if (crank == 0) {
        int total = 0;
        for (int q = 0; q < CL; ++q) total += sm.mcount[q];
        for (int i = total + tid; i < K; i += kThreads) {
          idx_out[i] = -1;
          if (top_out) top_out[i] = -__int_as_float(0x7f800000);
        }
        n_sel = min(total, K);
      }
    } else {
      if (!start_waited) {
        cluster_wait_acquire();
        start_waited = true;
      }
      // all-gather: every CTA receives every CTA's zero-padded sorted list
      for (int f = tid; f < CL * Kp; f += kThreads) {
        const int dst = f / Kp, i = f - dst * Kp;
        st_cluster_u64(map_to_rank(smem_u32(&sm.merge[crank * Kp + i]), dst), sm.run[cur][i]);
      }
      if (tid < CL) st_cluster_s32(map_to_rank(smem_u32(&sm.mcount[crank]), tid), run_n);
      cluster_arrive_release();
      cluster_wait_acquire();
      // Each CTA ranks its own candidates in the union: a group of CL lanes
      // per candidate, one lane per list, counts summed with shuffles.
      const int list = lane & (CL - 1);
      const int per_warp = 32 / CL;
      for (int c0 = warp * per_warp; c0 < run_n; c0 += kWarps * per_warp) {
        const int c = c0 + lane / CL;
        const bool have = c < run_n;
        const uint64_t k = have ? sm.merge[crank * Kp + c] : ~0ull;
        int cnt = count_greater_pow2(&sm.merge[list * Kp], Kp, k);
        for (int o = 1; o < CL; o <<= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
        if (have && list == 0 && cnt < Kout) emit(cnt, k);
      }
      if (crank == 0) {
        int total = 0;
        for (int q = 0; q < CL; ++q) total += sm.mcount[q];
        pad(min(total, Kout));
        n_sel = min(total, Kout);
      }
    }
    // the compact table of the output (kk_compact_table), written by one CTA
    // that holds the n selected logical indices sv[] and their pages spg[]
    // by output rank: each goes to the place given by the number of smaller
    // indices (they are distinct), tpk threads an entry splitting the count
    auto write_compact = [&](const int* sv, const int* spg, int n) {
      int tpk = 1;
      while (tpk < 32 && tpk * 2 * max(1, n) <= kThreads) tpk <<= 1;
      const int e = tid / tpk, part = tid & (tpk - 1);
      const int v = e < n ? sv[e] : -1;
      const int pgv = (v >= 0 && part == 0) ? spg[e] : -1;
      int rank = 0;
      if (v >= 0)
        for (int u = part; u < n; u += tpk) rank += sv[u] < v ? 1 : 0;
      for (int o = 1; o < tpk; o <<= 1) rank += __shfl_xor_sync(kFull, rank, o);
      int* sp_out = p.sel_pages + (long long)r * K;
      int* sl_out = p.sel_logical ? p.sel_logical + (long long)r * K : nullptr;
      if (v >= 0 && part == 0) {
        sp_out[rank] = pgv;
        if (sl_out) sl_out[rank] = v;
      }
      for (int i = n + tid; i < K; i += kThreads) {
        sp_out[i] = -1;
        if (sl_out) sl_out[i] = -1;
      }
      if (tid == 0 && p.sel_count) p.sel_count[r] = n;
    };
    if (p.sel_pages && S == 1) {
      // CTA 0 of the cluster received every output's index and page
      if (CL > 1) {
        cluster_arrive_release();
        cluster_wait_acquire();
      } else {
        __syncthreads();
      }
      if (crank == 0) write_compact(sel_v, sel_p, n_sel);
    }
    if (S > 1) {
      // Every CTA has written its part of this cluster's list: fence, meet,
      // then one thread counts this cluster in. The last cluster of the
      // request merges the S sorted lists and resets the counter.
      __threadfence();
      if (CL > 1) {
        if (!start_waited) {
          cluster_wait_acquire();
          start_waited = true;
        }
        cluster_arrive_release();
        cluster_wait_acquire();
      } else {
        __syncthreads();
      }
      if (crank == 0) {
        // count this cluster in; the last one merges and sets the counter
        // back to zero for the next call (a count at or past S means the
        // workspace was not zeroed before its first use: reported)
        if (tid == 0) {
          const unsigned long long seen = atomicAdd(p.split_ctr + r, 1ull);
          if (seen >= (unsigned long long)S) flag_error(p.err, kErrBadIndex);
          sm.wn[0] = seen == (unsigned long long)(S - 1) ? 1 : 0;
        }
        __syncthreads();
        if (sm.wn[0]) {
          __threadfence();
          const uint64_t* lists = p.split_keys + (long long)r * p.split_cap * Kp;
          if (Kp <= 32) {
            // each warp folds lists warp, warp + 8, ... (up to kSplitPerWarp,
            // loaded together into its shared-memory slots) into one
            // descending 32-key list, keeping the larger 32 of each pair;
            // then the eight results fold as a tree (4, 2, 1 warps). The
            // folds are loops, not unrolled: this code runs once per call,
            // from a cold instruction cache.
            uint64_t* mine = &sm.merge[warp * kSplitPerWarp * 32];
#pragma unroll
            for (int u = 0; u < kSplitPerWarp; ++u) {
              const int q = warp + u * kWarps;
              mine[u * 32 + lane] = (q < S && lane < Kp) ? __ldcg(lists + q * Kp + lane) : 0ull;
            }
            __syncwarp();
            const int nl = S > warp ? (S - warp + kWarps - 1) / kWarps : 0;  // this warp's lists
            uint64_t acc = mine[lane];
#pragma unroll 1
            for (int u = 1; u < nl; ++u) acc = warp_merge_top32(acc, mine[u * 32 + lane], lane);
            sm.wl[warp][lane] = acc;
#pragma unroll 1
            for (int h = kWarps / 2; h > 0; h >>= 1) {
              __syncthreads();
              if (warp < h) {
                acc = warp_merge_top32(acc, sm.wl[warp + h][lane], lane);
                sm.wl[warp][lane] = acc;
              }
            }
            // the merged list's indices and pages for the compact table
            // (sm.keys: free here, never written by another CTA)
            int* mv = reinterpret_cast<int*>(sm.keys);
            int* mp = mv + kMaxK;
            static_assert(sizeof(sm.keys) >= 2 * kMaxK * sizeof(int), "merged-list staging");
            if (warp == 0) {
              const bool have = lane < K && acc != 0ull && lane < Kout;
              if (lane < K) {
                const int v = have ? (int)(stab ? stab_key_index(acc) : key_index(acc)) : -1;
                idx_out[lane] = v;
                if (top_out)
                  top_out[lane] = have ? (stab ? stab_key_score(acc) : key_score(acc)) : -__int_as_float(0x7f800000);
                if (p.sel_pages && have) {
                  mv[lane] = v;
                  mp[lane] = p.bt.pages[off + v];
                }
              }
              const int n = __popc(__ballot_sync(kFull, have));
              if (lane == 0) sm.wn[1] = n;
            }
            if (tid == 0) p.split_ctr[r] = 0ull;  // ready for the next call (and graph replays)
            if (p.sel_pages) {
              __syncthreads();
              write_compact(mv, mp, sm.wn[1]);
            }
          } else {
            for (int f = tid; f < S * Kp; f += kThreads) sm.merge[f] = __ldcg(lists + f);
            __syncthreads();
            // pairwise rounds: lists q and q ^ 1 become list q / 2, cut to Kp
            // keys (the top K of a union lies in the union of its parts' top K);
            // a key's place in the pair is its own position plus the number of
            // larger keys in the other list
            constexpr int kPer = kMergeSlots / kThreads;  // keys a thread holds
            const int kp_log = __ffs(Kp) - 1;
            for (int n = S; n > 1; n = (n + 1) >> 1) {
              uint64_t key[kPer];
              int at[kPer];
#pragma unroll
              for (int u = 0; u < kPer; ++u) {
                const int f = tid + u * kThreads;
                key[u] = f < (n << kp_log) ? sm.merge[f] : 0ull;
                at[u] = -1;
                if (key[u] != 0ull) {
                  const int q = f >> kp_log, o = q ^ 1;
                  const int rank = (f & (Kp - 1)) + (o < n ? count_greater_pow2(&sm.merge[o << kp_log], Kp, key[u]) : 0);
                  if (rank < Kp) at[u] = ((q >> 1) << kp_log) + rank;
                }
              }
              __syncthreads();
              for (int f = tid; f < (((n + 1) >> 1) << kp_log); f += kThreads) sm.merge[f] = 0ull;
              __syncthreads();
#pragma unroll
              for (int u = 0; u < kPer; ++u)
                if (at[u] >= 0) sm.merge[at[u]] = key[u];
              __syncthreads();
            }
            int* mv = reinterpret_cast<int*>(sm.keys);
            int* mp = mv + kMaxK;
            static_assert(kMaxK <= kThreads, "one output a thread");
            const int i = tid;
            const uint64_t k = (i < K && i < Kout) ? sm.merge[i] : 0ull;
            if (i < K) {
              const int v = k ? (int)(stab ? stab_key_index(k) : key_index(k)) : -1;
              idx_out[i] = v;
              if (top_out) top_out[i] = k ? (stab ? stab_key_score(k) : key_score(k)) : -__int_as_float(0x7f800000);
              if (p.sel_pages && k) {
                mv[i] = v;
                mp[i] = p.bt.pages[off + v];
              }
            }
            if (tid == 0) p.split_ctr[r] = 0ull;
            if (p.sel_pages) {
              const int n = __syncthreads_count(k != 0ull);
              write_compact(mv, mp, n);
            }
          }
        }
      }
    }
  }
  if (!start_waited) cluster_wait_acquire();
}

// Blocks a request's clusters score: its table, or (hierarchy) the blocks of
// the kept Chunks, about max_blocks * permille_grid * permille_chunk / 10^6
// of them plus a Chunk.
long long hier_work(const StepParams& p) {
  long long work = p.bt.max_blocks;
  if (p.hier_grid)
    work = std::min<long long>(work, (long long)p.bt.max_blocks * p.permille[0] / 1000 * p.permille[1] / 1000 +
                                         p.chunk_pages);
  return work;
}

// Per-device launch setup of one instantiation: dynamic shared memory above
// 48 KB, non-portable cluster sizes, and the largest cluster size (<= 16)
// that the occupancy calculator says can be co-scheduled.
struct ClusterCaps {
  int active[kMaxCluster + 1];  // co-resident clusters of each size (0 = cannot launch)
};

template <typename T, int D, bool kFused>
cudaError_t setup_device(ClusterCaps* caps) {
  static std::mutex mu;
  static bool ready[64] = {};
  static ClusterCaps cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    const int smem = (int)sizeof(StepSmem<D>);
    e = cudaFuncSetAttribute(step_kernel<T, D, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(step_kernel<T, D, kFused>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    ClusterCaps c = {};
    for (int cl = 1; cl <= kMaxCluster; cl <<= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cl, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cl;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, step_kernel<T, D, kFused>, &cfg) != cudaSuccess) n = 0;
      (void)cudaGetLastError();  // an unsupported size is not an error here
      c.active[cl] = n;
    }
    cached[dev] = c;
    ready[dev] = true;
  }
  *caps = cached[dev];
  return cudaSuccess;
}

// CTAs per request: the largest cluster size (<= 16) at which all R
// requests' clusters are resident at once, limited by the merge buffer
// (CL * K) and by the work (at least 16 blocks per CTA); with more requests
// than that, single-CTA requests.
int pick_cluster(const StepParams& p, const ClusterCaps& caps) {
  const int per_cta_min = 16;
  const int Kp = p.K <= 1 ? 1 : 1 << (32 - __builtin_clz(p.K - 1));
  // Measured on GB300: past 8 CTAs the cluster's list exchange costs more
  // than the extra SMs return (7B: 10.5 us at 8 vs 11.3 at 16; 8 x 1024
  // blocks: 13.7 vs 18.5). A few very long requests take more SMs by
  // splitting over several clusters instead (one request of 65536 blocks:
  // 28.5 us at 16 CTAs x 16 clusters, 24.1 at 8 x 32). Short tables of few
  // requests do gain from 16 (one request of 256 blocks, anchor from the
  // ring: 6.9 -> 6.5 us).
  const long long work = hier_work(p);
  const int cap = work <= 512 ? 16 : 8;
  int best = 1;
  for (int cl = 2; cl <= cap; cl <<= 1) {
    if (caps.active[cl] < p.bt.R) break;
    if (cl * Kp > kMergeSlots / 2) break;
    if ((long long)cl * per_cta_min > work + per_cta_min) break;
    best = cl;
  }
  return best;
}

// Clusters per request: a few long requests leave most SMs idle at one
// cluster each, so their blocks are split over as many clusters as stay
// resident together, each keeping at least kSplitMinBlocks blocks per CTA
// (every cluster recomputes the anchor), within the scratch and the final
// merge buffer.
int pick_splits(const StepParams& p, const ClusterCaps& caps, int CL) {
  if (!(p.flags & (kStepScore | kStepTopK)) || !p.split_ctr || p.split_cap < 2) return 1;
  int S = caps.active[CL] / p.bt.R;
  // the hierarchy's coarse levels run in every CTA at once, so its few kept
  // blocks are spread thinner (measured, one request of 65536 blocks: 24
  // CTAs left 275 blocks each to the block level)
  const int min_blocks = p.hier_grid ? kHierSplitMinBlocks : kSplitMinBlocks;
  S = std::min<long long>(S, hier_work(p) / (CL * min_blocks));
  S = std::min(S, p.split_cap);
  return std::max(S, 1);
}

template <typename T, int D, bool kFused>
cudaError_t launch_typed(const StepParams& p0, cudaStream_t s) {
  ClusterCaps caps;
  cudaError_t e = setup_device<T, D, kFused>(&caps);
  if (e != cudaSuccess) return e;
  StepParams p = p0;
  p.wait_ns = wait_limit_ns();
  const int CL = pick_cluster(p, caps);
  p.splits = pick_splits(p, caps, CL);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, p.bt.R * p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(StepSmem<D>);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, step_kernel<T, D, kFused>, p);
}

}  // namespace
}  // namespace kk
