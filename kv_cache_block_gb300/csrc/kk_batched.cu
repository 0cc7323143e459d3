// Shared-pool scoring ("Key-Key Semantic Affinity" page, §5.1: every block
// representation scored against the anchors in one matrix product, then
// masked): R anchors against N pooled block vectors, each anchor restricted to
// the blocks its mask marks, top K per anchor.
//
// Kernel 1 is a persistent tcgen05 GEMM: TMA streams 128-block tiles of V
// (128-byte swizzle) past a resident 128-anchor tile of A, one thread issues
// eight 128x128x16 bf16 MMAs per tile into one of two TMEM fp32 accumulators,
// and four epilogue warps read them back (tcgen05.ld), divide by the norms
// (computed from the same shared-memory tiles), apply the ownership mask and write each
// owned candidate as a 64-bit key (score, pool id) into the anchor's segment
// for this tile, with the segment's count (no atomics: one writer each).
// Kernel 2 selects each anchor's top K from its list by radix select over the
// 64-bit keys (8-bit digits, most significant first), then sorts the K.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"
#include "kk_tcgen05.cuh"

namespace kk {
namespace {

constexpr int kBM = 128;  // anchors per tile
constexpr int kBN = 128;  // pool blocks per tile
constexpr int kD = 128;   // head_dim (two 64-element swizzle boxes)
constexpr int kBoxBytes = 128 * 128;   // 128 rows x 128 bytes
constexpr int kTileBytes = 2 * kBoxBytes;
constexpr int kStages = 4;             // V tiles in flight
constexpr int kEpiWarps = 8;           // two per TMEM lane quarter, 64 columns each
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kGemmThreads = 64 + kEpiThreads;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr uint32_t kTmemCols = 2 * kBN;  // two accumulators
constexpr int kStageFloats = kEpiWarps * 32 * 33;  // per-lane 32-column dump, padded
constexpr int kGemmSmem = kTileBytes * (1 + kStages) + kStageFloats * 4 + 8 * 128 * 4 + 256 + 1024;

struct GemmArgs {
  const uint32_t* mask;
  int R, N, mask_words, tiles;
  int* counts;      // [R][tiles] owned candidates of each anchor in each 128-block tile
  uint64_t* cand;   // [R][tiles][128] candidate keys, segment per (anchor, tile)
  int* err;
};

// Persistent, warp-specialised: CTA c owns M-tile (c % MT) of the anchors and
// N-tiles p, p + P, p + 2P, ... (p = c / MT, P = CTAs per M-tile). Warp 0
// streams V tiles through a kStages-deep TMA ring; warp 1 issues the MMAs of
// tile j into TMEM accumulator j % 2; eight epilogue warps take the V-row
// norms from the ring (then release the stage) and drain the other
// accumulator, so the epilogue of tile j overlaps the loads and MMAs of tile
// j + 1. Each epilogue warp drains 64 columns of its 32 TMEM lanes (anchors)
// without branches: every column's score is formed in registers and only
// owned columns are stored, at slots given by a popcount prefix of the mask.
__global__ void __launch_bounds__(kGemmThreads, 1)
    score_pool_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmV,
                      GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = base;               // A tile: two boxes (dims 0-63, 64-127)
  unsigned char* sV = base + kTileBytes;  // kStages V tiles
  float* s_dump = reinterpret_cast<float*>(base + kTileBytes * (1 + kStages));  // [warp][lane][33]
  float* s_part = s_dump + kStageFloats;  // [2 halves][128] sums of squares
  float* s_inv_a = s_part + 256;          // [128] 1 / ||A row||
  float* s_inv_v = s_inv_a + 128;         // [2 buffers][128] 1 / ||V row||
  float* s_part_a = s_inv_v + 256;        // [2 halves][128]
  uint64_t* bar = reinterpret_cast<uint64_t*>(s_part_a + 256);
  uint64_t* bar_a = bar;                         // A tile landed
  uint64_t* full = bar + 1;                      // [kStages] V tile landed
  uint64_t* empty = full + kStages;              // [kStages] V tile released (MMA + epilogue warps)
  uint64_t* acc_full = empty + kStages;          // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;            // [2] accumulator drained (epilogue warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int MT = (g.R + kBM - 1) / kBM;
  const int P = max(1, (int)gridDim.x / MT);
  const int m = blockIdx.x % MT, p = blockIdx.x / MT;
  if (p >= P) return;
  const int ntiles = p < g.tiles ? (g.tiles - p + P - 1) / P : 0;
  if (ntiles == 0) return;
  const int m0 = m * kBM;

  if (tid == 0) {
    mbar_init(bar_a, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1 + kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_flag = s_abort;
  auto fail = [&](int code) {
    *abort_flag = 1;
    flag_error(g.err, code);
  };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_a, kTileBytes);
      tma_load_2d(sA, &tmA, 0, m0, bar_a);
      tma_load_2d(sA + kBoxBytes, &tmA, 64, m0, bar_a);
      for (int j = 0; j < ntiles && !*abort_flag; ++j) {
        const int st = j % kStages;
        if (j >= kStages && !mbar_wait_bounded(&empty[st], ((j / kStages) & 1) ^ 1, kWaitLimitNs)) {
          fail(kErrTimeout);
          break;
        }
        const int n0 = (p + j * P) * kBN;
        unsigned char* dst = sV + st * kTileBytes;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        tma_load_2d(dst, &tmV, 0, n0, &full[st]);
        tma_load_2d(dst + kBoxBytes, &tmV, 64, n0, &full[st]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      if (!mbar_wait_bounded(bar_a, 0, kWaitLimitNs)) fail(kErrTimeout);
      for (int j = 0; j < ntiles && !*abort_flag; ++j) {
        const int st = j % kStages, b = j & 1;
        if (!mbar_wait_bounded(&full[st], (j / kStages) & 1, kWaitLimitNs) ||
            (j >= 2 && !mbar_wait_bounded(&acc_empty[b], ((j >> 1) & 1) ^ 1, kWaitLimitNs))) {
          fail(kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA), v0 = smem_u32(sV + st * kTileBytes);
        const uint32_t d = tmem + (uint32_t)(b * kBN);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t off = (uint32_t)((k >> 2) * kBoxBytes + (k & 3) * 32);
          mma_bf16(d, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(v0 + off), idesc, k > 0);
        }
        mma_commit(&empty[st]);
        mma_commit(&acc_full[b]);
      }
    }
  } else {
    const int ew = warp - 2;             // epilogue warp 0..7
    const int half = ew >> 2;            // which 64 columns this warp drains
    const int q4 = warp & 3;             // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;      // anchor row (TMEM lane) this thread drains
    const int r = m0 + row;
    const int nrow = ew * 32 + lane;     // norm work item: row nrow & 127, half nrow >> 7
    const int nr = nrow & 127, nh = nrow >> 7;
    // half of the squared norm of a 128-dim bf16 row stored as two 128-byte
    // swizzled rows: box `nh`, eight 16-byte chunks (rotated by lane to spread
    // banks; the order of a sum of squares does not matter)
    auto half_sq = [&](const unsigned char* tile) {
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int cc = (c + lane) & 7;
        const uint4 x = *reinterpret_cast<const uint4*>(tile + nh * kBoxBytes + nr * 128 + cc * 16);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = bf16_lo(xw[q]), hi = bf16_hi(xw[q]);
          acc = fmaf(lo, lo, fmaf(hi, hi, acc));
        }
      }
      return acc;
    };
    auto inv_norm = [](float sq) { return sq > 0.f ? 1.f / sqrtf(sq) : 0.f; };
    bool ok = mbar_wait_bounded(bar_a, 0, kWaitLimitNs);
    if (!ok) fail(kErrTimeout);
    s_part_a[nh * 128 + nr] = ok ? half_sq(sA) : 0.f;
    named_sync(1, kEpiThreads);
    if (nrow < 128) s_inv_a[nrow] = inv_norm(s_part_a[nrow] + s_part_a[128 + nrow]);
    named_sync(1, kEpiThreads);
    const float inv_a = s_inv_a[row];
    // ownership bits of this anchor's 128 columns of tile jj (limited to
    // columns < N); fetched two tiles ahead so their latency stays hidden
    auto mask_words = [&](int jj, uint32_t (&w)[4]) {
      const int n0 = (p + jj * P) * kBN;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int wi = n0 / 32 + c;
        uint32_t x = 0;
        if (jj < ntiles && r < g.R && wi < g.mask_words) x = g.mask[(long long)r * g.mask_words + wi];
        w[c] = x;
      }
    };
    auto limit_cols = [&](int n0, uint32_t (&w)[4]) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int lim = g.N - (n0 / 32 + c) * 32;
        if (lim < 32) w[c] &= lim <= 0 ? 0u : ((1u << lim) - 1u);
      }
    };
    uint32_t w_next[4], w_after[4];
    mask_words(0, w_next);
    mask_words(1, w_after);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kStages, b = j & 1;
      const int tile = p + j * P, n0 = tile * kBN;
      uint32_t w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        w[c] = w_next[c];
        w_next[c] = w_after[c];
      }
      mask_words(j + 2, w_after);
      limit_cols(n0, w);
      // V-row norms of this tile, then release the ring stage. The epilogue
      // warps leave the loop together (a lone warp leaving would strand the
      // others at the named barrier).
      ok = !*abort_flag && mbar_wait_bounded(&full[st], (j / kStages) & 1, kWaitLimitNs);
      s_part[nh * 128 + nr] = ok ? half_sq(sV + st * kTileBytes) : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (named_sync_or(1, kEpiThreads, !ok)) {
        if (!ok) fail(kErrTimeout);
        break;
      }
      if (nrow < 128) s_inv_v[b * 128 + nrow] = inv_norm(s_part[nrow] + s_part[128 + nrow]);
      ok = mbar_wait_bounded(&acc_full[b], (j >> 1) & 1, kWaitLimitNs);
      if (named_sync_or(1, kEpiThreads, !ok)) {  // tcgen05.ld below is warp-collective too
        if (!ok) fail(kErrTimeout);
        break;
      }
      tc_fence_after();
      uint32_t acc[2][32];
      const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(b * kBN + half * 64);
      tmem_ld32(taddr, acc[0]);
      tmem_ld32(taddr + 32, acc[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);  // the accumulator may be reused
      if (r < g.R && half == 0)
        g.counts[(long long)r * g.tiles + tile] = __popc(w[0]) + __popc(w[1]) + __popc(w[2]) + __popc(w[3]);
      uint64_t* out = g.cand + ((long long)r * g.tiles + tile) * kBN;
      int k = half ? __popc(w[0]) + __popc(w[1]) : 0;
      const float* inv_v = s_inv_v + b * 128 + half * 64;
      // Owned columns are sparse: dump the 32 accumulators of a chunk to this
      // lane's shared-memory row (stride 33: no bank conflicts) and visit only
      // the set mask bits.
      float* dump = s_dump + (ew * 32 + lane) * 33;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int i = 0; i < 32; ++i) dump[i] = __uint_as_float(acc[c][i]);
        uint32_t x = half ? w[2 + c] : w[c];
        // the first four owned columns as independent slots (they overlap),
        // then the rare remainder one by one
        int ib[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ib[u] = x ? __ffs(x) - 1 : -1;
          x &= x - 1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (ib[u] >= 0) {
            const int i = ib[u];
            float cosv = dump[i] * inv_a * inv_v[c * 32 + i];
            cosv = fminf(1.f, fmaxf(-1.f, cosv));
            out[k + u] = make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + half * 64 + c * 32 + i));
          }
        }
        k += (ib[0] >= 0) + (ib[1] >= 0) + (ib[2] >= 0) + (ib[3] >= 0);
        while (x) {
          const int i = __ffs(x) - 1;
          x &= x - 1;
          float cosv = dump[i] * inv_a * inv_v[c * 32 + i];
          cosv = fminf(1.f, fmaxf(-1.f, cosv));
          out[k++] = make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + half * 64 + c * 32 + i));
        }
      }
    }
  }

  // teardown: every role has left its loop; no MMA or TMEM read is pending
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- per-anchor top-K by radix select ------------------------------------
constexpr int kSelThreads = 256;
constexpr int kSelStage = 6144;  // keys of a row held in shared memory (48 KB)

// Visits every candidate key of row r, warp-uniformly (every lane of a warp
// runs the same iterations; `active` marks real keys), either from the
// shared-memory copy or, for rows too long for it, from the tile segments.
template <typename F>
__device__ __forceinline__ void for_each_key(bool staged, int n, const uint64_t* s_keys, const int* cnt,
                                             const uint64_t* seg, int tiles, F&& fn) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (staged) {
    for (int i0 = 0; i0 < n; i0 += kSelThreads) {
      const int i = i0 + tid;
      const bool active = i < n;
      fn(active, active ? s_keys[i] : 0ull);
    }
  } else {
    for (int t = warp; t < tiles; t += kSelThreads / 32) {
      const int c = min(max(cnt[t], 0), kBN);
      for (int j0 = 0; j0 < c; j0 += 32) {
        const int j = j0 + lane;
        const bool active = j < c;
        fn(active, active ? seg[(long long)t * kBN + j] : 0ull);
      }
    }
  }
}

constexpr int kBuckets = 2048;  // linear buckets over a row's score range
constexpr int kMaxTiles = 2048; // tiles of a row whose offsets are staged (N <= 262144)
constexpr int kTieCap = 512;    // boundary-bucket keys ranked exactly

__global__ void __launch_bounds__(kSelThreads) select_rows_kernel(const uint64_t* cand, const int* counts,
                                                                  int tiles, int K, int* idx_out,
                                                                  float* top_out, int* err) {
  extern __shared__ __align__(16) uint64_t s_keys[];  // [kSelStage]
  __shared__ int hist[kBuckets];
  __shared__ int s_bin, s_above;
  __shared__ int s_sel_n, s_tie_n;
  __shared__ int s_wsum[kSelThreads / 32];
  __shared__ int s_off[kMaxTiles + 1];
  __shared__ uint64_t s_lo[kSelThreads / 32], s_hi[kSelThreads / 32];
  __shared__ uint64_t s_sel[kMaxK];
  __shared__ uint64_t s_tie[kTieCap];
  __shared__ uint64_t s_wl[kSelThreads / 32][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int* cnt = counts + (long long)r * tiles;
  const uint64_t* seg = cand + (long long)r * tiles * kBN;

  // ---- row length and per-tile offsets: each thread sums a contiguous run
  // of tiles, an exclusive scan over the block gives the run's start, and the
  // run's tile offsets go to shared memory (rows of up to kMaxTiles tiles)
  const int tpt = (tiles + kSelThreads - 1) / kSelThreads;
  const int t_begin = min(tiles, tid * tpt), t_end = min(tiles, t_begin + tpt);
  int mine = 0;
  for (int t = t_begin; t < t_end; ++t) {
    int c = cnt[t];
    if (c < 0 || c > kBN) {
      flag_error(err, kErrBadIndex);
      c = min(max(c, 0), kBN);
    }
    mine += c;
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int base = incl - mine, n = 0;
#pragma unroll
  for (int w = 0; w < kSelThreads / 32; ++w) {
    if (w < warp) base += s_wsum[w];
    n += s_wsum[w];
  }
  const bool staged = n <= kSelStage && tiles <= kMaxTiles;
  if (staged) {
    int o = base;
    for (int t = t_begin; t < t_end; ++t) {
      s_off[t] = o;
      o += min(max(cnt[t], 0), kBN);
    }
    if (tid == 0) s_off[tiles] = n;
  }
  __syncthreads();

  // ---- stage the row compactly: key i lives in the last tile whose offset
  // is <= i (binary search), 16 independent loads per thread; and the key range
  uint64_t lo = ~0ull, hi = 0ull;
  if (staged) {
    for (int i0 = 0; i0 < n; i0 += kSelThreads * 16) {
      uint64_t v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        int t = 0;
        for (int step = kMaxTiles / 2; step > 0; step >>= 1)
          if (t + step <= tiles && s_off[t + step] <= i) t += step;
        v[u] = i < n ? seg[(long long)t * kBN + (i - s_off[t])] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        if (i < n) {
          s_keys[i] = v[u];
          lo = v[u] < lo ? v[u] : lo;
          hi = v[u] > hi ? v[u] : hi;
        }
      }
    }
  } else {
    for_each_key(false, n, s_keys, cnt, seg, tiles, [&](bool active, uint64_t k) {
      if (active) {
        lo = k < lo ? k : lo;
        hi = k > hi ? k : hi;
      }
    });
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t a = __shfl_xor_sync(kFull, lo, o), b = __shfl_xor_sync(kFull, hi, o);
    lo = a < lo ? a : lo;
    hi = b > hi ? b : hi;
  }
  if (lane == 0) {
    s_lo[warp] = lo;
    s_hi[warp] = hi;
  }
  for (int b = tid; b < kBuckets; b += kSelThreads) hist[b] = 0;
  if (tid == 0) {
    s_sel_n = 0;
    s_tie_n = 0;
  }
  __syncthreads();
  lo = s_lo[0];
  hi = s_hi[0];
#pragma unroll
  for (int w = 1; w < kSelThreads / 32; ++w) {
    lo = s_lo[w] < lo ? s_lo[w] : lo;
    hi = s_hi[w] > hi ? s_hi[w] : hi;
  }
  const int m = min(K, n);

  // ---- bucket pass: linear buckets over the score part of the keys (a
  // non-decreasing function of the key, so keys above the boundary bucket
  // are all selected and only the boundary bucket needs exact ranking)
  const uint32_t s_lo32 = (uint32_t)(lo >> 32), s_hi32 = (uint32_t)(hi >> 32);
  const float bscale = (float)kBuckets / ((float)(s_hi32 - s_lo32) + 1.f);
  auto bucket = [&](uint64_t k) {
    return min(kBuckets - 1, (int)((float)((uint32_t)(k >> 32) - s_lo32) * bscale));
  };
  bool fast = m > 0 && s_hi32 != s_lo32;
  if (fast) {
    for_each_key(staged, n, s_keys, cnt, seg, tiles, [&](bool active, uint64_t k) {
      if (active) atomicAdd(&hist[bucket(k)], 1);
    });
    __syncthreads();
    // suffix counts from the top bucket down: thread t owns buckets 8t .. 8t+7
    int local = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) local += hist[tid * 8 + b];
    int sfx = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(kFull, sfx, o);
      if (lane + o < 32) sfx += y;
    }
    if (lane == 0) s_wsum[warp] = sfx;  // total of this warp's buckets
    __syncthreads();
    int above = sfx - local;  // buckets above this thread's run
    for (int w = warp + 1; w < kSelThreads / 32; ++w) above += s_wsum[w];
    for (int b = 7; b >= 0; --b) {
      const int hb = hist[tid * 8 + b];
      if (above < m && above + hb >= m) {
        s_bin = tid * 8 + b;
        s_above = above;
      }
      above += hb;
    }
    __syncthreads();
    const int bstar = s_bin;
    for_each_key(staged, n, s_keys, cnt, seg, tiles, [&](bool active, uint64_t k) {
      if (!active) return;
      const int b = bucket(k);
      if (b > bstar) {
        const int p = atomicAdd(&s_sel_n, 1);
        if (p < kMaxK) s_sel[p] = k;
      } else if (b == bstar) {
        const int p = atomicAdd(&s_tie_n, 1);
        if (p < kTieCap) s_tie[p] = k;
      }
    });
    __syncthreads();
    const int ties = s_tie_n, need = m - s_above;
    if (ties <= kTieCap) {
      // exact rank among the boundary bucket's keys (distinct keys)
      for (int i = tid; i < ties; i += kSelThreads) {
        const uint64_t k = s_tie[i];
        int rank = 0;
        for (int q = 0; q < ties; ++q) rank += s_tie[q] > k;
        if (rank < need) s_sel[s_above + rank] = k;
      }
      __syncthreads();
    } else {
      fast = false;  // massive ties: fall back to the radix select
      __syncthreads();
      if (tid == 0) s_sel_n = 0;
      __syncthreads();
    }
  }
  if (!fast && m > 0) {
    // radix select on the 64-bit keys, 8-bit digits below the common prefix
    int need = m;
    const int common = lo != hi ? __clzll(lo ^ hi) : 64;
    uint64_t pmask = common >= 64 ? ~0ull : (common == 0 ? 0ull : ~0ull << (64 - common));
    uint64_t prefix = hi & pmask;
    if (common < 64) {
      for (int shift = 56 - ((common / 8) * 8); shift >= 0 && need > 0; shift -= 8) {
        hist[tid] = 0;
        __syncthreads();
        for_each_key(staged, n, s_keys, cnt, seg, tiles, [&](bool active, uint64_t k) {
          const int d = (active && (k & pmask) == prefix) ? (int)((k >> shift) & 255) : 256;
          const unsigned same = __match_any_sync(kFull, d);
          if (d < 256 && lane == __ffs(same) - 1) atomicAdd(&hist[d], __popc(same));
        });
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
              s_bin = lane * 8 + b;
              s_above = above;
            }
            above += hb;
          }
        }
        __syncthreads();
        const int b = s_bin;
        need -= s_above;
        prefix |= (uint64_t)b << shift;
        pmask |= (uint64_t)0xFF << shift;
        const bool exact = hist[b] == need;
        __syncthreads();
        if (exact) break;
      }
    }
    // the m largest keys are exactly those >= prefix
    for_each_key(staged, n, s_keys, cnt, seg, tiles, [&](bool active, uint64_t k) {
      if (active && k >= prefix) {
        const int p = atomicAdd(&s_sel_n, 1);
        if (p < kMaxK) s_sel[p] = k;
      }
    });
    __syncthreads();
  }
  const int sel = m;
  // ---- sort the selected keys: warp-sorted lists of 32, then rank in the union
  uint64_t key = tid < sel ? s_sel[tid] : 0ull;
  key = warp_sort_desc(key, lane);
  s_wl[warp][lane] = key;
  __syncthreads();
  int* io = idx_out + (long long)r * K;
  float* to = top_out ? top_out + (long long)r * K : nullptr;
  if (key != 0ull) {
    int pos[kSelThreads / 32];
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) pos[w] = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
#pragma unroll
      for (int w = 0; w < kSelThreads / 32; ++w) pos[w] += (s_wl[w][pos[w] + step] > key) ? step : 0;
    int rank = 0;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) rank += (s_wl[w][0] > key) ? pos[w] + 1 : 0;
    if (rank < K) {
      io[rank] = (int)key_index(key);
      if (to) to[rank] = key_score(key);
    }
  }
  for (int i = sel + tid; i < K; i += kSelThreads) {
    io[i] = -1;
    if (to) to[i] = -__int_as_float(0x7f800000);
  }
}

// ---- host ---------------------------------------------------------------
// Tensor map of a row-major bf16 [rows][128] matrix, boxes of 64 x 128.
bool make_map(CUtensorMap* map, const void* ptr, int rows) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t setup_gemm() {
  static std::mutex mu;
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    e = cudaFuncSetAttribute(score_pool_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(select_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(uint64_t) * kSelStage));
    if (e != cudaSuccess) return e;
    ready[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

size_t batched_workspace_bytes(int R, int N) {
  const size_t tiles = ((size_t)N + kBN - 1) / kBN;
  return ((sizeof(int) * (size_t)R * tiles + 255) & ~size_t(255)) + sizeof(uint64_t) * (size_t)R * tiles * kBN;
}

cudaError_t launch_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask, int R,
                                      int N, int K, int* idx, float* top, void* ws, int* err,
                                      cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int tiles = (N + kBN - 1) / kBN;
  int* counts = static_cast<int*>(ws);
  uint64_t* cand = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) +
                                               ((sizeof(int) * (size_t)R * tiles + 255) & ~size_t(255)));
  cudaError_t e = setup_gemm();
  if (e != cudaSuccess) return e;
  if (N > 0) {
    CUtensorMap ma, mv;
    if (!make_map(&ma, A, R) || !make_map(&mv, V, N)) return cudaErrorInvalidValue;
    GemmArgs g{mask, R, N, (N + 31) / 32, tiles, counts, cand, err};
    // one CTA per SM, split evenly across the M-tiles of the anchors
    const int MT = (R + kBM - 1) / kBM;
    const int P = std::max(1, std::min(tiles, sm_count() / MT));
    score_pool_kernel<<<MT * P, kGemmThreads, kGemmSmem, s>>>(ma, mv, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  select_rows_kernel<<<R, kSelThreads, sizeof(uint64_t) * kSelStage, s>>>(cand, counts, tiles, K, idx,
                                                                          top, err);
  return cudaGetLastError();
}

}  // namespace kk
