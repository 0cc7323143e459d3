// Shared-pool scoring ("Key-Key Semantic Affinity" page, §5.1: every block
// representation scored against the anchors in one matrix product, then
// masked): R anchors against N pooled block vectors, each anchor restricted to
// the blocks its mask marks, top K per anchor.
//
// Kernel 1 is a tcgen05 GEMM tile: TMA loads a 128-anchor x 128-dim tile of A
// and a 128-block tile of V into shared memory (128-byte swizzle), one thread
// issues eight 128x128x16 bf16 MMAs into a TMEM fp32 accumulator, and four
// epilogue warps read it back (tcgen05.ld), divide by the norms (computed from
// the same shared-memory tiles), apply the ownership mask and write each
// owned candidate as a 64-bit key (score, pool id) into the anchor's segment
// for this tile, with the segment's count (no atomics: one writer each).
// Kernel 2 selects each anchor's top K from its list by radix select over the
// 64-bit keys (8-bit digits, most significant first), then sorts the K.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"
#include "kk_tcgen05.cuh"

namespace kk {
namespace {

constexpr int kBM = 128;  // anchors per tile
constexpr int kBN = 128;  // pool blocks per tile
constexpr int kD = 128;   // head_dim (two 64-element swizzle boxes)
constexpr int kBoxBytes = 128 * 128;  // 128 rows x 128 bytes
constexpr int kGemmThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kTmemCols = 128;
constexpr int kGemmSmem = 4 * kBoxBytes + 2 * 128 * 4 + 64 + 1024;  // tiles, norms, barriers, alignment

struct GemmArgs {
  const uint32_t* mask;
  int R, N, mask_words, tiles;
  int* counts;      // [R][tiles] owned candidates of each anchor in each 128-block tile
  uint64_t* cand;   // [R][tiles][128] candidate keys, segment per (anchor, tile)
  int* err;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    score_pool_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmV,
                      GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = base;                   // two boxes of A: dims 0-63, 64-127
  unsigned char* sV = base + 2 * kBoxBytes;   // two boxes of V
  float* s_na = reinterpret_cast<float*>(base + 4 * kBoxBytes);
  float* s_nv = s_na + 128;
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(s_nv + 128);
  uint64_t* bar_mma = bar_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;

  if (tid == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
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

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar_full, 4 * kBoxBytes);
    tma_load_2d(sA, &tmA, 0, m0, bar_full);
    tma_load_2d(sA + kBoxBytes, &tmA, 64, m0, bar_full);
    tma_load_2d(sV, &tmV, 0, n0, bar_full);
    tma_load_2d(sV + kBoxBytes, &tmV, 64, n0, bar_full);
  } else if (warp == 1 && lane == 0) {
    if (mbar_wait_bounded(bar_full, 0, kWaitLimitNs)) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      const uint32_t a0 = smem_u32(sA), v0 = smem_u32(sV);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {
        const uint32_t off = (uint32_t)((k >> 2) * kBoxBytes + (k & 3) * 32);
        mma_bf16(tmem, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(v0 + off), idesc, k > 0);
      }
      mma_commit(bar_mma);
    } else {
      atomicExch(s_abort, 1);
      flag_error(g.err, kErrTimeout);
      mbar_arrive(bar_mma);  // release the epilogue
    }
  } else if (warp >= 2) {
    const int e = tid - 64;  // 0..127: norm row, then TMEM lane owner below
    const int q4 = warp & 3;            // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;     // anchor row within the tile
    const int r = m0 + row;
    // Ownership bits of this anchor's 128 columns (limited to columns < N)
    // and the row's write offset, both independent of the tiles: fetched
    // first so their latency hides behind the loads and the MMAs.
    uint32_t w[4];
    int total = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int wi = n0 / 32 + c;
      uint32_t x = 0;
      if (r < g.R && wi < g.mask_words) x = g.mask[(long long)r * g.mask_words + wi];
      const int lim = g.N - wi * 32;  // valid columns in this word
      if (lim < 32) x &= lim <= 0 ? 0u : ((1u << lim) - 1u);
      w[c] = x;
      total += __popc(x);
    }
    if (r < g.R) g.counts[(long long)r * g.tiles + blockIdx.x] = total;
    if (mbar_wait_bounded(bar_full, 0, kWaitLimitNs)) {
      // squared norms of A row e and V row e (16-byte chunks rotated by lane
      // to spread banks; the order of a sum of squares does not matter)
      float na = 0.f, nv = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int cc = (c + lane) & 15;
        const int off = (cc >> 3) * kBoxBytes + e * 128 + (cc & 7) * 16;
        const uint4 a = *reinterpret_cast<const uint4*>(sA + off);
        const uint4 v = *reinterpret_cast<const uint4*>(sV + off);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a_lo = bf16_lo(aw[q]), a_hi = bf16_hi(aw[q]);
          const float v_lo = bf16_lo(vw[q]), v_hi = bf16_hi(vw[q]);
          na = fmaf(a_lo, a_lo, fmaf(a_hi, a_hi, na));
          nv = fmaf(v_lo, v_lo, fmaf(v_hi, v_hi, nv));
        }
      }
      s_na[e] = sqrtf(na);
      s_nv[e] = sqrtf(nv);
    } else {
      atomicExch(s_abort, 1);
      flag_error(g.err, kErrTimeout);
    }
    named_sync(1, 128);
    bool mma_ok = mbar_wait_bounded(bar_mma, 0, kWaitLimitNs);
    if (!mma_ok) flag_error(g.err, kErrTimeout);
    // tcgen05.ld is warp-collective: the whole warp takes one decision
    mma_ok = __all_sync(kFull, mma_ok && *s_abort == 0);
    tc_fence_after();
    if (mma_ok) {
      uint64_t* out = g.cand + ((long long)r * g.tiles + blockIdx.x) * kBN;
      int k = 0;
      const float na = s_na[row];
      const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16);
      // The MMAs have consumed the V tile, so its shared memory stages each
      // lane's 32 accumulator columns; only the owned columns are then visited
      // (mask bits are sparse), by index into shared memory.
      // 4 warps x 32 lanes x 33 floats = 16.9 KB of the 32 KB V tile; each lane
      // writes and reads only its own row, so no synchronisation is needed
      float* stage = reinterpret_cast<float*>(sV) + ((warp - 2) * 32 + lane) * 33;
      uint32_t acc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(taddr + c * 32, acc[c]);  // whole warp, one wait
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[i] = __uint_as_float(acc[c][i]);
        uint32_t x = w[c];
        while (x) {
          const int i = __ffs(x) - 1;
          x &= x - 1;
          const int col = c * 32 + i;
          const float nv = s_nv[col];
          float cosv = (na > 0.f && nv > 0.f) ? stage[i] / (na * nv) : 0.f;
          cosv = fminf(1.f, fmaxf(-1.f, cosv));
          out[k++] = make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + col));
        }
      }
    }
  }

  // teardown: nothing may still read TMEM or wait on copies
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *s_abort) (void)mbar_wait_bounded(bar_full, 0, kWaitLimitNs);  // copies in flight
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
      const int c = cnt[t];
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major bf16 [rows][128] matrix, boxes of 64 x 128.
bool make_map(CUtensorMap* map, const void* ptr, int rows) {
  auto fn = encode_fn();
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
    dim3 grid(tiles, (R + kBM - 1) / kBM);
    score_pool_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(ma, mv, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  select_rows_kernel<<<R, kSelThreads, sizeof(uint64_t) * kSelStage, s>>>(cand, counts, tiles, K, idx, top,
                                                                          err);
  return cudaGetLastError();
}

}  // namespace kk
