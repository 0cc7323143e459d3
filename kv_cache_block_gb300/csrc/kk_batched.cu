// Shared-pool scoring ("Key-Key Semantic Affinity" page, §5.1: every block
// representation scored against the anchors in one matrix product, then
// masked): R anchors against N pooled block vectors, each anchor restricted to
// the blocks its mask marks, top K per anchor.
//
// Kernel 1 counts each anchor's owned blocks before every 128-block tile
// (prefix popcounts of the mask). Kernel 2 is a persistent tcgen05 GEMM: TMA
// streams 128-block tiles of V (128-byte swizzle) past a resident 128-anchor
// tile of A, one thread issues eight 128x128x16 bf16 MMAs per tile into one
// of four TMEM fp32 accumulators, and four epilogue groups of four warps read
// them back (tcgen05.ld), divide by the norms (computed from the same
// shared-memory tiles), apply the ownership mask and write each owned
// candidate as a 64-bit key (score, pool id) into the anchor's contiguous
// list, at the tile's offset from kernel 1 (no atomics: one writer a slot).
// Rows in front of the pool that every anchor scores (the coarse levels of
// the hierarchy) are written as a dense score matrix instead. Kernel 3
// selects each anchor's top K from its list (linear buckets over the score
// range, exact ranking of the boundary bucket, a radix select on the 64-bit
// keys for massive ties), then orders the K by counting. The three are
// chained by programmatic dependent launch.
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
constexpr int kStages = 3;             // V tiles in flight
constexpr int kGroups = 4;             // epilogue groups, each drains whole tiles
constexpr int kAccs = kGroups;         // TMEM accumulators (128 columns each), one per group
constexpr int kGroupThreads = 128;     // four warps: one per TMEM lane quarter
constexpr int kEpiThreads = kGroups * kGroupThreads;
constexpr int kGemmThreads = 64 + kEpiThreads;  // warp 0 TMA, warp 1 MMA, then the epilogue groups
constexpr uint32_t kTmemCols = kAccs * kBN;
constexpr int kDumpStride = 36;  // floats per lane row of the dump: 16-byte rows, no bank conflicts
constexpr int kDumpFloats = kEpiThreads * kDumpStride;
constexpr int kGemmSmem =
    1024 + kTileBytes * (1 + kStages) + kDumpFloats * 4 + kGroups * 2 * kBN * 4 + 256;

struct GemmArgs {
  const uint32_t* mask;
  int R, N, mask_words, tiles;
  int coarse_rows;  // rows before the pool's blocks that every anchor scores (0: none)
  int coarse_tiles; // tiles holding them (their rows come first, 128 per tile)
  float* coarse;    // [R][coarse_tiles * 128] their scores, dense
  const int* offsets;  // [R][mtiles + 1] owned blocks of each anchor before each block tile, then the total
  int mtiles;          // block tiles (128 pool blocks each)
  uint64_t* keys;      // [R][N] each anchor's candidate keys, contiguous, in pool order
  int mask_vec;     // mask rows allow 16-byte loads of a tile's four words
  unsigned long long wait_ns;  // limit of every bounded wait
  int* err;
};

// Starts fetching a tensor map (a __grid_constant__ kernel parameter) into
// the TMA unit's descriptor cache, so that the first copy does not wait for it.
__device__ __forceinline__ void tma_prefetch_map(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Sum of squares of one 128-dim bf16 row held as two 128-byte swizzled rows
// (one per box); the swizzle only permutes 16-byte chunks inside a row, and
// the order of a sum of squares does not matter. The chunk order is rotated
// by the row so that the eight rows a quarter-warp reads hit eight different
// bank groups; four chains for ILP.
__device__ __forceinline__ float row_sq(const unsigned char* tile, int row) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int pc = (c + row) & 7;
      const uint4 x = *reinterpret_cast<const uint4*>(tile + h * kBoxBytes + row * 128 + pc * 16);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = bf16_lo(xw[q]), hi = bf16_hi(xw[q]);
        acc[q] = fmaf(lo, lo, fmaf(hi, hi, acc[q]));
      }
    }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Persistent, warp-specialised: CTA c owns M-tile (c % MT) of the anchors and
// N-tiles p, p + P, p + 2P, ... (p = c / MT, P = CTAs per M-tile), split into
// four contiguous ranges, one per epilogue group of four warps, each group
// with its own TMEM accumulator. Warp 0 streams V tiles through a
// kStages-deep TMA ring and warp 1 issues the MMAs, both visiting the ranges
// round robin, so four tiles drain at once. A group computes its tile's V-row
// norms from the ring (then releases the stage), reads the accumulator (one
// anchor row per thread, tcgen05.ld), and writes each owned column as a
// 64-bit key (score, pool id) into its own segment of that anchor, in tile
// order, and the segment's length at the end. No atomics: every slot has one
// writer. kCoarse: the first tiles hold rows every anchor scores, written as
// dense scores.
template <bool kCoarse>
__global__ void __launch_bounds__(kGemmThreads, 1)
    score_pool_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmV,
                      GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned (the 128-byte swizzle atom); offset arithmetic on the
  // shared array keeps every derived pointer in the shared address space
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sA = base;               // A tile: two boxes (dims 0-63, 64-127)
  unsigned char* sV = base + kTileBytes;  // kStages V tiles
  float* s_dump = reinterpret_cast<float*>(base + kTileBytes * (1 + kStages));  // [thread][36]
  float* s_inv_v = s_dump + kDumpFloats;  // [group][2 buffers][128] 1 / ||V row||
  uint64_t* bar = reinterpret_cast<uint64_t*>(s_inv_v + kGroups * 2 * kBN);
  uint64_t* bar_a = bar;                  // A tile landed
  uint64_t* full = bar + 1;               // [kStages] V tile landed
  uint64_t* empty = full + kStages;       // [kStages] V tile released (MMA + the tile's group)
  uint64_t* acc_full = empty + kStages;   // [kAccs] accumulator ready
  uint64_t* acc_empty = acc_full + kAccs; // [kAccs] accumulator drained (the tile's group)
  uint64_t* epi_done = acc_empty + kAccs; // every epilogue warp has left its loop
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_done + 1);
  int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

  // the select kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int MT = (g.R + kBM - 1) / kBM;
  const int P = max(1, (int)gridDim.x / MT);
  const int m = blockIdx.x % MT, p = blockIdx.x / MT;
  if (p >= P) return;
  const int ntiles = p < g.tiles ? (g.tiles - p + P - 1) / P : 0;
  if (ntiles == 0) return;
  const int m0 = m * kBM;

  // The CTA's local tiles 0 .. ntiles-1 (global tile p + j * P) are split
  // into four contiguous ranges, one per epilogue group, and each group has
  // its own TMEM accumulator. The producer and the MMA issuer visit the
  // ranges round robin (sequence k: group k % 4, its (k / 4)-th tile), so
  // four tiles drain at once; q counts the tiles issued (its ring stage).
  auto range_lo = [&](int gg) { return gg * ntiles / kGroups; };
  auto range_len = [&](int gg) { return (gg + 1) * ntiles / kGroups - gg * ntiles / kGroups; };

  if (tid == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmV);
    mbar_init(bar_a, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1 + kGroupThreads / 32);
    }
    for (int b = 0; b < kAccs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kGroupThreads / 32);
    }
    mbar_init(epi_done, kEpiThreads / 32);
    *s_abort = 0;
    fence_mbar_init();
    // the A tile goes out before the TMEM allocation and the block barrier
    // (this thread is the producer)
    mbar_arrive_expect_tx(bar_a, kTileBytes);
    tma_load_2d(sA, &tmA, 0, m0, bar_a);
    tma_load_2d(sA + kBoxBytes, &tmA, 64, m0, bar_a);
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
      for (int k = 0, q = 0; q < ntiles && !*abort_flag; ++k) {
        const int gg = k % kGroups, i = k / kGroups;
        if (i >= range_len(gg)) continue;
        const int j = range_lo(gg) + i;
        const int st = q % kStages;
        if (q >= kStages && !mbar_wait_bounded(&empty[st], ((q / kStages) & 1) ^ 1, g.wait_ns)) {
          fail(kErrTimeout);
          break;
        }
        const int n0 = (p + j * P) * kBN;
        unsigned char* dst = sV + st * kTileBytes;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        tma_load_2d(dst, &tmV, 0, n0, &full[st]);
        tma_load_2d(dst + kBoxBytes, &tmV, 64, n0, &full[st]);
        ++q;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      if (!mbar_wait_bounded(bar_a, 0, g.wait_ns)) fail(kErrTimeout);
      for (int k = 0, q = 0; q < ntiles && !*abort_flag; ++k) {
        const int gg = k % kGroups, i = k / kGroups;
        if (i >= range_len(gg)) continue;
        const int st = q % kStages;
        if (!mbar_wait_bounded(&full[st], (q / kStages) & 1, g.wait_ns) ||
            (i >= 1 && !mbar_wait_bounded(&acc_empty[gg], (i - 1) & 1, g.wait_ns))) {
          fail(kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA), v0 = smem_u32(sV + st * kTileBytes);
        const uint32_t d = tmem + (uint32_t)(gg * kBN);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * kBoxBytes + (kk & 3) * 32);
          mma_bf16(d, desc_kmajor_sw128(a0 + off), desc_kmajor_sw128(v0 + off), idesc, kk > 0);
        }
        mma_commit(&empty[st]);
        mma_commit(&acc_full[gg]);
        ++q;
      }
    }
  } else {
    const int et = tid - 64;
    const int grp = et / kGroupThreads;       // epilogue group
    const int q4 = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;           // anchor row (TMEM lane) of this thread
    const int r = m0 + row;
    const int bar_id = 1 + grp;               // named barrier of the group
    float* inv_v_grp = s_inv_v + grp * 2 * kBN;
    const uint32_t dump = smem_u32(s_dump + et * kDumpStride);
    const int lo = range_lo(grp), len = range_len(grp);
    auto inv_norm = [](float sq) { return sq > 0.f ? 1.f / sqrtf(sq) : 0.f; };
    // ownership bits of this anchor's 128 columns of the CTA's local tile jj
    // (one 16-byte load when the rows allow it), loaded a tile ahead and
    // limited to columns < N only when the tile is drained, so that the load
    // is not waited for early. Coarse tiles (first) have no mask.
    const uint32_t* mrow = g.mask + (long long)(r < g.R ? r : 0) * g.mask_words;
    const int* orow = g.offsets + (long long)(r < g.R ? r : 0) * (g.mtiles + 1);
    auto mask_load = [&](int jj, uint32_t (&w)[4], int& o) {
      const int tile = p + jj * P;
      o = 0;
      if (kCoarse && tile < g.coarse_tiles) {
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = 0u;
        return;
      }
      const int mt = tile - g.coarse_tiles;
      if (jj < ntiles && r < g.R) o = orow[mt];
      const int wi0 = mt * (kBN / 32);
      if (g.mask_vec && jj < ntiles && r < g.R) {
        const uint4 x = *reinterpret_cast<const uint4*>(mrow + wi0);
        w[0] = x.x;
        w[1] = x.y;
        w[2] = x.z;
        w[3] = x.w;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          w[c] = (jj < ntiles && r < g.R && wi0 + c < g.mask_words) ? mrow[wi0 + c] : 0u;
      }
    };
    auto mask_finish = [&](int jj, uint32_t (&w)[4]) {
      const int wi0 = (p + jj * P - g.coarse_tiles) * (kBN / 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int lim = g.N - (wi0 + c) * 32;
        if (lim < 32) w[c] &= lim <= 0 ? 0u : ((1u << lim) - 1u);
      }
    };
    // An anchor's keys go to its contiguous list, each tile's at the offset
    // the offsets kernel (launched just before this grid) computed from the
    // mask; only the epilogue waits for that grid.
    uint64_t* list = g.keys + (long long)(r < g.R ? r : 0) * g.N;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t dump0 = dump - (uint32_t)(lane * kDumpStride * 4);  // lane 0's dump row in this warp
    uint32_t w_next[4];
    int o_next;
    mask_load(len > 0 ? lo : ntiles, w_next, o_next);
    bool ok = mbar_wait_bounded(bar_a, 0, g.wait_ns);
    if (!ok) fail(kErrTimeout);
    const float inv_a = ok ? inv_norm(row_sq(sA, row)) : 0.f;
    for (int i = 0; i < len; ++i) {
      const int j = lo + i;
      // this tile's place in the issue sequence: tiles of earlier rounds,
      // then those of the groups before this one in round i
      int q = 0;
#pragma unroll
      for (int gg = 0; gg < kGroups; ++gg) q += min(range_len(gg), i + (gg < grp ? 1 : 0));
      const int st = q % kStages;
      const int tile = p + j * P, n0 = tile * kBN;
      uint32_t w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = w_next[c];
      const int o_tile = o_next;
      mask_load(i + 1 < len ? j + 1 : ntiles, w_next, o_next);
      // V-row norms of this tile (one row per thread), then release the
      // ring stage. The group leaves the loop together (a lone warp leaving
      // would strand the others at the named barrier).
      ok = !*abort_flag && mbar_wait_bounded(&full[st], (q / kStages) & 1, g.wait_ns);
      float* inv_v = inv_v_grp + (i & 1) * kBN;
      inv_v[row] = ok ? inv_norm(row_sq(sV + st * kTileBytes, row)) : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      ok = ok && mbar_wait_bounded(&acc_full[grp], i & 1, g.wait_ns);
      if (named_sync_or(bar_id, kGroupThreads, !ok)) {  // also orders the inv_v writes before the reads
        if (!ok) fail(kErrTimeout);
        break;
      }
      tc_fence_after();
      const bool coarse = kCoarse && tile < g.coarse_tiles;
      if (!coarse) mask_finish(j, w);
      const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(grp * kBN);
      uint64_t* out = list + o_tile;
      int k = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t acc[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), acc);
        tmem_wait_ld();
        if (c == 3) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[grp]);  // the accumulator may be reused
        }
        if (coarse) {
          // every anchor scores every coarse row: the scores go out dense,
          // 128 bytes a thread per chunk
          if (r < g.R) {
            float* dst = g.coarse + (long long)r * g.coarse_tiles * kBN + n0 + c * 32;
            const float4* iv4 = reinterpret_cast<const float4*>(inv_v + c * 32);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 iv = iv4[e / 4];
              float4 sc;
              sc.x = fmaf(0.5f, fminf(1.f, fmaxf(-1.f, __uint_as_float(acc[e]) * iv.x * inv_a)), 0.5f);
              sc.y = fmaf(0.5f, fminf(1.f, fmaxf(-1.f, __uint_as_float(acc[e + 1]) * iv.y * inv_a)), 0.5f);
              sc.z = fmaf(0.5f, fminf(1.f, fmaxf(-1.f, __uint_as_float(acc[e + 2]) * iv.z * inv_a)), 0.5f);
              sc.w = fmaf(0.5f, fminf(1.f, fmaxf(-1.f, __uint_as_float(acc[e + 3]) * iv.w * inv_a)), 0.5f);
              *reinterpret_cast<float4*>(dst + e) = sc;
            }
          }
          continue;
        }
        uint32_t x = w[c];
        const unsigned rows = __ballot_sync(kFull, x != 0u);
        if (rows == 0u) continue;
        // the chunk goes to this thread's row of shared memory, then either
        // each thread writes its own row's keys (few per row), or, when the
        // warp has fewer owning rows than its busiest row has keys, the lanes
        // write one row at a time, lane e taking column e (coalesced)
        if (x != 0u) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) sts128(dump + e * 4, acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
        }
        if (__popc(rows) <= __reduce_max_sync(kFull, (unsigned)__popc(x))) {
          __syncwarp();
          const float iv = inv_v[c * 32 + lane];
          const unsigned long long my_out = reinterpret_cast<unsigned long long>(out + k);
          const uint32_t below = (1u << lane) - 1u;
          // four rows at a time, so their loads and math overlap
          for (unsigned rr = rows; rr != 0u;) {
            int qs[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              qs[u] = rr != 0u ? __ffs(rr) - 1 : -1;
              rr &= rr - 1u;
            }
            uint32_t xq[4];
            float aq[4], vq[4];
            unsigned long long oq[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = qs[u] < 0 ? 0 : qs[u];
              xq[u] = qs[u] < 0 ? 0u : __shfl_sync(kFull, x, q);
              aq[u] = __shfl_sync(kFull, inv_a, q);
              oq[u] = __shfl_sync(kFull, my_out, q);
              vq[u] = ((xq[u] >> lane) & 1u) ? lds_f32(dump0 + (uint32_t)(q * kDumpStride * 4 + lane * 4)) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if ((xq[u] >> lane) & 1u) {
                const float cosv = fminf(1.f, fmaxf(-1.f, vq[u] * iv * aq[u]));
                reinterpret_cast<uint64_t*>(oq[u])[__popc(xq[u] & below)] =
                    make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + c * 32 + lane));
              }
            }
          }
          k += __popc(x);
          __syncwarp();  // the dump rows are rewritten by the next chunk
          continue;
        }
        // this row's owned columns, four at a time (their loads and math
        // overlap)
        while (x) {
          int ib[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            ib[u] = x ? __ffs(x) - 1 : -1;
            x &= x - 1;
          }
          float v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] = ib[u] >= 0 ? lds_f32(dump + ib[u] * 4) * inv_v[c * 32 + ib[u]] : 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (ib[u] >= 0) {
              const float cosv = fminf(1.f, fmaxf(-1.f, v[u] * inv_a));
              out[k + u] = make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + c * 32 + ib[u]));
            }
          }
          k += (ib[0] >= 0) + (ib[1] >= 0) + (ib[2] >= 0) + (ib[3] >= 0);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(epi_done);  // this warp reads TMEM no more
  }

  // teardown: the TMEM is freed only after every epilogue warp has said (on
  // an mbarrier) that it reads no more; warps 0 and 1 reconverge first, as
  // lane 0 ran the producer / MMA loop alone
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!mbar_wait_bounded(epi_done, 0, g.wait_ns)) flag_error(g.err, kErrTimeout);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- per-anchor top-K ----------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kSelStage = 6144;                    // keys of a row held in registers,
constexpr int kRegKeys = kSelStage / kSelThreads;  // 24 per thread
constexpr int kBuckets = 2048;                     // linear buckets over a row's score range
constexpr int kTieCap = 512;                       // boundary-bucket keys ranked exactly

struct SelArgs {
  const uint64_t* keys;  // [R][cap] each anchor's candidate keys, contiguous
  const int* offsets;    // [R][mtiles + 1]: entry mtiles is the anchor's count
  int mtiles;
  long long cap;
  int K;
  int* idx;
  float* top;
  int* err;
};

// Visits every candidate key of a row, warp-uniformly (every lane of a warp
// runs the same iterations; `active` marks real keys): the path for rows
// longer than the register copy.
template <typename F>
__device__ __forceinline__ void for_each_row_key(const uint64_t* row, int n, F&& fn) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j0 = warp * 32; j0 < n; j0 += kSelThreads) {
    const int j = j0 + lane;
    const bool active = j < n;
    fn(active, active ? row[j] : 0ull);
  }
}

// One CTA per anchor. The row's keys go straight into registers (24 keys a
// thread, coalesced loads of the contiguous list). One pass of linear
// buckets over the row's score range finds the bucket holding the K-th key;
// keys above it are selected, the boundary bucket's keys are ranked exactly;
// the K winners are sorted (warp bitonic lists + merge ranks). Rows of more
// than 24 keys a thread take the same passes over the list, with a radix
// select on the 64-bit keys when a bucket holds too many ties.
__global__ void __launch_bounds__(kSelThreads) select_rows_kernel(const SelArgs a) {
  __shared__ int hist[kBuckets];
  __shared__ int s_bin, s_above;
  __shared__ int s_sel_n, s_tie_n;
  __shared__ int s_wsum[kSelThreads / 32];
  __shared__ uint64_t s_lo[kSelThreads / 32], s_hi[kSelThreads / 32];
  __shared__ uint64_t s_sel[kMaxK];
  __shared__ uint64_t s_tie[kTieCap];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int K = a.K;
  const uint64_t* row = a.keys + (long long)r * a.cap;

  for (int b = tid; b < kBuckets; b += kSelThreads) hist[b] = 0;
  if (tid == 0) {
    s_sel_n = 0;
    s_tie_n = 0;
  }
  // the candidates come from the GEMM grid launched just before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int n = a.offsets[(long long)r * (a.mtiles + 1) + a.mtiles];
  if (n < 0 || n > a.cap) {
    if (tid == 0) flag_error(a.err, kErrBadIndex);
    n = n < 0 ? 0 : (int)a.cap;
  }
  const bool staged = n <= kSelStage;

  // ---- this thread's keys (rows of at most 24 keys a thread): keys tid,
  // tid + 256, ... of the list (coalesced)
  uint64_t key[kRegKeys];
  uint32_t vmask = 0u;  // bit u: key[u] holds a candidate
  uint64_t lo = ~0ull, hi = 0ull;
  if (staged) {
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) {
      const int pos = tid + u * kSelThreads;
      key[u] = pos < n ? row[pos] : 0ull;
      vmask |= (pos < n ? 1u : 0u) << u;
    }
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) {
      if ((vmask >> u) & 1u) {
        lo = key[u] < lo ? key[u] : lo;
        hi = key[u] > hi ? key[u] : hi;
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) key[u] = 0ull;
    for_each_row_key(row, n, [&](bool active, uint64_t k) {
      if (active) {
        lo = k < lo ? k : lo;
        hi = k > hi ? k : hi;
      }
    });
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
  lo = s_lo[0];
  hi = s_hi[0];
#pragma unroll
  for (int w = 1; w < kSelThreads / 32; ++w) {
    lo = s_lo[w] < lo ? s_lo[w] : lo;
    hi = s_hi[w] > hi ? s_hi[w] : hi;
  }
  const int m = min(K, n);
  // visits every key of the row warp-uniformly: registers, or the list
  auto visit = [&](auto&& fn) {
    if (staged) {
#pragma unroll
      for (int u = 0; u < kRegKeys; ++u) fn(((vmask >> u) & 1u) != 0u, key[u]);
    } else {
      for_each_row_key(row, n, fn);
    }
  };

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
    visit([&](bool active, uint64_t k) {
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
    // keys above the boundary bucket to s_sel, the boundary bucket's to
    // s_tie; one shared-memory atomic per warp and list, a lane's slot is
    // the count of the keys of lower lanes (and earlier rounds) before it
    const unsigned below_me = (1u << lane) - 1u;
    if (staged) {
      // this thread's keys above / in the boundary bucket as bit masks, a
      // warp scan of their counts, one atomic per warp and list
      uint32_t m_above = 0, m_tie = 0;
#pragma unroll
      for (int u = 0; u < kRegKeys; ++u) {
        const int b = ((vmask >> u) & 1u) ? bucket(key[u]) : -1;
        m_above |= (b > bstar ? 1u : 0u) << u;
        m_tie |= (b == bstar ? 1u : 0u) << u;
      }
      const int c_above = __popc(m_above), c_tie = __popc(m_tie);
      int x_above = c_above, x_tie = c_tie;  // inclusive scans over the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(kFull, x_above, o), yt = __shfl_up_sync(kFull, x_tie, o);
        if (lane >= o) {
          x_above += ya;
          x_tie += yt;
        }
      }
      int p_sel = 0, p_tie = 0;
      if (lane == 31) {
        if (x_above) p_sel = atomicAdd(&s_sel_n, x_above);
        if (x_tie) p_tie = atomicAdd(&s_tie_n, x_tie);
      }
      p_sel = __shfl_sync(kFull, p_sel, 31) + x_above - c_above;
      p_tie = __shfl_sync(kFull, p_tie, 31) + x_tie - c_tie;
#pragma unroll
      for (int u = 0; u < kRegKeys; ++u) {
        if ((m_above >> u) & 1u) {
          if (p_sel < kMaxK) s_sel[p_sel] = key[u];
          ++p_sel;
        }
        if ((m_tie >> u) & 1u) {
          if (p_tie < kTieCap) s_tie[p_tie] = key[u];
          ++p_tie;
        }
      }
    } else {
      for_each_row_key(row, n, [&](bool active, uint64_t k) {
        const int b = active ? bucket(k) : -1;
        const unsigned ab = __ballot_sync(kFull, b > bstar), ti = __ballot_sync(kFull, b == bstar);
        int p_sel = 0, p_tie = 0;
        if (lane == 0) {
          if (ab) p_sel = atomicAdd(&s_sel_n, __popc(ab));
          if (ti) p_tie = atomicAdd(&s_tie_n, __popc(ti));
        }
        p_sel = __shfl_sync(kFull, p_sel, 0) + __popc(ab & below_me);
        p_tie = __shfl_sync(kFull, p_tie, 0) + __popc(ti & below_me);
        if (b > bstar && p_sel < kMaxK) s_sel[p_sel] = k;
        if (b == bstar && p_tie < kTieCap) s_tie[p_tie] = k;
      });
    }
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
        visit([&](bool active, uint64_t k) {
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
    visit([&](bool active, uint64_t k) {
      if (active && k >= prefix) {
        const int p = atomicAdd(&s_sel_n, 1);
        if (p < kMaxK) s_sel[p] = k;
      }
    });
    __syncthreads();
  }
  const int sel = m;
  // ---- order the selected keys: a key's place is the number of selected
  // keys above it (each thread reads the list in step, so the loads broadcast)
  int* io = a.idx + (long long)r * K;
  float* to = a.top ? a.top + (long long)r * K : nullptr;
  if (tid < sel) {
    const uint64_t mine_key = s_sel[tid];
    int rank = 0;
#pragma unroll 8
    for (int q = 0; q < sel; ++q) rank += s_sel[q] > mine_key ? 1 : 0;
    if (rank < K) {
      io[rank] = (int)key_index(mine_key);
      if (to) to[rank] = key_score(mine_key);
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
    e = cudaFuncSetAttribute(score_pool_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(score_pool_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    ready[dev] = true;
  }
  return cudaSuccess;
}

// Owned blocks of each anchor before each 128-block tile, and its total:
// offsets[r][t] = popcount of mask row r over tiles 0 .. t-1 (bits < N),
// offsets[r][mtiles] = the row's total. One CTA per anchor, a contiguous run
// of tiles per thread, then a block scan. This is where the GEMM's epilogue
// writes each tile's keys in the anchor's contiguous list.
__global__ void __launch_bounds__(kSelThreads) pool_offsets_kernel(const uint32_t* mask, int N, int mask_words,
                                                                   int mtiles, int mask_vec, int* offsets) {
  constexpr int kTilesPerThread = 4;  // a run of tiles loaded together (more: a second round)
  __shared__ int s_wsum[kSelThreads / 32];
  // the GEMM may be scheduled now: only its epilogue reads these offsets,
  // after waiting for this grid (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t* mrow = mask + (long long)r * mask_words;
  int* orow = offsets + (long long)r * (mtiles + 1);
  // owned blocks of tile t: its four mask words (one 16-byte load when the
  // rows allow it), bits past N dropped
  auto tile_count = [&](int t) {
    uint32_t w[4];
    if (mask_vec) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(mrow) + t);
      w[0] = x.x;
      w[1] = x.y;
      w[2] = x.z;
      w[3] = x.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = t * 4 + q < mask_words ? __ldg(mrow + t * 4 + q) : 0u;
    }
    int c = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int lim = N - (t * 4 + q) * 32;
      c += lim <= 0 ? 0 : __popc(lim >= 32 ? w[q] : (w[q] & ((1u << lim) - 1u)));
    }
    return c;
  };
  const int per = (mtiles + kSelThreads - 1) / kSelThreads;
  const int t0 = min(mtiles, tid * per), t1 = min(mtiles, t0 + per);
  int cnt[kTilesPerThread];
  int mine = 0;
#pragma unroll
  for (int u = 0; u < kTilesPerThread; ++u) {
    cnt[u] = t0 + u < t1 ? tile_count(t0 + u) : 0;
    mine += cnt[u];
  }
  for (int t = t0 + kTilesPerThread; t < t1; ++t) mine += tile_count(t);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int base = incl - mine, total = 0;
#pragma unroll
  for (int w = 0; w < kSelThreads / 32; ++w) {
    if (w < warp) base += s_wsum[w];
    total += s_wsum[w];
  }
#pragma unroll
  for (int u = 0; u < kTilesPerThread; ++u) {
    if (t0 + u < t1) {
      orow[t0 + u] = base;
      base += cnt[u];
    }
  }
  for (int t = t0 + kTilesPerThread; t < t1; ++t) {
    orow[t] = base;
    base += tile_count(t);
  }
  if (tid == 0) orow[mtiles] = total;
}

// Work split of the shared-pool scorer: MT M-tiles of 128 anchors, P CTAs
// per M-tile (one CTA per SM in all), CTA p of an M-tile taking tiles p,
// p + P, ... (split into kGroups contiguous ranges). The workspace holds the
// offsets [R][mtiles + 1], then each anchor's list of up to N keys.
struct PoolLayout {
  int tiles, MT, P, mtiles;
  size_t offsets_bytes, bytes;
};

PoolLayout pool_layout(int R, int rows, int N) {
  PoolLayout L;
  L.tiles = (rows + kBN - 1) / kBN;
  L.mtiles = (N + kBN - 1) / kBN;
  L.MT = (R + kBM - 1) / kBM;
  L.P = L.tiles == 0 ? 0 : std::max(1, std::min(L.tiles, sm_count() / std::max(1, L.MT)));
  L.offsets_bytes = (sizeof(int) * (size_t)R * (size_t)(L.mtiles + 1) + 255) & ~size_t(255);
  L.bytes = L.offsets_bytes + sizeof(uint64_t) * (size_t)R * (size_t)N;
  return L;
}

}  // namespace

size_t batched_workspace_bytes(int R, int rows, int N) { return pool_layout(R, rows, N).bytes; }

cudaError_t launch_pool_gemm(const uint16_t* A, const uint16_t* V, int rows, const uint32_t* mask, int R, int N,
                             int coarse_rows, float* coarse, void* ws, int* err, cudaStream_t s, PoolLists* out) {
  const PoolLayout L = pool_layout(R, rows, N);
  int* offsets = static_cast<int*>(ws);
  uint64_t* keys = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + L.offsets_bytes);
  *out = PoolLists{keys, offsets, L.mtiles, (long long)N};
  if (R == 0) return cudaSuccess;
  cudaError_t e = setup_gemm();
  if (e != cudaSuccess) return e;
  const int mask_words = (N + 31) / 32;
  const int mask_vec = (mask_words % 4 == 0 && reinterpret_cast<uintptr_t>(mask) % 16 == 0) ? 1 : 0;
  pool_offsets_kernel<<<R, kSelThreads, 0, s>>>(mask, N, mask_words, L.mtiles, mask_vec, offsets);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (L.P > 0) {
    CUtensorMap ma, mv;
    if (!make_map(&ma, A, R) || !make_map(&mv, V, rows)) return cudaErrorInvalidValue;
    GemmArgs g{mask, R, N, mask_words, L.tiles, coarse_rows, (rows - N) / kBN, coarse, offsets, L.mtiles, keys,
               mask_vec, wait_limit_ns(), err};
    // programmatic dependent launch: the GEMM's producer and MMA start while
    // the offsets kernel runs; the epilogue waits for it (griddepcontrol.wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(L.MT * L.P));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = g.coarse_tiles > 0 ? cudaLaunchKernelEx(&cfg, score_pool_kernel<true>, ma, mv, g)
                           : cudaLaunchKernelEx(&cfg, score_pool_kernel<false>, ma, mv, g);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask, int R,
                                      int N, int K, int* idx, float* top, void* ws, int* err,
                                      cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  PoolLists lists;
  cudaError_t e = launch_pool_gemm(A, V, N, mask, R, N, 0, nullptr, ws, err, s, &lists);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the select grid is scheduled while the
  // GEMM drains and waits (griddepcontrol.wait) for its results
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)R);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const SelArgs sa{lists.keys, lists.offsets, lists.mtiles, lists.cap, K, idx, top, err};
  return cudaLaunchKernelEx(&cfg, select_rows_kernel, sa);
}

}  // namespace kk
