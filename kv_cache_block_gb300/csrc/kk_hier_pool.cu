// Hierarchical selection Grid -> Chunk -> Page over a pool shared by many
// anchors ("Key-Key Semantic Affinity" page, §5.1): the representations of
// all three levels are rows of one matrix M, scored against every anchor in
// one tensor-core product, and boolean parent -> child masks filter them.
//
// M (bf16, 128 columns) holds the Grid rows [0, G), the Chunk rows [G, G+C),
// zero rows up to H = the next multiple of 128, then the pool's N blocks.
// A Chunk is chunk_pages consecutive pool blocks, a Grid grid_chunks
// consecutive Chunks; a Chunk's row is the mean of its blocks' rows and a
// Grid's the mean of its Chunks' (pool_reps_kernel, float32 sums rounded
// once to bf16).
//
// The product is the shared-pool GEMM of kk_batched.cu with the coarse rows
// in front: every anchor gets the scores of all coarse rows (a dense matrix)
// and a key (score, row) for each block its mask allows.
// hier_pool_select_kernel then takes one anchor per CTA: a coarse member is
// active when it covers an allowed block (and, for a Chunk, its Grid was
// kept); each level keeps ceil(n * permille / 1000) of its n active members
// by a radix select on the 64-bit keys; the allowed blocks of kept Chunks are
// listed in shared memory and the best of them written out.
#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kCols = 128;        // head_dim of the shared pool
constexpr int kRepThreads = 256;  // 16 column octets x 16 row slots
constexpr int kRepSlots = kRepThreads / (kCols / 8);
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPageStage = 4096;  // active blocks of an anchor listed in shared memory

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// Sum of rows [j0, j1) of the pool, columns 8*oct .. 8*oct+7, over the rows
// of this thread's slot (four rows in flight per thread).
__device__ __forceinline__ void sum_rows(const uint16_t* V, int j0, int j1, int slot, int oct, float (&acc)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int j = j0 + slot; j < j1; j += 4 * kRepSlots) {
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int jj = j + u * kRepSlots;
      x[u] = jj < j1 ? __ldg(reinterpret_cast<const uint4*>(V + (long long)jj * kCols + oct * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(w[q]);
        acc[2 * q + 1] += bf16_hi(w[q]);
      }
    }
  }
}

// CTA b < G: Grid b, the mean over its Chunks of each Chunk's mean block;
// G <= b < G + C: Chunk b - G; the last CTA zeroes rows [G + C, H).
__global__ void __launch_bounds__(kRepThreads) pool_reps_kernel(uint16_t* M, int N, int cp, int gc, int G, int C,
                                                               int H) {
  __shared__ float s_red[kRepSlots][kCols];
  const int b = blockIdx.x, tid = threadIdx.x;
  if (b == G + C) {
    for (long long i = tid; i < (long long)(H - G - C) * kCols; i += kRepThreads)
      M[(long long)(G + C) * kCols + i] = 0;
    return;
  }
  const uint16_t* V = M + (long long)H * kCols;
  const int oct = tid % (kCols / 8), slot = tid / (kCols / 8);
  float out[8];
  const int c0 = b < G ? b * gc : b - G;
  const int c1 = b < G ? min(C, c0 + gc) : c0 + 1;
#pragma unroll
  for (int e = 0; e < 8; ++e) out[e] = 0.f;
  for (int c = c0; c < c1; ++c) {
    const int j0 = c * cp, j1 = min(N, j0 + cp);
    float part[8];
    sum_rows(V, j0, j1, slot, oct, part);
    const float inv = 1.f / (float)(j1 - j0);
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = fmaf(part[e], inv, out[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_red[slot][oct * 8 + e] = out[e];
  __syncthreads();
  if (tid < kCols) {
    float x = 0.f;
#pragma unroll
    for (int q = 0; q < kRepSlots; ++q) x += s_red[q][tid];
    M[(long long)b * kCols + tid] = f32_to_bf16_rn(x / (float)(c1 - c0));
  }
}

struct HierPoolArgs {
  PoolLists lists;
  const float* coarse;   // [R][H] scores of the coarse rows
  const uint32_t* mask;  // [R][ceil(N/32)]
  int N, G, C, H, cp, gc;
  int permille[3];
  int K;
  int* idx;   // [R][K] pool ids
  float* top; // [R][K] or null
  int* kept;  // [R] or null
  int* err;
};

// Whether any bit in [lo, hi) of a mask row is set (lo < hi).
__device__ __forceinline__ bool range_any(const uint32_t* row, int lo, int hi) {
  const int w0 = lo >> 5, w1 = (hi - 1) >> 5;
  for (int w = w0; w <= w1; ++w) {
    uint32_t x = __ldg(row + w);
    if (w == w0) x &= kFull << (lo & 31);
    if (w == w1 && (hi & 31)) x &= (1u << (hi & 31)) - 1u;
    if (x) return true;
  }
  return false;
}

__device__ __forceinline__ bool bit(const uint32_t* bits, int i) { return (bits[i >> 5] >> (i & 31)) & 1u; }

// The smallest key T such that exactly k of the keys `visit` offers as
// active are >= T (keys distinct, 1 <= k <= active count): a radix select on
// 8-bit digits, most significant first, stopping as soon as a digit's bucket
// holds exactly the keys still needed. visit(fn) calls fn(active, key) for
// every candidate this thread owns.
template <typename Visit>
__device__ uint64_t radix_kth(Visit&& visit, int k, int* hist, int* s_pick) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t prefix = 0ull, pmask = 0ull;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
    __syncthreads();
    visit([&](bool active, uint64_t key) {
      if (active && (key & pmask) == prefix) atomicAdd(&hist[(int)((key >> shift) & 255)], 1);
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
          s_pick[0] = lane * 8 + b;
          s_pick[1] = above;
        }
        above += hb;
      }
    }
    __syncthreads();
    const int b = s_pick[0];
    need -= s_pick[1];
    prefix |= (uint64_t)b << shift;
    pmask |= (uint64_t)0xFF << shift;
    const bool exact = hist[b] == need;
    __syncthreads();
    if (exact) break;
  }
  return prefix;
}

__global__ void __launch_bounds__(kThreads) hier_pool_select_kernel(const HierPoolArgs a) {
  extern __shared__ __align__(16) uint64_t s_dyn[];
  uint64_t* s_pk = s_dyn;                                              // [kPageStage] active block keys
  float* s_cs = reinterpret_cast<float*>(s_dyn + kPageStage);          // [kHierPoolCoarseMax] coarse scores
  auto coarse_key = [&](int x) { return make_key(s_cs[x], (uint32_t)x); };
  __shared__ uint32_t s_call[kHierPoolCoarseMax / 32];  // Chunks covering an allowed block
  __shared__ uint32_t s_gall[kHierPoolCoarseMax / 32];  // Grids covering an allowed block
  __shared__ uint32_t s_ckept[kHierPoolCoarseMax / 32];
  __shared__ uint32_t s_gkept[kHierPoolCoarseMax / 32];
  __shared__ int hist[256], s_pick[2], s_tmp[kWarps], s_np, s_nout;
  __shared__ uint64_t s_out[kMaxK];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G, C = a.C, N = a.N;
  const int nco = G + C;
  const int cwords = (C + 31) / 32, gwords = (G + 31) / 32;
  for (int w = tid; w < cwords; w += kThreads) {
    s_call[w] = 0u;
    s_ckept[w] = 0u;
  }
  for (int w = tid; w < gwords; w += kThreads) {
    s_gall[w] = 0u;
    s_gkept[w] = 0u;
  }
  if (tid == 0) {
    s_np = 0;
    s_nout = 0;
  }
  // Chunks (then Grids) that cover an allowed block; the mask is an input,
  // not a result of the GEMM, so this overlaps the GEMM's tail
  const uint32_t* mrow = a.mask + (long long)r * ((N + 31) / 32);
  __syncthreads();
  for (int c = tid; c < C; c += kThreads)
    if (range_any(mrow, c * a.cp, min(N, (c + 1) * a.cp))) atomicOr(&s_call[c >> 5], 1u << (c & 31));
  __syncthreads();
  for (int g = tid; g < G; g += kThreads) {
    bool any = false;
    for (int c = g * a.gc; c < min(C, (g + 1) * a.gc) && !any; ++c) any = bit(s_call, c);
    if (any) atomicOr(&s_gall[g >> 5], 1u << (g & 31));
  }

  // the keys come from the GEMM grid launched just before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t* row = a.lists.keys + (long long)r * a.lists.cap;
  int ntot = a.lists.offsets[(long long)r * (a.lists.mtiles + 1) + a.lists.mtiles];
  if (ntot < 0 || ntot > a.lists.cap) {
    if (tid == 0) flag_error(a.err, kErrBadIndex);
    ntot = ntot < 0 ? 0 : (int)a.lists.cap;
  }
  // the coarse rows' scores, as keys (score, row)
  for (int x = tid; x < nco; x += kThreads) s_cs[x] = a.coarse[(long long)r * a.H + x];
  __syncthreads();

  // ---- Grids, then Chunks: keep ceil(n * permille / 1000) of the n active
  auto level = [&](int base, int n, auto&& active, uint32_t* kept_bits, int q) {
    int na = 0;
    for (int i = tid; i < n; i += kThreads) na += active(i) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) na += __shfl_xor_sync(kFull, na, o);
    if (lane == 0) s_tmp[warp] = na;
    __syncthreads();
    na = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) na += s_tmp[w];
    __syncthreads();
    const int m = (int)(((long long)na * q + 999) / 1000);
    if (m == 0) return;
    const uint64_t T = radix_kth(
        [&](auto&& fn) {
          for (int i = tid; i < n; i += kThreads) fn(active(i), coarse_key(base + i));
        },
        m, hist, s_pick);
    for (int i = tid; i < n; i += kThreads)
      if (active(i) && coarse_key(base + i) >= T) atomicOr(&kept_bits[i >> 5], 1u << (i & 31));
    __syncthreads();
  };
  level(0, G, [&](int g) { return bit(s_gall, g); }, s_gkept, a.permille[0]);
  level(G, C, [&](int c) { return bit(s_call, c) && bit(s_gkept, c / a.gc); }, s_ckept, a.permille[1]);

  // ---- blocks: the allowed blocks of kept Chunks (the segments hold only
  // blocks' keys), listed in shared memory while they fit
  auto page_active = [&](uint64_t k) {
    const long long i = (long long)key_index(k) - a.H;
    return i >= 0 && i < N && bit(s_ckept, (int)(i / a.cp));
  };
  // Each thread takes keys tid, tid + 256, ... of the anchor's list
  // (coalesced), eight loads in flight.
  auto visit_run = [&](auto&& fn) {
    constexpr int kBatch = 8;
    for (int p0 = tid; p0 < ntot; p0 += kBatch * kThreads) {
      uint64_t v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int pos = p0 + u * kThreads;
        v[u] = pos < ntot ? row[pos] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (p0 + u * kThreads < ntot) fn(page_active(v[u]), v[u]);
    }
  };
  visit_run([&](bool act, uint64_t k) {
    if (act) {
      const int q = atomicAdd(&s_np, 1);
      if (q < kPageStage) s_pk[q] = k;
    }
  });
  __syncthreads();
  const int np = s_np;
  const bool staged = np <= kPageStage;
  const int m_keep = (int)(((long long)np * a.permille[2] + 999) / 1000);
  const int m = min(a.K, m_keep);
  auto visit_pages = [&](auto&& fn) {
    if (staged) {
      for (int i = tid; i < np; i += kThreads) fn(true, s_pk[i]);
    } else {
      visit_run(fn);
    }
  };
  if (m > 0) {
    const uint64_t T = radix_kth(visit_pages, m, hist, s_pick);
    visit_pages([&](bool act, uint64_t k) {
      if (act && k >= T) {
        const int q = atomicAdd(&s_nout, 1);
        if (q < kMaxK) s_out[q] = k;
      }
    });
    __syncthreads();
  }
  // ---- the m winners in order: a key's place is the number of winners
  // above it (each thread reads the list in step, so the loads broadcast)
  const int got = min(s_nout, kMaxK);
  if (tid == 0 && got != m) flag_error(a.err, kErrBadIndex);  // the select lost or gained a key
  int* io = a.idx + (long long)r * a.K;
  float* to = a.top ? a.top + (long long)r * a.K : nullptr;
  const int mm = min(m, got);
  if (tid < mm) {
    const uint64_t mine = s_out[tid];
    int rank = 0;
#pragma unroll 8
    for (int q = 0; q < mm; ++q) rank += s_out[q] > mine ? 1 : 0;
    if (rank < a.K) {
      io[rank] = (int)(key_index(mine) - (uint32_t)a.H);
      if (to) to[rank] = key_score(mine);
    }
  }
  for (int i = m + tid; i < a.K; i += kThreads) {
    io[i] = -1;
    if (to) to[i] = -__int_as_float(0x7f800000);
  }
  if (tid == 0 && a.kept) a.kept[r] = m_keep;
}

}  // namespace

size_t hier_pool_workspace_bytes(int R, int N, int cp, int gc) {
  const int H = hier_pool_coarse_rows(N, cp, gc);
  const size_t gemm = (batched_workspace_bytes(R, H + N, N) + 255) & ~size_t(255);
  return gemm + sizeof(float) * (size_t)R * (size_t)H;
}

int hier_pool_coarse_rows(int N, int cp, int gc) {
  if (N <= 0) return 0;
  const int C = (N + cp - 1) / cp, G = (C + gc - 1) / gc;
  return (G + C + 127) / 128 * 128;
}

cudaError_t launch_hier_pool_reps(uint16_t* M, int N, int cp, int gc, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  const int C = (N + cp - 1) / cp, G = (C + gc - 1) / gc;
  const int H = hier_pool_coarse_rows(N, cp, gc);
  pool_reps_kernel<<<G + C + 1, kRepThreads, 0, s>>>(M, N, cp, gc, G, C, H);
  return cudaGetLastError();
}

cudaError_t launch_hier_select_pool(const uint16_t* A, const uint16_t* M, const uint32_t* mask, int R, int N,
                                    int cp, int gc, const int* permille, int K, int* idx, float* top, int* kept,
                                    void* ws, int* err, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int C = N > 0 ? (N + cp - 1) / cp : 0, G = C > 0 ? (C + gc - 1) / gc : 0;
  const int H = hier_pool_coarse_rows(N, cp, gc);
  PoolLists lists;
  float* coarse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                           ((batched_workspace_bytes(R, H + N, N) + 255) & ~size_t(255)));
  cudaError_t e = launch_pool_gemm(A, M, H + N, mask, R, N, G + C, coarse, ws, err, s, &lists);
  if (e != cudaSuccess) return e;
  constexpr int kDyn = (int)(sizeof(uint64_t) * kPageStage + sizeof(float) * kHierPoolCoarseMax);
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(hier_pool_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
    if (e != cudaSuccess) return e;
    // as much shared memory as the SM has, so that several anchors share an SM
    e = cudaFuncSetAttribute(hier_pool_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  HierPoolArgs ha{lists, coarse, mask, N, G, C, H, cp, gc, {permille[0], permille[1], permille[2]}, K, idx, top, kept, err};
  // programmatic dependent launch: scheduled while the GEMM drains
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)R);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDyn;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hier_pool_select_kernel, ha);
}

}  // namespace kk
