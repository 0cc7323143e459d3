// Hierarchical selection Grid -> Chunk -> Page ("Key-Key Semantic Affinity"
// page, §5.1): a Chunk is `chunk_pages` consecutive blocks of a request, a
// Grid `grid_chunks` consecutive Chunks; a Chunk's representation is the
// mean of its blocks' v_b and a Grid's the mean of its Chunks'
// representations. Every level is scored with the same affinity; a level
// keeps ceil(n * permille / 1000) of its n active members, and only the
// children of kept parents are active at the next level.
//
// grid_reps_kernel builds the Grid level from the Chunk level (the Chunk
// level is kk_coarse_means over the blocks). hier_select_kernel runs the
// three levels for one request per CTA: score the level's active members
// (one warp per member, 16-byte loads), sort their 64-bit keys (score, index)
// in shared memory, keep the best share and mark it; the last level's kept
// blocks are written in kk_topk order.
#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// grid[r][g][d] = mean over chunks c in [g*gc, min((g+1)*gc, C_r)) of
// chunk[r][c][d] (float64 sum), zero past the request's last Grid.
__global__ void __launch_bounds__(kThreads) grid_reps_kernel(const float* chunk, int D, int c_max, int g_max,
                                                             Table bt, int chunk_pages, int grid_chunks,
                                                             float* grid) {
  const int g = blockIdx.x, r = blockIdx.y;
  const int nb = bt.offsets[r + 1] - bt.offsets[r];
  const int C = nb > 0 ? (nb + chunk_pages - 1) / chunk_pages : 0;
  const int c0 = g * grid_chunks, c1 = min(C, c0 + grid_chunks);
  float* out = grid + ((long long)r * g_max + g) * D;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    double acc = 0.0;
    for (int c = c0; c < c1; ++c) acc += (double)chunk[((long long)r * c_max + c) * D + d];
    out[d] = c1 > c0 ? (float)(acc / (double)(c1 - c0)) : 0.f;
  }
}

struct HierArgs {
  const float* vb;
  int vb_rows, D;
  Table bt;
  const float* chunk;  // [R][c_max][D]
  const float* grid;   // [R][g_max][D]
  int c_max, g_max;
  const float* va;     // [R][D]
  int chunk_pages, grid_chunks;
  int permille[3];
  int K;
  int* idx;       // [R][K]
  float* top;     // [R][K] or null
  int* kept;      // [R] or null: blocks the last level keeps
  int* err;
};

// kPer consecutive floats of a global row through the read-only path.
template <int kPer>
__device__ __forceinline__ void load_row_slice(const float* q, float (&x)[kPer]) {
  if constexpr (kPer == 8) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(q)), b = __ldg(reinterpret_cast<const float4*>(q) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else if constexpr (kPer == 4) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(q));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  } else if constexpr (kPer == 2) {
    const float2 a = __ldg(reinterpret_cast<const float2*>(q));
    x[0] = a.x; x[1] = a.y;
  } else {
    x[0] = __ldg(q);
  }
}

// Descending bitonic sort of n keys (padded with 0 to a power of two).
__device__ void sort_desc(uint64_t* keys, int n) {
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  for (int i = n + threadIdx.x; i < p2; i += kThreads) keys[i] = 0ull;
  __syncthreads();
  for (int k = 2; k <= p2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < p2; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) hier_select_kernel(const HierArgs a) {
  constexpr int kPer = D / 32;
  extern __shared__ __align__(16) uint64_t s_keys[];  // [kHierMax]
  __shared__ float s_va[D];
  __shared__ uint32_t s_gbits[kHierMax / 32];  // kept Grids
  __shared__ uint32_t s_cbits[kHierMax / 32];  // kept Chunks
  __shared__ int s_wsum[kWarps];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int off = a.bt.offsets[r];
  int nb = a.bt.offsets[r + 1] - off;
  if (nb < 0 || nb > a.bt.max_blocks) {
    if (tid == 0) flag_error(a.err, kErrBadIndex);
    nb = 0;
  }
  const int C = nb > 0 ? (nb + a.chunk_pages - 1) / a.chunk_pages : 0;
  const int G = C > 0 ? (C + a.grid_chunks - 1) / a.grid_chunks : 0;
  for (int d = tid; d < D; d += kThreads) s_va[d] = a.va[(long long)r * D + d];
  for (int i = tid; i < kHierMax / 32; i += kThreads) {
    s_gbits[i] = 0u;
    s_cbits[i] = 0u;
  }
  __syncthreads();
  float na2 = 0.f;
  float va_l[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    va_l[e] = s_va[lane * kPer + e];
    na2 = fmaf(va_l[e], va_l[e], na2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) na2 += __shfl_xor_sync(kFull, na2, o);
  const float na = sqrtf(na2);

  // keys of up to 16 members whose representations are rows[0..16) (null:
  // empty) in one pass: per-lane partial dots and squared norms, one
  // transposed warp reduction, lane u < 16 forms member u's key
  auto score_keys16 = [&](const float* const (&rows)[16], const uint32_t (&ids)[16]) -> uint64_t {
    float part[32];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      float dot = 0.f, n2 = 0.f;
      if (rows[u]) {
        float x[kPer];
        load_row_slice<kPer>(rows[u] + lane * kPer, x);
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          dot = fmaf(va_l[e], x[e], dot);
          n2 = fmaf(x[e], x[e], n2);
        }
      }
      part[u] = dot;
      part[16 + u] = n2;
    }
#pragma unroll
    for (int n = 32; n > 1; n >>= 1) {
      const int o = n >> 1;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? part[i] : part[i + n / 2];
        const float keep = upper ? part[i + n / 2] : part[i];
        part[i] = keep + __shfl_xor_sync(kFull, send, o);
      }
    }
    const float n2 = __shfl_down_sync(kFull, part[0], 16);
    float cosv = 0.f;
    if (na2 > 0.f && n2 > 0.f) cosv = part[0] / (na * sqrtf(n2));
    cosv = fminf(1.f, fmaxf(-1.f, cosv));
    uint32_t id = 0;
#pragma unroll
    for (int u = 0; u < 16; ++u) id = lane == u ? ids[u] : id;
    return make_key(fmaf(0.5f, cosv, 0.5f), id);
  };

  // One level: the active members are the children of the kept parents
  // (parent p holds members [p * fan, min((p + 1) * fan, n_members)); every
  // parent is kept when `pbits` is null). They are scored (representation
  // row_of(m)) and sorted, and the best ceil(n * permille / 1000) are marked
  // in `bits` (when given); returns the number kept.
  auto level = [&](int n_parents, int fan, int n_members, const uint32_t* pbits, auto&& row_of, uint32_t* bits,
                   int permille) -> int {
    // list the active members' indices in s_keys (each slot becomes the
    // member's key below): one thread per parent, a block scan of the counts
    int n = 0;
    for (int base = 0; base < n_parents; base += kThreads) {
      const int p = base + tid;
      int cnt = 0;
      if (p < n_parents && (!pbits || ((pbits[p >> 5] >> (p & 31)) & 1u)))
        cnt = max(0, min(fan, n_members - p * fan));
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_wsum[warp] = incl;
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        before += w < warp ? s_wsum[w] : 0;
        total += s_wsum[w];
      }
      const int slot = n + before + incl - cnt;
      for (int c = 0; c < cnt; ++c) s_keys[slot + c] = (uint64_t)(uint32_t)(p * fan + c);  // index for now
      n += total;
      __syncthreads();
    }
    // score the active members, sixteen per warp at a time, replacing each
    // slot by the member's key
    for (int i0 = warp * 16; i0 < n; i0 += kWarps * 16) {
      const float* rows[16];
      uint32_t ids[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const bool have = i0 + u < n;
        ids[u] = have ? (uint32_t)s_keys[i0 + u] : 0u;
        rows[u] = have ? row_of((int)ids[u]) : nullptr;
      }
      __syncwarp();
      const uint64_t key = score_keys16(rows, ids);
      if (lane < 16 && i0 + lane < n) s_keys[i0 + lane] = key;
    }
    __syncthreads();
    sort_desc(s_keys, n);
    const int k = (int)(((long long)n * permille + 999) / 1000);
    if (bits)
      for (int i = tid; i < k; i += kThreads) {
        const uint32_t m = key_index(s_keys[i]);
        atomicOr(&bits[m >> 5], 1u << (m & 31));
      }
    __syncthreads();
    return k;
  };

  const long long rrow = (long long)r;
  level(G, 1, G, nullptr, [&](int g) { return a.grid + (rrow * a.g_max + g) * D; }, s_gbits, a.permille[0]);
  level(G, a.grid_chunks, C, s_gbits, [&](int c) { return a.chunk + (rrow * a.c_max + c) * D; }, s_cbits,
        a.permille[1]);
  const int kp = level(
      C, a.chunk_pages, nb, s_cbits,
      [&](int j) -> const float* {
        const int pg = a.bt.pages[off + j];
        if (pg < 0 || pg >= a.vb_rows) {
          flag_error(a.err, kErrBadIndex);
          return nullptr;
        }
        return a.vb + (long long)pg * D;
      },
      nullptr, a.permille[2]);
  int* io = a.idx + (long long)r * a.K;
  float* to = a.top ? a.top + (long long)r * a.K : nullptr;
  for (int i = tid; i < a.K; i += kThreads) {
    const bool have = i < kp;
    io[i] = have ? (int)key_index(s_keys[i]) : -1;
    if (to) to[i] = have ? key_score(s_keys[i]) : -__int_as_float(0x7f800000);
  }
  if (tid == 0 && a.kept) a.kept[r] = kp;
}

template <int D>
cudaError_t launch_select_t(const HierArgs& a, cudaStream_t s) {
  constexpr int smem = kHierMax * (int)sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(hier_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  hier_select_kernel<D><<<a.bt.R, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grid_reps(const float* chunk, int D, int c_max, int g_max, const Table& bt, int chunk_pages,
                             int grid_chunks, float* grid, cudaStream_t s) {
  if (bt.R == 0 || g_max == 0) return cudaSuccess;
  grid_reps_kernel<<<dim3(g_max, bt.R), kThreads, 0, s>>>(chunk, D, c_max, g_max, bt, chunk_pages, grid_chunks,
                                                          grid);
  return cudaGetLastError();
}

cudaError_t launch_hier_select(const float* vb, int D, int vb_rows, const Table& bt, const float* chunk,
                               const float* grid, int c_max, int g_max, const float* va, int chunk_pages,
                               int grid_chunks, const int* permille, int K, int* idx, float* top, int* kept,
                               int* err, cudaStream_t s) {
  if (bt.R == 0) return cudaSuccess;
  HierArgs a{vb, vb_rows, D, bt, chunk, grid, c_max, g_max, va, chunk_pages, grid_chunks,
             {permille[0], permille[1], permille[2]}, K, idx, top, kept, err};
  switch (D) {
    case 32: return launch_select_t<32>(a, s);
    case 64: return launch_select_t<64>(a, s);
    case 128: return launch_select_t<128>(a, s);
    case 256: return launch_select_t<256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kk
