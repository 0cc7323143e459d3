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
// three levels for one request per thread-block cluster (one CTA unless a
// few long requests leave SMs idle): every CTA lists the level's active
// members, scores its share (sixteen per warp, one transposed reduction) and
// stores the 64-bit keys (score, index) into the leader's shared memory; the
// leader finds the k-th largest key (one counting pass for short lists, else
// a radix select), keeps the best share and sends the kept bitmap to every
// CTA. The last level's first K kept blocks are written in kk_topk order:
// ranked at the leader, or, when a cluster scored a long last level and at
// most 32 are written, folded from every CTA's top-32 list.
#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"
#include "kk_warp.cuh"

namespace kk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHierOut = 2048;  // output blocks ordered by rank counting (more: a full sort)

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

__device__ __forceinline__ uint64_t lds_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// Descending bitonic sort of n keys in shared memory (padded with 0 to a
// power of two). Each stage walks the p2/2 compare-exchange pairs, eight per
// thread at a time: all eight pairs are loaded before any is stored, so the
// loads overlap.
__device__ __forceinline__ void sort_desc(uint64_t* keys_ptr, int n) {
  constexpr int kBatch = 8;
  const uint32_t keys = smem_u32(keys_ptr);
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  for (int i = n + threadIdx.x; i < p2; i += kThreads) sts_u64(keys + i * 8, 0ull);
  __syncthreads();
  const int pairs = p2 >> 1;
  for (int k = 2; k <= p2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int q0 = threadIdx.x; q0 < pairs; q0 += kThreads * kBatch) {
        int lo[kBatch];
        uint64_t a[kBatch], b[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int q = q0 + u * kThreads;
          lo[u] = q < pairs ? (((q & ~(j - 1)) << 1) | (q & (j - 1))) : -1;  // j is a power of two
          a[u] = lo[u] >= 0 ? lds_u64(keys + lo[u] * 8) : 0ull;
          b[u] = lo[u] >= 0 ? lds_u64(keys + (lo[u] + j) * 8) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (lo[u] < 0) continue;
          const bool desc = (lo[u] & k) == 0;
          if (desc ? (a[u] < b[u]) : (a[u] > b[u])) {
            sts_u64(keys + lo[u] * 8, b[u]);
            sts_u64(keys + (lo[u] + j) * 8, a[u]);
          }
        }
      }
      __syncthreads();
    }
  }
}

// The smallest key T such that exactly k of keys[0..n) (distinct, in shared
// memory) are >= T. Up to one key a thread: T is the key with k - 1 keys
// above it (one pass of counting). Longer lists: a radix select on 8-bit
// digits, the first just below the bits every key shares (found by a min /
// max pass, so no pass is spent on a digit every key has in common), stopping
// as soon as a digit's bucket holds exactly the keys still needed. `hist` is
// 256 ints of shared memory, `s_sel` two ints; k in [1, n].
__device__ __forceinline__ uint64_t kth_largest(const uint64_t* keys_ptr, int n, int k, int* hist, int* s_sel) {
  __shared__ uint64_t s_lo[kWarps], s_hi[kWarps], s_res;
  const uint32_t keys = smem_u32(keys_ptr);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n <= kThreads) {
    if (tid < n) {
      const uint64_t key = lds_u64(keys + tid * 8);
      int above = 0;
#pragma unroll 8
      for (int q = 0; q < n; ++q) above += lds_u64(keys + q * 8) > key ? 1 : 0;
      if (above == k - 1) s_res = key;
    }
    __syncthreads();
    const uint64_t res = s_res;
    __syncthreads();  // s_res is rewritten by the next call
    return res;
  }
  uint64_t lo = ~0ull, hi = 0ull;
  for (int i = tid; i < n; i += kThreads) {
    const uint64_t key = lds_u64(keys + i * 8);
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
  if (lo == hi) return lo;
  const int common = __clzll(lo ^ hi);  // leading bits every key shares
  uint64_t pmask = common == 0 ? 0ull : ~0ull << (64 - common);
  uint64_t prefix = hi & pmask;
  int need = k;
  for (int shift = 56 - common;; shift -= 8) {
    const int sh = shift < 0 ? 0 : shift;  // the last digit may overlap bits already fixed
    for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint64_t key = lds_u64(keys + i * 8);
      if ((key & pmask) == prefix) atomicAdd(&hist[(int)((key >> sh) & 255)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // counts above each lane's 8 buckets (255 .. 0 from the top)
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) hier_select_kernel(const HierArgs a) {
  constexpr int kPer = D / 32;
  extern __shared__ __align__(16) uint64_t s_keys[];  // [kHierMax] level list, then [kHierOut] output stage
  __shared__ float s_va[D];
  __shared__ uint32_t s_gbits[kHierMax / 32];  // kept Grids
  __shared__ uint32_t s_cbits[kHierMax / 32];  // kept Chunks
  __shared__ int s_wsum[kWarps];
  __shared__ int s_hist[256], s_sel[2], s_cnt;
  const int r = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CL = (int)cluster_size(), crank = (int)cluster_rank();
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
  // parent is kept when `pbits` is null). Every CTA of the cluster lists
  // them; CTA c scores its share and stores the keys into the leader's
  // list; the leader sorts, keeps the best ceil(n * permille / 1000), marks
  // them in `bits` (when given) and copies those words to every CTA. Returns
  // the number kept.
  int n_last = 0;  // members of the most recent level
  auto level = [&](int n_parents, int fan, int n_members, const uint32_t* pbits, auto&& row_of, auto&& prep,
                   uint32_t* bits, int n_bits, int permille) -> int {
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
      if (fan >= 32) {
        // wide parents: the warp writes each listed parent's members together
        for (unsigned todo = __ballot_sync(kFull, cnt > 0); todo != 0u; todo &= todo - 1u) {
          const int src = __ffs(todo) - 1;
          const int c_src = __shfl_sync(kFull, cnt, src), s_src = __shfl_sync(kFull, slot, src);
          const int m0 = __shfl_sync(kFull, p, src) * fan;
          for (int c = lane; c < c_src; c += 32) s_keys[s_src + c] = (uint64_t)(uint32_t)(m0 + c);
        }
      } else {
        for (int c = 0; c < cnt; ++c) s_keys[slot + c] = (uint64_t)(uint32_t)(p * fan + c);  // index for now
      }
      n += total;
      __syncthreads();
    }
    // every CTA has its list before any key lands in the leader's
    cluster_arrive_release();
    cluster_wait_acquire();
    // score this CTA's share, sixteen members per warp at a time
    const int i_lo = (int)((long long)n * crank / CL), i_hi = (int)((long long)n * (crank + 1) / CL);
    const uint32_t keys0 = map_to_rank(smem_u32(s_keys), 0);
    prep(i_lo, i_hi);
    for (int i0 = i_lo + warp * 16; i0 < i_hi; i0 += kWarps * 16) {
      const float* rows[16];
      uint32_t ids[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const bool have = i0 + u < i_hi;
        const uint64_t e = have ? s_keys[i0 + u] : 0ull;
        ids[u] = (uint32_t)e;
        rows[u] = have ? row_of(e) : nullptr;
      }
      __syncwarp();
      const uint64_t key = score_keys16(rows, ids);
      if (lane < 16 && i0 + lane < i_hi) {
        st_cluster_u64(keys0 + (uint32_t)((i0 + lane) * 8), key);
        s_keys[i0 + lane] = key;  // this CTA's own copy of its share (the leader's is the same slot)
      }
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    int k = (int)(((long long)n * permille + 999) / 1000);
    n_last = n;
    if (crank == 0 && bits && k > 0) {
      // the kept members: the k largest keys
      const uint64_t thr = kth_largest(s_keys, n, k, s_hist, s_sel);
      for (int i = tid; i < n; i += kThreads) {
        const uint64_t key = s_keys[i];
        if (key >= thr) {
          const uint32_t m = key_index(key);
          atomicOr(&bits[m >> 5], 1u << (m & 31));
        }
      }
      __syncthreads();
    }
    if (crank == 0) {
      if (bits) {
        for (int q = 1; q < CL; ++q)
          for (int i = tid; i < (n_bits + 31) / 32; i += kThreads)
            st_cluster_s32(map_to_rank(smem_u32(&bits[i]), q), (int)bits[i]);
      }
    }
    if (bits) {  // the kept bits reach every CTA before the next level
      cluster_arrive_release();
      cluster_wait_acquire();
    }
    return k;
  };

  // A list entry holds the member's index in its low half; the block level
  // first loads the CTA's share of page ids together into the high halves,
  // so that scoring does not wait for them one group at a time.
  const long long rrow = (long long)r;
  auto no_prep = [](int, int) {};
  level(G, 1, G, nullptr, [&](uint64_t e) { return a.grid + (rrow * a.g_max + (uint32_t)e) * D; }, no_prep, s_gbits,
        G, a.permille[0]);
  level(G, a.grid_chunks, C, s_gbits, [&](uint64_t e) { return a.chunk + (rrow * a.c_max + (uint32_t)e) * D; },
        no_prep, s_cbits, C, a.permille[1]);
  const int kp = level(
      C, a.chunk_pages, nb, s_cbits,
      [&](uint64_t e) -> const float* {
        const int pg = (int)(uint32_t)(e >> 32);
        if (pg < 0 || pg >= a.vb_rows) {
          flag_error(a.err, kErrBadIndex);
          return nullptr;
        }
        return a.vb + (long long)pg * D;
      },
      [&](int i_lo, int i_hi) {
        constexpr int kBatch = 4;
        for (int i0 = i_lo + tid; i0 < i_hi; i0 += kBatch * kThreads) {
          int pg[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kThreads;
            pg[u] = i < i_hi ? a.bt.pages[off + (int)(uint32_t)s_keys[i]] : 0;
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kThreads;
            if (i < i_hi) s_keys[i] = (uint64_t)(uint32_t)s_keys[i] | ((uint64_t)(uint32_t)pg[u] << 32);
          }
        }
        __syncthreads();
      },
      nullptr, 0, a.permille[2]);
  // the first m = min(K, kp) blocks of the last level in kk_topk order
  int* io = a.idx + (long long)r * a.K;
  float* to = a.top ? a.top + (long long)r * a.K : nullptr;
  const int m = min(a.K, kp);
  const int n3 = n_last;
  if (m > 0 && m <= 32 && CL > 1 && n3 > kThreads) {
    // The 32 largest keys of a long list scored by a cluster: every CTA
    // folds the share it scored into one descending 32-key list (runs of 32
    // sorted by warps, the larger 32 of each pair kept, then a tree over the
    // warps) and sends it to the leader, which folds the CL lists the same
    // way. (A short list is ranked at the leader in one counting pass.)
    __shared__ uint64_t s_wl[kWarps][32];
    uint64_t* inbox = s_keys + kHierMax;  // [CL][32] at the leader
    const int i_lo = (int)((long long)n3 * crank / CL), i_hi = (int)((long long)n3 * (crank + 1) / CL);
    uint64_t acc = 0ull;
    for (int c0 = i_lo + warp * 32; c0 < i_hi; c0 += kWarps * 32) {
      const uint64_t k = c0 + lane < i_hi ? s_keys[c0 + lane] : 0ull;
      acc = warp_merge_top32(acc, warp_sort_desc(k, lane), lane);
    }
    auto fold_warps = [&]() {
      s_wl[warp][lane] = acc;
      for (int h = kWarps / 2; h > 0; h >>= 1) {
        __syncthreads();
        if (warp < h) {
          acc = warp_merge_top32(acc, s_wl[warp + h][lane], lane);
          s_wl[warp][lane] = acc;
        }
      }
    };
    fold_warps();
    if (warp == 0) st_cluster_u64(map_to_rank(smem_u32(&inbox[crank * 32 + lane]), 0), acc);
    cluster_arrive_release();
    cluster_wait_acquire();
    if (crank != 0) return;
    acc = 0ull;
    for (int q = warp; q < CL; q += kWarps) acc = warp_merge_top32(acc, inbox[q * 32 + lane], lane);
    fold_warps();
    if (warp == 0 && lane < a.K) {
      const bool have = lane < m;
      io[lane] = have ? (int)key_index(acc) : -1;
      if (to) to[lane] = have ? key_score(acc) : -__int_as_float(0x7f800000);
    }
    for (int i = 32 + tid; i < a.K; i += kThreads) {
      io[i] = -1;
      if (to) to[i] = -__int_as_float(0x7f800000);
    }
    if (tid == 0 && a.kept) a.kept[r] = kp;
    return;
  }
  if (crank != 0) return;
  if (m > 0 && m <= kHierOut) {
    // the m largest keys, staged past the level's list, each written at its
    // rank among them
    const uint64_t thr = kth_largest(s_keys, n3, m, s_hist, s_sel);
    uint64_t* stage = s_keys + kHierMax;
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    for (int i = tid; i < n3; i += kThreads) {
      const uint64_t key = s_keys[i];
      if (key >= thr) stage[atomicAdd(&s_cnt, 1)] = key;
    }
    __syncthreads();
    for (int i = tid; i < m; i += kThreads) {
      const uint64_t key = stage[i];
      int rank = 0;
      for (int q = 0; q < m; ++q) rank += stage[q] > key;
      io[rank] = (int)key_index(key);
      if (to) to[rank] = key_score(key);
    }
  } else if (m > 0) {  // a very long output: sort the whole level
    sort_desc(s_keys, n3);
    for (int i = tid; i < m; i += kThreads) {
      io[i] = (int)key_index(s_keys[i]);
      if (to) to[i] = key_score(s_keys[i]);
    }
  }
  for (int i = m + tid; i < a.K; i += kThreads) {
    io[i] = -1;
    if (to) to[i] = -__int_as_float(0x7f800000);
  }
  if (tid == 0 && a.kept) a.kept[r] = kp;
}

template <int D>
cudaError_t launch_select_t(const HierArgs& a, cudaStream_t s) {
  constexpr int smem = (kHierMax + kHierOut) * (int)sizeof(uint64_t);
  static std::mutex mu;
  static int caps[64][kMaxCluster + 1];  // co-resident clusters of each size, per device (-1: not yet asked)
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      e = cudaFuncSetAttribute(hier_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(hier_select_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
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
        if (cudaOccupancyMaxActiveClusters(&n, hier_select_kernel<D>, &cfg) != cudaSuccess) n = 0;
        (void)cudaGetLastError();  // an unsupported size is not an error here
        caps[dev][cl] = n;
      }
      ready[dev] = true;
    }
  }
  // A cluster per request splits each level's scoring over CL SMs: worth it
  // only for a few long requests (otherwise one CTA per request already
  // fills the GPU).
  int cl = 1;
  const int sms = sm_count();
  for (int c = 2; c <= kMaxCluster; c <<= 1)
    if ((long long)a.bt.R * c <= sms && a.bt.max_blocks >= 256 * c && caps[dev][c] >= a.bt.R) cl = c;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl, a.bt.R);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hier_select_kernel<D>, a);
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
