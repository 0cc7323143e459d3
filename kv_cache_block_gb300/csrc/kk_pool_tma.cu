// Block pooling of many blocks at once ("Key-Key Semantic Affinity" page,
// §2.2 step 1 and §5.2 steps 2-3; per-(layer, head) weights per §3.3 finding
// 2): the same v_b as pool_kernel in kk_pool.cu, from a persistent kernel
// built for writes of hundreds to many thousands of blocks.
//
// One CTA per SM owns a contiguous, balanced range of whole blocks. Warp 0
// streams each block's Keys through a ring of shared-memory stages with tiled
// TMA loads of a 5-D view of the paged cache (dims, token, head, page, layer,
// the last four in order of stride); eight consumer warps sum every stage's
// rows. The bytes in flight per SM are set by the ring (six 32 KB stages), not
// by how many CTAs are resident, so the SMs that still hold blocks at the end
// of a launch draw the bandwidth the finished ones no longer use.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"
#include "kk_tcgen05.cuh"

namespace kk {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = 32 + kConsumers;
constexpr int kStageBytes = 32768;
constexpr int kStages = 6;
constexpr int kRowsPerThread = kStageBytes / (kConsumers * 16);  // 16-byte vectors per thread per stage
constexpr int kMaxD = 256;
constexpr int kTmaSmem = 1024 + kStages * kStageBytes + kMaxLH * 4 + 2 * kConsumerWarps * kMaxD * 4 +
                         2 * kStages * 8 + 16;

// The four strided axes of a K cache; each sits at one of the tensor map's
// positions 1..4 (position 0 is the contiguous axis of the D dims).
enum Dim { kTok = 0, kHead = 1, kPage = 2, kLayer = 3 };

struct PoolTmaArgs {
  const int* pages;
  const int* n_valid;
  const float* head_w;  // [n_sets][L*H] or null (uniform)
  int n_sets;
  const int* w_set;
  float* vb;
  int n;
  int L, H, bs, num_pages;
  int tb, hb, lb;     // tokens, heads and layers per box (tb | bs, hb | H, lb | L)
  int nhb, nlb;       // boxes per block along heads and layers
  int pos[4];         // tensor-map position (1..4) of each Dim
  int ext[5];         // box extent at each tensor-map position
  unsigned long long wait_ns;  // limit of every bounded wait
  long long skip_box;          // failure-detection tests: CTA 0 leaves this box uncopied (-1: none)
  int* err;
};

struct BlockMeta {
  int page, n, wsel;
  bool ok;
};

__device__ __forceinline__ BlockMeta block_meta(const PoolTmaArgs& a, long long i) {
  BlockMeta m;
  m.page = a.pages[i];
  m.n = a.n_valid[i];
  m.wsel = (a.head_w && a.w_set) ? a.w_set[i] : 0;
  m.ok = !(m.n < 0 || m.n > a.bs || m.page < 0 || m.page >= a.num_pages ||
           (a.head_w && (m.wsel < 0 || m.wsel >= a.n_sets)));
  return m;
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Value of tensor-map position p (1..4) for box coordinates given per Dim.
__device__ __forceinline__ int coord_at(const PoolTmaArgs& a, int p, int tok, int head, int page, int layer) {
  return a.pos[kTok] == p ? tok : a.pos[kHead] == p ? head : a.pos[kPage] == p ? page : layer;
}

template <typename T, int D, bool kWeighted>
__global__ void __launch_bounds__(kTmaThreads, 1)
    pool_tma_kernel(const __grid_constant__ CUtensorMap tm, const PoolTmaArgs a) {
  constexpr int ES = elem_bytes<T>();
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int V16 = D / EPV;              // 16-byte vectors per row
  constexpr int RSTEP = kConsumers / V16;   // rows covered by one pass of the consumers
  static_assert(V16 >= 1 && V16 <= 32 && (32 % V16) == 0, "row must be 16..512 bytes");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  float* s_w = reinterpret_cast<float*>(base + kStages * kStageBytes);  // [L*H] weights of the block
  float* s_red = s_w + kMaxLH;                                          // [2][warps][D]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_red + 2 * kConsumerWarps * kMaxD);
  uint64_t* empty = full + kStages;
  int* s_abort = reinterpret_cast<int*>(empty + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long b0 = (long long)a.n * blockIdx.x / gridDim.x;
  const long long b1 = (long long)a.n * (blockIdx.x + 1) / gridDim.x;
  const int LH = a.L * a.H;
  const uint32_t box_bytes = (uint32_t)(a.tb * a.hb * a.lb * D * ES);

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = s_abort;

  if (warp == 0) {
    // ---- producer: one thread issues every box of the CTA's blocks --------
    if (lane == 0) {
      uint32_t k = 0;  // boxes issued
      bool alive = true;
      BlockMeta nx = b0 < b1 ? block_meta(a, b0) : BlockMeta{0, 0, 0, false};
      for (long long i = b0; i < b1 && alive; ++i) {
        const BlockMeta m = nx;
        if (i + 1 < b1) nx = block_meta(a, i + 1);
        if (!m.ok) continue;
        const int nt = (m.n + a.tb - 1) / a.tb;
        for (int lbi = 0; lbi < a.nlb && alive; ++lbi)
          for (int hbi = 0; hbi < a.nhb && alive; ++hbi)
            for (int tbi = 0; tbi < nt; ++tbi) {
              const int st = (int)(k % kStages);
              if ((k >= kStages && !mbar_wait_bounded(&empty[st], ((k / kStages) & 1) ^ 1, a.wait_ns)) ||
                  *abort_flag) {
                if (!*abort_flag) flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
                alive = false;
                break;
              }
              if (blockIdx.x == 0 && (long long)k == a.skip_box) {
                ++k;  // no copy and no arrival: the consumers' wait for this box runs out
                continue;
              }
              const int ct = tbi * a.tb, ch = hbi * a.hb, cl = lbi * a.lb;
              mbar_arrive_expect_tx(&full[st], box_bytes);
              tma_load_5d(stages + st * kStageBytes, &tm, 0, coord_at(a, 1, ct, ch, m.page, cl),
                          coord_at(a, 2, ct, ch, m.page, cl), coord_at(a, 3, ct, ch, m.page, cl),
                          coord_at(a, 4, ct, ch, m.page, cl), &full[st]);
              ++k;
            }
      }
      // no copy may still be writing shared memory when the CTA exits: every
      // box of the last kStages is waited for, each wait bounded (a box whose
      // wait runs out does not end the drain of the ones after it)
      for (uint32_t j = k > (uint32_t)kStages ? k - kStages : 0; j < k; ++j)
        if (!mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, a.wait_ns)) flag_error(a.err, kErrTimeout);
    }
    return;
  }

  // ---- consumers ------------------------------------------------------------
  const int ct = tid - 32, cw = ct >> 5;
  const int col = ct % V16, r0 = ct / V16;
  const int rows = a.tb * a.hb * a.lb;
  // this thread's rows of a box: token offset and (layer, head) offset of each
  int t_off[kRowsPerThread], s_off[kRowsPerThread];
#pragma unroll
  for (int j = 0; j < kRowsPerThread; ++j) {
    int rr = r0 + j * RSTEP, q[5] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int p = 1; p <= 4; ++p) {
      q[p] = rr % a.ext[p];
      rr /= a.ext[p];
    }
    int qt = 0, qh = 0, ql = 0;
#pragma unroll
    for (int p = 1; p <= 4; ++p) {
      if (a.pos[kTok] == p) qt = q[p];
      if (a.pos[kHead] == p) qh = q[p];
      if (a.pos[kLayer] == p) ql = q[p];
    }
    const bool in_box = r0 + j * RSTEP < rows;
    t_off[j] = in_box ? qt : a.bs;  // rows past the box are never valid tokens
    s_off[j] = in_box ? ql * a.H + qh : 0;
  }
  const uint32_t stage0 = smem_u32(stages) + (uint32_t)(r0 * D * ES + col * 16);
  uint32_t k = 0;
  int nred = 0;
  // Every consumer thread walks the same blocks and boxes and meets the same
  // named barriers whatever happens; after a failed wait a warp only stops
  // touching the ring (the error word says why).
  bool alive = true;
  BlockMeta nx = b0 < b1 ? block_meta(a, b0) : BlockMeta{0, 0, 0, false};
  for (long long i = b0; i < b1; ++i) {
    const BlockMeta m = nx;
    if (i + 1 < b1) nx = block_meta(a, i + 1);
    if (!m.ok) {
      if (ct == 0) flag_error(a.err, kErrBadIndex);
      continue;
    }
    if (kWeighted) {
      named_sync(1, kConsumers);  // the previous block's weights are no longer read
      for (int s = ct; s < LH; s += kConsumers) s_w[s] = a.head_w[(long long)m.wsel * LH + s];
      named_sync(1, kConsumers);
    }
    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
    const int nt = (m.n + a.tb - 1) / a.tb;
    for (int lbi = 0; lbi < a.nlb; ++lbi)
      for (int hbi = 0; hbi < a.nhb; ++hbi)
        for (int tbi = 0; tbi < nt; ++tbi, ++k) {
          if (!alive) continue;
          const int st = (int)(k % kStages);
          bool ok = !*abort_flag && mbar_wait_bounded(&full[st], (k / kStages) & 1, a.wait_ns);
          ok = __all_sync(kFull, ok);
          if (!ok) {
            if (lane == 0 && !*abort_flag) flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
            alive = false;
            continue;
          }
          const uint32_t sp = stage0 + (uint32_t)(st * kStageBytes);
          const int tleft = m.n - tbi * a.tb;  // valid tokens from this box's first
          const int sbase = lbi * a.lb * a.H + hbi * a.hb;
          uint4 v[kRowsPerThread];
#pragma unroll
          for (int j = 0; j < kRowsPerThread; ++j)
            v[j] = (r0 + j * RSTEP < rows) ? lds16(sp + (uint32_t)(j * RSTEP * D * ES)) : make_uint4(0, 0, 0, 0);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
          for (int j = 0; j < kRowsPerThread; ++j) {
            if (t_off[j] < tleft) {
              float f[EPV];
              Vec16<T>::unpack(v[j], f);
              const float w = kWeighted ? s_w[sbase + s_off[j]] : 1.f;
#pragma unroll
              for (int e = 0; e < EPV; ++e) acc[e] = fmaf(w, f[e], acc[e]);
            }
          }
        }
    // sum the lanes that share a dim range, then the warps
#pragma unroll
    for (int e = 0; e < EPV; ++e)
#pragma unroll
      for (int o = V16; o < 32; o <<= 1) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
    float* red = s_red + (nred & 1) * kConsumerWarps * D;
    if (lane < V16) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) red[cw * D + col * EPV + e] = acc[e];
    }
    named_sync(1, kConsumers);
    if (!*abort_flag) {
      const float scale = m.n == 0 ? 0.f : (kWeighted ? 1.f / (float)m.n : 1.f / ((float)m.n * (float)LH));
      for (int d = ct; d < D; d += kConsumers) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) s += red[w * D + d];
        a.vb[(long long)m.page * D + d] = s * scale;
      }
    }
    ++nred;
  }
}

// ---- per-(layer, head) sums for the head-variance weights -----------------
// The same ring over the blocks of a block table, writing for every block g
// and (layer, head) slice s the token sum S[g][s][:] and the sum of squares
// Q[g][s] (the inputs of the variance weights). A box holds at most eight
// slices, tokens innermost; each slice of a box is summed by one consumer
// warp (rotated from box to box), which keeps its sums in registers across
// the slice's token boxes and writes them once.
struct SliceTmaArgs {
  Table bt;
  long long total;  // blocks in S / Q (offsets[R])
  int L, H, bs, num_pages;
  int tb, hb, lb, nhb, nlb;
  int pos[4];
  float* S;
  float* Q;
  unsigned long long wait_ns;
  int* err;
};

struct SliceBlock {
  int page, n;
  bool ok, bad;
  bool zero;  // a valid table entry whose page id is out of range: its sums are written as zero
};

// Block g of the table; r is the request holding it, advanced monotonically.
__device__ __forceinline__ SliceBlock slice_block(const SliceTmaArgs& a, long long g, int& r) {
  while (r < a.bt.R && a.bt.offsets[r + 1] <= g) ++r;
  SliceBlock m{0, 0, false, false, false};
  if (r >= a.bt.R) return m;
  const int off = a.bt.offsets[r], nb = a.bt.offsets[r + 1] - off, T = a.bt.seq_lens[r];
  if (off < 0 || nb < 0 || nb > a.bt.max_blocks || (long long)off + nb > a.total || T < 0 ||
      nb != (T + a.bs - 1) / a.bs || g < off) {
    m.bad = true;
    return m;
  }
  m.page = a.bt.pages[g];
  m.n = min(a.bs, T - (int)(g - off) * a.bs);
  m.bad = m.page < 0 || m.page >= a.num_pages;
  m.zero = m.bad;
  m.ok = !m.bad && m.n > 0;
  return m;
}

// first request holding block g (offsets non-decreasing)
__device__ __forceinline__ int request_of(const Table& bt, long long g) {
  int lo = 0, hi = bt.R;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (bt.offsets[mid + 1] <= g) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

template <typename T, int D>
__global__ void __launch_bounds__(kTmaThreads, 1)
    pool_tma_slices_kernel(const __grid_constant__ CUtensorMap tm, const SliceTmaArgs a) {
  constexpr int ES = elem_bytes<T>();
  constexpr int EPV = Vec16<T>::kElems;
  constexpr int V16 = D / EPV;
  constexpr int RPW = 32 / V16;  // rows one warp covers per pass
  static_assert(V16 >= 1 && V16 <= 32 && (32 % V16) == 0, "row must be 16..512 bytes");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  int* s_abort = reinterpret_cast<int*>(empty + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long b0 = a.total * blockIdx.x / gridDim.x;
  const long long b1 = a.total * (blockIdx.x + 1) / gridDim.x;
  const int LH = a.L * a.H;
  const int nsub = a.hb * a.lb;
  const uint32_t box_bytes = (uint32_t)(a.tb * nsub * D * ES);

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = s_abort;
  int r = b0 < b1 ? request_of(a.bt, b0) : a.bt.R;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t k = 0;
      bool alive = true;
      for (long long g = b0; g < b1 && alive; ++g) {
        const SliceBlock m = slice_block(a, g, r);
        if (!m.ok) continue;
        const int nt = (m.n + a.tb - 1) / a.tb;
        for (int lbi = 0; lbi < a.nlb && alive; ++lbi)
          for (int hbi = 0; hbi < a.nhb && alive; ++hbi)
            for (int tbi = 0; tbi < nt; ++tbi) {
              const int st = (int)(k % kStages);
              if ((k >= kStages && !mbar_wait_bounded(&empty[st], ((k / kStages) & 1) ^ 1, a.wait_ns)) ||
                  *abort_flag) {
                if (!*abort_flag) flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
                alive = false;
                break;
              }
              const int ct = tbi * a.tb, ch = hbi * a.hb, cl = lbi * a.lb;
              mbar_arrive_expect_tx(&full[st], box_bytes);
              tma_load_5d(stages + st * kStageBytes, &tm, 0, ct, ch, a.pos[kPage] == 3 ? m.page : cl,
                          a.pos[kPage] == 3 ? cl : m.page, &full[st]);
              ++k;
            }
      }
      for (uint32_t j = k > (uint32_t)kStages ? k - kStages : 0; j < k; ++j)
        if (!mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, a.wait_ns)) flag_error(a.err, kErrTimeout);
    }
    return;
  }

  // ---- consumers: warp cw sums the slice `sub` of a box with
  // (sub + unit) % 8 == cw, unit counting the (layer, head) box groups
  const int cw = warp - 1;
  const int col = lane % V16, rg = lane / V16;
  uint32_t k = 0, unit = 0;
  bool alive = true;
  for (long long g = b0; g < b1; ++g) {
    const SliceBlock m = slice_block(a, g, r);
    if (!m.ok) {
      if (m.bad && cw == 0 && lane == 0) flag_error(a.err, kErrBadIndex);
      if (m.zero) {
        // the request's variance sums read this block as zero rather than
        // whatever an earlier call left in the scratch
        const int ct = tid - 32;
        for (int i = ct; i < LH * D; i += kConsumers) a.S[g * LH * D + i] = 0.f;
        for (int i = ct; i < LH; i += kConsumers) a.Q[g * LH + i] = 0.f;
      }
      continue;
    }
    const int nt = (m.n + a.tb - 1) / a.tb;
    for (int lbi = 0; lbi < a.nlb; ++lbi)
      for (int hbi = 0; hbi < a.nhb; ++hbi, ++unit) {
        const int sub = (int)((cw + kConsumerWarps - (int)(unit % kConsumerWarps)) % kConsumerWarps);
        const bool mine = sub < nsub;
        float acc[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
        float q = 0.f;
        for (int tbi = 0; tbi < nt; ++tbi, ++k) {
          if (!alive) continue;
          const int st = (int)(k % kStages);
          bool ok = !*abort_flag && mbar_wait_bounded(&full[st], (k / kStages) & 1, a.wait_ns);
          ok = __all_sync(kFull, ok);
          if (!ok) {
            if (lane == 0 && !*abort_flag) flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
            alive = false;
            continue;
          }
          if (mine) {
            const int tvalid = min(a.tb, m.n - tbi * a.tb);
            const uint32_t rows = smem_u32(stages + st * kStageBytes) + (uint32_t)((sub * a.tb) * D * ES + col * 16);
#pragma unroll 4
            for (int t = rg; t < tvalid; t += RPW) {
              const uint4 v = lds16(rows + (uint32_t)(t * D * ES));
              float f[EPV];
              Vec16<T>::unpack(v, f);
#pragma unroll
              for (int e = 0; e < EPV; ++e) {
                acc[e] += f[e];
                q = fmaf(f[e], f[e], q);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (mine && alive) {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
#pragma unroll
            for (int o = V16; o < 32; o <<= 1) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(kFull, q, o);
          const int ll = sub / a.hb, hh = sub - ll * a.hb;
          const int sl = (lbi * a.lb + ll) * a.H + hbi * a.hb + hh;
          float* dst = a.S + ((long long)g * LH + sl) * D + col * EPV;
          if (rg == 0) {
#pragma unroll
            for (int e = 0; e < EPV; e += 4)
              *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
          }
          if (lane == 0) a.Q[(long long)g * LH + sl] = q;
        }
      }
  }
}

template <typename T, int D, bool kWeighted>
cudaError_t launch_t(const CUtensorMap& tm, const PoolTmaArgs& a, int grid, cudaStream_t s) {
  static std::mutex mu;
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      e = cudaFuncSetAttribute(pool_tma_kernel<T, D, kWeighted>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTmaSmem);
      if (e != cudaSuccess) return e;
      ready[dev] = true;
    }
  }
  pool_tma_kernel<T, D, kWeighted><<<grid, kTmaThreads, kTmaSmem, s>>>(tm, a);
  return cudaGetLastError();
}

template <typename T, bool kWeighted>
cudaError_t dispatch_d(int D, const CUtensorMap& tm, const PoolTmaArgs& a, int grid, cudaStream_t s) {
  switch (D) {
    case 32: return launch_t<T, 32, kWeighted>(tm, a, grid, s);
    case 64: return launch_t<T, 64, kWeighted>(tm, a, grid, s);
    case 128: return launch_t<T, 128, kWeighted>(tm, a, grid, s);
    case 256: return sizeof(T) == 2 ? launch_t<bf16_t, 256, kWeighted>(tm, a, grid, s) : cudaErrorNotSupported;
    default: return cudaErrorNotSupported;
  }
}

int largest_divisor_at_most(int x, int cap) {
  for (int d = std::min(x, cap); d > 1; --d)
    if (x % d == 0) return d;
  return 1;
}

}  // namespace

namespace {

// Box and tensor map of a paged cache for the TMA pools: box = tokens first,
// then whole heads, then whole layers, up to one stage and max_sub (layer,
// head) slices; the four strided axes sorted by stride.
struct TmaPlan {
  int tb, hb, lb;
  int pos[4];
  int ext[5];
  CUtensorMap tm;
};

bool plan_tma(const KCache& kc, int max_sub, TmaPlan* pl) {
  const int ES = kc.dtype == 1 ? 2 : 4;
  const long long row_bytes = (long long)kc.D * ES;
  if (kc.D > kMaxD || row_bytes % 16 != 0 || row_bytes > 512 || (reinterpret_cast<uintptr_t>(kc.base) & 15))
    return false;
  const long long stride[4] = {kc.sT * ES, kc.sH * ES, kc.sP * ES, kc.sL * ES};
  for (long long b : stride)
    if (b <= 0 || b % 16 != 0 || b >= (1ll << 40)) return false;
  const int rows_cap = (int)std::min<long long>(kStageBytes / row_bytes, 1 << 30);
  int tb = kc.bs;
  if (tb > rows_cap) {
    if ((kc.bs & (kc.bs - 1)) != 0) return false;
    tb = rows_cap;  // a power of two dividing bs
  }
  if (tb > 256) tb = 256;
  if (kc.bs % tb != 0) return false;
  const int hb = tb == kc.bs ? largest_divisor_at_most(kc.H, std::min({256, rows_cap / tb, max_sub})) : 1;
  const int lb = (tb == kc.bs && hb == kc.H)
                     ? largest_divisor_at_most(kc.L, std::min({256, rows_cap / (tb * hb), max_sub / hb}))
                     : 1;
  pl->tb = tb;
  pl->hb = hb;
  pl->lb = lb;
  const long long extent[4] = {kc.bs, kc.H, kc.num_pages, kc.L};
  const int box[4] = {tb, hb, 1, lb};
  int order[4] = {kTok, kHead, kPage, kLayer};
  std::stable_sort(order, order + 4, [&](int x, int y) { return stride[x] < stride[y]; });
  cuuint64_t dims[5] = {(cuuint64_t)kc.D, 0, 0, 0, 0};
  cuuint64_t strides[4] = {};
  cuuint32_t bdim[5] = {(cuuint32_t)kc.D, 0, 0, 0, 0};
  pl->ext[0] = kc.D;
  for (int p = 1; p <= 4; ++p) {
    const int d = order[p - 1];
    pl->pos[d] = p;
    dims[p] = (cuuint64_t)extent[d];
    strides[p - 1] = (cuuint64_t)stride[d];
    bdim[p] = (cuuint32_t)box[d];
    pl->ext[p] = box[d];
  }
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  return encode &&
         encode(&pl->tm, kc.dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5,
                const_cast<void*>(kc.base), dims, strides, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_slices_t(const CUtensorMap& tm, const SliceTmaArgs& a, int grid, cudaStream_t s) {
  static std::mutex mu;
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
      e = cudaFuncSetAttribute(pool_tma_slices_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaSmem);
      if (e != cudaSuccess) return e;
      ready[dev] = true;
    }
  }
  pool_tma_slices_kernel<T, D><<<grid, kTmaThreads, kTmaSmem, s>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool_tma(const KCache& kc, const int* pages, const int* n_valid, int n,
                            const float* head_w, int n_sets, const int* w_set, float* vb, int* err,
                            cudaStream_t s) {
  const int sms = sm_count();
  if (n < sms) return cudaErrorNotSupported;  // too few blocks for one per SM: the cluster path splits them
  TmaPlan pl;
  if (!plan_tma(kc, 256, &pl)) return cudaErrorNotSupported;
  PoolTmaArgs a = {};
  a.pages = pages;
  a.n_valid = n_valid;
  a.head_w = head_w;
  a.n_sets = n_sets;
  a.w_set = w_set;
  a.vb = vb;
  a.n = n;
  a.L = kc.L;
  a.H = kc.H;
  a.bs = kc.bs;
  a.num_pages = kc.num_pages;
  a.tb = pl.tb;
  a.hb = pl.hb;
  a.lb = pl.lb;
  a.nhb = kc.H / pl.hb;
  a.nlb = kc.L / pl.lb;
  a.err = err;
  a.wait_ns = wait_limit_ns();
  a.skip_box = take_skip_box();
  for (int i = 0; i < 4; ++i) a.pos[i] = pl.pos[i];
  for (int i = 0; i < 5; ++i) a.ext[i] = pl.ext[i];
  const int grid = std::min(n, sms);
  if (kc.dtype == 1)
    return head_w ? dispatch_d<bf16_t, true>(kc.D, pl.tm, a, grid, s) : dispatch_d<bf16_t, false>(kc.D, pl.tm, a, grid, s);
  return head_w ? dispatch_d<float, true>(kc.D, pl.tm, a, grid, s) : dispatch_d<float, false>(kc.D, pl.tm, a, grid, s);
}

cudaError_t launch_pool_tma_slices(const KCache& kc, const Table& bt, long long total_blocks, float* S, float* Q,
                                   int* err, cudaStream_t s) {
  const int sms = sm_count();
  if (total_blocks < sms) return cudaErrorNotSupported;
  TmaPlan pl;
  if (!plan_tma(kc, kConsumerWarps, &pl)) return cudaErrorNotSupported;
  if (pl.pos[kTok] != 1 || pl.pos[kHead] != 2) return cudaErrorNotSupported;  // slices must be contiguous rows
  SliceTmaArgs a = {};
  a.bt = bt;
  a.total = total_blocks;
  a.L = kc.L;
  a.H = kc.H;
  a.bs = kc.bs;
  a.num_pages = kc.num_pages;
  a.tb = pl.tb;
  a.hb = pl.hb;
  a.lb = pl.lb;
  a.nhb = kc.H / pl.hb;
  a.nlb = kc.L / pl.lb;
  for (int i = 0; i < 4; ++i) a.pos[i] = pl.pos[i];
  a.S = S;
  a.Q = Q;
  a.err = err;
  a.wait_ns = wait_limit_ns();
  const int grid = (int)std::min<long long>(total_blocks, sms);
  if (kc.dtype == 1) {
    switch (kc.D) {
      case 32: return launch_slices_t<bf16_t, 32>(pl.tm, a, grid, s);
      case 64: return launch_slices_t<bf16_t, 64>(pl.tm, a, grid, s);
      case 128: return launch_slices_t<bf16_t, 128>(pl.tm, a, grid, s);
      case 256: return launch_slices_t<bf16_t, 256>(pl.tm, a, grid, s);
    }
  } else {
    switch (kc.D) {
      case 32: return launch_slices_t<float, 32>(pl.tm, a, grid, s);
      case 64: return launch_slices_t<float, 64>(pl.tm, a, grid, s);
      case 128: return launch_slices_t<float, 128>(pl.tm, a, grid, s);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace kk
