// Shared-pool scoring ("Key-Key Semantic Affinity" page, §5.1: every block
// representation scored against the anchors in one matrix product, then
// masked): R anchors against N pooled block vectors, each anchor restricted to
// the blocks its mask marks, top K per anchor.
//
// Kernel 1 is a tcgen05 GEMM tile: TMA loads a 128-anchor x 128-dim tile of A
// and a 128-block tile of V into shared memory (128-byte swizzle), one thread
// issues eight 128x128x16 bf16 MMAs into a TMEM fp32 accumulator, and four
// epilogue warps read it back (tcgen05.ld), divide by the norms (computed from
// the same shared-memory tiles), apply the ownership mask and append each
// owned candidate as a 64-bit key (score, pool id) to its anchor's list.
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
  int R, N, mask_words;
  int* counts;      // [R] candidates appended per anchor
  uint64_t* cand;   // [R][N] candidate keys
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
    const int q4 = warp & 3;            // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;     // anchor row within the tile
    const int r = m0 + row;
    if (mma_ok) {
      // ownership bits of this anchor's 128 columns, limited to columns < N
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
      int k = 0;
      if (total > 0) k = atomicAdd(&g.counts[r], total);
      uint64_t* out = g.cand + (long long)r * g.N;
      const float na = s_na[row];
      const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t acc[32];
        tmem_ld32(taddr + c * 32, acc);  // all lanes of the warp take part
        tmem_wait_ld();
        if (w[c] == 0) continue;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if ((w[c] >> i) & 1u) {
            const int col = c * 32 + i;
            const float nv = s_nv[col];
            const float dot = __uint_as_float(acc[i]);
            float cosv = (na > 0.f && nv > 0.f) ? dot / (na * nv) : 0.f;
            cosv = fminf(1.f, fmaxf(-1.f, cosv));
            out[k++] = make_key(fmaf(0.5f, cosv, 0.5f), (uint32_t)(n0 + col));
          }
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

__global__ void __launch_bounds__(kSelThreads) select_rows_kernel(const uint64_t* cand, long long stride,
                                                                  const int* counts, int K, int* idx_out,
                                                                  float* top_out, int* err) {
  __shared__ int hist[256];
  __shared__ int s_bin, s_above;
  __shared__ int s_sel_n;
  __shared__ uint64_t s_sel[kMaxK];
  __shared__ uint64_t s_wl[kSelThreads / 32][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  int n = counts[r];
  if (n < 0 || n > stride) {
    if (tid == 0) flag_error(err, kErrBadIndex);
    n = n < 0 ? 0 : (int)stride;
  }
  const uint64_t* keys = cand + (long long)r * stride;
  int need = min(K, n);
  const int m = need;
  uint64_t prefix = 0, pmask = 0;
  // Find the m-th largest key: at each digit, the bin where the count of
  // larger keys crosses `need`; stop once that bin holds exactly what is left.
  for (int shift = 56; shift >= 0 && need > 0; shift -= 8) {
    hist[tid] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kSelThreads) {
      const int i = i0 + tid;
      int d = 256;  // no bin
      if (i < n) {
        const uint64_t k = keys[i];
        if ((k & pmask) == prefix) d = (int)((k >> shift) & 255);
      }
      const unsigned same = __match_any_sync(kFull, d);
      if (d < 256 && lane == __ffs(same) - 1) atomicAdd(&hist[d], __popc(same));
    }
    __syncthreads();
    if (warp == 0) {
      // suffix counts from the top bin down: lane l owns bins 8l .. 8l+7
      int local = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) local += hist[lane * 8 + b];
      int incl = local;  // sum over lanes >= this lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(kFull, incl, o);
        if (lane + o < 32) incl += y;
      }
      int above = incl - local;  // bins above this lane's block
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
  // the m largest keys are exactly those >= prefix
  if (tid == 0) s_sel_n = 0;
  __syncthreads();
  if (m > 0) {
    for (int i = tid; i < n; i += kSelThreads) {
      const uint64_t k = keys[i];
      if (k >= prefix) {
        const int pos = atomicAdd(&s_sel_n, 1);
        if (pos < kMaxK) s_sel[pos] = k;
      }
    }
  }
  __syncthreads();
  const int sel = min(s_sel_n, m);
  // sort the selected keys: warp-sorted lists of 32, then rank in the union
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
    ready[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

size_t batched_workspace_bytes(int R, int N) {
  return ((sizeof(int) * (size_t)R + 255) & ~size_t(255)) + sizeof(uint64_t) * (size_t)R * (size_t)N;
}

cudaError_t launch_score_pool_batched(const uint16_t* A, const uint16_t* V, const uint32_t* mask, int R,
                                      int N, int K, int* idx, float* top, void* ws, int* err,
                                      cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  int* counts = static_cast<int*>(ws);
  uint64_t* cand = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) +
                                               ((sizeof(int) * (size_t)R + 255) & ~size_t(255)));
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int) * (size_t)R, s);
  if (e != cudaSuccess) return e;
  if (N > 0) {
    CUtensorMap ma, mv;
    if (!make_map(&ma, A, R) || !make_map(&mv, V, N)) return cudaErrorInvalidValue;
    if ((e = setup_gemm()) != cudaSuccess) return e;
    GemmArgs g{mask, R, N, (N + 31) / 32, counts, cand, err};
    dim3 grid((N + kBN - 1) / kBN, (R + kBM - 1) / kBM);
    score_pool_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(ma, mv, g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  select_rows_kernel<<<R, kSelThreads, 0, s>>>(cand, N, counts, K, idx, top, err);
  return cudaGetLastError();
}

}  // namespace kk
