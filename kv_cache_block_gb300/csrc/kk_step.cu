// One decode step of the Key-Key selector ("Key-Key Semantic Affinity" page,
// §5.2 steps 1-4): pool the anchor from the last W tokens' Keys, score every
// block of the request's table by (1 + cos(v_b, v_anchor)) / 2 (§2.2 step 3,
// §3.2), and keep the top K (§5.2 step 4).
//
// A request is served by one thread-block cluster of CL CTAs. The CTAs split
// the anchor's (layer, head) slices and the request's blocks; partial anchors
// and partial top-K lists travel through distributed shared memory, so a whole
// step is one launch with no global scratch. Every stage can be switched off,
// which gives kk_anchor, kk_score, kk_topk and kk_score_topk from the same code.
#include <mutex>

#include "kk_device.cuh"
#include "kk_internal.h"

namespace kk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kThreads;  // candidates per top-K tile
constexpr int kUnroll = 8;

template <int D>
struct StepSmem {
  float part[kMaxCluster][D];  // anchor partial of each CTA of the cluster
  float wpart[kWarps][D];
  float va[D];
  long long tok[kMaxW];  // byte offset of each anchor token row (page, slot)
  float w[kMaxLH];
  int pg[kTile];
  uint64_t keys[kTile];
  uint64_t wl[kWarps][32];
  int wn[kWarps];
  uint64_t run[2][kMaxK];
  uint64_t merge[kMergeSlots];
  int mcount[kMaxCluster];
};

// D floats per row: each lane holds D/32 of them.
template <int D>
struct RowSlice {
  static constexpr int kPer = D / 32;
  float v[kPer];
  __device__ __forceinline__ void load(const float* row, int lane) {
    const float* p = row + lane * kPer;
    if (kPer == 8) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(p));
      const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if (kPer == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(p));
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if (kPer == 2) {
      const float2 a = __ldg(reinterpret_cast<const float2*>(p));
      v[0] = a.x; v[1] = a.y;
    } else {
      v[0] = __ldg(p);
    }
  }
  __device__ __forceinline__ void load_shared(const float* row, int lane) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[e] = row[lane * kPer + e];
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[e] = 0.f;
  }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) step_kernel(StepParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StepSmem<D>& sm = *reinterpret_cast<StepSmem<D>*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.y;
  const int CL = (int)cluster_size();
  const int crank = CL > 1 ? (int)cluster_rank() : 0;
  const bool do_anchor = p.flags & kStepAnchor;
  const bool do_score = p.flags & kStepScore;
  const bool do_topk = p.flags & kStepTopK;
  const bool from_scores = p.flags & kStepTopKFromScores;
  const int K = p.K;

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

  // ---- stage 1: anchor -----------------------------------------------------
  constexpr bool kAnchorFits = D <= 32 * Vec16<T>::kElems;  // a row is at most 32 vectors
  if (kAnchorFits && do_anchor) {
    constexpr int EPV = Vec16<T>::kElems;
    constexpr int V16 = kAnchorFits ? D / EPV : 32;
    constexpr int RPW = 32 / V16;
    constexpr int ES = elem_bytes<T>();
    const int vec = lane % V16, tl = lane / V16;
    const int LH = p.kc.L * p.kc.H;
    const int w_eff = min(p.W, T_r);
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
      for (int s = tid; s < LH; s += kThreads) sm.w[s] = p.head_w[(long long)r * LH + s];
    __syncthreads();

    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
    const char* kbase = reinterpret_cast<const char*>(p.kc.base) + vec * 16;
    for (int s = crank + CL * warp; s < LH; s += CL * kWarps) {
      const int l = s / p.kc.H, h = s - l * p.kc.H;
      const char* sbase = kbase + ((long long)l * p.kc.sL + (long long)h * p.kc.sH) * ES;
      float ps[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) ps[e] = 0.f;
      for (int i0 = 0; i0 < w_eff; i0 += kUnroll * RPW) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = i0 + u * RPW + tl;
          const long long o = (i < w_eff) ? sm.tok[i] : -1;
          v[u] = ld_stream16(sbase + (o >= 0 ? o : 0), o >= 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          float f[EPV];
          Vec16<T>::unpack(v[u], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) ps[e] += f[e];
        }
      }
      const float wt = p.head_w ? sm.w[s] : 1.f;
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[e] = fmaf(wt, ps[e], acc[e]);
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
      if (crank == 0 && p.va_out) p.va_out[(long long)r * D + tid] = v;
    }
    __syncthreads();
  } else if (do_score) {
    if (tid < D) sm.va[tid] = p.va_in[(long long)r * D + tid];
    __syncthreads();
  }

  // ---- stage 2: scores and the CTA's top-K over its share of the blocks --
  int run_n = 0, cur = 0;
  if (do_score || from_scores) {
    const int chunk = (nb + CL - 1) / CL;
    const int j0 = min(nb, crank * chunk);
    const int j1 = min(nb, j0 + chunk);
    RowSlice<D> a;
    float na2 = 0.f;
    if (do_score) {
      a.load_shared(sm.va, lane);
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < RowSlice<D>::kPer; ++e) t = fmaf(a.v[e], a.v[e], t);
      na2 = warp_sum(t);
    }
    const float na = sqrtf(na2);
    for (int tile0 = j0; tile0 < j1; tile0 += kTile) {
      const int tcount = min(kTile, j1 - tile0);
      if (do_score) {
        {
          int pg = -1;
          if (tid < tcount) {
            pg = p.bt.pages[off + tile0 + tid];
            if (pg < 0 || pg >= p.vb_rows) {
              flag_error(p.err, kErrBadIndex);
              pg = -1;
            }
          }
          sm.pg[tid] = pg;
        }
        __syncthreads();
        // warp w scores tile slots [32w, 32w + 32)
        for (int i0 = 0; i0 < 32; i0 += kUnroll) {
          RowSlice<D> b[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int pg = sm.pg[warp * 32 + i0 + u];
            if (pg >= 0)
              b[u].load(p.vb + (long long)pg * D, lane);
            else
              b[u].zero();
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int slot = warp * 32 + i0 + u;
            float dot = 0.f, n2 = 0.f;
#pragma unroll
            for (int e = 0; e < RowSlice<D>::kPer; ++e) {
              dot = fmaf(a.v[e], b[u].v[e], dot);
              n2 = fmaf(b[u].v[e], b[u].v[e], n2);
            }
            dot = warp_sum(dot);
            n2 = warp_sum(n2);
            if (lane == 0) {
              uint64_t key = 0;
              if (slot < tcount) {
                float cosv = 0.f;
                if (na2 > 0.f && n2 > 0.f) cosv = dot / (na * sqrtf(n2));
                cosv = fminf(1.f, fmaxf(-1.f, cosv));
                const float sc = fmaf(0.5f, cosv, 0.5f);
                const int j = tile0 + slot;
                if (p.scores_out) p.scores_out[off + j] = sc;
                if (sm.pg[slot] >= 0) key = make_key(sc, (uint32_t)j);
              }
              sm.keys[slot] = key;
            }
          }
        }
      } else {
        const int j = tile0 + tid;
        sm.keys[tid] = (tid < tcount) ? make_key(p.scores_in[off + j], (uint32_t)j) : 0ull;
      }
      if (!do_topk) {
        __syncthreads();
        continue;
      }
      __syncthreads();
      // merge this tile into the running top-K list (sorted, descending)
      uint64_t key = sm.keys[tid];
      const uint64_t thr = (run_n == K) ? sm.run[cur][K - 1] : 0ull;
      if (key <= thr) key = 0ull;
      if (!__syncthreads_or(key != 0ull)) continue;
      key = warp_sort_desc(key, lane);
      sm.wl[warp][lane] = key;
      const int cnt = __popc(__ballot_sync(kFull, key != 0ull));
      if (lane == 0) sm.wn[warp] = cnt;
      __syncthreads();
      const int nxt = cur ^ 1;
      if (key != 0ull) {
        int rank = lane + count_greater(sm.run[cur], run_n, key);
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
          if (w != warp) rank += count_greater(sm.wl[w], sm.wn[w], key);
        if (rank < K) sm.run[nxt][rank] = key;
      }
      if (tid < run_n) {
        const uint64_t x = sm.run[cur][tid];
        int rank = tid;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) rank += count_greater(sm.wl[w], sm.wn[w], x);
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
    if (CL == 1) {
      for (int i = tid; i < K; i += kThreads) {
        const bool have = i < run_n;
        const uint64_t k = have ? sm.run[cur][i] : 0ull;
        idx_out[i] = have ? (int)key_index(k) : -1;
        if (top_out) top_out[i] = have ? key_score(k) : -__int_as_float(0x7f800000);
      }
    } else {
      if (!start_waited) {
        cluster_wait_acquire();
        start_waited = true;
      }
      for (int i = tid; i < run_n; i += kThreads)
        st_cluster_u64(map_to_rank(smem_u32(&sm.merge[crank * K + i]), 0), sm.run[cur][i]);
      if (tid == 0) st_cluster_s32(map_to_rank(smem_u32(&sm.mcount[crank]), 0), run_n);
      cluster_arrive_release();
      cluster_wait_acquire();
      if (crank == 0) {
        int total = 0;
        for (int q = 0; q < CL; ++q) total += sm.mcount[q];
        for (int f = tid; f < CL * K; f += kThreads) {
          const int q = f / K, i = f - q * K;
          if (i >= sm.mcount[q]) continue;
          const uint64_t k = sm.merge[q * K + i];
          int rank = i;
          for (int o = 0; o < CL; ++o)
            if (o != q) rank += count_greater(&sm.merge[o * K], sm.mcount[o], k);
          if (rank < K) {
            idx_out[rank] = (int)key_index(k);
            if (top_out) top_out[rank] = key_score(k);
          }
        }
        for (int i = total + tid; i < K; i += kThreads) {
          idx_out[i] = -1;
          if (top_out) top_out[i] = -__int_as_float(0x7f800000);
        }
      }
    }
  }
  if (!start_waited) cluster_wait_acquire();
}

// Per-device launch setup of one instantiation: dynamic shared memory above
// 48 KB, non-portable cluster sizes, and the largest cluster size (<= 16)
// that the occupancy calculator says can be co-scheduled.
template <typename T, int D>
cudaError_t setup_device(int* max_cluster) {
  static std::mutex mu;
  static int cached[64] = {};  // 0 = not set up yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    const int smem = (int)sizeof(StepSmem<D>);
    e = cudaFuncSetAttribute(step_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(step_kernel<T, D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int best = 1;
    for (int cl = kMaxCluster; cl > 1; cl >>= 1) {
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
      if (cudaOccupancyMaxActiveClusters(&n, step_kernel<T, D>, &cfg) == cudaSuccess && n > 0) {
        best = cl;
        break;
      }
      (void)cudaGetLastError();  // clear a sticky-free error from an unsupported size
    }
    cached[dev] = best;
  }
  *max_cluster = cached[dev];
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t launch_typed(const StepParams& p, int CL, cudaStream_t s) {
  int max_cl = 1;
  cudaError_t e = setup_device<T, D>(&max_cl);
  if (e != cudaSuccess) return e;
  while (CL > max_cl) CL >>= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, p.bt.R);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(StepSmem<D>);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<T, D>, p);
}

// CTAs per request: enough CTAs to cover the GPU's 152 SMs about twice,
// at most 16, and no more than the merge buffer (CL * K) or the work allows.
int pick_cluster(const StepParams& p) {
  int CL = 1;
  const int per_cta_min = 16;  // blocks scored by a CTA, at least
  while (CL < kMaxCluster && (long long)p.bt.R * CL < 2 * 152 && 2 * CL * p.K <= kMergeSlots &&
         (long long)2 * CL * per_cta_min <= (long long)p.bt.max_blocks + per_cta_min)
    CL *= 2;
  return CL;
}

}  // namespace

cudaError_t launch_step(const StepParams& p, cudaStream_t s) {
  if (p.bt.R == 0) return cudaSuccess;
  const int CL = pick_cluster(p);
  const bool bf16 = (p.flags & kStepAnchor) && p.kc.dtype == 1;
#define KK_STEP_CASE(DD)                                                          \
  if (p.D == DD) return bf16 ? launch_typed<bf16_t, DD>(p, CL, s) : launch_typed<float, DD>(p, CL, s);
  KK_STEP_CASE(32)
  KK_STEP_CASE(64)
  KK_STEP_CASE(128)
  KK_STEP_CASE(256)
#undef KK_STEP_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kk
