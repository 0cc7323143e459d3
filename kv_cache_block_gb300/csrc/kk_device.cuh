// Device helpers shared by the selector kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "kk_internal.h"

namespace kk {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ---- error word ---------------------------------------------------------
// Kernels record the first device-side error here and skip the bad item.
__device__ __forceinline__ void flag_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- element decode -------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 16-byte streaming load of data read once (no L1 allocation, 256 B L2
// prefetch), predicated: returns zeros and touches no memory when !pred.
// Not volatile, so several of them can be in flight before the first use.
__device__ __forceinline__ uint4 ld_stream16(const void* p, bool pred) {
  uint4 v;
  asm("{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
      "@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "r"((int)pred));
  return v;
}

// Elements held by one 16-byte vector, as float32.
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};
struct bf16_t {};  // tag: bf16 stored as raw 16-bit patterns
template <>
struct Vec16<bf16_t> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x);
    f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y);
    f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z);
    f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w);
    f[7] = bf16_hi(v.w);
  }
};
template <typename T>
__host__ __device__ constexpr int elem_bytes() {
  return 16 / Vec16<T>::kElems;
}

// ---- selection keys -------------------------------------------------------
// A candidate is a 64-bit key: the score mapped to an order-preserving
// unsigned integer in the high word, and the bitwise complement of its index
// in the low word, so that a larger key means a higher score, and among equal
// scores the lower index. Key 0 is never produced for a real candidate and
// marks an empty slot.
__device__ __forceinline__ uint32_t f32_to_ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_to_f32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint64_t make_key(float score, uint32_t idx) {
  return ((uint64_t)f32_to_ordered(score) << 32) | (uint64_t)(~idx);
}
__device__ __forceinline__ uint32_t key_index(uint64_t k) { return ~(uint32_t)k; }
__device__ __forceinline__ float key_score(uint64_t k) { return ordered_to_f32((uint32_t)(k >> 32)); }

// Key of a candidate ranked by stability first: the count of high steps (6
// bits), then the score (a non-negative float's 31 bits, which order like
// the float), then the complement of the index in 27 bits. Indices stay
// below 2^27 - 1, so a real key is never 0.
__device__ __forceinline__ uint64_t make_stab_key(uint32_t high_steps, float score, uint32_t idx) {
  const uint32_t sb = __float_as_uint(fmaxf(score, 0.f)) & 0x7FFFFFFFu;
  return ((uint64_t)high_steps << 58) | ((uint64_t)sb << kStabIdxBits) | (uint64_t)(kStabIdxMask - idx);
}
__device__ __forceinline__ uint32_t stab_key_index(uint64_t k) { return kStabIdxMask - (uint32_t)(k & kStabIdxMask); }
__device__ __forceinline__ float stab_key_score(uint64_t k) {
  return __uint_as_float((uint32_t)(k >> kStabIdxBits) & 0x7FFFFFFFu);
}

// Bitonic sort of one key per lane across a warp, descending (lane 0 largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(kFull, x, j);
      const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
      x = keep_max ? (x > o ? x : o) : (x < o ? x : o);
    }
  }
  return x;
}

// Number of entries greater than `key` (> 0) in a descending list of distinct
// keys stored in `cap` slots (cap a power of two), unused slots holding 0.
// Branch-free with a fixed number of steps, so searches in several lists can
// be interleaved by the compiler instead of running as serial chains.
__device__ __forceinline__ int count_greater_pow2(const uint64_t* list, int cap, uint64_t key) {
  int pos = 0;
  for (int step = cap >> 1; step > 0; step >>= 1) pos += (list[pos + step] > key) ? step : 0;
  return (list[0] > key) ? pos + 1 : 0;
}

// ---- thread-block clusters (distributed shared memory) --------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(saddr), "r"(rank));
  return out;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---- mbarrier and bulk (TMA) copies --------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes an initialised mbarrier visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of the barrier for at most `limit_ns` nanoseconds.
// Returns false on timeout; never spins unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completes as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Every spin on an mbarrier is bounded: kernels take the limit as an
// argument (1 s unless a diagnostic call set another; the host side keeps it).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

}  // namespace kk
