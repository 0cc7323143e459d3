// Allocation-free variant of the weighted pool. Its scratch (per-slice token
// sums, sums of squares and head variances) lives in a file-scope device
// array that the library owns, so a caller that cannot allocate device memory
// can still run the weighted write path. The kernels are the ones
// kk_pool_blocks_weighted launches; only where the scratch comes from differs.
#include <mutex>

#include "../../include/kk.h"
#include "kk_internal.h"

namespace kk {
kk_status check_weighted_args(const kk_kcache_desc* kc, const kk_block_table* bt,
                              int32_t total_blocks, const float* head_w_out, const float* vb,
                              KCache* c, Table* t);
}  // namespace kk

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB, held by every GPU that loads the library

static __device__ __align__(256) unsigned char g_kk_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::mutex mu;
  static void* ptr[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kk_static_scratch) != cudaSuccess) return nullptr;
    ptr[dev] = p;
  }
  return ptr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" kk_status kk_pool_blocks_weighted_static(const kk_kcache_desc* kc,
                                                    const kk_block_table* bt,
                                                    int32_t total_blocks, float* head_w_out,
                                                    float* vb, cudaStream_t stream) {
  kk::KCache c;
  kk::Table t;
  kk_status st = kk::check_weighted_args(kc, bt, total_blocks, head_w_out, vb, &c, &t);
  if (st != KK_OK) return st;
  if (t.R == 0) return KK_OK;
  const int LH = c.L * c.H;
  const size_t s_bytes = round256(sizeof(float) * (size_t)total_blocks * LH * c.D);
  const size_t q_bytes = round256(sizeof(float) * (size_t)total_blocks * LH);
  const size_t v_bytes = round256(sizeof(double) * (size_t)t.R * LH);
  if (s_bytes + q_bytes + v_bytes > kStaticScratchBytes) return KK_ERR_UNSUPPORTED;
  char* base = static_cast<char*>(scratch_address());
  if (!base) return KK_ERR_CUDA;
  int* err = kk::device_error_word();
  if (!err) return KK_ERR_CUDA;
  // Every scratch byte a kernel reads is written earlier in the same call, so
  // nothing left by a previous call needs clearing.
  float* S = reinterpret_cast<float*>(base);
  float* Q = reinterpret_cast<float*>(base + s_bytes);
  double* var = reinterpret_cast<double*>(base + s_bytes + q_bytes);
  cudaError_t e = kk::launch_pool_slices(c, t, total_blocks, S, Q, err, stream);
  if (e == cudaSuccess) e = kk::launch_head_var(c, t, total_blocks, S, Q, var, err, stream);
  if (e == cudaSuccess) e = kk::launch_finalize_weights(c, t, total_blocks, var, head_w_out, stream);
  if (e == cudaSuccess) e = kk::launch_combine(c, t, total_blocks, S, head_w_out, vb, err, stream);
  return e == cudaSuccess ? KK_OK : KK_ERR_CUDA;
}
