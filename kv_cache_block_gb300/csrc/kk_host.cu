// Host helpers shared by the kernel files: the driver's tensor-map encoder
// (reached through the runtime, so the library needs no -lcuda) and the SM
// count of the current device.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kk_internal.h"

namespace kk {

void* tensor_map_encoder() {
  static std::once_flag once;
  static void* fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] > 0) return cached[dev];
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    cached[dev] = n;
  }
  return n;
}

}  // namespace kk
