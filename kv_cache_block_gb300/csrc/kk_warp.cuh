// Warp-wide sorted key lists (one 64-bit key per lane, lane 0 largest).
#ifndef KK_WARP_CUH_
#define KK_WARP_CUH_

#include <cstdint>

#include "kk_device.cuh"

namespace kk {

// The 32 largest of two descending warp-wide lists (one key per lane, lane 0
// largest), descending: pairing a[i] with b[31 - i] and keeping the larger
// gives a bitonic sequence that holds the 32 largest; a bitonic merge sorts it.
__device__ __forceinline__ uint64_t warp_merge_top32(uint64_t a, uint64_t b, int lane) {
  const uint64_t br = __shfl_sync(kFull, b, 31 - lane);
  uint64_t x = a > br ? a : br;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(kFull, x, j);
    x = (lane & j) == 0 ? (x > o ? x : o) : (x < o ? x : o);
  }
  return x;
}

}  // namespace kk

#endif  // KK_WARP_CUH_
