// Seeded synthetic-input generator (GPU side). Not part of the scoring
// library: it only draws test and benchmark inputs. It implements the same
// definition as synth/__init__.py (SplitMix64 counters, Irwin-Hall noise,
// fl32(cs + fl32(sigma * noise)), bf16 by round-to-nearest-even), bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float noise_of(uint64_t key, uint64_t ctr) {
  int64_t total = 0;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    uint64_t h = mix64(key + (3ull * ctr + (uint64_t)(k + 1)) * kGolden);
    total += (int64_t)(h & 0xFFFF) + (int64_t)((h >> 16) & 0xFFFF) + (int64_t)((h >> 32) & 0xFFFF) +
             (int64_t)(h >> 48);
  }
  const int32_t num = (int32_t)(2 * total + 12 - 786432);
  return __fmul_rn((float)num, 7.62939453125e-06f);  // 2^-17, exact
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t r = ((u >> 16) & 1u) + 0x7FFFu;
  return (uint16_t)((u + r) >> 16);
}

__global__ void gen_paged_kernel(void* base, int dtype, int L, int H, int D, int bs, long long sL,
                                 long long sP, long long sH, long long sT, const int* pages,
                                 const int* n_valid, const int* topic, const long long* tok0,
                                 long long total_elems, const float* cs, const float* sigma,
                                 uint64_t key) {
  // element order: block g, layer l, head h, token t, dim d (d fastest)
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_elems;
       i += (long long)gridDim.x * blockDim.x) {
    long long q = i;
    const int d = (int)(q % D);
    q /= D;
    const int t = (int)(q % bs);
    q /= bs;
    const int h = (int)(q % H);
    q /= H;
    const int l = (int)(q % L);
    const long long g = q / L;
    if (t >= n_valid[g]) continue;
    const long long tok = tok0[g] + t;
    const uint64_t ctr = (uint64_t)(((tok * L + l) * H + h) * D + d);
    const float nz = noise_of(key, ctr);
    const float v = __fadd_rn(cs[(long long)topic[g] * D + d], __fmul_rn(sigma[l * H + h], nz));
    const long long off = l * sL + (long long)pages[g] * sP + h * sH + t * sT + d;
    if (dtype == 0)
      reinterpret_cast<float*>(base)[off] = v;
    else
      reinterpret_cast<uint16_t*>(base)[off] = bf16_rne_bits(v);
  }
}

__global__ void gen_rows_kernel(void* out, int dtype, long long N, int D, const int* topic,
                                const float* cs, float sigma, uint64_t key) {
  const long long total = N * D;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / D;
    const int d = (int)(i % D);
    const float nz = noise_of(key, (uint64_t)i);
    const float v = __fadd_rn(cs[(long long)topic[row] * D + d], __fmul_rn(sigma, nz));
    if (dtype == 0)
      reinterpret_cast<float*>(out)[i] = v;
    else
      reinterpret_cast<uint16_t*>(out)[i] = bf16_rne_bits(v);
  }
}

__global__ void fill_u32_kernel(uint32_t* p, long long n, uint32_t v) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = v;
}

int grid_for(long long n) {
  long long g = (n + 255) / 256;
  if (g > 152LL * 64) g = 152LL * 64;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

int kks_gen_paged(void* base, int dtype, int L, int H, int D, int bs, long long sL, long long sP,
                  long long sH, long long sT, const int* pages, const int* n_valid, const int* topic,
                  const long long* tok0, int nblocks, const float* cs, const float* sigma,
                  unsigned long long key, cudaStream_t stream) {
  if (!base || L <= 0 || H <= 0 || D <= 0 || bs <= 0 || nblocks < 0) return 1;
  if (nblocks == 0) return 0;
  const long long total = (long long)nblocks * L * H * bs * D;
  gen_paged_kernel<<<grid_for(total), 256, 0, stream>>>(base, dtype, L, H, D, bs, sL, sP, sH, sT,
                                                        pages, n_valid, topic, tok0, total, cs,
                                                        sigma, key);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int kks_gen_rows(void* out, int dtype, long long N, int D, const int* topic, const float* cs,
                 float sigma, unsigned long long key, cudaStream_t stream) {
  if (!out || N < 0 || D <= 0) return 1;
  if (N == 0) return 0;
  gen_rows_kernel<<<grid_for(N * D), 256, 0, stream>>>(out, dtype, N, D, topic, cs, sigma, key);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int kks_fill_u32(void* p, long long n, unsigned int v, cudaStream_t stream) {
  if (!p || n < 0) return 1;
  if (n == 0) return 0;
  fill_u32_kernel<<<grid_for(n), 256, 0, stream>>>(reinterpret_cast<uint32_t*>(p), n, v);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
