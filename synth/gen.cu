// CUDA side of the seeded input generator (same definition as synth/__init__.py):
// SplitMix64 words of counter (i + 1 + stream*2^40 + seed*2^48) * GAMMA, Irwin-Hall
// standard normals from the four 16-bit fields, float32 mu + sigma*z with one multiply
// and one add (no contraction), then round-to-nearest-even to bf16 / f16.
// It holds no attention arithmetic; it only lets large inputs be drawn on the device.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint32_t seed, uint32_t stream, uint64_t i) {
  const uint64_t base = 1ull + ((uint64_t)stream << 40) + ((uint64_t)seed << 48);
  return mix64((i + base) * 0x9E3779B97F4A7C15ull);
}

__device__ __forceinline__ float normal(uint32_t seed, uint32_t stream, uint64_t i, float mu, float sigma,
                                        bool affine) {
  const uint64_t w = word(seed, stream, i);
  const int64_t s = (int64_t)((w & 0xFFFF) + ((w >> 16) & 0xFFFF) + ((w >> 32) & 0xFFFF) + (w >> 48)) - 131070;
  float z = __fmul_rn((float)s, __uint_as_float(0x37DDB3D7u));
  if (affine) z = __fadd_rn(__fmul_rn(z, sigma), mu);
  return z;
}

__global__ void fill_normal(void* out, long long n, long long start, uint32_t seed, uint32_t stream,
                            float mu, float sigma, int affine, int dtype) {
  for (long long j = blockIdx.x * (long long)blockDim.x + threadIdx.x; j < n;
       j += (long long)gridDim.x * blockDim.x) {
    const float z = normal(seed, stream, (uint64_t)(start + j), mu, sigma, affine != 0);
    if (dtype == 1) static_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(z);
    else if (dtype == 0) static_cast<__half*>(out)[j] = __float2half_rn(z);
    else static_cast<float*>(out)[j] = z;
  }
}

// lse[p, rh] for the standalone combine workload: N(mu, sigma), set to -inf with
// probability `drop` per entry and for every p of a row-head drawn with `row_drop`.
__global__ void fill_lse(float* out, int P, long long RH, uint32_t seed, uint32_t s_val, uint32_t s_drop,
                         uint32_t s_row, float mu, float sigma, uint32_t drop_thresh, uint32_t row_thresh) {
  const long long n = (long long)P * RH;
  for (long long j = blockIdx.x * (long long)blockDim.x + threadIdx.x; j < n;
       j += (long long)gridDim.x * blockDim.x) {
    const long long rh = j % RH;
    float v = normal(seed, s_val, (uint64_t)j, mu, sigma, true);
    const bool d = (uint32_t)(word(seed, s_drop, (uint64_t)j) >> 32) < drop_thresh;
    const bool r = (uint32_t)(word(seed, s_row, (uint64_t)rh) >> 32) < row_thresh;
    out[j] = (d || r) ? -INFINITY : v;
  }
}

}  // namespace

extern "C" {

// dtype: 0 f16, 1 bf16, 2 f32.  Elements [start, start+n) of (seed, stream).
int synth_fill_normal(void* out, long long n, long long start, unsigned seed, unsigned stream, float mu,
                      float sigma, int dtype, void* cuda_stream) {
  if (n <= 0) return 0;
  const int affine = (mu != 0.f || sigma != 1.f) ? 1 : 0;
  fill_normal<<<152 * 8, 256, 0, (cudaStream_t)cuda_stream>>>(out, n, start, seed, stream, mu, sigma, affine,
                                                             dtype);
  return (int)cudaGetLastError();
}

int synth_fill_lse(float* out, int P, long long RH, unsigned seed, unsigned s_val, unsigned s_drop,
                   unsigned s_row, float mu, float sigma, unsigned drop_thresh, unsigned row_thresh,
                   void* cuda_stream) {
  fill_lse<<<152 * 8, 256, 0, (cudaStream_t)cuda_stream>>>(out, P, RH, seed, s_val, s_drop, s_row, mu, sigma,
                                                          drop_thresh, row_thresh);
  return (int)cudaGetLastError();
}

}  // extern "C"
