// Packing of the optional Boolean attention mask: one byte per (query, key) in, one bit
// per key out ("Streaming attention and online state", section "Attention as a
// consumer": the worked kernel takes an optional Boolean M x N mask).
//
// Row r of the input is the byte row mask + r * row_stride (nonzero byte = the key is
// visible); row r of the output is mask_words(Nkv) 32-bit words at bits + r * W, bit j
// of word w standing for key 32*w + j.  Bits past Nkv are written as zero.  One thread
// writes one word, so a warp reads 1 KB of consecutive bytes of a row and writes 128
// consecutive bytes.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace oattn {
namespace {

// Four mask bytes -> four bits (byte i -> bit i): each nonzero byte becomes 1, and one
// multiply gathers the four byte-aligned ones into bits 24..27 (the partial products
// land on distinct bit positions, so no carries mix them).
__device__ __forceinline__ uint32_t bits4(uint32_t x) {
  const uint32_t ones = __vcmpne4(x, 0u) & 0x01010101u;
  return (ones * 0x01020408u) >> 24;
}

__device__ __forceinline__ uint32_t bits16(uint4 u) {
  return bits4(u.x) | (bits4(u.y) << 4) | (bits4(u.z) << 8) | (bits4(u.w) << 12);
}

__global__ void __launch_bounds__(256)
    mask_pack_kernel(const uint8_t* __restrict__ mask, uint32_t* __restrict__ bits, long long rows, int nkv,
                     long long row_stride, int W, int vec) {
  const long long i = blockIdx.x * 256LL + threadIdx.x;
  if (i >= rows * W) return;
  const long long r = i / W;
  const int w = (int)(i - r * W);
  const int k0 = 32 * w;
  uint32_t out = 0u;
  if (k0 < nkv) {
    const uint8_t* src = mask + r * row_stride + k0;
    if (vec && k0 + 32 <= nkv) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      out = bits16(__ldg(s4)) | (bits16(__ldg(s4 + 1)) << 16);
    } else {
      const int n = min(32, nkv - k0);
      for (int j = 0; j < n; ++j) out |= (src[j] != 0 ? 1u : 0u) << j;
    }
  }
  bits[i] = out;
}

}  // namespace

cudaError_t launch_mask_pack(const uint8_t* mask, uint32_t* bits, long long rows, int nkv, long long row_stride,
                             cudaStream_t st) {
  const int W = mask_words(nkv);
  const long long total = rows * W;
  if (total <= 0) return cudaSuccess;
  const long long blocks = (total + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int vec = (reinterpret_cast<uintptr_t>(mask) % 16 == 0) && (row_stride % 16 == 0);
  mask_pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(mask, bits, rows, nkv, row_stride, W, vec);
  return cudaGetLastError();
}

}  // namespace oattn
