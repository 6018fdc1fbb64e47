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

// Block summary of a packed mask: for each mask head (b, h), block of 256 query rows p and
// key tile j of 128 keys, bit j of word j / 32 of the block's words is set iff some row
// of the block has some bit set in the tile's 16 bytes.  One CTA of 8 warps per (word,
// block, mask head): warp w ORs rows 32 w .. 32 w + 31 of the block, lane = key tile
// (one 512-byte coalesced load per row), and the warps' ballots are ORed in shared memory.
__global__ void __launch_bounds__(256)
    mask_blocks_kernel(const uint32_t* __restrict__ bits, long long sb, long long sh, long long sq, int Hm, int nq,
                       int nblk, int ntiles, int wpb, uint32_t* __restrict__ blocks) {
  __shared__ uint32_t s_word;
  const int word = blockIdx.x % wpb;
  const int p = (blockIdx.x / wpb) % nblk;
  const int mh = blockIdx.x / wpb / nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_word = 0u;
  __syncthreads();
  const int b = mh / Hm, h = mh - b * Hm;
  const int j = word * 32 + lane;
  const int r0 = p * 256 + warp * 32;
  const int nr = min(32, nq - r0);
  uint32_t acc = 0u;
  if (j < ntiles && nr > 0) {
    const uint32_t* base = bits + b * sb + h * sh + (long long)r0 * sq + 4 * j;
    for (int i0 = 0; i0 < nr && acc == 0u; i0 += 8) {
      uint4 w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = i0 + i < nr ? __ldg(reinterpret_cast<const uint4*>(base + (long long)(i0 + i) * sq))
                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc |= w[i].x | w[i].y | w[i].z | w[i].w;
    }
  }
  const uint32_t marks = __ballot_sync(0xffffffffu, acc != 0u);
  if (lane == 0 && marks != 0u) atomicOr(&s_word, marks);
  __syncthreads();
  if (threadIdx.x == 0) blocks[blockIdx.x] = s_word;  // = ((mh * nblk) + p) * wpb + word
}

}  // namespace

long long mask_blocks_words(int B, int H, int nq, int nkv, long long sb, long long sh) {
  if (B <= 0 || H <= 0 || nq <= 0 || nkv <= 0) return 0;
  const long long heads = (long long)(sb ? B : 1) * (sh ? H : 1);
  return heads * ((nq + 255) / 256) * mask_block_wpb(nkv);
}

cudaError_t launch_mask_blocks(const uint32_t* bits, long long sb, long long sh, long long sq, int B, int H, int nq,
                               int nkv, uint32_t* blocks, cudaStream_t st) {
  if (B <= 0 || H <= 0 || nq <= 0 || nkv <= 0) return cudaSuccess;
  const int Hm = sh ? H : 1;
  const long long total = mask_blocks_words(B, H, nq, nkv, sb, sh);  // one CTA per word
  if (total > 0x7fffffffLL) return cudaErrorInvalidValue;
  mask_blocks_kernel<<<(unsigned)total, 256, 0, st>>>(bits, sb, sh, sq, Hm, nq, (nq + 255) / 256, (nkv + 127) / 128,
                                                       mask_block_wpb(nkv), blocks);
  return cudaGetLastError();
}

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
