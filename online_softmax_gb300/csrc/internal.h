// Launchers shared between the translation units of the library (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace oattn {

enum DType : int { kF16 = 0, kBF16 = 1, kF32 = 2 };

// ---- splitk_combine (combine.cu)
bool combine_supported(int depth, int in_dt);
// pdl: launch as a programmatic dependent of the previous kernel on the stream (the
// combine's blocks wait for that grid's completion before their first read).
cudaError_t launch_combine(const void* o_partial, const float* lse_partial, void* o,
                           float* lse_out, int P, long long RH, int depth, int in_dt, int out_dt,
                           float lse_scale, bool pdl, cudaStream_t st);

// ---- self-test of the bounded-wait failure path (selftest.cu)
cudaError_t launch_selftest_wait(unsigned int* status, int* flags, cudaStream_t st);

// ---- the optional Boolean mask, packed one bit per key (mask.cu packs it)
// Row (b, h, q) of the mask starts at bits + b*sb + h*sh + q*sq (32-bit words; a stride
// of 0 broadcasts); bit j of word w is key 32*w + j, set = visible.  A row holds
// mask_words(Nkv) = 4*ceil(Nkv/128) words, so a 128-key tile is one aligned 16-byte load.
struct MaskArgs {
  const uint32_t* bits;  // nullptr: no mask
  long long sb, sh, sq;
  int H;                 // heads per batch entry (splits the flattened b*H + h index)
};
inline int mask_words(int nkv) { return 4 * ((nkv + 127) / 128); }
cudaError_t launch_mask_pack(const uint8_t* mask, uint32_t* bits, long long rows, int nkv,
                             long long row_stride, cudaStream_t st);

// Block summary of a packed mask (one bit per mask head, block of 256 query rows and key
// tile of 128: set iff some row of the block sees some key of the tile).  A mask stride of
// 0 shares the mask, and so its summary, along that axis; the words of (b, h, block p)
// are bits + b * sb + h * sh + p * wpb.
struct MaskBlocks {
  const uint32_t* bits;  // nullptr: no summary
  long long sb, sh;
  int wpb;               // words per block
};
inline int mask_block_wpb(int nkv) { return ((nkv + 127) / 128 + 31) / 32; }
long long mask_blocks_words(int B, int H, int nq, int nkv, long long sb, long long sh);
cudaError_t launch_mask_blocks(const uint32_t* bits, long long sb, long long sh, long long sq, int B, int H, int nq,
                               int nkv, uint32_t* blocks, cudaStream_t st);

// ---- in-kernel split-K merge: the last CTA to finish a group of P partitions merges
// them.  counters[g] counts the arrivals of group g (one per row-head in decode, one per
// (head, pair of query tiles) in the tcgen05 split mode); the last arrival resets it to 0.
struct FusedMerge {
  unsigned int* counters;  // nullptr: no merge (partials only)
  void* o;                 // [BH, Nq, D] in the input dtype
  float* lse;              // [BH, Nq] natural log, or nullptr
};

// ---- one-query split-K decode on CUDA cores (decode.cu)
struct DecodeArgs {
  const void* q;       // [BH, D]
  const void* k;       // [BH, Nkv, D]
  const void* v;       // [BH, Nkv, D]
  void* o_partial;     // [P, BH, D] f32 or input dtype
  float* lse_partial;  // [P, BH] base 2
  long long BH;
  int Nkv, D, P, chunk;
  float scale_log2;    // scale * log2(e)
  int dtype;           // kF16 / kBF16
  int partial_dtype;   // kF32 / input dtype
  MaskArgs mask;       // optional; row q = 0 of each (b, h)
  FusedMerge fused;    // optional in-kernel merge
  unsigned int* status;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

// ---- tcgen05 attention forward / split-K partitions (attn_fwd_d*.cu)
struct AttnArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [BH, N, D], boxes of 128 or BN rows
  CUtensorMap tm_o;              // plain mode: output map (box of 128 rows); split: unused
  void* o;            // plain: [BH, N, D] dtype;  split: [P, BH*N, D] partial dtype
  float* lse;         // plain: [BH, N] natural log (nullable);  split: [P, BH*N] base 2
  int BH, N, Nkv, D;
  int causal;
  float scale_log2;
  int P, chunk;       // split mode when P > 0
  int out_f32;        // split mode: o_partial is float32
  MaskArgs mask;      // optional (key tiles of 128 only)
  MaskBlocks mblocks; // optional block summary of the mask (plain mode)
  FusedMerge fused;   // split mode: optional in-kernel merge
  unsigned int* status;
};
// Instantiated per head dimension in attn_fwd_d{16,32,64,128}.cu.
cudaError_t launch_attn_d16(const AttnArgs& a, int block_n, int bf16, cudaStream_t st);
cudaError_t launch_attn_d32(const AttnArgs& a, int block_n, int bf16, cudaStream_t st);
cudaError_t launch_attn_d64(const AttnArgs& a, int block_n, int bf16, cudaStream_t st);
cudaError_t launch_attn_d128(const AttnArgs& a, int block_n, int bf16, cudaStream_t st);

}  // namespace oattn
