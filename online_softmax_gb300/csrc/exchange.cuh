// Cross-warp max / sum of one FP32 value per thread through shared memory with a
// single named barrier per call ("fa4_ws_exchange4", the Mojo softmax-warp function:
// "everyone reduces" over a double-buffered window selected by the parity of a
// monotone exchange counter).
//
// Every thread writes its partial into slot (g * ROWS + local_row) of the window for
// (warpgroup, seq & 1), all 128 threads of the warpgroup meet at one named barrier,
// then every thread folds the M_PACK slots of its row in the fixed order
// g = 0 .. M_PACK-1.  The fixed order makes the result bit-identical in every warp.
//
// One barrier suffices because consecutive calls alternate buffers: a warp that runs
// ahead writes the other buffer, and it cannot come back to this buffer before every
// warp has passed the next call's barrier, which a warp reaches only after it has read
// this buffer.  This holds only if `seq` increases by one on every call made by the
// warpgroup for its whole lifetime (never reset between phases).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace oattn {

template <int M_PACK, int ROWS, bool IS_MAX>
__device__ __forceinline__ float ws_exchange(float partial, uint32_t local_row, uint32_t g,
                                             uint32_t wg, uint32_t seq, float* xchg,
                                             uint32_t barrier_id) {
  static_assert(M_PACK * ROWS == 128, "the slot map must cover the warpgroup's 128 threads");
  float* buf = xchg + (wg * 2u + (seq & 1u)) * 128u;
  buf[g * ROWS + local_row] = partial;
  named_bar_sync(barrier_id, 128);
  float r = buf[local_row];
#pragma unroll
  for (int i = 1; i < M_PACK; ++i) {
    const float x = buf[i * ROWS + local_row];
    r = IS_MAX ? fmaxf(r, x) : r + x;
  }
  return r;
}

}  // namespace oattn
