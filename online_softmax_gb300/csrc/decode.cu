// Split-K attention for one query row per head (decode), on CUDA cores.
//
// One CTA handles one (head, key partition) pair: four compute warps (one warpgroup)
// share the query row, and a fifth warp streams the partition's K and V rows through
// a ring of shared-memory stages with bulk asynchronous copies (the rows of a
// partition are contiguous, so each stage is two plain cp.async.bulk transfers).
// With a single query row the work is a matrix-vector product bound by HBM
// bandwidth, so it stays off the tensor cores.
//
// Per key tile every warp scores its own 8 keys (lane l holds D/32 elements of q and
// of each key row; a butterfly reduce-scatter finishes the 8 dot products with 9
// shuffles and leaves key k's score in lanes 4k..4k+3), the four warps agree on
// the tile maximum through the single-barrier cross-warp exchange ("fa4_ws_exchange4"),
// and then all warps update the running maximum identically.  Because that maximum is
// bit-identical in every warp, each warp can keep its own partial denominator and
// numerator in one common scale, and the end of the partition merges them with plain
// sums (the exchange's "add" for l, a shared-memory sum for the D-vector).
//
// The recurrence is the one of "Streaming attention and online state" (Online
// statistics): m' = max(m, tile max), alpha = 2^(m - m'), p = 2^(s - m'),
// l' = alpha*l + sum p, o' = alpha*o + p V, in base 2 on scores pre-multiplied by
// scale*log2(e).  The rescale is lazy: the maximum in use only moves when the new
// maximum exceeds it by more than kTau, so p <= 2^kTau and the FP32 state cannot
// overflow; the result is the same up to rounding.  p stays FP32 for the P.V products
// here (there is no 16-bit operand to feed).
//
// The optional Boolean mask (one bit per key, packed) hides keys like the partition
// bounds do: their score is -inf.  Lane i of every warp holds the mask word of tile
// t0 + i for a window of 32 tiles; the tile's word is broadcast by a shuffle.
//
// Outputs: o_partial[p, bh, :] = o / l and lse_partial[p, bh] = m + log2(l), or +0 and
// -inf when the partition holds no visible key.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "exchange.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace oattn {
namespace {

constexpr int kTK = 32;          // keys per stage
constexpr int kKeysPerWarp = 8;  // kTK / 4 warps
constexpr int kStages = 2;
constexpr int kThreads = 160;    // 4 compute warps + 1 copy warp
constexpr float kTau = 8.0f;     // lazy-rescale threshold (log2 units)

// EPL consecutive 16-bit elements (8, 4 or 2 bytes, naturally aligned) widened to FP32.
template <int EPL, bool BF16>
__device__ __forceinline__ void load_row(const uint16_t* p, float (&x)[EPL]) {
  uint32_t w[(EPL + 1) / 2];
  if constexpr (EPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x; w[1] = u.y;
  } else if constexpr (EPL == 2) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    w[0] = *p;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    x[i] = (i & 1) ? unpack_hi<BF16>(w[i / 2]) : unpack_lo<BF16>(w[i / 2]);
}

template <int D>
struct DecodeSmem {
  alignas(128) uint16_t k[kStages][kTK * D];
  alignas(128) uint16_t v[kStages][kTK * D];
  float red[4][D];
  float xchg[2 * 2 * 128];
  float lse_all[256];  // fused merge: the P partition LSEs of this row-head
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
  int last;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads)
    decode_splitk_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                         const uint16_t* __restrict__ v, void* __restrict__ o_partial,
                         float* __restrict__ lse_partial, long long BH, int Nkv, int P, int chunk,
                         float scale_log2, int partial_f32, const MaskArgs mk, const FusedMerge fm,
                         unsigned int* status) {
  constexpr int EPL = D >= 32 ? D / 32 : 1;   // elements of a row per lane
  constexpr int LANES = D >= 32 ? 32 : D;     // lanes holding row elements
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long bh = blockIdx.x / P;
  const int part = blockIdx.x % P;
  const int lo = min(part * chunk, Nkv);
  const int hi = min(lo + chunk, Nkv);
  const int nkeys = hi - lo;
  const int ntiles = (nkeys + kTK - 1) / kTK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 4);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &sm.abort;

  if (warp == 4) {
    // ------------------------------------------------------------ copy warp
    if (lane == 0) {
      const size_t row_bytes = (size_t)D * 2;
      const uint8_t* kb = reinterpret_cast<const uint8_t*>(k) + ((size_t)bh * Nkv + lo) * row_bytes;
      const uint8_t* vb = reinterpret_cast<const uint8_t*>(v) + ((size_t)bh * Nkv + lo) * row_bytes;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages;
        const uint32_t use = t / kStages;
        if (!mbar_wait(&sm.empty[s], (use & 1u) ^ 1u, abort, status, kErrWaitLoad)) break;
        const int nk = min(kTK, nkeys - t * kTK);
        const uint32_t bytes = (uint32_t)(nk * row_bytes);
        mbar_arrive_expect_tx(&sm.full[s], 2 * bytes);
        bulk_load(sm.k[s], kb + (size_t)t * kTK * row_bytes, bytes, &sm.full[s]);
        bulk_load(sm.v[s], vb + (size_t)t * kTK * row_bytes, bytes, &sm.full[s]);
        issued = t + 1;
      }
      // Drain: every copy this thread started must land before the CTA exits.
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_drain(&sm.full[t % kStages], (uint32_t)(t / kStages) & 1u, status);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    float qv[EPL], o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      o[e] = 0.f;
      qv[e] = 0.f;
    }
    if (lane < LANES) load_row<EPL, BF16>(q + bh * D + lane * EPL, qv);
    float m = -INFINITY;  // running max in use (log2 units of the scaled score)
    float l = 0.f;        // this warp's partial denominator
    uint32_t seq = 0;     // monotone exchange counter of the warpgroup
    const uint32_t* mrow = nullptr;  // mask word of the partition's first key tile
    if (mk.bits != nullptr) {
      const long long b = bh / mk.H, h = bh - b * mk.H;
      mrow = mk.bits + b * mk.sb + h * mk.sh + (lo >> 5);
    }
    uint32_t mwin = ~0u;  // lane i: mask word of tile (t & ~31) + i

    for (int t = 0; t < ntiles; ++t) {
      const int s = t % kStages;
      if (mrow != nullptr && (t & 31) == 0) mwin = (t + lane < ntiles) ? __ldg(mrow + t + lane) : 0u;
      const uint32_t mword = __shfl_sync(0xffffffffu, mwin, t & 31);
      // On a failed wait the warp keeps going through the loop without touching the
      // stage, so that all four warps still meet at every exchange barrier.
      const bool ok = mbar_wait(&sm.full[s], (uint32_t)(t / kStages) & 1u, abort, status, kErrWaitFull);
      const uint16_t* ks = sm.k[s];
      const uint16_t* vs = sm.v[s];
      const int key0 = t * kTK + warp * kKeysPerWarp;  // first key of this warp, partition-relative

      // Partial dot products of this lane's EPL elements with the warp's 8 keys.
      float dp[kKeysPerWarp];
#pragma unroll
      for (int i = 0; i < kKeysPerWarp; ++i) {
        dp[i] = 0.f;
        if (ok && lane < LANES) {  // rows past the partition end hold stale data: masked below
          float kf[EPL];
          load_row<EPL, BF16>(ks + (warp * kKeysPerWarp + i) * D + lane * EPL, kf);
#pragma unroll
          for (int e = 0; e < EPL; ++e) dp[i] = fmaf(qv[e], kf[e], dp[i]);
        }
      }
      // Butterfly reduce-scatter: after the xor-16/8/4 halving steps and two xor
      // reductions, lanes 4k..4k+3 hold the full dot product of key k (9 shuffles for 8
      // keys instead of 5 per key).
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
      float e4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float send = b4 ? dp[j] : dp[j + 4];
        const float keep = b4 ? dp[j + 4] : dp[j];
        e4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
      float f2[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float send = b3 ? e4[j] : e4[j + 2];
        const float keep = b3 ? e4[j + 2] : e4[j];
        f2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      float g = (b2 ? f2[1] : f2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? f2[0] : f2[1], 4);
      g += __shfl_xor_sync(0xffffffffu, g, 2);
      g += __shfl_xor_sync(0xffffffffu, g, 1);
      const int my_key = (lane >> 2) & 7;  // key of this lane's score within the warp's 8
      const bool valid = ok && key0 + my_key < nkeys && ((mword >> (warp * kKeysPerWarp + my_key)) & 1u);
      const float sc = valid ? g * scale_log2 : -INFINITY;
      float tmax = sc;  // max over the 8 keys (lanes of one key agree)
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      // All four warps agree on the tile maximum (bit-identical result everywhere).
      tmax = ws_exchange<4, 32, true>(tmax, lane, warp, 0, seq++, sm.xchg, 1);
      const float mnew = fmaxf(m, tmax);
      if (mnew - m > kTau) {  // identical decision in every thread
        const float alpha = (m == -INFINITY) ? 0.f : ex2(m - mnew);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] *= alpha;
        m = mnew;
      }
      const float base = (m == -INFINITY) ? 0.f : m;
      const float pk = ex2(sc - base);  // 0 for masked keys
      // Sum over the 8 keys: the xor-4/8/16 partners hold the 8 different keys, so each
      // key is counted once in every lane.
      float psum = pk;
      psum += __shfl_xor_sync(0xffffffffu, psum, 4);
      psum += __shfl_xor_sync(0xffffffffu, psum, 8);
      psum += __shfl_xor_sync(0xffffffffu, psum, 16);
      l += psum;
#pragma unroll
      for (int i = 0; i < kKeysPerWarp; ++i) {
        const float p = __shfl_sync(0xffffffffu, pk, 4 * i);
        if (ok && key0 + i < nkeys && lane < LANES) {  // warp-uniform except the lane test
          float vf[EPL];
          load_row<EPL, BF16>(vs + (warp * kKeysPerWarp + i) * D + lane * EPL, vf);
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[e] = fmaf(p, vf[e], o[e]);
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&sm.empty[s]);
    }

    // Merge the four warps: one common scale, so plain sums.
    const float ltot = ws_exchange<4, 32, false>(l, lane, warp, 0, seq++, sm.xchg, 1);
    if (lane < LANES) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) sm.red[warp][lane * EPL + e] = o[e];
    }
    named_bar_sync(1, 128);
    if (tid < D) {
      const float sum = ((sm.red[0][tid] + sm.red[1][tid]) + sm.red[2][tid]) + sm.red[3][tid];
      const float y = (ltot > 0.f) ? sum / ltot : 0.f;
      const size_t idx = ((size_t)part * BH + bh) * D + tid;
      if (partial_f32) {
        static_cast<float*>(o_partial)[idx] = y + 0.f;
      } else {
        uint16_t b;
        if (BF16) b = __bfloat16_as_ushort(__float2bfloat16_rn(y + 0.f));
        else b = __half_as_ushort(__float2half_rn(y + 0.f));
        static_cast<uint16_t*>(o_partial)[idx] = b;
      }
    }
    if (tid == 0) lse_partial[(size_t)part * BH + bh] = (ltot > 0.f) ? m + lg2(ltot) : -INFINITY;
  }
  if (fm.counters == nullptr) {
    __syncthreads();
    return;
  }

  // ---- in-kernel merge ("Streaming attention and online state", Online statistics:
  // independent summaries merge by rescaling each with exp(m_i - m); here each partition
  // is already normalised, so the weights are 2^(lse_p - G) as in "fa4_splitk_combine").
  // The CTA's partial is published before its arrival is counted (barrier, then one
  // release fence and the counter update by thread 0); the CTA that arrives last
  // acquires the others' partials the same way and reads them back (from L2).
  __syncthreads();
  if (tid == 0) {
    fence_acq_rel_gpu();
    sm.last = atomicAdd(fm.counters + bh, 1u) == (unsigned)(P - 1);
    if (sm.last) {
      fence_acq_rel_gpu();
      fm.counters[bh] = 0u;  // ready for the next call
    }
  }
  __syncthreads();
  if (!sm.last) return;
  for (int p = tid; p < P; p += kThreads) sm.lse_all[p] = __ldcg(lse_partial + (size_t)p * BH + bh);
  __syncthreads();
  float mstar = -INFINITY;
  for (int p = 0; p < P; ++p) mstar = fmaxf(mstar, sm.lse_all[p]);
  float G = -INFINITY;
  if (mstar != -INFINITY) {
    float sum = 0.f;
    for (int p = 0; p < P; ++p) sum += ex2(sm.lse_all[p] - mstar);  // 2^-inf = 0
    G = mstar + lg2(sum);
  }
  if (tid < D) {
    float acc = 0.f;
    if (G != -INFINITY) {
      // Eight partitions per step, their loads issued together (independent L2 reads).
      constexpr int kU = 8;
      for (int p0 = 0; p0 < P; p0 += kU) {
        float x[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          const int p = p0 + j;
          x[j] = 0.f;
          if (p < P) {
            const size_t idx = ((size_t)p * BH + bh) * D + tid;
            if (partial_f32) {
              x[j] = __ldcg(static_cast<const float*>(o_partial) + idx);
            } else {
              const unsigned short b = __ldcg(static_cast<const unsigned short*>(o_partial) + idx);
              x[j] = BF16 ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          const int p = p0 + j;
          // an empty partition (lse -inf) contributes nothing
          if (p < P && sm.lse_all[p] != -INFINITY) acc = fmaf(ex2(sm.lse_all[p] - G), x[j], acc);
        }
      }
    }
    const uint16_t y = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(acc + 0.f))
                            : __half_as_ushort(__float2half_rn(acc + 0.f));
    static_cast<uint16_t*>(fm.o)[(size_t)bh * D + tid] = y;
  }
  if (tid == 0 && fm.lse != nullptr) fm.lse[bh] = G * 0.6931471805599453f;
}

template <int D, bool BF16>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  auto kern = decode_splitk_kernel<D, BF16>;
  const int smem = (int)sizeof(DecodeSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = a.BH * a.P;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(
      static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
      static_cast<const uint16_t*>(a.v), a.o_partial, a.lse_partial, a.BH, a.Nkv, a.P, a.chunk,
      a.scale_log2, a.partial_dtype == kF32 ? 1 : 0, a.mask, a.fused, a.status);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_dt(const DecodeArgs& a, cudaStream_t st) {
  switch (a.D) {
    case 16: return launch_t<16, BF16>(a, st);
    case 32: return launch_t<32, BF16>(a, st);
    case 64: return launch_t<64, BF16>(a, st);
    case 128: return launch_t<128, BF16>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.BH <= 0 || a.P <= 0) return cudaSuccess;
  return a.dtype == kBF16 ? launch_dt<true>(a, st) : launch_dt<false>(a, st);
}

}  // namespace oattn
