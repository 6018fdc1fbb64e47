// Split-K LSE-weighted combine ("fa4_splitk_combine", the Mojo module doc for the SM100
// workspace combine): one warp per output row-head rh, reducing over P partitions
//   m* = max_p lse_p,  G = log2(sum_p 2^(lse_p - m*)) + m*,
//   scale_p = 2^(lse_p - G),  O[d] = sum_p scale_p * o_partial[p, rh, d].
//
// Structure on GB300: the LSE reduction is done once per warp into per-lane
// registers (lane l keeps partitions l, l+32, ...; five xor shuffles for the max and
// five for the sum); each partition's scale is then broadcast from its owning lane
// with one indexed shuffle, and the depth vector of the next partition step is loaded
// (128-bit loads) before the current one is folded in; the first steps are requested
// before the LSE reduction, whose loads they do not depend on.  Ladder sizes P in
// {2, 4, 8, 16, 32} get fully unrolled instances; any other P runs a runtime-bound loop.
// Rows shorter than a warp of 128-bit vectors:
//   * at P = 2 and 4 every lane owns one vector of a row-head and folds all partitions
//     itself, several row-heads per warp with all loads in flight;
//   * rows of 16 vectors (16-bit data at depth 128), any other P: half a warp owns a
//     row-head end to end (two per warp; at P = 8 two row-heads per half-warp), so
//     nothing is summed across half-warps;
//   * other short rows: the warp splits into 32/LPP groups that take consecutive
//     partitions of one row-head and are summed at the end.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace oattn {
namespace {

constexpr int kCombineWarps = 8;  // row-heads per 256-thread block

// Programmatic dependent launch ("fa4_splitk_combine", PDL paragraph): when the combine
// is launched as a dependent of the split-K producer, its blocks may start while the
// producer's last blocks are still running; every thread waits here, before its first
// read, until the producer grid has completed and its writes are visible.  The
// producer issues no early trigger, so the release is its completion.  Without a
// programmatic dependency the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kern` with the programmatic-stream-serialisation attribute when pdl is set.
template <typename Kern, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, Kern kern, dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
constexpr int kMaxP = 256;
constexpr int kLseSlots = kMaxP / 32;

template <typename T> struct Vec;  // one 16-byte vector of T
template <> struct Vec<float> { static constexpr int E = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int E = 8; };
template <> struct Vec<__half> { static constexpr int E = 8; };

// Widen one raw 16-byte vector of T to floats.
template <typename T>
__device__ __forceinline__ void widen_vec(const uint4 u, float (&x)[Vec<T>::E]) {
  if constexpr (Vec<T>::E == 4) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  } else {
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = unpack_lo<BF>(w[i]);
      x[2 * i + 1] = unpack_hi<BF>(w[i]);
    }
  }
}

template <typename T, int E>
__device__ __forceinline__ void store_vec(T* p, const float (&x)[E]) {
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int i = 0; i < E; i += 4)
      *reinterpret_cast<float4*>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  } else {
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    if constexpr (E == 8) {
      uint4 u;
      u.x = pack2<BF>(x[0], x[1]); u.y = pack2<BF>(x[2], x[3]);
      u.z = pack2<BF>(x[4], x[5]); u.w = pack2<BF>(x[6], x[7]);
      *reinterpret_cast<uint4*>(p) = u;
    } else {
      uint2 u;
      u.x = pack2<BF>(x[0], x[1]); u.y = pack2<BF>(x[2], x[3]);
      *reinterpret_cast<uint2*>(p) = u;
    }
  }
}

// TIn/TOut element types; LPP lanes per partition row; VPL 16-byte vectors per lane;
// P_STATIC > 0: exact partition count, fully unrolled; 0: runtime P (<= kMaxP).
template <typename TIn, typename TOut, int LPP, int VPL, int P_STATIC>
__global__ void __launch_bounds__(kCombineWarps * 32)
    splitk_combine_kernel(const TIn* __restrict__ o_partial, const float* __restrict__ lse_partial,
                          TOut* __restrict__ out, float* __restrict__ lse_out, int P_rt,
                          long long RH, float lse_scale) {
  constexpr int E = Vec<TIn>::E;
  constexpr int PPS = 32 / LPP;               // partitions folded per step
  constexpr int DEPTH = LPP * VPL * E;
  constexpr int SLOTS = P_STATIC > 0 ? (P_STATIC + 31) / 32 : kLseSlots;
  const int P = P_STATIC > 0 ? P_STATIC : P_rt;

  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long rh = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (rh >= RH) return;  // whole warp leaves together

  const int sub = lane / LPP;  // which partition of a step this lane folds
  const int li = lane % LPP;
  const TIn* base = o_partial + rh * DEPTH + li * E;
  const long long pstride = RH * (long long)DEPTH;
  const int steps = (P + PPS - 1) / PPS;

  // Raw 16-byte vectors of step `step` (partition step*PPS + sub); zeros past the last
  // partition.  They stay packed until folded, which halves the registers that the
  // prefetch buffers need for 16-bit inputs.
  auto fetch = [&](int step, uint4 (&x)[VPL]) {
    const int p = step * PPS + sub;
#pragma unroll
    for (int v = 0; v < VPL; ++v)
      x[v] = (p < P) ? __ldcs(reinterpret_cast<const uint4*>(base + p * pstride + v * LPP * E))
                     : make_uint4(0u, 0u, 0u, 0u);
  };
  float acc[VPL][E];
#pragma unroll
  for (int v = 0; v < VPL; ++v)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[v][e] = 0.f;
  auto fold = [&](float sc, const uint4 (&x)[VPL]) {
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float w[E];
      widen_vec<TIn>(x[v], w);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[v][e] = fmaf(sc, (sc != 0.f) ? w[e] : 0.f, acc[v][e]);
    }
  };

  // The partition vectors do not depend on the LSE reduction: the first ones are
  // requested before it, so both memory latencies overlap.
  constexpr int STATIC_STEPS = P_STATIC > 0 ? (P_STATIC + PPS - 1) / PPS : 0;
  constexpr int AHEAD = STATIC_STEPS > 0 ? (STATIC_STEPS <= 8 ? STATIC_STEPS : 2) : 4;
  uint4 pre[AHEAD][VPL];
#pragma unroll
  for (int i = 0; i < AHEAD; ++i) fetch(i, pre[i]);

  // ---- LSE reduction, once, into per-lane registers
  float lse[SLOTS];
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int p = s * 32 + lane;
    lse[s] = (p < P) ? __ldg(lse_partial + (long long)p * RH + rh) : -INFINITY;
    m = fmaxf(m, lse[s]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const bool dead = (m == -INFINITY);
  const float msafe = dead ? 0.f : m;
  float sum = 0.f;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) sum += ex2(lse[s] - msafe);  // ex2(-inf) = +0
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float G = dead ? -INFINITY : lg2(sum) + msafe;
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) lse[s] = dead ? 0.f : ex2(lse[s] - G);  // now scale_p

  // ---- weighted accumulation
  if constexpr (P_STATIC > 0) {
    if constexpr (STATIC_STEPS <= 8) {
      // everything is already in flight: fold in order
#pragma unroll
      for (int step = 0; step < STATIC_STEPS; ++step) {
        const int p = step * PPS + sub;
        const float sc = __shfl_sync(0xffffffffu, lse[(step * PPS) / 32], p & 31);
        fold(p < P ? sc : 0.f, pre[step]);
      }
    } else {
      // two steps ahead through a register ring (indices are compile-time after unrolling)
#pragma unroll
      for (int step = 0; step < STATIC_STEPS; ++step) {
        const int p = step * PPS + sub;
        const float sc = __shfl_sync(0xffffffffu, lse[(step * PPS) / 32], p & 31);
        uint4 cur[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) cur[v] = pre[step % AHEAD][v];
        if (step + AHEAD < STATIC_STEPS) fetch(step + AHEAD, pre[step % AHEAD]);
        fold(p < P ? sc : 0.f, cur);
      }
    }
  } else {
    // Runtime P: a partition's scale would need a run-time register index, so the
    // warp parks its per-lane scales in its own shared-memory row and every lane reads
    // the one it needs (a broadcast read).  Vectors stream in chunks of four steps,
    // the next chunk requested before the current one is folded.
    __shared__ float s_scale[kCombineWarps][kMaxP];
    float* my = s_scale[threadIdx.x >> 5];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
      if (s * 32 + lane < P) my[s * 32 + lane] = lse[s];
    __syncwarp();
    uint4 nxt[AHEAD][VPL];
    for (int c0 = 0; c0 < steps; c0 += 2 * AHEAD) {
      // pre holds steps c0 .. c0+3; request c0+4 .. c0+7 into nxt
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) fetch(c0 + AHEAD + i, nxt[i]);
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) {
        const int p = (c0 + i) * PPS + sub;
        fold(p < P ? my[p] : 0.f, pre[i]);
      }
      // request c0+8 .. c0+11 into pre, fold nxt
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) fetch(c0 + 2 * AHEAD + i, pre[i]);
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) {
        const int p = (c0 + AHEAD + i) * PPS + sub;
        fold(p < P ? my[p] : 0.f, nxt[i]);
      }
    }
  }

  // ---- fold the PPS partition groups of the warp together and store
#pragma unroll
  for (int o = LPP; o < 32; o <<= 1)
#pragma unroll
    for (int v = 0; v < VPL; ++v)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[v][e] += __shfl_xor_sync(0xffffffffu, acc[v][e], o);

  if (sub == 0) {
    TOut* dst = out + rh * DEPTH + li * E;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float y[E];
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = dead ? 0.f : acc[v][e] + 0.f;
      store_vec<TOut, E>(dst + v * LPP * E, y);
    }
  }
  if (lse_out != nullptr && lane == 0) lse_out[rh] = dead ? -INFINITY : G * lse_scale;
}

// Small P (a ladder rung of at most 4 partitions): a warp owns RPW row-heads and puts
// every load of all of them in flight before reducing any, so that the few bytes per
// row-head do not leave the warp waiting on one dependent load chain after another.
template <typename TIn, typename TOut, int LPP, int VPL, int P_STATIC, int RPW>
__global__ void __launch_bounds__(kCombineWarps * 32)
    splitk_combine_small_kernel(const TIn* __restrict__ o_partial, const float* __restrict__ lse_partial,
                                TOut* __restrict__ out, float* __restrict__ lse_out, long long RH,
                                float lse_scale) {
  constexpr int E = Vec<TIn>::E;
  constexpr int PPS = 32 / LPP;
  constexpr int DEPTH = LPP * VPL * E;
  constexpr int STEPS = (P_STATIC + PPS - 1) / PPS;
  static_assert(P_STATIC <= 32, "one LSE per lane");
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long rh0 = ((long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5)) * RPW;
  if (rh0 >= RH) return;  // whole warp leaves together
  const int sub = lane / LPP;
  const int li = lane % LPP;
  const long long pstride = RH * (long long)DEPTH;

  uint4 x[RPW][STEPS][VPL];
  float lse[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const long long rh = rh0 + r;
    const bool valid = rh < RH;
    const TIn* base = o_partial + rh * DEPTH + li * E;
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int p = st * PPS + sub;
#pragma unroll
      for (int v = 0; v < VPL; ++v)
        x[r][st][v] = (valid && p < P_STATIC)
                          ? __ldcs(reinterpret_cast<const uint4*>(base + p * pstride + v * LPP * E))
                          : make_uint4(0u, 0u, 0u, 0u);
    }
    lse[r] = (valid && lane < P_STATIC) ? __ldg(lse_partial + (long long)lane * RH + rh) : -INFINITY;
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const long long rh = rh0 + r;
    // Only lanes 0..P-1 hold an LSE: reduce over that many lanes, then broadcast.
    constexpr int W = P_STATIC <= 1 ? 1 : (P_STATIC <= 2 ? 2 : (P_STATIC <= 4 ? 4 : 32));
    float m = lse[r];
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    m = __shfl_sync(0xffffffffu, m, 0);
    const bool dead = (m == -INFINITY);
    const float msafe = dead ? 0.f : m;
    float sum = ex2(lse[r] - msafe);
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    sum = __shfl_sync(0xffffffffu, sum, 0);
    const float G = dead ? -INFINITY : lg2(sum) + msafe;
    const float scale = dead ? 0.f : ex2(lse[r] - G);
    float acc[VPL][E];
#pragma unroll
    for (int v = 0; v < VPL; ++v)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[v][e] = 0.f;
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      const int p = st * PPS + sub;
      float sc = __shfl_sync(0xffffffffu, scale, p & 31);
      sc = p < P_STATIC ? sc : 0.f;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        float w[E];
        widen_vec<TIn>(x[r][st][v], w);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[v][e] = fmaf(sc, (sc != 0.f) ? w[e] : 0.f, acc[v][e]);
      }
    }
#pragma unroll
    for (int o = LPP; o < 32; o <<= 1)
#pragma unroll
      for (int v = 0; v < VPL; ++v)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[v][e] += __shfl_xor_sync(0xffffffffu, acc[v][e], o);
    if (rh < RH) {
      if (sub == 0) {
        TOut* dst = out + rh * DEPTH + li * E;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          float y[E];
#pragma unroll
          for (int e = 0; e < E; ++e) y[e] = dead ? 0.f : acc[v][e] + 0.f;
          store_vec<TOut, E>(dst + v * LPP * E, y);
        }
      }
      if (lse_out != nullptr && lane == 0) lse_out[rh] = dead ? -INFINITY : G * lse_scale;
    }
  }
}

// Small P with short rows (NV < 32 vectors of 16 bytes per partition row): each lane owns
// one vector of the row and folds all P partitions into it itself, so nothing crosses
// lanes but the broadcast LSE loads; a warp covers 32/NV row-heads per pass and RPW
// passes, with every load of all of them in flight before the first fold.
template <typename TIn, typename TOut, int NV, int P_STATIC, int RPW>
__global__ void __launch_bounds__(kCombineWarps * 32)
    splitk_combine_lane_kernel(const TIn* __restrict__ o_partial, const float* __restrict__ lse_partial,
                               TOut* __restrict__ out, float* __restrict__ lse_out, long long RH,
                               float lse_scale) {
  constexpr int E = Vec<TIn>::E;
  constexpr int G = 32 / NV;  // row-heads per pass
  constexpr int DEPTH = NV * E;
  static_assert(NV < 32 && 32 % NV == 0, "a row-head takes a whole number of lanes");
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long rh0 = ((long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5)) * (RPW * G);
  if (rh0 >= RH) return;  // whole warp leaves together
  const int g = lane / NV, li = lane % NV;
  const long long pstride = RH * (long long)DEPTH;

  uint4 x[RPW][P_STATIC];
  float lse[RPW][P_STATIC];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const long long rh = rh0 + r * G + g;
    const bool valid = rh < RH;
    const TIn* base = o_partial + rh * DEPTH + li * E;
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p)
      x[r][p] = valid ? __ldcs(reinterpret_cast<const uint4*>(base + p * pstride)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p) lse[r][p] = valid ? __ldg(lse_partial + (long long)p * RH + rh) : -INFINITY;
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const long long rh = rh0 + r * G + g;
    float m = lse[r][0];
#pragma unroll
    for (int p = 1; p < P_STATIC; ++p) m = fmaxf(m, lse[r][p]);
    const bool dead = (m == -INFINITY);
    const float msafe = dead ? 0.f : m;
    float sum = 0.f;
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p) sum += ex2(lse[r][p] - msafe);
    const float Gl = dead ? -INFINITY : lg2(sum) + msafe;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p) {
      const float sc = dead ? 0.f : ex2(lse[r][p] - Gl);
      float w[E];
      widen_vec<TIn>(x[r][p], w);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(sc, (sc != 0.f) ? w[e] : 0.f, acc[e]);
    }
    if (rh < RH) {
      float y[E];
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = dead ? 0.f : acc[e] + 0.f;
      store_vec<TOut, E>(out + rh * DEPTH + li * E, y);
      if (lse_out != nullptr && li == 0) lse_out[rh] = dead ? -INFINITY : Gl * lse_scale;
    }
  }
}

// Rows shorter than a warp of 16-byte vectors (LPP < 32 lanes per row, e.g. 16-bit data
// at depth 128): each group of LPP lanes owns one row-head end to end, 32/LPP row-heads
// per warp.  The LSE reduction and the scale broadcasts stay inside the group
// (width-LPP shuffles), every lane folds all P partitions of its 16-byte vector, and
// nothing is summed across groups at the end.  AHEAD partition vectors per lane are in
// flight while the current one is folded.
template <typename TIn, typename TOut, int LPP, int P_STATIC>
__global__ void __launch_bounds__(kCombineWarps * 32)
    splitk_combine_group_kernel(const TIn* __restrict__ o_partial, const float* __restrict__ lse_partial,
                                TOut* __restrict__ out, float* __restrict__ lse_out, int P_rt, long long RH,
                                float lse_scale) {
  constexpr int E = Vec<TIn>::E;
  constexpr int G = 32 / LPP;  // row-heads per warp
  constexpr int DEPTH = LPP * E;
  constexpr int SLOTS = P_STATIC > 0 ? (P_STATIC + LPP - 1) / LPP : kMaxP / LPP;
  constexpr int AHEAD = 8;
  static_assert(LPP < 32 && 32 % LPP == 0, "a row-head takes a whole number of lanes");
  static_assert(P_STATIC > 0 || G * kMaxP * kCombineWarps * 4 <= 32768, "runtime-P scales fit shared memory");
  const int P = P_STATIC > 0 ? P_STATIC : P_rt;

  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long rh0 = ((long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5)) * G;
  if (rh0 >= RH) return;  // whole warp leaves together
  const int g = lane / LPP, li = lane % LPP;
  const long long rh = rh0 + g;
  const bool valid = rh < RH;
  const TIn* base = o_partial + rh * DEPTH + li * E;
  const long long pstride = RH * (long long)DEPTH;
  auto load = [&](int p) {
    return (valid && p < P) ? __ldcs(reinterpret_cast<const uint4*>(base + p * pstride)) : make_uint4(0u, 0u, 0u, 0u);
  };

  // The first partition vectors are requested before the LSE reduction.
  uint4 x[AHEAD];
#pragma unroll
  for (int i = 0; i < AHEAD; ++i) x[i] = load(i);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  auto fold = [&](float sc, const uint4 v) {
    float w[E];
    widen_vec<TIn>(v, w);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(sc, (sc != 0.f) ? w[e] : 0.f, acc[e]);
  };
  bool dead;
  float Gl;
  if constexpr (P_STATIC > 0) {
    // ---- LSE reduction inside the group: lane li keeps partitions li, li + LPP, ...
    float lse[SLOTS];
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int p = s * LPP + li;
      lse[s] = (valid && p < P) ? __ldg(lse_partial + (long long)p * RH + rh) : -INFINITY;
      m = fmaxf(m, lse[s]);
    }
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    dead = (m == -INFINITY);
    const float msafe = dead ? 0.f : m;
    float sum = 0.f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) sum += ex2(lse[s] - msafe);  // ex2(-inf) = +0
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    Gl = dead ? -INFINITY : lg2(sum) + msafe;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) lse[s] = dead ? 0.f : ex2(lse[s] - Gl);  // now scale_p
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p) {
      const float sc = __shfl_sync(0xffffffffu, lse[p / LPP], p % LPP, LPP);
      const uint4 cur = x[p % AHEAD];
      if (p + AHEAD < P_STATIC) x[p % AHEAD] = load(p + AHEAD);
      fold(sc, cur);
    }
  } else {
    // Runtime P: the group's LSEs, then its scales, live in its own shared-memory row
    // (a run-time register index would spill), so no per-lane arrays are kept; the
    // vectors stream through one rolling buffer of AHEAD.
    __shared__ float s_scale[kCombineWarps][G][kMaxP];
    float* my = s_scale[threadIdx.x >> 5][g];
    float m = -INFINITY;
    for (int p = li; p < P; p += LPP) {
      const float v = valid ? __ldg(lse_partial + (long long)p * RH + rh) : -INFINITY;
      my[p] = v;
      m = fmaxf(m, v);
    }
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    dead = (m == -INFINITY);
    const float msafe = dead ? 0.f : m;
    float sum = 0.f;
    for (int p = li; p < P; p += LPP) sum += ex2(my[p] - msafe);
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    Gl = dead ? -INFINITY : lg2(sum) + msafe;
    for (int p = li; p < P; p += LPP) my[p] = dead ? 0.f : ex2(my[p] - Gl);
    __syncwarp();
    for (int p0 = 0; p0 < P; p0 += AHEAD) {
#pragma unroll
      for (int i = 0; i < AHEAD; ++i) {
        const uint4 cur = x[i];
        x[i] = load(p0 + AHEAD + i);
        if (p0 + i < P) fold(my[p0 + i], cur);
      }
    }
  }
  if (valid) {
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = dead ? 0.f : acc[e] + 0.f;
    store_vec<TOut, E>(out + rh * DEPTH + li * E, y);
    if (lse_out != nullptr && li == 0) lse_out[rh] = dead ? -INFINITY : Gl * lse_scale;
  }
}

// Rows of LPP < 32 vectors, small ladder P: each group of LPP lanes owns RPG row-heads
// (interleaved with the other groups', so that a warp's loads of one step are
// contiguous) and puts the loads of all of them in flight before folding any, so that
// short kernels keep more bytes moving per warp.
template <typename TIn, typename TOut, int LPP, int P_STATIC, int RPG>
__global__ void __launch_bounds__(kCombineWarps * 32)
    splitk_combine_group_multi_kernel(const TIn* __restrict__ o_partial, const float* __restrict__ lse_partial,
                                      TOut* __restrict__ out, float* __restrict__ lse_out, long long RH,
                                      float lse_scale) {
  constexpr int E = Vec<TIn>::E;
  constexpr int G = 32 / LPP;
  constexpr int DEPTH = LPP * E;
  static_assert(P_STATIC <= LPP, "one LSE per lane of the group");
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long rh0 = ((long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5)) * G * RPG;
  if (rh0 >= RH) return;  // whole warp leaves together
  const int g = lane / LPP, li = lane % LPP;
  const long long pstride = RH * (long long)DEPTH;
  uint4 x[RPG][P_STATIC];
  float lse[RPG];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const long long rh = rh0 + r * G + g;
    const bool valid = rh < RH;
    const TIn* base = o_partial + rh * DEPTH + li * E;
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p)
      x[r][p] = valid ? __ldcs(reinterpret_cast<const uint4*>(base + p * pstride)) : make_uint4(0u, 0u, 0u, 0u);
    lse[r] = (valid && li < P_STATIC) ? __ldg(lse_partial + (long long)li * RH + rh) : -INFINITY;
  }
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const long long rh = rh0 + r * G + g;
    float m = lse[r];
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const bool dead = (m == -INFINITY);
    const float msafe = dead ? 0.f : m;
    float sum = ex2(lse[r] - msafe);
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float Gl = dead ? -INFINITY : lg2(sum) + msafe;
    const float scale = dead ? 0.f : ex2(lse[r] - Gl);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int p = 0; p < P_STATIC; ++p) {
      const float sc = __shfl_sync(0xffffffffu, scale, p, LPP);
      float w[E];
      widen_vec<TIn>(x[r][p], w);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(sc, (sc != 0.f) ? w[e] : 0.f, acc[e]);
    }
    if (rh < RH) {
      float y[E];
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = dead ? 0.f : acc[e] + 0.f;
      store_vec<TOut, E>(out + rh * DEPTH + li * E, y);
      if (lse_out != nullptr && li == 0) lse_out[rh] = dead ? -INFINITY : Gl * lse_scale;
    }
  }
}

template <typename TIn, typename TOut, int LPP, int VPL>
cudaError_t launch_p(const void* op, const float* lp, void* o, float* lo, int P, long long RH,
                     float lse_scale, bool pdl, cudaStream_t st) {
  const dim3 grid((unsigned)((RH + kCombineWarps - 1) / kCombineWarps));
  const dim3 block(kCombineWarps * 32);
  auto* a = static_cast<const TIn*>(op);
  auto* c = static_cast<TOut*>(o);
  // Row-heads per warp at P = 2 and 4 (measured): with 16-bit rows of one vector per lane
  // fewer row-heads per warp, hence more warps, keep more of HBM busy at P = 2.
  constexpr bool kWide = sizeof(TIn) == 2 && VPL == 1;
  constexpr int R2 = kWide ? 4 : 8, R4 = 4;
  const dim3 grid_small2((unsigned)((RH + kCombineWarps * R2 - 1) / (kCombineWarps * R2)));
  const dim3 grid_small4((unsigned)((RH + kCombineWarps * R4 - 1) / (kCombineWarps * R4)));
  cudaError_t e;
  // Short rows at P = 2 and 4: one lane per vector, P partitions folded in the lane,
  // 8 partition vectors in flight per lane (RPW = 8 / P passes).
  constexpr int kLaneG = 32 / LPP;
  const dim3 grid_lane2((unsigned)((RH + kCombineWarps * 4 * kLaneG - 1) / (kCombineWarps * 4 * kLaneG)));
  const dim3 grid_lane4((unsigned)((RH + kCombineWarps * 2 * kLaneG - 1) / (kCombineWarps * 2 * kLaneG)));
  if constexpr (LPP == 16 && VPL == 1) {
    // Rows of 16 vectors at P = 8: two row-heads per half-warp, all 16 loads in flight
    // (measured 1.01 of the copy peak against 0.96 with one; at P = 2 the lane kernel
    // below stays ahead of 4 or 8 row-heads per half-warp).
    if (P == 8) {
      constexpr int kRpg = 2;
      const dim3 grid_m((unsigned)((RH + kCombineWarps * kLaneG * kRpg - 1) / (kCombineWarps * kLaneG * kRpg)));
      e = launch_maybe_pdl(pdl, splitk_combine_group_multi_kernel<TIn, TOut, LPP, 8, kRpg>, grid_m, block, st, a, lp,
                           c, lo, RH, lse_scale);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
  }
  if constexpr (LPP < 32 && VPL == 1) {
    if (P == 2 || P == 4) {
      e = (P == 2) ? launch_maybe_pdl(pdl, splitk_combine_lane_kernel<TIn, TOut, LPP, 2, 4>, grid_lane2, block, st, a, lp, c, lo, RH, lse_scale)
                   : launch_maybe_pdl(pdl, splitk_combine_lane_kernel<TIn, TOut, LPP, 4, 2>, grid_lane4, block, st, a, lp, c, lo, RH, lse_scale);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
  }
  if constexpr (LPP == 16 && VPL == 1) {
    // Rows of 16 vectors (16-bit data at depth 128), any other P: half a warp per row-head.
    const dim3 grid_group((unsigned)((RH + kCombineWarps * kLaneG - 1) / (kCombineWarps * kLaneG)));
    switch (P) {
      case 8: e = launch_maybe_pdl(pdl, splitk_combine_group_kernel<TIn, TOut, LPP, 8>, grid_group, block, st, a, lp, c, lo, P, RH, lse_scale); break;
      case 16: e = launch_maybe_pdl(pdl, splitk_combine_group_kernel<TIn, TOut, LPP, 16>, grid_group, block, st, a, lp, c, lo, P, RH, lse_scale); break;
      case 32: e = launch_maybe_pdl(pdl, splitk_combine_group_kernel<TIn, TOut, LPP, 32>, grid_group, block, st, a, lp, c, lo, P, RH, lse_scale); break;
      default: e = launch_maybe_pdl(pdl, splitk_combine_group_kernel<TIn, TOut, LPP, 0>, grid_group, block, st, a, lp, c, lo, P, RH, lse_scale); break;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  switch (P) {
    case 2: e = launch_maybe_pdl(pdl, splitk_combine_small_kernel<TIn, TOut, LPP, VPL, 2, R2>, grid_small2, block, st, a, lp, c, lo, RH, lse_scale); break;
    case 4: e = launch_maybe_pdl(pdl, splitk_combine_small_kernel<TIn, TOut, LPP, VPL, 4, R4>, grid_small4, block, st, a, lp, c, lo, RH, lse_scale); break;
    case 8: e = launch_maybe_pdl(pdl, splitk_combine_kernel<TIn, TOut, LPP, VPL, 8>, grid, block, st, a, lp, c, lo, P, RH, lse_scale); break;
    case 16: e = launch_maybe_pdl(pdl, splitk_combine_kernel<TIn, TOut, LPP, VPL, 16>, grid, block, st, a, lp, c, lo, P, RH, lse_scale); break;
    case 32: e = launch_maybe_pdl(pdl, splitk_combine_kernel<TIn, TOut, LPP, VPL, 32>, grid, block, st, a, lp, c, lo, P, RH, lse_scale); break;
    default: e = launch_maybe_pdl(pdl, splitk_combine_kernel<TIn, TOut, LPP, VPL, 0>, grid, block, st, a, lp, c, lo, P, RH, lse_scale); break;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_depth(const void* op, const float* lp, void* o, float* lo, int P, long long RH,
                         int depth, float lse_scale, bool pdl, cudaStream_t st) {
  constexpr int E = Vec<TIn>::E;
  const int nvec = depth / E;  // 16-byte vectors per partition row
  switch (nvec) {
    case 2: return launch_p<TIn, TOut, 2, 1>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    case 4: return launch_p<TIn, TOut, 4, 1>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    case 8: return launch_p<TIn, TOut, 8, 1>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    case 16: return launch_p<TIn, TOut, 16, 1>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    case 32: return launch_p<TIn, TOut, 32, 1>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    case 64: return launch_p<TIn, TOut, 32, 2>(op, lp, o, lo, P, RH, lse_scale, pdl, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename TIn>
cudaError_t launch_out(const void* op, const float* lp, void* o, float* lo, int P, long long RH,
                       int depth, int out_dt, float lse_scale, bool pdl, cudaStream_t st) {
  switch (out_dt) {
    case kF32: return launch_depth<TIn, float>(op, lp, o, lo, P, RH, depth, lse_scale, pdl, st);
    case kBF16: return launch_depth<TIn, __nv_bfloat16>(op, lp, o, lo, P, RH, depth, lse_scale, pdl, st);
    case kF16: return launch_depth<TIn, __half>(op, lp, o, lo, P, RH, depth, lse_scale, pdl, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool combine_supported(int depth, int in_dt) {
  const int E = (in_dt == kF32) ? 4 : 8;
  if (depth % E) return false;
  const int nvec = depth / E;
  return nvec == 2 || nvec == 4 || nvec == 8 || nvec == 16 || nvec == 32 || nvec == 64;
}

cudaError_t launch_combine(const void* o_partial, const float* lse_partial, void* o, float* lse_out,
                           int P, long long RH, int depth, int in_dt, int out_dt, float lse_scale, bool pdl,
                           cudaStream_t st) {
  if (RH <= 0) return cudaSuccess;
  switch (in_dt) {
    case kF32: return launch_out<float>(o_partial, lse_partial, o, lse_out, P, RH, depth, out_dt, lse_scale, pdl, st);
    case kBF16: return launch_out<__nv_bfloat16>(o_partial, lse_partial, o, lse_out, P, RH, depth, out_dt, lse_scale, pdl, st);
    case kF16: return launch_out<__half>(o_partial, lse_partial, o, lse_out, P, RH, depth, out_dt, lse_scale, pdl, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oattn
