// Tiled attention forward with the online-softmax recurrence on tcgen05 tensor cores.
//
// What it computes ("A3. Tiled attention with online normalization", sections "Keep
// three quantities for each query row" and "Masks that preserve the recurrence";
// "Streaming attention and online state", section "Online statistics"): for every
// query row a running maximum m, denominator l and FP32 numerator o are carried over
// key tiles; each tile gives m' = max(m, rowmax s), alpha = exp(m - m'),
// p = exp(s - m'), l' = alpha l + rowsum p, o' = alpha o + p V; after the last tile the
// output is o / l and the row's log-sum-exp is m + log l.  Masked scores (keys past the
// end, keys after the query when causal, keys outside the split-K partition, keys the
// optional Boolean mask hides) are -inf and give p = 0; a row that saw no key ends
// with l = 0 and stores 0 and -inf.
//
// How it maps onto one GB300 SM (one CTA per SM: 193 KB of shared memory and all 512
// TMEM columns at D = 128):
//   * A CTA owns two 128-row query tiles of one head (and one split-K partition in
//     split mode).  Warps 0-3 and 4-7 are two softmax warpgroups, one per query tile;
//     thread r of a warpgroup owns row r, which is TMEM lane r, so row max and row sum
//     need no shuffles.  Warp 8 issues TMA copies, warp 9 issues the MMAs (all its
//     lanes walk the issue loop, one elected lane issues), warp 10 watches the K/V
//     copies for the MMA issuer (see below); warps 10-11 also complete
//     the third warpgroup so that setmaxnreg can move its registers to the softmax
//     warpgroups (216 per softmax thread).
//   * Q tiles are copied once; K and V tiles stream through a ring of shared-memory
//     slots (K in even, V in odd slots) filled by cp.async.bulk.tensor with the
//     128/64/32-byte swizzle that matches the tcgen05 shared-memory descriptors.
//     Keys past the end of the sequence arrive as zeros (out-of-bounds fill).
//   * S_t = Q_t K^T is a kind::f16 MMA (M=128, N=BN, K=D) into TMEM columns
//     [t*BN, (t+1)*BN).  The softmax threads read their row (tcgen05.ld), mask with
//     -inf, compute p = 2^(s*scale*log2e - m) with one FMA and one ex2.approx each,
//     sum the FP32 p, round p to the input dtype (cvt.rn, round to nearest even) and
//     write it back over S (tcgen05.st) as the A operand of
//     O_t += P V (M=128, N=D, K=BN, A from TMEM, B = V tile read MN-major).
//   * The MMA issuer is the critical path: one MMA of M=128, N=128, K=16 takes the
//     tensor pipe 64 cycles, about as long as issuing it takes.  The issue loop runs on
//     all 32 lanes of warp 9 with the issuing lane picked once by elect.sync, so every
//     descriptor and address is warp-uniform (a lone-thread loop measured 5% slower).
//     The issuer waits once per group: bar_p[t] counts the
//     128 softmax threads of tile t AND a watcher thread that has seen V_j and K_(j+1)
//     land, so one completed phase means "P_t(j) written, PV_t(j) and S_t(j+1) may
//     start".  The watcher never arrives for phase j before phase j - 1 completed.
//   * The issue order S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ... lets one
//     warpgroup's softmax run while the tensor pipe works on the other tile.  A
//     commit after S_t(j+1) also covers PV_t(j) (commits track every earlier MMA of the
//     issuing thread), so when the softmax sees S_t(j+1) it may rescale O_t safely.
//   * The stabiliser is lazy: m only has to keep p = 2^(x - m) bounded, so the common
//     path computes no row maximum at all.  A warp takes the maximum only while some
//     row has seen no key, or when a tile's row sum of p exceeds kPBound (2^15); then
//     it redoes that tile against the exact new maximum and rescales O (TMEM load,
//     multiply by alpha, store) and l.  Exact arithmetic is unchanged.
//   * The epilogue writes o / l into the query tile's own (now free) shared memory in
//     the swizzled layout of the output tensor map and stores it with one TMA copy per
//     row chunk (rows past the end are clipped by the copy).  Split-K partials are
//     stored directly from registers (FP32 or 16-bit).
//   * The optional Boolean M x N mask ("Streaming attention and online state", section
//     "Attention as a consumer") arrives packed one bit per key: each softmax thread
//     reads the 16 bytes of its row that cover the key tile while it waits for the
//     tile's scores, and turns the hidden scores to -inf with selects; a warp whose 32
//     rows see the whole tile skips the selects.  Before the key loop the softmax warps
//     scan the mask once and mark the key tiles that some row of the CTA sees; every
//     role then walks the marked tiles only (key tile 0 is always visited).
//   * CTAs are ordered in groups of kHeadGroup heads: within a group the query-tile
//     pairs run longest first (causal), and the few heads in flight keep their K/V in
//     L2 instead of streaming every head's K/V from HBM for every pair.
//
//   * Launches are programmatic dependents of the previous kernel on the stream: every
//     CTA lets the next grid be scheduled as soon as it starts, and waits for the
//     previous grid (griddepcontrol.wait) before its first global access.
//
// Every wait is bounded (see ptx.cuh); a thread that gives up marks the CTA aborted,
// everyone leaves its loop, copies and MMAs in flight are drained, TMEM is freed.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace oattn {

constexpr int pow2_at_least(int x, int p = 32) { return p >= x ? p : pow2_at_least(x, p * 2); }

template <int D, int BN>
struct AttnCfg {
  static constexpr int D_ = D, BN_ = BN;
  static constexpr int BM = 128;
  static constexpr int SW = D * 2 >= 128 ? 128 : D * 2;   // swizzle span = bytes per smem row
  static constexpr int CH = SW / 2;                        // elements per row chunk (TMA box x)
  static constexpr int NCH = D / CH;                       // chunks per row
  static constexpr uint32_t SWZ = SW == 128 ? kSwizzle128B : (SW == 64 ? kSwizzle64B : kSwizzle32B);
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int BUDGET = 200 * 1024;
  static constexpr int NSLOT_RAW = ((BUDGET - 2 * Q_BYTES) / KV_BYTES) & ~1;
  static constexpr int NSLOT = NSLOT_RAW > 8 ? 8 : NSLOT_RAW;
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + NSLOT * KV_BYTES;
  static constexpr int COL_S0 = 0, COL_S1 = BN, COL_O0 = 2 * BN, COL_O1 = 2 * BN + D;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + 2 * D);
  static constexpr int THREADS = 384;       // 2 softmax warpgroups + 1 copy/MMA warpgroup
  static constexpr int REGS_LAUNCH = 168;   // 65536 / 384 rounded down to a multiple of 8
  static constexpr int REGS_SOFTMAX = 216;  // after setmaxnreg.inc
  static constexpr int REGS_OTHER = 72;     // after setmaxnreg.dec
  // Per SM sub-partition: two softmax warps and one other warp share what three warps
  // had at launch (2*216 + 72 = 3*168).
  static_assert(2 * REGS_SOFTMAX + REGS_OTHER <= 3 * REGS_LAUNCH, "register split exceeds the launch pool");
  static_assert(NSLOT >= 4, "need at least two K/V tile pairs in flight");
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(BN % 32 == 0 && D % 16 == 0, "tile shapes");
};

// Bound on a tile's row sum of p = 2^(x - m) before the stabiliser m must move (keeps
// every p, and the 16-bit P operand, far from overflow; f16 stops at 65504).
constexpr float kPBound = 32768.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kHeadGroup = 8;

// Compiler fence: the registers filled by earlier tcgen05.ld are valid only after
// tcgen05.wait::ld; routing them through this empty asm (placed after the wait) keeps
// every use behind it.
__device__ __forceinline__ void reg_fence32(uint32_t* v) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]),
                 "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]),
                 "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}
__device__ __forceinline__ void reg_fence16(uint32_t* v) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Load NC consecutive TMEM columns of this thread's lane (NC = 16 or a multiple of 32):
// every load is issued first, then one wait.
template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&u)[NC]) {
  if constexpr (NC % 32 == 0) {
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) tmem_ld_x32(taddr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) reg_fence32(&u[c * 32]);
  } else {
    static_assert(NC == 16, "16 or a multiple of 32 columns");
    tmem_ld_x16(taddr, u);
    tmem_wait_ld();
    reg_fence16(u);
  }
}

// Multiply NC TMEM columns of this lane by a (read, scale, write back; the caller
// waits for the stores).
template <int NC>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, float a) {
  constexpr int W = NC % 32 == 0 ? 32 : 16;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    uint32_t u[W];
    tmem_load_cols<W>(taddr + c * W, u);
#pragma unroll
    for (int i = 0; i < W; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * a);
    if constexpr (W == 32) tmem_st_x32(taddr + c * W, u); else tmem_st_x16(taddr + c * W, u);
  }
}

// Store 16 or 32 output values of a row to global memory: FP32 or 16-bit (RNE).
template <int NV, bool BF16>
__device__ __forceinline__ void store_row_chunk(void* dst, const float (&y)[NV], bool f32) {
  if (f32) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) d[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < NV / 8; ++i) {
      uint4 w;
      w.x = pack2<BF16>(y[8 * i + 0], y[8 * i + 1]);
      w.y = pack2<BF16>(y[8 * i + 2], y[8 * i + 3]);
      w.z = pack2<BF16>(y[8 * i + 4], y[8 * i + 5]);
      w.w = pack2<BF16>(y[8 * i + 6], y[8 * i + 7]);
      d[i] = w;
    }
  }
}

// Byte offset of 16-byte unit u of row r inside one swizzled row chunk (rows of SW
// bytes): the XOR of address bits [4, 4+log2(SW/16)) with bits [7, ...), the pattern
// the TMA copies and the MMA descriptors use (chunk bases are 1024-byte aligned).
template <int SW>
__device__ __forceinline__ uint32_t swizzled(uint32_t r, uint32_t u) {
  const uint32_t off = r * SW + u * 16;
  return off ^ (((off >> 7) & (SW / 16 - 1)) << 4);
}

// Wait (once) for ring entry n (K_j at n = 2j, V_j at n = 2j+1); `ready` remembers the
// highest entry already waited for.
template <int NSLOT>
__device__ __forceinline__ bool wait_kv(uint64_t* full, int n, int& ready, volatile int* abort,
                                        unsigned int* status) {
  if (n <= ready) return true;
  if (!mbar_wait(&full[n % NSLOT], (uint32_t)(n / NSLOT) & 1u, abort, status, kErrWaitFull)) return false;
  ready = n;
  return true;
}

// Shared-memory descriptors are split into a 32-bit low word (start address >> 4 and
// leading byte offset >> 4) and a high word (stride byte offset >> 4, the fixed 0b001 and
// the swizzle mode) that is the same for every operand here.  Consecutive K steps only
// move the start address, so each MMA costs one 32-bit add on a precomputed low word:
// the issuer must keep up with 64-cycle MMAs.
template <class C>
__device__ __forceinline__ uint32_t desc_hi() {
  return (uint32_t)(((8 * C::SW) >> 4) & 0x3FFF) | (1u << 14) | (C::SWZ << 29);
}
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t desc64(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}

// S_t = Q_t K^T with K in ring entry `entry`: D/16 MMAs of K = 16 (32 bytes of each
// operand row), walking the swizzled row chunks.
template <class C, bool BF16>
__device__ __forceinline__ void issue_qk_e(uint32_t tmem, uint32_t q_addr, uint32_t kv_addr, int t, int entry,
                                           uint64_t* bar) {
  constexpr uint32_t IDESC = idesc_f16(128, C::BN_, BF16, false);
  constexpr int KPC = C::CH / 16;  // K steps per row chunk
  const uint32_t hi = desc_hi<C>();
  const uint32_t a0 = desc_lo(q_addr, 16);
  const uint32_t b0 = desc_lo(kv_addr + (entry % C::NSLOT) * C::KV_BYTES, 16);
  const uint32_t d = tmem + (t ? C::COL_S1 : C::COL_S0);
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < C::D_ / 16; ++kk) {
    const uint32_t off = (kk % KPC) * 32;
    const uint32_t c = kk / KPC;
    mma_ss_lo(d, a0 + ((c * C::BM * C::SW + off) >> 4), b0 + ((c * C::BN_ * C::SW + off) >> 4), hi, IDESC,
              kk > 0 ? 1u : 0u);
  }
  tc_commit(bar);
}
// K_j sits in ring entry 2j.
template <class C, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t q_addr, uint32_t kv_addr, int t, int j,
                                         uint64_t* bar) {
  issue_qk_e<C, BF16>(tmem, q_addr, kv_addr, t, 2 * j, bar);
}

// O_t (+)= P_t V with V in ring entry `entry`: BN/16 MMAs of K = 16 keys, P read from
// TMEM (8 packed columns per step), V read MN-major (16 key rows per step; the leading
// byte offset steps between the 64-column chunks of D).  `acc` = O already holds
// earlier tiles.
template <class C, bool BF16>
__device__ __forceinline__ void issue_pv_e(uint32_t tmem, uint32_t kv_addr, int t, int entry, bool acc) {
  constexpr uint32_t IDESC = idesc_f16(128, C::D_, BF16, true);
  const uint32_t hi = desc_hi<C>();
  const uint32_t b0 = desc_lo(kv_addr + (entry % C::NSLOT) * C::KV_BYTES, C::BN_ * C::SW);
  const uint32_t d = tmem + (t ? C::COL_O1 : C::COL_O0);
  const uint32_t p = tmem + (t ? C::COL_S1 : C::COL_S0);
  tc_fence_after();
#pragma unroll
  for (int kb = 0; kb < C::BN_ / 16; ++kb)
    mma_ts_lo(d, p + kb * 8, b0 + ((kb * 16 * C::SW) >> 4), hi, IDESC, (acc || kb > 0) ? 1u : 0u);
}
// V_j sits in ring entry 2j + 1.
template <class C, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t kv_addr, int t, int j) {
  issue_pv_e<C, BF16>(tmem, kv_addr, t, 2 * j + 1, j > 0);
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the bulk stores of this thread have read their shared-memory source (the
// global writes complete on their own before the kernel does).
__device__ __forceinline__ void bulk_wait_group_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// In-kernel split-K merge of one query row (rh = flat row-head index, RH row-heads per
// partition): G = log2 sum_p 2^lse_p over the partitions, found in one pass with a
// running maximum ("Streaming attention and online state", Online statistics, applied
// to the partition summaries), then O = sum_p 2^(lse_p - G) O_p in 32-column chunks
// ("fa4_splitk_combine").  Partitions with lse_p = -inf are skipped; a row with no
// visible key anywhere gets +0 and -inf.  The partials were written by other CTAs in
// this launch, so they are read through L2 (ld.global.cg), never a stale L1 line.
template <int D, bool BF16>
__device__ __forceinline__ void merge_row(const void* o_partial, const float* lse_partial, bool part_f32, int P,
                                          size_t RH, size_t rh, void* o_final, float* lse_final) {
  float m = -INFINITY, sum = 0.f;
  for (int p = 0; p < P; ++p) {
    const float l = __ldcg(lse_partial + (size_t)p * RH + rh);
    if (l == -INFINITY) continue;
    if (l > m) {
      sum = fmaf(sum, ex2(m - l), 1.f);  // ex2(-inf) = 0 on the first live partition
      m = l;
    } else {
      sum += ex2(l - m);
    }
  }
  const float G = (m == -INFINITY) ? -INFINITY : m + lg2(sum);
  constexpr int W = D < 32 ? D : 32;
#pragma unroll 1
  for (int c = 0; c < D / W; ++c) {
    float acc[W];
#pragma unroll
    for (int i = 0; i < W; ++i) acc[i] = 0.f;
    if (G != -INFINITY) {
      // Two partitions per step, their loads issued together (independent L2 reads).
#pragma unroll 1
      for (int p0 = 0; p0 < P; p0 += 2) {
        float x[2][W];
        float w[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int p = p0 + u;
          const float l = p < P ? __ldcg(lse_partial + (size_t)p * RH + rh) : -INFINITY;
          w[u] = ex2(l - G);  // 0 for an empty partition (or none)
          const size_t base = ((size_t)min(p, P - 1) * RH + rh) * D + (size_t)c * W;
          if (part_f32) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(o_partial) + base);
#pragma unroll
            for (int i = 0; i < W / 4; ++i) {
              const float4 v4 = __ldcg(src + i);
              x[u][4 * i] = v4.x;
              x[u][4 * i + 1] = v4.y;
              x[u][4 * i + 2] = v4.z;
              x[u][4 * i + 3] = v4.w;
            }
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(o_partial) + base);
#pragma unroll
            for (int i = 0; i < W / 8; ++i) {
              const uint4 v4 = __ldcg(src + i);
              const uint32_t xw[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                x[u][8 * i + 2 * j] = unpack_lo<BF16>(xw[j]);
                x[u][8 * i + 2 * j + 1] = unpack_hi<BF16>(xw[j]);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (w[u] != 0.f) {  // skip empty partitions: their data never enters the sum
#pragma unroll
            for (int i = 0; i < W; ++i) acc[i] = fmaf(w[u], x[u][i], acc[i]);
          }
      }
    }
#pragma unroll
    for (int i = 0; i < W; ++i) acc[i] += 0.f;
    store_row_chunk<W, BF16>(static_cast<uint16_t*>(o_final) + rh * D + (size_t)c * W, acc, false);
  }
  if (lse_final != nullptr) lse_final[rh] = G * kLn2;
}

// 16 bytes of the packed mask (read-only path; rows of a shared mask stay in L2).
// Key tiles marked in a bitmap (bit j of word j/32 = key tile j): how many of tiles
// [0, n) are marked, and the first marked tile at or after `from` (callers walk at most
// as many tiles as are marked; past the last word the walk returns the end index).
constexpr int kNeedWords = 64;  // key tiles a CTA can skip over: 64 * 32 = 2048
constexpr int kListWords = 256; // persistent masked kernel: summary words of one CTA's items
__device__ __forceinline__ int count_marked(const uint32_t* need, int n) {
  int c = 0;
  for (int w = 0; w * 32 < n; ++w) {
    uint32_t bits = need[w];
    if (n - w * 32 < 32) bits &= (1u << (n - w * 32)) - 1u;
    c += __popc(bits);
  }
  return c;
}
__device__ __forceinline__ int next_marked(const uint32_t* need, int from, int nwords = kNeedWords) {
  int w = from >> 5;
  if (w >= nwords) return nwords * 32;
  uint32_t bits = need[w] & (~0u << (from & 31));
  while (bits == 0u) {
    if (++w >= nwords) return nwords * 32;
    bits = need[w];
  }
  return w * 32 + __ffs(bits) - 1;
}

// One key tile of one query row (the calling thread's TMEM lane): read S, hide the keys
// the optional mask hides (MASK; `w` = this row's 16 mask bytes for the tile), the keys
// at or past kv_hi and, when causal, after the query; then p = 2^(s*scale*log2e - m),
// the FP32 row sum into l, and P rounded to the input dtype written back over S.
//
// The stabiliser m only has to keep every p = 2^(x - m) finite and within the 16-bit P
// operand's range; it need not be the row maximum.  So the common path takes no row
// maximum: it computes p against the current m in registers and accepts the tile when
// every row sum of p in the warp is at most kPBound (p <= row sum).  Otherwise, and
// while some row of the warp has seen no key, the tile is done against the exact
// maximum: the scores are read again from TMEM (P is only stored once the tile is
// accepted, so S is still there), O and l are rescaled by alpha = 2^(m - m')
// (`rescale_ok`: O holds earlier tiles) and p is computed again.  Exact arithmetic is
// unchanged.  Not keeping the raw scores for that rare second pass leaves the
// registers free for the scale, exponential, sum and packing stages of all columns to
// overlap.
template <class C, bool MASK>
__device__ __forceinline__ void load_scores(uint32_t taddr, int key0, int row, int row0, int kv_hi, int causal,
                                            uint4 w, float (&s)[C::BN_]) {
  constexpr int BN = C::BN_;
  uint32_t u[BN];
  tmem_load_cols<BN>(taddr, u);
#pragma unroll
  for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(u[c]);
  if constexpr (MASK) {
    const bool whole = (w.x & w.y & w.z & w.w) == ~0u;
    if (!__all_sync(0xffffffffu, whole)) {  // a warp whose rows see the whole tile skips this
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int c = 0; c < BN; ++c) s[c] = ((ww[c >> 5] >> (c & 31)) & 1u) ? s[c] : -INFINITY;
    }
  }
  if ((key0 + BN > kv_hi) || (causal && key0 + BN - 1 > row0)) {
    // key key0 + c is used when it is below kv_hi and, causal, at most the query row
    const int lim = (causal ? min(kv_hi, row + 1) : kv_hi) - key0;
#pragma unroll
    for (int c = 0; c < BN; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
  }
}

// p = 2^(s*scale_log2 + nbase) for a whole tile, in place: the scale-and-shift on pairs
// (f32x2 FMA), the exponentials on the MUFU, the FP32 row sum on pairs (f32x2 add, four
// chains) and the 16-bit packing (RNE) into pk.  All columns are independent, so the
// stages of different columns overlap.
template <int BN, bool BF16>
__device__ __forceinline__ float exp_pack(float (&s)[BN], float scale_log2, float nbase, uint32_t (&pk)[BN / 2]) {
#pragma unroll
  for (int i = 0; i < BN / 2; ++i)
    ffma2(s[2 * i], s[2 * i + 1], s[2 * i], s[2 * i + 1], scale_log2, scale_log2, nbase, nbase);
#pragma unroll
  for (int i = 0; i < BN; ++i) s[i] = ex2(s[i]);
  float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < BN / 2; ++i) {
    fadd2(sum8[2 * (i & 3)], sum8[2 * (i & 3) + 1], s[2 * i], s[2 * i + 1]);
    pk[i] = pack2<BF16>(s[2 * i], s[2 * i + 1]);
  }
  return ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
}

template <int BN>
__device__ __forceinline__ void store_p(uint32_t taddr, const uint32_t (&pk)[BN / 2]) {
  if constexpr (BN / 2 >= 32) {
#pragma unroll
    for (int c = 0; c < BN / 64; ++c)
      tmem_st_x32(taddr + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
  } else {
    tmem_st_x16(taddr, pk);
  }
  tmem_wait_st();
}


template <class C, bool BF16, bool MASK>
__device__ __forceinline__ void softmax_tile(uint32_t trow, uint32_t col_s, uint32_t col_o, bool rescale_ok,
                                             int key0, int row, int row0, int kv_hi, int causal, float scale_log2,
                                             uint4 w, float& m, float& l) {
  constexpr int BN = C::BN_;
  static_assert((BN - 8) % 16 == 8, "the row maximum walks 8 columns, then pairs of 8");
  if (__all_sync(0xffffffffu, m != -INFINITY)) {
    float s[BN];
    uint32_t pk[BN / 2];
    load_scores<C, MASK>(trow + col_s, key0, row, row0, kv_hi, causal, w, s);
    const float rowsum = exp_pack<BN, BF16>(s, scale_log2, -m, pk);
    if (__all_sync(0xffffffffu, rowsum <= kPBound)) {  // NaN/inf fail the test
      store_p<BN>(trow + col_s, pk);
      l += rowsum;
      return;
    }
  }
  float s[BN];
  uint32_t pk[BN / 2];
  load_scores<C, MASK>(trow + col_s, key0, row, row0, kv_hi, causal, w, s);
  // row max: 8 independent chains of three-input max
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
  for (int c = 8; c + 16 <= BN; c += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[BN - 8 + i]);
  const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
  const float mnew = fmaxf(m, mx * scale_log2);
  const float alpha = (mnew == m) ? 1.f : ex2(m - mnew);  // ex2(-inf) = 0
  m = mnew;
  const float rowsum = exp_pack<BN, BF16>(s, scale_log2, (m == -INFINITY) ? 0.f : -m, pk);
  store_p<BN>(trow + col_s, pk);
  // O is rescaled last, when the scores and P no longer occupy registers (PV of this
  // tile starts only after the arrival that follows)
  if (rescale_ok && __any_sync(0xffffffffu, alpha != 1.f)) {
    tmem_scale_cols<C::D_>(trow + col_o, alpha);
    tmem_wait_st();
  }
  l = l * alpha + rowsum;
}

__device__ __forceinline__ uint4 ld_mask16(const uint32_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// What one CTA owns: a head, a pair of 128-row query tiles and (split mode) a key
// partition, its key range and the key tiles each query tile needs before any mask
// skipping.  CTA index -> (head, pair, partition) in groups of kHeadGroup heads, pairs
// longest first when causal.
struct CtaPlan {
  int bh, pair, part, kv_lo, kv_hi, row0_0, row0_1, nkv0, nkv1;
};
template <int BM, int BN>
__device__ __forceinline__ CtaPlan cta_plan(long long idx, int BH, int N, int Nkv, int causal, int nparts, int chunk,
                                            bool split) {
  CtaPlan c;
  const int npairs = (N + 2 * BM - 1) / (2 * BM);
  c.part = (int)(idx % nparts);
  idx /= nparts;
  const int group = (int)(idx / ((long long)kHeadGroup * npairs));
  const int gheads = min(kHeadGroup, BH - group * kHeadGroup);
  const int within = (int)(idx - (long long)group * kHeadGroup * npairs);
  const int pair_rank = within / gheads;
  c.bh = group * kHeadGroup + within % gheads;
  c.pair = causal ? (npairs - 1 - pair_rank) : pair_rank;
  c.kv_lo = split ? min(c.part * chunk, Nkv) : 0;
  c.kv_hi = split ? min(c.kv_lo + chunk, Nkv) : Nkv;
  c.row0_0 = c.pair * 2 * BM;
  c.row0_1 = c.row0_0 + BM;
  // key tiles needed by the query tile starting at row0; 0 if the tile is empty
  auto tiles_for = [&](int row0) -> int {
    if (row0 >= N) return 0;
    const int last_row = min(row0 + BM - 1, N - 1);
    const int key_end = causal ? min(c.kv_hi, last_row + 1) : c.kv_hi;
    return key_end > c.kv_lo ? (key_end - c.kv_lo + BN - 1) / BN : 0;
  };
  c.nkv0 = tiles_for(c.row0_0);
  c.nkv1 = tiles_for(c.row0_1);
  return c;
}

// ptxas keeps every value that is live across a setmaxnreg in local memory.  So each
// role derives what it needs again after its setmaxnreg, from sources that are not
// registers: the thread and CTA indices (read afresh, so the compiler cannot reuse the
// earlier reads), the kernel parameters and shared memory.
__device__ __forceinline__ int tid_fresh() {
  int v;
  asm volatile("mov.u32 %0, %%tid.x;" : "=r"(v));
  return v;
}
__device__ __forceinline__ int ctaid_fresh() {
  int v;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(v));
  return v;
}
__device__ __forceinline__ uint32_t lds_fresh(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}

template <int D, int BN, bool BF16, bool MASK, bool SPLIT>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    void* __restrict__ out, float* __restrict__ lse_out, int BH, int N, int Nkv, int causal,
                    float scale_log2, int P, int chunk, int out_f32, const MaskArgs mk, const FusedMerge fm,
                    int ahead, unsigned int* status) {
  static_assert(!MASK || BN == 128, "the packed mask is read in 128-key tiles");
  // Programmatic dependent launch: the next kernel on the stream may be scheduled once
  // every CTA of this grid has started (its CTAs then take the SMs this grid's last
  // wave frees); it waits for this grid's completion before touching memory, as this
  // grid waits for the previous one below.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = AttnCfg<D, BN>;
  constexpr int BM = C::BM;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[NSLOT], bar_empty[NSLOT];
  __shared__ uint64_t bar_q, bar_s[2], bar_p[2], bar_o[2], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_last;
  __shared__ uint32_t s_need[MASK ? kNeedWords : 1];  // masked instances: key tiles to visit

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  uint8_t* sKV = smem + 2 * C::Q_BYTES;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- which query tiles, head and key range this CTA owns
  constexpr bool split = SPLIT;  // split-K partitions (P > 0) or the plain forward
  const int nparts = split ? P : 1;
  const CtaPlan pl = cta_plan<BM, BN>(blockIdx.x, BH, N, Nkv, causal, nparts, chunk, split);
  const int bh = pl.bh, kv_lo = pl.kv_lo;
  const int row0_0 = pl.row0_0, row0_1 = pl.row0_1;
  const int nkv0_all = pl.nkv0, nkv1_all = pl.nkv1;
  const int nkv_all = max(nkv0_all, nkv1_all);  // key tiles in range, before any skipping
  // With the optional mask, key tiles that no row of this CTA sees are skipped by every
  // role.  They are only known after the set-up, so only the first key tile (always
  // visited) is loaded before it; its copy overlaps the scan of the mask.
  const bool skip = MASK && nkv_all <= 32 * kNeedWords;

  // ---- set-up: barriers, TMEM
  if (warp == 9) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  // The copy thread sets up the barriers and starts the copies of Q and of the first ring
  // of K/V tiles before the CTA-wide barrier, so they overlap the TMEM allocation.
  const int first = min(skip ? 2 : NSLOT, 2 * nkv_all);  // K/V loads issued before the CTA barrier
  if (warp == 8 && lane == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_q, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 129);  // 128 softmax threads + the K/V watcher
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(&bar_done, 1);
    if constexpr (MASK) {
      for (int i = 0; i < kNeedWords; ++i) s_need[i] = 0u;
      if (skip && nkv_all > 0) s_need[0] = 1u;  // key tile 0: loaded before the scan
    }
    s_abort = 0;
    fence_mbar_init();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // previous grid done and visible
    if (nkv_all > 0) {
      mbar_arrive_expect_tx(&bar_q, (nkv0_all > 0 ? C::Q_BYTES : 0) + (nkv1_all > 0 ? C::Q_BYTES : 0));
      for (int t = 0; t < 2; ++t)
        if ((t ? nkv1_all : nkv0_all) > 0)
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(smem + t * C::Q_BYTES + c * BM * C::SW, &tm_q, &bar_q, c * C::CH, t ? row0_1 : row0_0, bh);
      for (int n = 0; n < first; ++n) {  // the ring starts empty: no wait
        mbar_arrive_expect_tx(&bar_full[n], C::KV_BYTES);
        const CUtensorMap* map = (n & 1) ? &tm_v : &tm_k;
        uint8_t* dst = sKV + n * C::KV_BYTES;
        for (int c = 0; c < C::NCH; ++c) tma_load_3d(dst + c * BN * C::SW, map, &bar_full[n], c * C::CH, kv_lo + (n >> 1) * BN, bh);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // before any global access
  volatile int* abort = &s_abort;

  // Masked instances: the softmax warps mark every key tile that some row of theirs
  // sees (lane = key tile, one coalesced 512-byte load per row and 32 tiles, 8 rows at a
  // time until the lane has seen a visible key; the key tiles a causal query tile cannot
  // reach are not looked at), then every role counts and walks the
  // marked tiles only (tile 0 is always marked: it is already on its way).  A skipped
  // tile has no visible key for any row of the CTA, so leaving it out changes no result.
  if constexpr (MASK) {
    if (skip) {
      if (warp < 8) {
        const int tt = warp >> 2;
        const int rbase = (tt ? row0_1 : row0_0) + (warp & 3) * 32;
        const int n_t = tt ? nkv1_all : nkv0_all;
        const int b = bh / mk.H, h = bh - b * mk.H;
        const uint32_t* base = mk.bits + b * mk.sb + h * mk.sh + (kv_lo >> 5);
        for (int g = 0; g * 32 < n_t; ++g) {
          const int j = g * 32 + lane;
          uint32_t acc = 0u;
          // The first 8 rows, then the other 24 only for lanes that have not yet seen a
          // visible key: a tile that is needed usually shows it at once, and only tiles
          // that end up skipped are read for all 32 rows (in two rounds).
          auto scan_rows = [&](auto nrows_c, int r0) {
            constexpr int NR = decltype(nrows_c)::value;
            uint4 w[NR];
#pragma unroll
            for (int i = 0; i < NR; ++i) {
              const int row = rbase + r0 + i;
              w[i] = row < N ? ld_mask16(base + (long long)row * mk.sq + 4 * j) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < NR; ++i) acc |= w[i].x | w[i].y | w[i].z | w[i].w;
          };
          if (j < n_t) scan_rows(std::integral_constant<int, 8>{}, 0);
          if (__any_sync(0xffffffffu, j < n_t && acc == 0u) && j < n_t && acc == 0u)
            scan_rows(std::integral_constant<int, 24>{}, 8);
          const uint32_t marks = __ballot_sync(0xffffffffu, acc != 0u);
          if (lane == 0 && marks != 0u) atomicOr(&s_need[g], marks);
        }
      }
      __syncthreads();
    }
  }

  // Registers move from the copy/MMA warpgroup to the softmax warpgroups.  Each
  // setmaxnreg sits at the top of its role's branch so that the register allocator
  // sees the new limit for all of that role's code.
  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_OTHER) : "memory");
    // Everything the role uses, derived again after setmaxnreg (see tid_fresh).
    const int tid = tid_fresh();
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const CtaPlan pl = cta_plan<BM, BN>(ctaid_fresh(), BH, N, Nkv, causal, nparts, chunk, split);
    const int bh = pl.bh, pair = pl.pair, part = pl.part, kv_lo = pl.kv_lo, kv_hi = pl.kv_hi;
    const int row0_0 = pl.row0_0, row0_1 = pl.row0_1;
    const int nkv_all = max(pl.nkv0, pl.nkv1);
    const bool skip = MASK && nkv_all <= 32 * kNeedWords;
    const int first = min(skip ? 2 : NSLOT, 2 * nkv_all);
    const int nkv0 = (MASK && skip) ? count_marked(s_need, pl.nkv0) : pl.nkv0;
    const int nkv1 = (MASK && skip) ? count_marked(s_need, pl.nkv1) : pl.nkv1;
    const int nkv_max = max(nkv0, nkv1);
    const uint32_t tmem = lds_fresh(&s_tmem);
    (void)pair; (void)part; (void)kv_hi; (void)row0_0; (void)row0_1; (void)first; (void)lane;

    if (warp == 8 && lane == 0 && nkv_all > 0) {
      // ============================================================== TMA producer
      // Warm L2 with the Q tiles of the CTA `ahead` launches later (one wave on), which
      // is about when this SM or another picks it up: its first loads then hit L2.
      if (ahead > 0 && (long long)ctaid_fresh() + ahead < (long long)gridDim.x) {
        const CtaPlan ahead_pl = cta_plan<BM, BN>((long long)ctaid_fresh() + ahead, BH, N, Nkv, causal, nparts, chunk,
                                                  split);
        for (int t = 0; t < 2; ++t)
          if (ahead_pl.row0_0 + t * BM < N)
            for (int c = 0; c < C::NCH; ++c) tma_prefetch_3d(&tm_q, c * C::CH, ahead_pl.row0_0 + t * BM, ahead_pl.bh);
      }
      int issued = first;
      int ktile = first > 0 ? 0 : -1;  // masked instances: the marked key tile of K/V load n
      for (int n = first; n < 2 * nkv_max; ++n) {
        const int slot = n % NSLOT;
        const uint32_t use = n / NSLOT;
        if (!mbar_wait(&bar_empty[slot], (use & 1u) ^ 1u, abort, status, kErrWaitLoad)) break;
        mbar_arrive_expect_tx(&bar_full[slot], C::KV_BYTES);
        const CUtensorMap* map = (n & 1) ? &tm_v : &tm_k;
        int tile_n = n >> 1;
        if constexpr (MASK) {
          if (skip) {
            if ((n & 1) == 0) ktile = next_marked(s_need, ktile + 1);
            tile_n = ktile;
          }
        }
        const int key0 = kv_lo + tile_n * BN;
        uint8_t* dst = sKV + slot * C::KV_BYTES;
        for (int c = 0; c < C::NCH; ++c) tma_load_3d(dst + c * BN * C::SW, map, &bar_full[slot], c * C::CH, key0, bh);
        issued = n + 1;
      }
      // Drain the copies still in flight before the CTA may exit.
      mbar_drain(&bar_q, 0, status);
      for (int n = max(0, issued - NSLOT); n < issued; ++n)
        mbar_drain(&bar_full[n % NSLOT], (uint32_t)(n / NSLOT) & 1u, status);
    } else if (warp == 9 && nkv_max > 0) {
      // ============================================================== MMA issuer
      // Every lane walks the loop and waits; the elected lane issues MMAs and commits.
      const bool leader = elect_one_lane();
      const uint32_t q_addr0 = smem_u32(smem), q_addr1 = q_addr0 + C::Q_BYTES;
      const uint32_t kv_addr = smem_u32(sKV);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_q, 0, abort, status, kErrWaitFull));
      int k_ready = -1;
      if (ok && nkv0 > 0) {
        ok = __all_sync(0xffffffffu, wait_kv<NSLOT>(bar_full, 0, k_ready, abort, status));
        if (ok && leader) issue_qk<C, BF16>(tmem, q_addr0, kv_addr, 0, 0, &bar_s[0]);
      }
      if (ok && nkv1 > 0) {
        ok = __all_sync(0xffffffffu, wait_kv<NSLOT>(bar_full, 0, k_ready, abort, status));
        if (ok && leader) issue_qk<C, BF16>(tmem, q_addr1, kv_addr, 1, 0, &bar_s[1]);
      }
      if (ok && leader) tc_commit(&bar_empty[0]);  // K_0 is free once both S(0) are done
      __syncwarp();
      for (int j = 0; ok && j < nkv_max; ++j) {
        for (int t = 0; t < 2; ++t) {
          const int nkv_t = t ? nkv1 : nkv0;
          if (j >= nkv_t) continue;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_p[t], (uint32_t)j & 1u, abort, status, kErrWaitP));
          if (!ok) break;
          if (leader) {
            issue_pv<C, BF16>(tmem, kv_addr, t, j);
            if (j == nkv_t - 1) tc_commit(&bar_o[t]);
            if (j + 1 < nkv_t) issue_qk<C, BF16>(tmem, t ? q_addr1 : q_addr0, kv_addr, t, j + 1, &bar_s[t]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) {
          tc_commit(&bar_empty[(2 * j + 1) % NSLOT]);                      // V_j consumed
          if (j + 1 < nkv_max) tc_commit(&bar_empty[(2 * j + 2) % NSLOT]);  // K_{j+1} consumed
        }
        __syncwarp();
      }
      // Drain every MMA this warp issued before TMEM is released.
      if (leader) {
        tc_commit(&bar_done);
        mbar_drain(&bar_done, 0, status);
      }
      __syncwarp();
    } else if (warp == 10 && lane == 0 && nkv_max > 0) {
      // ============================================================== K/V watcher
      // Waits for the copies of V_j and K_(j+1) and adds one arrival to bar_p[t], so
      // that the MMA issuer needs a single wait (P_t(j) written and its operands
      // loaded) before PV_t(j) and S_t(j+1): the issuer is on the critical path.
      bool ok = true;
      for (int j = 0; ok && j < nkv_max; ++j)
        for (int t = 0; ok && t < 2; ++t) {
          const int nkv_t = t ? nkv1 : nkv0;
          if (j >= nkv_t) continue;
          // never arrive for phase j before phase j - 1 of bar_p[t] has completed
          if (j > 0) ok = mbar_wait(&bar_p[t], (uint32_t)(j - 1) & 1u, abort, status, kErrWaitP);
          const int nv = 2 * j + 1;
          if (ok) ok = mbar_wait(&bar_full[nv % NSLOT], (uint32_t)(nv / NSLOT) & 1u, abort, status, kErrWaitFull);
          if (ok && j + 1 < nkv_t) {
            const int nk = 2 * (j + 1);
            ok = mbar_wait(&bar_full[nk % NSLOT], (uint32_t)(nk / NSLOT) & 1u, abort, status, kErrWaitFull);
          }
          if (ok) mbar_arrive(&bar_p[t]);
        }
    }
    // warp 11 and the other lanes: nothing to do (they donate registers)
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_SOFTMAX) : "memory");
    // Everything the role uses, derived again after setmaxnreg (see tid_fresh).
    const int tid = tid_fresh();
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const CtaPlan pl = cta_plan<BM, BN>(ctaid_fresh(), BH, N, Nkv, causal, nparts, chunk, split);
    const int bh = pl.bh, pair = pl.pair, part = pl.part, kv_lo = pl.kv_lo, kv_hi = pl.kv_hi;
    const int row0_0 = pl.row0_0, row0_1 = pl.row0_1;
    const int nkv_all = max(pl.nkv0, pl.nkv1);
    const bool skip = MASK && nkv_all <= 32 * kNeedWords;
    const int first = min(skip ? 2 : NSLOT, 2 * nkv_all);
    const int nkv0 = (MASK && skip) ? count_marked(s_need, pl.nkv0) : pl.nkv0;
    const int nkv1 = (MASK && skip) ? count_marked(s_need, pl.nkv1) : pl.nkv1;
    const int nkv_max = max(nkv0, nkv1);
    const uint32_t tmem = lds_fresh(&s_tmem);
    (void)pair; (void)part; (void)kv_hi; (void)row0_0; (void)row0_1; (void)first; (void)lane;

    // ================================================================ softmax warpgroups
    const int t = warp >> 2;    // query tile of this warpgroup
    const int quad = warp & 3;  // TMEM lane quadrant = rows 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;
    const int row0 = t ? row0_1 : row0_0;
    const int nkv = t ? nkv1 : nkv0;
    const int row = row0 + r;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t col_s = t ? C::COL_S1 : C::COL_S0;
    const uint32_t col_o = t ? C::COL_O1 : C::COL_O0;
    float m = -INFINITY;  // running max in use, log2 units of scale*s
    float l = 0.f;
    bool ok = true;
    // This row's packed mask words from the partition's first key; tile j's 16 bytes
    // are loaded before the wait for S_t(j), so the load overlaps the wait.
    const uint32_t* mrow = nullptr;
    if constexpr (MASK) {
      if (row < N) {
        const int b = bh / mk.H, h = bh - b * mk.H;
        mrow = mk.bits + b * mk.sb + h * mk.sh + (long long)row * mk.sq + (kv_lo >> 5);
      }
    }

    if (row0 < N) {
      // key tile of the next iteration (masked instances skip unmarked tiles) and, masked,
      // this row's mask words for it: fetched one iteration ahead to hide the load
      int tn = (MASK && skip) ? next_marked(s_need, 0) : 0;
      uint4 wn = make_uint4(~0u, ~0u, ~0u, ~0u);
      if constexpr (MASK) {
        if (mrow != nullptr && nkv > 0) wn = ld_mask16(mrow + 4 * tn);
      }
      for (int j = 0; j < nkv; ++j) {
        const int tj = tn;
        const uint4 w = wn;
        if (j + 1 < nkv) {
          tn = (MASK && skip) ? next_marked(s_need, tn + 1) : j + 1;
          if constexpr (MASK) {
            if (mrow != nullptr) wn = ld_mask16(mrow + 4 * tn);
          }
        }
        ok = mbar_wait(&bar_s[t], (uint32_t)j & 1u, abort, status, kErrWaitS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        softmax_tile<C, BF16, MASK>(trow, col_s, col_o, j > 0, kv_lo + tj * BN, row, row0, kv_hi, causal, scale_log2, w,
                                    m, l);
        tc_fence_before();
        mbar_arrive(&bar_p[t]);
      }

      // ---- epilogue: o / l and the log-sum-exp of the row
      if (ok && nkv > 0) {
        ok = mbar_wait(&bar_o[t], 0, abort, status, kErrWaitO);
        ok = __all_sync(0xffffffffu, ok);
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      constexpr int W = D % 32 == 0 ? 32 : 16;
      if (ok && nkv > 0) tc_fence_after();
      if constexpr (!split) {
        // o / l -> 16-bit -> this tile's Q buffer (free now: the last S_t finished before
        // the last PV_t) in the output map's swizzled layout -> TMA store.  Every warp of
        // the warpgroup reaches the barrier, aborted or not; the store is skipped when
        // the CTA aborted.
        uint8_t* tile = smem + t * C::Q_BYTES;
        if (ok) {
#pragma unroll
          for (int c = 0; c < D / W; ++c) {
            uint32_t u[W];
            if (!MASK || nkv > 0) {
              tmem_load_cols<W>(trow + col_o + c * W, u);
            } else {  // every key tile of this query tile was skipped: o = +0
#pragma unroll
              for (int i = 0; i < W; ++i) u[i] = 0u;
            }
            uint32_t w[W / 2];
#pragma unroll
            for (int i = 0; i < W / 2; ++i)
              w[i] = pack2<BF16>(__uint_as_float(u[2 * i]) * inv + 0.f, __uint_as_float(u[2 * i + 1]) * inv + 0.f);
#pragma unroll
            for (int v16 = 0; v16 < W / 8; ++v16) {
              const int col = c * W + v16 * 8;  // first element of this 16-byte unit
              const int ch = col / C::CH;
              const int unit = (col % C::CH) / 8;
              *reinterpret_cast<uint4*>(tile + ch * BM * C::SW + swizzled<C::SW>(r, unit)) =
                  make_uint4(w[4 * v16], w[4 * v16 + 1], w[4 * v16 + 2], w[4 * v16 + 3]);
            }
          }
          fence_proxy_async_smem();
        }
        named_bar_sync(1 + t, 128);
        if (r == 0 && *abort == 0) {
          for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_o, tile + c * BM * C::SW, c * C::CH, row0, bh);
          bulk_commit_group();
          bulk_wait_group_read_0();
        }
        if (ok && row < N && lse_out != nullptr) {
          const float lse2 = (l > 0.f) ? m + lg2(l) : -INFINITY;
          lse_out[(size_t)bh * N + row] = lse2 * kLn2;
        }
      } else if (ok) {
        {
          const bool f32 = out_f32 != 0;
          const size_t grow_idx = (size_t)part * BH * N + (size_t)bh * N + row;
          const size_t esz = f32 ? 4 : 2;
          uint8_t* dst = static_cast<uint8_t*>(out) + grow_idx * D * esz;
#pragma unroll
          for (int c = 0; c < D / W; ++c) {
            float y[W];
            if (nkv > 0) {
              uint32_t u[W];
              tmem_load_cols<W>(trow + col_o + c * W, u);
#pragma unroll
              for (int i = 0; i < W; ++i) y[i] = __uint_as_float(u[i]) * inv + 0.f;
            } else {
#pragma unroll
              for (int i = 0; i < W; ++i) y[i] = 0.f;
            }
            if (row < N) store_row_chunk<W, BF16>(dst + (size_t)c * W * esz, y, f32);
          }
          if (row < N && lse_out != nullptr) lse_out[grow_idx] = (l > 0.f) ? m + lg2(l) : -INFINITY;
        }
      }
    }
    if (split && fm.counters != nullptr) {  // (compiled into the split instances only)
      // In-kernel merge: the CTA that finishes last among the P partitions of this
      // (head, tile pair) merges its 256 rows.  Both softmax warpgroups take part (an
      // empty second tile included) so that the barriers always complete.
      // Publication: barrier, then one release fence and the counter update by thread 0;
      // the last CTA's thread 0 fences again (acquire) before the barrier that releases
      // the merge.
      named_bar_sync(3, 256);
      const long long g = (long long)bh * ((N + 2 * BM - 1) / (2 * BM)) + pair;
      if (tid == 0) {
        fence_acq_rel_gpu();
        s_last = atomicAdd(fm.counters + g, 1u) == (unsigned)(P - 1);
        if (s_last) {
          fence_acq_rel_gpu();
          fm.counters[g] = 0u;  // ready for the next call
        }
      }
      named_bar_sync(3, 256);
      if (s_last) {
        if (row < N)
          merge_row<D, BF16>(out, lse_out, out_f32 != 0, P, (size_t)BH * N, (size_t)bh * N + row, fm.o, fm.lse);
      }
    }
  }

  // ---- tear-down: everyone is done with TMEM before it is released
  tc_fence_before();
  __syncthreads();
  if ((tid_fresh() >> 5) == 9) {
    tc_fence_after();
    tmem_dealloc(lds_fresh(&s_tmem), C::TMEM_COLS);
  }
}

// ============================================================================
// Persistent plain forward (no mask, no split, key tiles of 128).
//
// The same warp roles and per-tile code as attn_fwd_kernel, but one CTA per SM walks a
// list of work items instead of one CTA per item, so the fixed cost of a CTA (set-up,
// TMEM allocation, the ramp to the first score tile, the tail after the last one and the
// hand-over of the SM to the next CTA) is paid once per SM: the K/V ring and every
// barrier's phase run on from one item to the next, the next item's Q tiles are loaded
// as soon as the current item's last S MMAs have read Q, and its first S MMAs follow
// the current item's last PV MMAs without a gap.
//
// Work units: a unit is one head's query-tile pair, or (causal) the two pairs p and
// npairs - 1 - p of one head, which together take 2 npairs + 2 key-tile iterations
// whatever p is (N a multiple of 256), so that every unit holds the same work; CTA b takes units b, b + G,
// b + 2G, ... (G = CTAs) in groups of kHeadGroup heads, so the heads in flight keep
// their K/V in L2.  O leaves through one 32 KB staging tile that the two query tiles
// use in turn (tile 0 then tile 1 of every item, an empty tile passing its turn).
struct WorkItem {
  int bh, row0_0, row0_1, nkv0, nkv1;
};
// Item s (0 or 1) of unit u; false when the unit has no such item.
template <int BM, int BN>
__device__ __forceinline__ bool unit_item(int u, int s, int BH, int N, int causal, int npairs, int upH,
                                          WorkItem& it) {
  const int group = u / (kHeadGroup * upH);
  const int gheads = min(kHeadGroup, BH - group * kHeadGroup);
  const int within = u - group * kHeadGroup * upH;
  const int rank = within / gheads;
  int pair;
  if (causal) {
    const int far = npairs - 1 - rank;  // the longer pair first
    if (s == 0) pair = far;
    else if (rank < far) pair = rank;
    else return false;
  } else {
    if (s > 0) return false;
    pair = rank;
  }
  it.bh = group * kHeadGroup + within % gheads;
  it.row0_0 = pair * 2 * BM;
  it.row0_1 = it.row0_0 + BM;
  auto tiles_for = [&](int row0) -> int {
    if (row0 >= N) return 0;
    const int last_row = min(row0 + BM - 1, N - 1);
    const int key_end = causal ? last_row + 1 : N;
    return (key_end + BN - 1) / BN;
  };
  it.nkv0 = tiles_for(it.row0_0);
  it.nkv1 = tiles_for(it.row0_1);
  return true;
}

// Item s of the i-th unit of this CTA: its summary words at list + (2 i + s) * wpb (zeros
// where the unit has no such item).  Not inlined, so that none of its values stays live
// into the roles (each role re-derives what it needs after setmaxnreg).
template <int BM, int BN>
__device__ __noinline__ void fill_item_list(uint32_t* list, int BH, int N, int causal, int H, const uint32_t* bits,
                                            long long sb, long long sh, int wpb) {
  const int npairs = (N + 2 * BM - 1) / (2 * BM);
  const int upH = causal ? (npairs + 1) / 2 : npairs;
  const int nunits = BH * upH;
  const int G = gridDim.x;
  const int nlist = min(2 * ((nunits - (int)blockIdx.x + G - 1) / G) * wpb, kListWords);
  for (int x = threadIdx.x; x < nlist; x += blockDim.x) {
    const int i = x / (2 * wpb), s2 = (x / wpb) & 1, w = x % wpb;
    WorkItem it;
    uint32_t v = 0u;
    if (unit_item<BM, BN>((int)blockIdx.x + i * G, s2, BH, N, causal, npairs, upH, it)) {
      const int b = it.bh / H, h = it.bh - b * H;
      v = bits[b * sb + h * sh + (long long)(it.row0_0 / (2 * BM)) * wpb + w];
    }
    list[x] = v;
  }
}

// Masked form (MASK): the block summary of the mask (one bit per block of 256 query rows
// and key tile) gives each item the key tiles it visits: marked tiles within its reach,
// counted and walked alike by every role.  A query tile whose tiles are all unmarked
// writes o = +0 and lse = -inf for its rows.
template <int D, bool BF16, bool MASK>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                            float* __restrict__ lse_out, int BH, int N, int causal, float scale_log2,
                            const MaskArgs mk, const MaskBlocks mb, unsigned int* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using C = AttnCfg<D, 128>;
  constexpr int BM = C::BM;
  constexpr int BN = 128;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[NSLOT], bar_empty[NSLOT];
  __shared__ uint64_t bar_q, bar_qfree, bar_s[2], bar_p[2], bar_o[2], bar_wr[2], bar_stg, bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint32_t s_list[MASK ? kListWords : 1];  // masked: summary words of this CTA's items

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  uint8_t* sKV = smem + 2 * C::Q_BYTES;
  uint8_t* stg = sKV + NSLOT * C::KV_BYTES;  // output staging tile (one query tile)

  if ((threadIdx.x >> 5) == 9) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qfree, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 129);  // 128 softmax threads + the K/V watcher
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_wr[t], 128);  // the 128 rows of tile t written to the staging tile
    }
    mbar_init(&bar_stg, 1);
    mbar_init(&bar_done, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // previous grid done and visible
  volatile int* abort = &s_abort;
  const int npairs = (N + 2 * BM - 1) / (2 * BM);
  const int upH = causal ? (npairs + 1) / 2 : npairs;  // units per head
  const int nunits = BH * upH;
  // Masked: item s of this CTA's i-th unit finds its summary words at s_list + (2 i + s)
  // * wpb (zeros where the unit has no such item); the launch keeps them within the list.
  if constexpr (MASK) {
    fill_item_list<BM, BN>(s_list, BH, N, causal, mk.H, mb.bits, mb.sb, mb.sh, mb.wpb);
    __syncthreads();
  }

  if ((threadIdx.x >> 5) >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_OTHER) : "memory");
    const int tid = tid_fresh();
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b0 = ctaid_fresh();
    const int G = gridDim.x;
    const uint32_t tmem = lds_fresh(&s_tmem);

    if (warp == 8 && lane == 0) {
      // ============================================================== TMA producer
      int n = 0;       // ring loads issued (K_j of an item in entry base + 2j, V_j in base + 2j + 1)
      int q_armed = 0; // Q phases started
      bool ok = true;
      int ui = 0;      // units begun
      for (int u = b0; ok && u < nunits; u += G, ++ui) {
        // warm L2 with the Q tiles of this CTA's next unit
        if (u + G < nunits)
          for (int s2 = 0; s2 < 2; ++s2) {
            WorkItem nx;
            if (!unit_item<BM, BN>(u + G, s2, BH, N, causal, npairs, upH, nx)) break;
            for (int t = 0; t < 2; ++t)
              if ((t ? nx.nkv1 : nx.nkv0) > 0)
                for (int c = 0; c < C::NCH; ++c) tma_prefetch_3d(&tm_q, c * C::CH, t ? nx.row0_1 : nx.row0_0, nx.bh);
          }
        for (int s2 = 0; ok && s2 < 2; ++s2) {
          WorkItem it;
          if (!unit_item<BM, BN>(u, s2, BH, N, causal, npairs, upH, it)) break;
          const uint32_t* list = s_list + (MASK ? (2 * ui + s2) * mb.wpb : 0);
          const int nkv0 = MASK ? count_marked(list, it.nkv0) : it.nkv0;
          const int nkv1 = MASK ? count_marked(list, it.nkv1) : it.nkv1;
          const int nkv_max = max(nkv0, nkv1);
          if (nkv_max == 0) continue;
          // Q_t of this item may overwrite the previous item's only once its S MMAs are done
          if (q_armed > 0) ok = mbar_wait(&bar_qfree, (uint32_t)(q_armed - 1) & 1u, abort, status, kErrWaitLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_q, (nkv0 > 0 ? C::Q_BYTES : 0) + (nkv1 > 0 ? C::Q_BYTES : 0));
          ++q_armed;
          for (int t = 0; t < 2; ++t)
            if ((t ? nkv1 : nkv0) > 0)
              for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(smem + t * C::Q_BYTES + c * BM * C::SW, &tm_q, &bar_q, c * C::CH, t ? it.row0_1 : it.row0_0,
                            it.bh);
          int ktile = -1;  // key tile of the K/V pair being loaded
          for (int m = 0; m < 2 * nkv_max; ++m, ++n) {
            const int slot = n % NSLOT;
            const uint32_t use = n / NSLOT;
            ok = mbar_wait(&bar_empty[slot], (use & 1u) ^ 1u, abort, status, kErrWaitLoad);
            if (!ok) break;
            mbar_arrive_expect_tx(&bar_full[slot], C::KV_BYTES);
            const CUtensorMap* map = (m & 1) ? &tm_v : &tm_k;
            if ((m & 1) == 0) ktile = MASK ? next_marked(list, ktile + 1, mb.wpb) : m >> 1;
            uint8_t* dst = sKV + slot * C::KV_BYTES;
            for (int c = 0; c < C::NCH; ++c) tma_load_3d(dst + c * BN * C::SW, map, &bar_full[slot], c * C::CH, ktile * BN, it.bh);
          }
        }
      }
      // Drain the copies still in flight before the CTA may exit.
      if (q_armed > 0) mbar_drain(&bar_q, (uint32_t)(q_armed - 1) & 1u, status);
      for (int e = max(0, n - NSLOT); e < n; ++e) mbar_drain(&bar_full[e % NSLOT], (uint32_t)(e / NSLOT) & 1u, status);
    } else if (warp == 9) {
      // ============================================================== MMA issuer
      // Every lane walks the loop and waits; the elected lane issues MMAs and commits.
      const bool leader = elect_one_lane();
      const uint32_t q_addr0 = smem_u32(smem), q_addr1 = q_addr0 + C::Q_BYTES;
      const uint32_t kv_addr = smem_u32(sKV);
      int nb = 0;               // ring entry of the current item's K_0
      int k = 0;                // items begun
      int cp0 = 0, cp1 = 0;     // phases of bar_p[0], bar_p[1] consumed
      bool ok = true;
      int ui = 0;               // units begun
      for (int u = b0; ok && u < nunits; u += G, ++ui) {
        for (int s2 = 0; ok && s2 < 2; ++s2) {
          WorkItem it;
          if (!unit_item<BM, BN>(u, s2, BH, N, causal, npairs, upH, it)) break;
          const uint32_t* list = s_list + (MASK ? (2 * ui + s2) * mb.wpb : 0);
          const int nkv0 = MASK ? count_marked(list, it.nkv0) : it.nkv0;
          const int nkv1 = MASK ? count_marked(list, it.nkv1) : it.nkv1;
          const int nkv_max = max(nkv0, nkv1);
          if (nkv_max == 0) continue;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_q, (uint32_t)k & 1u, abort, status, kErrWaitFull));
          if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_full[nb % NSLOT], (uint32_t)(nb / NSLOT) & 1u, abort, status,
                                                   kErrWaitFull));
          if (!ok) break;
          if (leader) {
            if (nkv0 > 0) issue_qk_e<C, BF16>(tmem, q_addr0, kv_addr, 0, nb, &bar_s[0]);
            if (nkv1 > 0) issue_qk_e<C, BF16>(tmem, q_addr1, kv_addr, 1, nb, &bar_s[1]);
            tc_commit(&bar_empty[nb % NSLOT]);  // K_0 is free once both S(0) are done
            if (nkv_max == 1) tc_commit(&bar_qfree);
          }
          __syncwarp();
          for (int j = 0; ok && j < nkv_max; ++j) {
            for (int t = 0; t < 2; ++t) {
              const int nkv_t = t ? nkv1 : nkv0;
              if (j >= nkv_t) continue;
              const int cp = t ? cp1++ : cp0++;
              ok = __all_sync(0xffffffffu, mbar_wait(&bar_p[t], (uint32_t)cp & 1u, abort, status, kErrWaitP));
              if (!ok) break;
              if (leader) {
                issue_pv_e<C, BF16>(tmem, kv_addr, t, nb + 2 * j + 1, j > 0);
                if (j == nkv_t - 1) tc_commit(&bar_o[t]);
                if (j + 1 < nkv_t) issue_qk_e<C, BF16>(tmem, t ? q_addr1 : q_addr0, kv_addr, t, nb + 2 * j + 2, &bar_s[t]);
              }
              __syncwarp();
            }
            if (!ok) break;
            if (leader) {
              tc_commit(&bar_empty[(nb + 2 * j + 1) % NSLOT]);                      // V_j consumed
              if (j + 1 < nkv_max) tc_commit(&bar_empty[(nb + 2 * j + 2) % NSLOT]);  // K_{j+1} consumed
              if (j + 2 == nkv_max) tc_commit(&bar_qfree);  // this item's last S MMAs are issued
            }
            __syncwarp();
          }
          nb += 2 * nkv_max;
          ++k;
        }
      }
      // Drain every MMA this warp issued before TMEM is released.
      if (leader) {
        tc_commit(&bar_done);
        mbar_drain(&bar_done, 0, status);
      }
      __syncwarp();
    } else if (warp == 10 && lane == 0) {
      // ============================================================== K/V watcher
      // One arrival on bar_p[t] per group once V_j and K_(j+1) have landed, never for a
      // phase before the previous phase of bar_p[t] completed (see attn_fwd_kernel).
      int nb = 0, cp0 = 0, cp1 = 0;
      bool ok = true;
      int ui = 0;  // units begun
      for (int u = b0; ok && u < nunits; u += G, ++ui) {
        for (int s2 = 0; ok && s2 < 2; ++s2) {
          WorkItem it;
          if (!unit_item<BM, BN>(u, s2, BH, N, causal, npairs, upH, it)) break;
          const uint32_t* list = s_list + (MASK ? (2 * ui + s2) * mb.wpb : 0);
          const int nkv0 = MASK ? count_marked(list, it.nkv0) : it.nkv0;
          const int nkv1 = MASK ? count_marked(list, it.nkv1) : it.nkv1;
          const int nkv_max = max(nkv0, nkv1);
          if (nkv_max == 0) continue;
          for (int j = 0; ok && j < nkv_max; ++j)
            for (int t = 0; ok && t < 2; ++t) {
              const int nkv_t = t ? nkv1 : nkv0;
              if (j >= nkv_t) continue;
              const int cp = t ? cp1++ : cp0++;
              if (cp > 0) ok = mbar_wait(&bar_p[t], (uint32_t)(cp - 1) & 1u, abort, status, kErrWaitP);
              const int ev = nb + 2 * j + 1;
              if (ok) ok = mbar_wait(&bar_full[ev % NSLOT], (uint32_t)(ev / NSLOT) & 1u, abort, status, kErrWaitFull);
              if (ok && j + 1 < nkv_t) {
                const int ek = nb + 2 * j + 2;
                ok = mbar_wait(&bar_full[ek % NSLOT], (uint32_t)(ek / NSLOT) & 1u, abort, status, kErrWaitFull);
              }
              if (ok) mbar_arrive(&bar_p[t]);
            }
          nb += 2 * nkv_max;
        }
      }
    }
    // warp 11 and the other lanes: nothing to do (they donate registers)
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_SOFTMAX) : "memory");
    // ================================================================ softmax warpgroups
    const int tid = tid_fresh();
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b0 = ctaid_fresh();
    const int G = gridDim.x;
    const int t = warp >> 2;    // query tile of this warpgroup
    const int quad = warp & 3;  // TMEM lane quadrant = rows 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;
    const uint32_t trow = lds_fresh(&s_tmem) + ((uint32_t)(quad * 32) << 16);
    const uint32_t col_s = t ? C::COL_S1 : C::COL_S0;
    const uint32_t col_o = t ? C::COL_O1 : C::COL_O0;
    const uint4 all_keys = make_uint4(~0u, ~0u, ~0u, ~0u);
    int cs = 0;  // phases of bar_s[t] consumed
    int co = 0;  // phases of bar_o[t] consumed
    int turn = 0;  // staging turns passed (two per item: tile 0, then tile 1)
    int cw = 0;    // phases of bar_wr[t] consumed
    bool ok = true;
    int ui = 0;  // units begun
    for (int u = b0; ok && u < nunits; u += G, ++ui) {
      for (int s2 = 0; ok && s2 < 2; ++s2) {
        WorkItem it;
        if (!unit_item<BM, BN>(u, s2, BH, N, causal, npairs, upH, it)) break;
        if (max(it.nkv0, it.nkv1) == 0) continue;
        const uint32_t* list = s_list + (MASK ? (2 * ui + s2) * mb.wpb : 0);
        const int reach = t ? it.nkv1 : it.nkv0;  // key tiles before any skipping (0: no rows)
        const int nkv = MASK ? count_marked(list, reach) : reach;
        const int row0 = t ? it.row0_1 : it.row0_0;
        const int row = row0 + r;
        // this row's packed mask words (rows past N see every key of the visited tiles)
        const uint32_t* mrow = nullptr;
        if (MASK && row < N) {
          const int b = it.bh / mk.H, h = it.bh - b * mk.H;
          mrow = mk.bits + b * mk.sb + h * mk.sh + (long long)row * mk.sq;
        }
        float m = -INFINITY;  // running max in use, log2 units of scale*s
        float l = 0.f;
        // Masked: the key tile of the next iteration and this row's mask words for it are
        // fetched one iteration ahead, so the load's latency hides behind a whole tile.
        int tn = MASK ? next_marked(list, 0, mb.wpb) : 0;
        uint4 wn = all_keys;
        if (MASK && mrow != nullptr && nkv > 0) wn = ld_mask16(mrow + 4 * tn);
        for (int j = 0; j < nkv; ++j) {
          const int tj = MASK ? tn : j;  // key tile of iteration j
          const uint4 w = wn;
          if (MASK && j + 1 < nkv) {
            tn = next_marked(list, tn + 1, mb.wpb);
            if (mrow != nullptr) wn = ld_mask16(mrow + 4 * tn);
          }
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[t], (uint32_t)cs & 1u, abort, status, kErrWaitS));
          ++cs;
          if (!ok) break;
          tc_fence_after();
          softmax_tile<C, BF16, MASK>(trow, col_s, col_o, j > 0, tj * BN, row, row0, N, causal, scale_log2, w, m, l);
          tc_fence_before();
          mbar_arrive(&bar_p[t]);
        }
        if (!ok) break;
        if (nkv > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_o[t], (uint32_t)co & 1u, abort, status, kErrWaitO));
          ++co;
        }
        // the staging tile is free once the previous turn's store has read it
        const int my_turn = turn + t;
        if (ok && my_turn > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_stg, (uint32_t)(my_turn - 1) & 1u, abort, status, kErrWaitO));
        if (!ok) break;
        if (reach > 0) {
          tc_fence_after();
          const float inv = (l > 0.f) ? 1.f / l : 0.f;
          constexpr int W = D % 32 == 0 ? 32 : 16;
#pragma unroll
          for (int c = 0; c < D / W; ++c) {
            uint32_t uo[W];
            if (!MASK || nkv > 0) {
              tmem_load_cols<W>(trow + col_o + c * W, uo);
            } else {  // every key tile of this query tile was skipped: o = +0
#pragma unroll
              for (int i = 0; i < W; ++i) uo[i] = 0u;
            }
            uint32_t w[W / 2];
#pragma unroll
            for (int i = 0; i < W / 2; ++i)
              w[i] = pack2<BF16>(__uint_as_float(uo[2 * i]) * inv + 0.f, __uint_as_float(uo[2 * i + 1]) * inv + 0.f);
#pragma unroll
            for (int v16 = 0; v16 < W / 8; ++v16) {
              const int col = c * W + v16 * 8;
              const int ch = col / C::CH;
              const int unit = (col % C::CH) / 8;
              *reinterpret_cast<uint4*>(stg + ch * BM * C::SW + swizzled<C::SW>(r, unit)) =
                  make_uint4(w[4 * v16], w[4 * v16 + 1], w[4 * v16 + 2], w[4 * v16 + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&bar_wr[t]);  // this row is in the staging tile
          if (r == 0) {
            // all 128 rows written (a bounded wait, unlike a named barrier): store the tile
            ok = mbar_wait(&bar_wr[t], (uint32_t)cw & 1u, abort, status, kErrWaitO);
            if (ok && *abort == 0) {
              for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_o, stg + c * BM * C::SW, c * C::CH, row0, it.bh);
              bulk_commit_group();
              bulk_wait_group_read_0();
            }
            mbar_arrive(&bar_stg);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);  // lane 0 of quadrant 0 decided for its warp
          ++cw;
          if (row < N && lse_out != nullptr) {
            const float lse2 = (l > 0.f) ? m + lg2(l) : -INFINITY;
            lse_out[(size_t)it.bh * N + row] = lse2 * kLn2;
          }
        } else if (r == 0) {
          mbar_arrive(&bar_stg);  // an empty tile passes its turn
        }
        turn += 2;
        if (!ok) break;
      }
    }
    // the stores issued by this warpgroup complete before the grid does
  }

  // ---- tear-down: everyone is done with TMEM before it is released
  tc_fence_before();
  __syncthreads();
  if ((tid_fresh() >> 5) == 9) {
    tc_fence_after();
    tmem_dealloc(lds_fresh(&s_tmem), C::TMEM_COLS);
  }
}

// Streaming multiprocessors of the current device (0 if it cannot be queried).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int D, int BN, bool BF16, bool MASK = false, bool SPLIT = false>
cudaError_t launch_attn_inst(const AttnArgs& a, cudaStream_t st) {
  using C = AttnCfg<D, BN>;
  auto kern = attn_fwd_kernel<D, BN, BF16, MASK, SPLIT>;
  // The shared-memory attribute belongs to the function on one device: it is set once
  // per device (one bit each; devices past 63 set it on every launch).
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || !(attr_set.load(std::memory_order_acquire) & bit)) {
    // The setmaxnreg split draws on the registers the CTA was launched with: refuse to
    // launch a build whose register count would make setmaxnreg.inc wait forever.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < C::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  const long long npairs = (a.N + 2 * C::BM - 1) / (2 * C::BM);
  const long long blocks = npairs * a.BH * (a.P > 0 ? a.P : 1);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // Launched as a programmatic dependent of the previous kernel on the stream.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.o, a.lse, a.BH, a.N, a.Nkv, a.causal,
                         a.scale_log2, a.P, a.chunk, a.out_f32, a.mask, a.fused, sm_count(), a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Grid of the persistent kernel: one CTA per SM, or one per unit when there are fewer.
inline long long persist_units(const AttnArgs& a) {
  const long long npairs = (a.N + 2 * 128LL - 1) / (2 * 128LL);
  return (a.causal ? (npairs + 1) / 2 : npairs) * a.BH;
}
inline int persist_grid(long long units) {
  const int sms = sm_count();
  return (int)(units < sms ? units : (sms > 0 ? sms : 1));
}
// The masked persistent form keeps the summary words of all of a CTA's items in shared
// memory: two item slots per unit of the CTA, mblocks.wpb words each.
inline bool persist_mask_fits(const AttnArgs& a) {
  const long long units = persist_units(a);
  if (units <= 0 || a.mblocks.bits == nullptr || a.mblocks.wpb <= 0) return false;
  const long long g = persist_grid(units);
  return 2 * ((units + g - 1) / g) * a.mblocks.wpb <= kListWords;
}

template <int D, bool BF16, bool MASK>
cudaError_t launch_persist(const AttnArgs& a, cudaStream_t st) {
  using C = AttnCfg<D, 128>;
  constexpr int SMEM = C::SMEM_BYTES + C::Q_BYTES;  // + the output staging tile
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  auto kern = attn_fwd_persist_kernel<D, BF16, MASK>;
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || !(attr_set.load(std::memory_order_acquire) & bit)) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < C::REGS_LAUNCH) return cudaErrorInvalidConfiguration;  // see launch_attn_inst
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  const long long units = persist_units(a);
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (MASK && !persist_mask_fits(a)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)persist_grid(units));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.lse, a.BH, a.N, a.causal, a.scale_log2,
                         a.mask, a.mblocks, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn_d(const AttnArgs& a, int block_n, int bf16, cudaStream_t st) {
  const bool mask = a.mask.bits != nullptr;
  // The plain forward with key tiles of 128 runs persistent (one CTA per SM walking the
  // work units), masked too when the mask's block summary is given and fits; the other
  // forms launch one CTA per query-tile pair.
  if (a.P == 0 && !mask && block_n == 128)
    return bf16 ? launch_persist<D, true, false>(a, st) : launch_persist<D, false, false>(a, st);
  if (a.P == 0 && mask && block_n == 128 && persist_mask_fits(a))
    return bf16 ? launch_persist<D, true, true>(a, st) : launch_persist<D, false, true>(a, st);
  if (a.P > 0) {  // split-K partitions: key tiles of 128
    if (block_n != 128) return cudaErrorInvalidValue;
    if (mask)
      return bf16 ? launch_attn_inst<D, 128, true, true, true>(a, st) : launch_attn_inst<D, 128, false, true, true>(a, st);
    return bf16 ? launch_attn_inst<D, 128, true, false, true>(a, st) : launch_attn_inst<D, 128, false, false, true>(a, st);
  }
  if (mask) {
    if (block_n != 128) return cudaErrorInvalidValue;
    return bf16 ? launch_attn_inst<D, 128, true, true>(a, st) : launch_attn_inst<D, 128, false, true>(a, st);
  }
  switch (block_n) {
    case 32: return bf16 ? launch_attn_inst<D, 32, true>(a, st) : launch_attn_inst<D, 32, false>(a, st);
    case 64: return bf16 ? launch_attn_inst<D, 64, true>(a, st) : launch_attn_inst<D, 64, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace oattn
