// C ABI entry points: argument checks, TMA descriptors, dispatch to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/oattn.h"
#include "internal.h"

namespace oattn {
namespace {

// Device status word: a bounded wait that gives up records its site code here.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::atomic<unsigned int*> g_status_ptr[kMaxDevices] = {};
std::mutex g_setup_mutex;

// Device address of the status word for the current device (looked up once per device).
unsigned int* status_ptr(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (g_status_ptr[dev] == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_status_ptr[dev] == nullptr) {
      void* p = nullptr;
      *err = cudaGetSymbolAddress(&p, g_status_word);
      if (*err != cudaSuccess) return nullptr;
      g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
  }
  return g_status_ptr[dev];
}

// Streams and events of the host-buffer entry point, created once per device (they are
// scheduling resources, not memory; kept until the process exits).
// A call holds `lock` while it enqueues, so that the record of an event and the waits on
// it are not interleaved with another host thread's call on the same device.
struct Pipe {
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, loaded = nullptr, done = nullptr, finished = nullptr;
  std::mutex lock;
};
Pipe g_pipe[kMaxDevices];

Pipe* pipe_for_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  Pipe& p = g_pipe[dev];
  if (p.finished == nullptr) {
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    if ((*err = cudaStreamCreateWithFlags(&p.in, sf)) != cudaSuccess ||
        (*err = cudaStreamCreateWithFlags(&p.comp, sf)) != cudaSuccess ||
        (*err = cudaStreamCreateWithFlags(&p.out, sf)) != cudaSuccess ||
        (*err = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess ||
        (*err = cudaEventCreateWithFlags(&p.loaded, ef)) != cudaSuccess ||
        (*err = cudaEventCreateWithFlags(&p.done, ef)) != cudaSuccess ||
        (*err = cudaEventCreateWithFlags(&p.finished, ef)) != cudaSuccess)
      return nullptr;
  }
  return &p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D tiled map over a [BH, rows, D] 16-bit tensor; box = (min(D,64) elements, box_rows, 1)
// with the swizzle whose span equals the box row (32, 64 or 128 bytes).  Rows past
// `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int BH, int rows, int D, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int ch = D >= 64 ? 64 : D;
  const CUtensorMapSwizzle swz = ch * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : ch * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_32B;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint32_t box[3] = {(cuuint32_t)ch, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool supported_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }
bool is16(oattn_dtype t) { return t == OATTN_F16 || t == OATTN_BF16; }
bool valid_dtype(oattn_dtype t) { return t == OATTN_F16 || t == OATTN_BF16 || t == OATTN_F32; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;

cudaError_t launch_attn(const AttnArgs& a, int block_n, bool bf16, cudaStream_t st) {
  switch (a.D) {
    case 16: return launch_attn_d16(a, block_n, bf16, st);
    case 32: return launch_attn_d32(a, block_n, bf16, st);
    case 64: return launch_attn_d64(a, block_n, bf16, st);
    case 128: return launch_attn_d128(a, block_n, bf16, st);
    default: return cudaErrorInvalidValue;
  }
}

// Size, dtype and scale checks first; pointer checks only when there is data to touch
// (an empty problem may come with null pointers, as empty tensors have).
oattn_status attn_common_checks(const void* q, const void* k, const void* v, int B, int H, int Nq,
                                int Nkv, int D, float scale, oattn_dtype dtype) {
  if (B < 1 || H < 1 || Nq < 0 || Nkv < 0 || D < 1) return OATTN_ERR_INVALID_ARG;
  if ((long long)B * H > 0x7fffffffLL) return OATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return OATTN_ERR_INVALID_ARG;
  if (!is16(dtype)) return OATTN_ERR_UNSUPPORTED;
  if (!supported_d(D)) return OATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return OATTN_OK;
  if (!q || (Nkv > 0 && (!k || !v))) return OATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return OATTN_ERR_INVALID_ARG;
  if (Nq > (1 << 24) || Nkv > (1 << 24)) return OATTN_ERR_UNSUPPORTED;
  return OATTN_OK;
}

// The packed mask: 16-byte aligned words, strides in words that keep every 128-key
// tile of a row on a 16-byte boundary.
oattn_status mask_checks(const unsigned int* bits, long long sb, long long sh, long long sq) {
  if (!bits || !aligned(bits, 16)) return OATTN_ERR_INVALID_ARG;
  if (sb < 0 || sh < 0 || sq < 0 || sb % 4 || sh % 4 || sq % 4) return OATTN_ERR_INVALID_ARG;
  return OATTN_OK;
}

MaskArgs mask_args(const unsigned int* bits, long long sb, long long sh, long long sq, int H) {
  MaskArgs m{};
  m.bits = reinterpret_cast<const uint32_t*>(bits);
  m.sb = sb;
  m.sh = sh;
  m.sq = sq;
  m.H = H;
  return m;
}

oattn_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                           int N, int D, int causal, float scale, oattn_dtype dtype, int block_n,
                           const MaskArgs& mk, cudaStream_t st, const MaskBlocks& mblocks = MaskBlocks{}) {
  oattn_status s = attn_common_checks(q, k, v, B, H, N, N, D, scale, dtype);
  if (s != OATTN_OK) return s;
  if (block_n == 0) block_n = 128;
  if (block_n != 32 && block_n != 64 && block_n != 128) return OATTN_ERR_INVALID_ARG;
  if (N == 0) return OATTN_OK;
  if (!o || !aligned(o, 16) || (lse && !aligned(lse, 4))) return OATTN_ERR_INVALID_ARG;
  cudaError_t e;
  AttnArgs a{};
  a.status = status_ptr(&e);
  if (!a.status) return OATTN_ERR_CUDA;
  const bool bf16 = dtype == OATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, bf16, BH, N, D, 128) || !make_map(&a.tm_k, k, bf16, BH, N, D, block_n) ||
      !make_map(&a.tm_v, v, bf16, BH, N, D, block_n) || !make_map(&a.tm_o, o, bf16, BH, N, D, 128))
    return OATTN_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.Nkv = N;
  a.D = D;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * kLog2e;
  a.P = 0;
  a.chunk = 0;
  a.out_f32 = 0;
  a.mask = mk;
  a.mblocks = mblocks;
  return launch_attn(a, block_n, bf16, st) == cudaSuccess ? OATTN_OK : OATTN_ERR_CUDA;
}

oattn_status attn_fwd_splitk_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                  int H, int Nq, int Nkv, int D, int causal, float scale, oattn_dtype dtype,
                                  int P, void* o_partial, float* lse_partial, oattn_dtype partial_dtype,
                                  const MaskArgs& mk, unsigned int* counters, cudaStream_t st) {
  oattn_status s = attn_common_checks(q, k, v, B, H, Nq, Nkv, D, scale, dtype);
  if (s != OATTN_OK) return s;
  if (causal && Nq != Nkv) return OATTN_ERR_INVALID_ARG;
  if (P < 1 || P > 256) return OATTN_ERR_INVALID_ARG;
  if (partial_dtype != OATTN_F32 && partial_dtype != dtype) return OATTN_ERR_INVALID_ARG;
  if (lse && !o) return OATTN_ERR_INVALID_ARG;
  if (o && !combine_supported(D, partial_dtype)) return OATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return OATTN_OK;
  if (!o_partial || !lse_partial) return OATTN_ERR_INVALID_ARG;
  if (!aligned(o_partial, 16) || !aligned(lse_partial, 4)) return OATTN_ERR_INVALID_ARG;
  if (o && (!aligned(o, 16) || (lse && !aligned(lse, 4)))) return OATTN_ERR_INVALID_ARG;
  if (counters && (!o || !aligned(counters, 4))) return OATTN_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* status = status_ptr(&e);
  if (!status) return OATTN_ERR_CUDA;
  const int BH = B * H;
  const int chunk = splitk_chunk(Nkv, P);
  const bool bf16 = dtype == OATTN_BF16;
  FusedMerge fm{};
  if (counters) {
    fm.counters = counters;
    fm.o = o;
    fm.lse = lse;
  }
  cudaError_t le;
  if (Nq == 1) {
    // One query row per head: matrix-vector work, streamed on CUDA cores.  (Causal with
    // Nq == Nkv == 1 sees its single key, the same as non-causal.)
    DecodeArgs d{};
    d.q = q; d.k = k; d.v = v;
    d.o_partial = o_partial;
    d.lse_partial = lse_partial;
    d.BH = BH; d.Nkv = Nkv; d.D = D; d.P = P; d.chunk = chunk;
    d.scale_log2 = scale * kLog2e;
    d.dtype = dtype;
    d.partial_dtype = partial_dtype;
    d.mask = mk;
    d.fused = fm;
    d.status = status;
    le = launch_decode(d, st);
  } else {
    AttnArgs a{};
    a.status = status;
    // With no keys the K/V maps are never read; q stands in as a valid base address.
    const void* kb = Nkv > 0 ? k : q;
    const void* vb = Nkv > 0 ? v : q;
    if (!make_map(&a.tm_q, q, bf16, BH, Nq, D, 128) || !make_map(&a.tm_k, kb, bf16, BH, Nkv, D, 128) ||
        !make_map(&a.tm_v, vb, bf16, BH, Nkv, D, 128))
      return OATTN_ERR_CUDA;
    a.tm_o = a.tm_q;  // split mode stores its partials without a tensor map
    a.o = o_partial;
    a.lse = lse_partial;
    a.BH = BH; a.N = Nq; a.Nkv = Nkv; a.D = D;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * kLog2e;
    a.P = P;
    a.chunk = chunk;
    a.out_f32 = partial_dtype == OATTN_F32 ? 1 : 0;
    a.mask = mk;
    a.fused = fm;
    le = launch_attn(a, 128, bf16, st);
  }
  if (le != cudaSuccess) return OATTN_ERR_CUDA;
  if (o && !counters) {
    // The combine is a programmatic dependent of the producer just launched on this stream.
    le = launch_combine(o_partial, lse_partial, o, lse, P, (long long)BH * Nq, D, partial_dtype, dtype,
                        kLn2f, true, st);
    if (le != cudaSuccess) return OATTN_ERR_CUDA;
  }
  return OATTN_OK;
}

}  // namespace
}  // namespace oattn

using namespace oattn;

extern "C" {

int splitk_chunk(int Nkv, int P) {
  if (Nkv <= 0 || P <= 0) return 0;
  const long long per = (Nkv + (long long)P - 1) / P;
  return (int)(((per + 127) / 128) * 128);
}

const char* oattn_status_string(oattn_status s) {
  switch (s) {
    case OATTN_OK: return "ok";
    case OATTN_ERR_INVALID_ARG: return "invalid argument";
    case OATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case OATTN_ERR_CUDA: return "CUDA error";
    case OATTN_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

oattn_status oattn_device_error(int* code) {
  if (!code) return OATTN_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* p = status_ptr(&e);
  if (!p) return OATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return OATTN_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return OATTN_ERR_CUDA;
  *code = (int)v;
  return v ? OATTN_ERR_TIMEOUT : OATTN_OK;
}

oattn_status oattn_selftest_wait(int* flags, struct CUstream_st* stream) {
  if (flags != nullptr && !aligned(flags, 4)) return OATTN_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* p = status_ptr(&e);
  if (!p) return OATTN_ERR_CUDA;
  return launch_selftest_wait(p, flags, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? OATTN_OK
                                                                                               : OATTN_ERR_CUDA;
}

oattn_status attn_fwd_bn(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int D, int causal, float scale, oattn_dtype dtype, int block_n,
                         struct CUstream_st* stream) {
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, block_n, MaskArgs{},
                       reinterpret_cast<cudaStream_t>(stream));
}

oattn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int N, int D, int causal, float scale, oattn_dtype dtype, struct CUstream_st* stream) {
  return attn_fwd_bn(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, 0, stream);
}

oattn_status attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                           void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d, int B, int H, int N, int D,
                           int causal, float scale, oattn_dtype dtype, int chunk_heads,
                           struct CUstream_st* stream) {
  oattn_status s = attn_common_checks(q_d, k_d, v_d, B, H, N, N, D, scale, dtype);
  if (s != OATTN_OK) return s;
  if (chunk_heads < 0) return OATTN_ERR_INVALID_ARG;
  if (N == 0) return OATTN_OK;
  if (!q_h || !k_h || !v_h || !o_h || !o_d || !aligned(o_d, 16)) return OATTN_ERR_INVALID_ARG;
  if ((lse_h == nullptr) != (lse_d == nullptr) || (lse_d && !aligned(lse_d, 4))) return OATTN_ERR_INVALID_ARG;
  cudaError_t e;
  Pipe* p = pipe_for_device(&e);
  if (!p) return OATTN_ERR_CUDA;
  std::lock_guard<std::mutex> enqueue(p->lock);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const long long BH = (long long)B * H;
  const long long ch = chunk_heads > 0 ? chunk_heads : (BH + 7) / 8;
  const size_t head_bytes = (size_t)N * D * 2, lse_bytes = (size_t)N * 4;
  auto off = [](const void* base, size_t bytes) { return static_cast<const char*>(base) + bytes; };
  auto offm = [](void* base, size_t bytes) { return static_cast<char*>(base) + bytes; };
  // Everything starts after the work already queued on the caller's stream.
  if (cudaEventRecord(p->start, st) != cudaSuccess || cudaStreamWaitEvent(p->in, p->start, 0) != cudaSuccess)
    return OATTN_ERR_CUDA;
  // Work queued on the caller's stream afterwards waits for everything enqueued here
  // (on success the copy-out stream already follows the other two; after a failure part
  // way through, all three are joined so that no copy outlives the call's buffers).
  auto join = [&]() {
    return cudaEventRecord(p->loaded, p->in) == cudaSuccess && cudaStreamWaitEvent(st, p->loaded, 0) == cudaSuccess &&
           cudaEventRecord(p->done, p->comp) == cudaSuccess && cudaStreamWaitEvent(st, p->done, 0) == cudaSuccess &&
           cudaEventRecord(p->finished, p->out) == cudaSuccess && cudaStreamWaitEvent(st, p->finished, 0) == cudaSuccess;
  };
  oattn_status result = OATTN_OK;
  for (long long h0 = 0, nh = 0; h0 < BH && result == OATTN_OK; h0 += nh) {
    nh = (h0 + ch <= BH) ? ch : BH - h0;
    const size_t o0 = (size_t)h0 * head_bytes, n0 = (size_t)nh * head_bytes;
    // Copy in (one copy per tensor), attention on these heads, copy out: three streams,
    // so the copies of one chunk overlap the attention of its neighbours.
    if (cudaMemcpyAsync(offm(q_d, o0), off(q_h, o0), n0, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
        cudaMemcpyAsync(offm(k_d, o0), off(k_h, o0), n0, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
        cudaMemcpyAsync(offm(v_d, o0), off(v_h, o0), n0, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
        cudaEventRecord(p->loaded, p->in) != cudaSuccess || cudaStreamWaitEvent(p->comp, p->loaded, 0) != cudaSuccess) {
      result = OATTN_ERR_CUDA;
      break;
    }
    result = attn_fwd_impl(offm(q_d, o0), offm(k_d, o0), offm(v_d, o0), offm(o_d, o0),
                           lse_d ? reinterpret_cast<float*>(offm(lse_d, (size_t)h0 * lse_bytes)) : nullptr, 1,
                           (int)nh, N, D, causal, scale, dtype, 128, MaskArgs{}, p->comp);
    if (result != OATTN_OK) break;
    if (cudaEventRecord(p->done, p->comp) != cudaSuccess || cudaStreamWaitEvent(p->out, p->done, 0) != cudaSuccess ||
        cudaMemcpyAsync(offm(o_h, o0), off(o_d, o0), n0, cudaMemcpyDeviceToHost, p->out) != cudaSuccess ||
        (lse_d && cudaMemcpyAsync(offm(lse_h, (size_t)h0 * lse_bytes), off(lse_d, (size_t)h0 * lse_bytes),
                                  (size_t)nh * lse_bytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess))
      result = OATTN_ERR_CUDA;
  }
  if (!join() && result == OATTN_OK) result = OATTN_ERR_CUDA;
  return result;
}

oattn_status splitk_combine(const void* o_partial, const float* lse_partial, void* o, float* lse_out,
                            int P, int rows, int heads, int depth, oattn_dtype in_dtype,
                            oattn_dtype out_dtype, struct CUstream_st* stream) {
  if (!o_partial || !lse_partial || !o) return OATTN_ERR_INVALID_ARG;
  if (P < 1 || P > 256 || rows < 1 || heads < 1 || depth < 1) return OATTN_ERR_INVALID_ARG;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return OATTN_ERR_INVALID_ARG;
  if (!aligned(o_partial, 16) || !aligned(o, 16) || !aligned(lse_partial, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return OATTN_ERR_INVALID_ARG;
  if (!combine_supported(depth, in_dtype)) return OATTN_ERR_UNSUPPORTED;
  const long long RH = (long long)rows * heads;
  return launch_combine(o_partial, lse_partial, o, lse_out, P, RH, depth, in_dtype, out_dtype, 1.0f, false,
                        reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? OATTN_OK
             : OATTN_ERR_CUDA;
}

oattn_status attn_fwd_splitk(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                             int H, int Nq, int Nkv, int D, int causal, float scale, oattn_dtype dtype,
                             int P, void* o_partial, float* lse_partial, oattn_dtype partial_dtype,
                             struct CUstream_st* stream) {
  return attn_fwd_splitk_impl(q, k, v, o, lse, B, H, Nq, Nkv, D, causal, scale, dtype, P, o_partial,
                              lse_partial, partial_dtype, MaskArgs{}, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int attn_mask_words(int Nkv) { return Nkv < 0 ? 0 : mask_words(Nkv); }

oattn_status attn_mask_pack(const void* mask, unsigned int* bits, long long rows, int Nkv, long long row_stride,
                            struct CUstream_st* stream) {
  if (rows < 0 || Nkv < 0) return OATTN_ERR_INVALID_ARG;
  if (rows == 0 || Nkv == 0) return OATTN_OK;
  if (!mask || !bits || !aligned(bits, 16) || row_stride < Nkv) return OATTN_ERR_INVALID_ARG;
  if (rows > (1LL << 40)) return OATTN_ERR_UNSUPPORTED;
  return launch_mask_pack(static_cast<const uint8_t*>(mask), reinterpret_cast<uint32_t*>(bits), rows, Nkv,
                          row_stride, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? OATTN_OK
             : OATTN_ERR_CUDA;
}

oattn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int N, int D, int causal, float scale, oattn_dtype dtype,
                             const unsigned int* mask_bits, long long mask_stride_b, long long mask_stride_h,
                             long long mask_stride_q, struct CUstream_st* stream) {
  if (N > 0) {
    const oattn_status s = mask_checks(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q);
    if (s != OATTN_OK) return s;
  }
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, 128,
                       mask_args(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q, H),
                       reinterpret_cast<cudaStream_t>(stream));
}

long long attn_mask_blocks_words(int B, int H, int Nq, int Nkv, long long mask_stride_b, long long mask_stride_h) {
  return mask_blocks_words(B, H, Nq, Nkv, mask_stride_b, mask_stride_h);
}

oattn_status attn_mask_blocks(const unsigned int* mask_bits, long long mask_stride_b, long long mask_stride_h,
                              long long mask_stride_q, int B, int H, int Nq, int Nkv, unsigned int* blocks,
                              struct CUstream_st* stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nkv < 0) return OATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || Nq == 0 || Nkv == 0) return OATTN_OK;
  const oattn_status s = mask_checks(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q);
  if (s != OATTN_OK) return s;
  if (!blocks || !aligned(blocks, 4)) return OATTN_ERR_INVALID_ARG;
  if (mask_blocks_words(B, H, Nq, Nkv, mask_stride_b, mask_stride_h) > 0x7fffffffLL) return OATTN_ERR_UNSUPPORTED;
  return launch_mask_blocks(reinterpret_cast<const uint32_t*>(mask_bits), mask_stride_b, mask_stride_h,
                            mask_stride_q, B, H, Nq, Nkv, reinterpret_cast<uint32_t*>(blocks),
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? OATTN_OK
             : OATTN_ERR_CUDA;
}

oattn_status attn_fwd_masked_blocks(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int N, int D, int causal, float scale, oattn_dtype dtype,
                                    const unsigned int* mask_bits, long long mask_stride_b, long long mask_stride_h,
                                    long long mask_stride_q, const unsigned int* blocks, struct CUstream_st* stream) {
  MaskBlocks mb{};
  if (N > 0) {
    const oattn_status s = mask_checks(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q);
    if (s != OATTN_OK) return s;
    if (!blocks || !aligned(blocks, 4)) return OATTN_ERR_INVALID_ARG;
    const int wpb = mask_block_wpb(N);
    const long long nblk = (N + 255) / 256;
    const long long hm = mask_stride_h ? H : 1;
    mb.bits = reinterpret_cast<const uint32_t*>(blocks);
    mb.wpb = wpb;
    mb.sh = mask_stride_h ? nblk * wpb : 0;
    mb.sb = mask_stride_b ? hm * nblk * wpb : 0;
  }
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, 128,
                       mask_args(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q, H),
                       reinterpret_cast<cudaStream_t>(stream), mb);
}

oattn_status attn_fwd_splitk_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                    int H, int Nq, int Nkv, int D, int causal, float scale, oattn_dtype dtype,
                                    int P, void* o_partial, float* lse_partial, oattn_dtype partial_dtype,
                                    const unsigned int* mask_bits, long long mask_stride_b,
                                    long long mask_stride_h, long long mask_stride_q,
                                    struct CUstream_st* stream) {
  if (Nq > 0 && Nkv > 0) {
    const oattn_status s = mask_checks(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q);
    if (s != OATTN_OK) return s;
  }
  // With no keys every row is empty whatever the mask says: run unmasked.
  const MaskArgs mk = Nkv > 0 ? mask_args(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q, H) : MaskArgs{};
  return attn_fwd_splitk_impl(q, k, v, o, lse, B, H, Nq, Nkv, D, causal, scale, dtype, P, o_partial,
                              lse_partial, partial_dtype, mk, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int attn_splitk_counters(int B, int H, int Nq) {
  if (B < 1 || H < 1 || Nq < 1) return 0;
  const long long n = (long long)B * H * (Nq == 1 ? 1 : (Nq + 255) / 256);
  return n > 0x7fffffffLL ? -1 : (int)n;
}

oattn_status attn_fwd_splitk_fused(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                   int H, int Nq, int Nkv, int D, int causal, float scale, oattn_dtype dtype,
                                   int P, void* o_partial, float* lse_partial, oattn_dtype partial_dtype,
                                   unsigned int* counters, const unsigned int* mask_bits, long long mask_stride_b,
                                   long long mask_stride_h, long long mask_stride_q, struct CUstream_st* stream) {
  if (Nq > 0 && (!o || !counters)) return OATTN_ERR_INVALID_ARG;
  MaskArgs mk{};
  if (mask_bits && Nq > 0 && Nkv > 0) {
    const oattn_status s = mask_checks(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q);
    if (s != OATTN_OK) return s;
    mk = mask_args(mask_bits, mask_stride_b, mask_stride_h, mask_stride_q, H);
  }
  return attn_fwd_splitk_impl(q, k, v, o, lse, B, H, Nq, Nkv, D, causal, scale, dtype, P, o_partial,
                              lse_partial, partial_dtype, mk, counters, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
