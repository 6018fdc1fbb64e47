// attn_fwd_splitk_noalloc: split-K attention whose partition workspace lives in a fixed
// device array inside this library, for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a plugin running inside a host framework
// that owns every byte of device memory through its own pool, or a latency-critical
// caller that cannot afford the implicit device synchronisation an allocation may
// cause.  attn_fwd_splitk needs two caller-owned scratch buffers (o_partial and
// lse_partial); this entry point takes only the inputs and the outputs and keeps the
// partials in the static array below.
//
// The array is a module global: every GPU that loads the library holds it (41 MiB)
// until the process exits, whether or not this entry point is ever called.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/oattn.h"

namespace {

// Capacity of the shared workspace, in floats.
constexpr long long kNoallocPartialFloats = 10LL * 1024 * 1024;  // o_partial: 40 MiB
constexpr long long kNoallocLseFloats = 256LL * 1024;            // lse_partial: 1 MiB

static __device__ __align__(256) float g_noalloc_partial[kNoallocPartialFloats];
static __device__ __align__(256) float g_noalloc_lse[kNoallocLseFloats];

constexpr int kMaxDevices = 64;
float* g_partial_ptr[kMaxDevices] = {};
float* g_lse_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

// Device addresses of the two arrays for the current device.  In host code the array
// names are host-side stand-ins, not device addresses, so they are looked up once per
// device with that device current.
bool noalloc_scratch(float** partial, float** lse) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_partial_ptr[dev] == nullptr || g_lse_ptr[dev] == nullptr) {
    void* p = nullptr;
    void* l = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partial) != cudaSuccess) return false;
    if (cudaGetSymbolAddress(&l, g_noalloc_lse) != cudaSuccess) return false;
    g_partial_ptr[dev] = static_cast<float*>(p);
    g_lse_ptr[dev] = static_cast<float*>(l);
  }
  *partial = g_partial_ptr[dev];
  *lse = g_lse_ptr[dev];
  return true;
}

}  // namespace

extern "C" oattn_status attn_fwd_splitk_noalloc(const void* q, const void* k, const void* v, void* o,
                                                float* lse, int B, int H, int Nq, int Nkv, int D,
                                                int causal, float scale, oattn_dtype dtype, int P,
                                                struct CUstream_st* stream) {
  if (Nq > 0 && !o) return OATTN_ERR_INVALID_ARG;  // the merged output is the only result
  if (B < 1 || H < 1 || Nq < 0 || P < 1) return OATTN_ERR_INVALID_ARG;
  const long long rows = (long long)B * H * Nq;
  if ((long long)P * rows * D > kNoallocPartialFloats || (long long)P * rows > kNoallocLseFloats)
    return OATTN_ERR_UNSUPPORTED;  // beyond the fixed workspace
  // An empty problem still goes through attn_fwd_splitk, which checks every other
  // argument (dtype, D, scale, P) and then returns without touching the device; the
  // workspace address is only looked up when there is work.
  float* partial = nullptr;
  float* lse_partial = nullptr;
  if (Nq > 0 && !noalloc_scratch(&partial, &lse_partial)) return OATTN_ERR_CUDA;
  // Every partition row is rewritten by each call, so nothing needs clearing first.
  return attn_fwd_splitk(q, k, v, o, lse, B, H, Nq, Nkv, D, causal, scale, dtype, P, partial, lse_partial,
                         OATTN_F32, stream);
}
