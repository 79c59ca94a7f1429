// attn_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or cannot own a workspace buffer
// across calls: code running under an allocator that forbids new device
// allocations (a serving process that fixed its memory budget up front), or a
// plugin whose host hands out no device allocations.  For them the fp32 dQ
// accumulator of the backward lives in a file-scope device array of this
// translation unit instead of a caller-provided workspace.  The source pages
// have no counterpart for this entry point.
//
// The array has a module of its own: with lazy module loading (the CUDA
// default) the driver reserves its 32 MiB on a device only when the first
// attn_bwd_noalloc call there looks up its address, so processes that never
// call this entry point do not hold it.  Once reserved, it stays until the
// process exits (with CUDA_MODULE_LOADING=EAGER every device holds it from
// context creation).  In host code `g_bwd_noalloc_scratch` is only a stand-in
// for the symbol; its device address is looked up once per device, with that
// device current, by cudaGetSymbolAddress.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace bss {
namespace {

constexpr size_t kNoAllocScratchFloats = size_t(8) << 20;   // 32 MiB of fp32
static __device__ __align__(256) float g_bwd_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_scratch_ptr[kNoAllocMaxDevices] = {nullptr};

// Device address of the scratch on the current device (looked up on first use;
// the cached addresses assume the CUDA context is not reset while the library
// is in use).
attn_status_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  char msg[200];
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    set_error_text(msg);
    return ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc: device %d is beyond the %d devices it keeps "
             "a scratch address for", dev, kNoAllocMaxDevices);
    set_error_text(msg);
    return ATTN_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch);
    if (e != cudaSuccess) {
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(g_bwd_noalloc_scratch): %s",
               cudaGetErrorString(e));
      set_error_text(msg);
      return ATTN_ERR_CUDA;
    }
    g_noalloc_scratch_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_noalloc_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace bss

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* dout,
                                          void* dq, void* dk, void* dv, float* delta, int B, int H,
                                          int H_kv, int L, int d, float scale, int causal,
                                          void* stream) {
  using namespace bss;
  if (B < 1 || H < 1 || L < 0) return ATTN_ERR_INVALID_ARG;
  const size_t need = static_cast<size_t>(B) * H * static_cast<size_t>(L) * (d > 0 ? d : 0);
  if (need > kNoAllocScratchFloats) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "attn_bwd_noalloc: B*H*L*d = %zu exceeds the static scratch of %zu floats; "
             "use attn_bwd with a caller-provided workspace",
             need, kNoAllocScratchFloats);
    set_error_text(msg);
    return ATTN_ERR_WORKSPACE;
  }
  float* scratch = nullptr;
  attn_status_t s = noalloc_scratch(&scratch);
  if (s != ATTN_OK) return s;
  // attn_bwd clears the accumulator on the stream before it is used
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, scratch,
                  kNoAllocScratchFloats * sizeof(float), B, H, H_kv, L, d, scale, causal, stream);
}
