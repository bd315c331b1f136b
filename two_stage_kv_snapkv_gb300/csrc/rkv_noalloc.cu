// rkv_decode_hsa_noalloc: the HSA decode step for callers that cannot allocate
// device memory.
//
// Some callers have no way to provide a workspace at the point of the call: code
// running as a plug-in inside another engine that owns every device allocation and
// hands out none, or a latency-critical loop that must never reach cudaMalloc
// (which can synchronise the whole device).  For them this entry point runs the
// same decode step as rkv_decode_hsa with its scratch taken from one fixed array
// compiled into the library, so the call itself allocates nothing.
//
// The array costs kNoAllocScratchBytes (32 MiB) of device memory on every GPU that
// loads the library, for as long as the process lives.  All calls share it.
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "rkv.h"
#include "rkv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 128;

// The scratch itself.  In host code this name is only a stand-in for the symbol,
// not a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
// The looked-up address per device, with the context it was looked up in: after a
// cudaDeviceReset the device gets a new primary context, the old address is stale,
// and the next call looks it up again.
struct Slot {
  CUcontext ctx;
  void* ptr;
};
Slot g_scratch[kMaxDevices];

// The current context of the calling thread (cuCtxGetCurrent, taken from the driver
// through the runtime so the library needs no link against libcuda).
cudaError_t current_context(CUcontext* out) {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  if (!get) return cudaErrorNotSupported;
  return get(out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch on the current device: looked up on the first call in
// each (device, context), then reused.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CUcontext ctx = nullptr;
  if (current_context(&ctx) != cudaSuccess) ctx = nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  Slot& sl = g_scratch[dev];
  if (!sl.ptr || !ctx || sl.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the primary context current if none was
    if (e != cudaSuccess) return e;
    if (current_context(&ctx) != cudaSuccess) ctx = nullptr;
    sl.ptr = p;
    sl.ctx = ctx;
  }
  *out = sl.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" rkv_status rkv_decode_hsa_noalloc(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq,
                                             const int32_t* k1, const int32_t* k2, float scale, float* out,
                                             int32_t* sel_channels, int32_t* sel_pages,
                                             int32_t sel_pages_stride, void* stream) {
  if (!cache) {
    rkv::set_last_error("rkv_decode_hsa_noalloc: cache is NULL");
    return RKV_ERR_INVALID_ARG;
  }
  const size_t need = rkv_decode_workspace_size(cache->B, Hq, cache->Hkv, cache->max_pages);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "rkv_decode_hsa_noalloc: this cache needs %zu bytes of scratch but the built-in scratch holds %zu "
             "(32 MiB); use rkv_decode_hsa with a workspace",
             need, kNoAllocScratchBytes);
    rkv::set_last_error(msg);
    return RKV_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "rkv_decode_hsa_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    rkv::set_last_error(msg);
    return RKV_ERR_CUDA;
  }
  // Nothing in the scratch has to start at zero: every byte the decode step reads
  // was written earlier in the same step.
  return rkv_decode_hsa(cache, q, Hq, k1, k2, scale, out, sel_channels, sel_pages, sel_pages_stride, ws,
                        kNoAllocScratchBytes, stream);
}
