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

#include "rkv.h"
#include "rkv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 128;

// The scratch itself.  In host code this name is only a stand-in for the symbol,
// not a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
