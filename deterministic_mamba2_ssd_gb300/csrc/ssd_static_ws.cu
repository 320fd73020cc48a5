// ssd_static_ws.cu -- a backward entry point for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they need the backward: code running inside a pre-sized memory
// arena that must not grow, plugins whose host forbids allocation after
// start-up, or hard real-time loops where an allocation could block.  Such
// callers still own their inputs and outputs but cannot provide the
// backward's scratch workspace.  For them this file keeps the scratch in one
// fixed-size array in device global memory (kStaticScratchBytes), which every
// GPU that loads the library holds until the process exits.
//
// Set-up: the first call on a device, with that device current, looks the
// array's device address up (cudaGetSymbolAddress) and caches it; later
// calls reuse it.  That first call should therefore come before any stream
// capture on the device.  The cached address belongs to the device context
// it was looked up in: after cudaDeviceReset (or any teardown of the primary
// context) the module is loaded again at a new address, and this entry point
// must not be called again in that process.  Calls share the array and it keeps the previous
// call's contents; the backward clears what must start at zero itself.  Calls
// whose work overlaps on the GPU (different streams without ordering) race
// on the array and must not be made.
#include <cuda_runtime.h>

#include <mutex>

#include "mamba2_ssd.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

// Host code may only name this array to look its device address up; the
// symbol itself is a host-side stand-in, not a device pointer.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (set up once per device).
ssd_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" {

size_t mamba2_ssd_static_scratch_bytes(void) { return kStaticScratchBytes; }

ssd_status mamba2_ssd_bwd_static_scratch(const ssd_saved *saved, const void *dout, float *dx, float *ddt,
                                         float *dA, float *dB, float *dC, float *dD, float *dinit, int config,
                                         void *stream) {
  if (!saved) return SSD_ERR_HANDLE;
  const size_t need = mamba2_ssd_bwd_workspace_size(&saved->dims, config, SSD_VARIANT_DETERMINISTIC);
  if (need == 0) return SSD_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return SSD_ERR_WORKSPACE;
  void *ws = nullptr;
  const ssd_status st = scratch_address(&ws);
  if (st != SSD_OK) return st;
  return mamba2_ssd_bwd(saved, dout, dx, ddt, dA, dB, dC, dD, dinit, ws, kStaticScratchBytes, config,
                        SSD_VARIANT_DETERMINISTIC, stream);
}

// The backward's device-side status word lives at the start of its workspace,
// here the static array; this reads it the way mamba2_ssd_bwd_check does.
ssd_status mamba2_ssd_static_scratch_check(const ssd_dims *dims, int config, void *stream) {
  if (config < 0 || config >= mamba2_ssd_num_configs(dims)) return SSD_ERR_INVALID_ARG;   // 0 configs: bad dims
  void *ws = nullptr;
  const ssd_status st = scratch_address(&ws);
  if (st != SSD_OK) return st;
  return mamba2_ssd_bwd_check(dims, config, ws, stream);
}

}  // extern "C"
