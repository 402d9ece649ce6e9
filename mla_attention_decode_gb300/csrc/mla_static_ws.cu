// mla_static_ws.cu -- mla_decode_fwd_static: mla_decode_fwd with its workspace
// in a device array owned by this library, for callers that cannot allocate
// device memory (see include/mla_decode.h).
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mla_decode.h"

namespace {

// The shared workspace.  Every GPU that loads the library holds these bytes
// until the process exits.  Host code must not use the name as an address (on
// the host it only stands for the symbol): the device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_address[kMaxDevices] = {};  // device address of g_static_workspace, per device ordinal

// Device address of the shared workspace on the current device; looked up once
// per device (the first call on a device does it) and cached.
int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_address[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_address[dev] = p;
  }
  *out = g_address[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_fwd_static(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                                     const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse,
                                     float sm_scale, const mla_plan* plan, int32_t* device_error, void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (mla_decode_workspace_bytes(plan) > MLA_STATIC_WORKSPACE_BYTES) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  int rc = static_workspace(&ws);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word (first 4 bytes) must start at zero; the rest is written
  // before it is read within one call
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  rc = mla_decode_fwd(q, kv, kv_scale, scale_stride, kv_indptr, qo_indptr, out, lse, sm_scale, plan, ws,
                      MLA_STATIC_WORKSPACE_BYTES, stream);
  if (rc != MLA_OK) return rc;
  if (device_error &&
      cudaMemcpyAsync(device_error, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
