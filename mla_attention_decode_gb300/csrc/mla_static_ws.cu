// mla_static_ws.cu -- mla_decode_fwd_static: mla_decode_fwd with its workspace
// in a device array owned by this library, for callers that cannot allocate
// device memory (see include/mla_decode.h).
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_decode.h"

namespace {

// The shared workspace.  Every GPU that loads the library holds these bytes
// until the process exits.  Host code must not use the name as an address (on
// the host it only stands for the symbol): the device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The device address of g_static_workspace is looked up once per device and
// kept together with the id of the context it belongs to.  A new context on
// the device (the application called cudaDeviceReset, or the primary context
// was released and created again) loads the module again, possibly at another
// address: the id then differs and the address is looked up again.
struct Entry {
  void* address = nullptr;
  unsigned long long ctx_id = 0;
};
std::mutex g_mutex;
Entry g_entry[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points for the current context's id, fetched through the
// runtime once (the library links only the runtime).
struct CtxIdApi {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
const CtxIdApi& ctx_api() {
  static const CtxIdApi api = []() {
    CtxIdApi a;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
    return a;
  }();
  return api;
}

// Id of the current context (0 when there is none or it cannot be read).
unsigned long long current_ctx_id() {
  const CtxIdApi& a = ctx_api();
  if (!a.get_current || !a.get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (a.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (a.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the shared workspace on the current device.  The first
// call on a device (and the first after its context changed) looks it up with
// cudaGetSymbolAddress, which also loads the module into the context.
int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  Entry& e = g_entry[dev];
  const unsigned long long id = current_ctx_id();
  if (!e.address || id == 0 || id != e.ctx_id) {
    void* p = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&p, g_static_workspace);
    if (rc != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      e.address = nullptr;
      return MLA_ERR_CUDA;
    }
    e.address = p;
    // the look-up made the device's primary context current if none was
    e.ctx_id = current_ctx_id();
  }
  *out = e.address;
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
