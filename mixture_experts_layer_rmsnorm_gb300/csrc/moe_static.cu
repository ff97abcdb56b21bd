// moe_static.cu -- moe_forward_static_scratch: the layer forward with its
// scratch in a fixed device array owned by this library, for callers that
// cannot allocate device memory themselves.
//
// Which callers, and why: some hosts hand every byte of device memory to
// their own pool or run under a fixed memory budget decided at start-up, so a
// library cannot ask them for a workspace; others (plain C callers, plug-ins)
// have no device allocator of their own; and latency-critical callers avoid
// cudaMalloc/cudaFree in the serving loop because those calls can block,
// take driver locks and synchronise the device.  For them this file keeps
// the scratch in a file-scope __device__ array of MOE_STATIC_SCRATCH_BYTES.
// Every GPU that loads the library holds that array until the process exits.
//
// The host cannot use the array's name as a device address (in host code it
// names a host-side stand-in).  So once per device, with that device
// current, the first call asks the runtime for the array's device address
// with cudaGetSymbolAddress and keeps it; later calls on that device reuse it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "moe_forward_impl.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device (set up once per device).
moe_status static_scratch_of_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status moe_static_scratch_bytes(size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = static_cast<size_t>(MOE_STATIC_SCRATCH_BYTES);
  return MOE_OK;
}

// The error word at the start of the array (the workspace layout puts it at
// offset 0), read after the stream has finished the caller's work.
extern "C" MOE_API moe_status moe_static_scratch_device_status(moe_stream_t stream, int32_t* detail) {
  void* scratch = nullptr;
  const moe_status st = static_scratch_of_current_device(&scratch);
  if (st != MOE_OK) return st;
  return moe_device_status(scratch, MOE_STATIC_SCRATCH_BYTES, stream, detail);
}

extern "C" MOE_API moe_status moe_forward_static_scratch(const moe_shape* shape, const moe_bf16* x, const moe_bf16* g_norm,
                                                 const float* w_router, const float* router_bias,
                                                 const moe_bf16* w13, const moe_bf16* w2, moe_bf16* y,
                                                 moe_stream_t stream) {
  size_t need = 0;
  const moe_status st = moe_workspace_size(shape, &need);
  if (st != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if (need > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;  // shape needs more than the fixed array
  void* scratch = nullptr;
  const moe_status s2 = static_scratch_of_current_device(&scratch);
  if (s2 != MOE_OK) return s2;
  return moe::forward_impl(shape, x, g_norm, w_router, router_bias, w13, w2, y, scratch, MOE_STATIC_SCRATCH_BYTES,
                           stream, nullptr);
}
