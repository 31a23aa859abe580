// zl_decode_attn_noalloc: zl_decode_attn for callers that cannot allocate
// device memory. The split-KV scratch lives in a fixed array that the library
// itself carries in device memory, so the caller passes only inputs and outputs.
//
// Who needs this: a caller embedded in a host process that has already
// reserved all device memory for its own pool, a plugin interface that hands
// the kernel no scratch allocator, or a latency-critical loop that cannot
// afford cudaMalloc (which may synchronise the device). None of them can
// provide the caller-owned workspace that zl_decode_attn requires.
#include "../../include/zl_decode_attn.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// The scratch every zl_decode_attn_noalloc call uses. Each GPU that loads the
// library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_workspace[ZL_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

// Device address of g_noalloc_workspace on `device` (which must be current).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device and cached. Returns nullptr on failure.
void* workspace_on(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_ptr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_workspace) != cudaSuccess) return nullptr;
    g_device_ptr[device] = ptr;
  }
  return g_device_ptr[device];
}

}  // namespace

extern "C" zl_status zl_decode_attn_noalloc(const zl_decode_attn_params* params,
                                            zl_stream_t stream) {
  if (!params || params->struct_size != sizeof(zl_decode_attn_params)) return ZL_ERR_INVALID_ARG;
  zl_decode_attn_params p = *params;
  p.workspace = nullptr;
  p.workspace_bytes = 0;
  size_t need = 0;
  zl_status st = zl_decode_attn_workspace_size(&p, &need);
  if (st != ZL_OK) return st;
  if (need > size_t(ZL_NOALLOC_WORKSPACE_BYTES)) return ZL_ERR_WORKSPACE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return ZL_ERR_CUDA;
  void* ws = workspace_on(device);
  if (!ws) return ZL_ERR_CUDA;
  p.workspace = ws;
  p.workspace_bytes = ZL_NOALLOC_WORKSPACE_BYTES;
  return zl_decode_attn(&p, stream);
}
