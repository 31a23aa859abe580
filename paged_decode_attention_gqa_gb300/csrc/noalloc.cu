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

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace {

// The scratch every zl_decode_attn_noalloc call uses. Each GPU that loads the
// library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_workspace[ZL_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Per device: the context the address below was looked up in (its unique id,
// which the driver never reuses within a process) and the array's address
// there.
struct Setup {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
std::mutex g_mutex;
Setup g_setup[kMaxDevices];

// The unique id of the calling thread's current context (0 if unavailable).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_workspace on `device` (which must be current).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device, and again if the device's context has changed
// since (after a cudaDeviceReset the module is loaded anew and the array may
// sit elsewhere). Returns nullptr on failure.
void* workspace_on(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  // 0 when the runtime has not made a context current on this thread yet; the
  // lookup below does (and the id is read again after it).
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  Setup& s = g_setup[device];
  if (!s.ptr || ctx == 0 || s.ctx_id != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_workspace) != cudaSuccess) return nullptr;
    s.ptr = ptr;
    s.ctx_id = ctx ? ctx : current_context_id();
  }
  return s.ptr;
}

}  // namespace

extern "C" zl_status zl_decode_attn_noalloc(const zl_decode_attn_params* params,
                                            zl_stream_t stream) {
  if (!params || params->struct_size != sizeof(zl_decode_attn_params)) return ZL_ERR_INVALID_ARG;
  zl_decode_attn_params p = *params;
  p.workspace = nullptr;
  p.workspace_bytes = 0;
  constexpr size_t kCap = size_t(ZL_NOALLOC_WORKSPACE_BYTES);
  size_t need = 0;
  zl_status st = zl_decode_attn_workspace_size(&p, &need);
  if (st != ZL_OK) return st;
  if (need > kCap && p.num_ctas == 0) {
    // The default grid's partial slots do not fit: take the largest grid
    // whose workspace does (the need grows by the same number of bytes per
    // CTA; rounding of the regions to 256 bytes is settled by the check
    // loop). Results do not depend on the grid beyond fp32 rounding.
    size_t n1 = 0, n2 = 0;
    p.num_ctas = 1;
    if ((st = zl_decode_attn_workspace_size(&p, &n1)) != ZL_OK) return st;
    p.num_ctas = 2;
    if ((st = zl_decode_attn_workspace_size(&p, &n2)) != ZL_OK) return st;
    if (n1 > kCap || n2 <= n1) return ZL_ERR_WORKSPACE;
    const size_t per_cta = n2 - n1;
    size_t k = 1 + (kCap - n1) / per_cta;
    if (k > 65535) k = 65535;
    for (;; --k) {
      p.num_ctas = int32_t(k);
      if ((st = zl_decode_attn_workspace_size(&p, &need)) != ZL_OK) return st;
      if (need <= kCap || k == 1) break;
    }
  }
  if (need > kCap) return ZL_ERR_WORKSPACE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return ZL_ERR_CUDA;
  void* ws = workspace_on(device);
  if (!ws) return ZL_ERR_CUDA;
  p.workspace = ws;
  p.workspace_bytes = kCap;
  // The single-launch merge counts arrivals in the first 8 * B * Hkv bytes,
  // which must start at zero; the array keeps whatever the previous call left
  // there (partials of a call without the flag, or of a larger shape), so
  // clear them on the stream first. cudaMemsetAsync allocates nothing.
  if (p.flags & ZL_DECODE_SINGLE_LAUNCH) {
    const size_t counters = size_t(p.B) * size_t(p.Hkv) * 8;
    if (counters > kCap) return ZL_ERR_WORKSPACE;
    if (cudaMemsetAsync(ws, 0, counters, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return ZL_ERR_CUDA;
  }
  return zl_decode_attn(&p, stream);
}
