// moe_quantize_e4m3_noalloc: the dynamic per-tensor E4M3 quantisation with its
// scratch (the per-CTA partial maxima of |x|) in a static device array owned by
// this library instead of a caller buffer.
//
// For callers that cannot allocate device memory at the point of the call:
// code that runs where cudaMalloc is not allowed or must not block (for
// example while another component owns every device allocation, or on a
// latency-critical thread that cannot take the allocator's implicit device
// synchronisation), and that therefore cannot provide the scratch buffer
// moe_quantize_e4m3 asks for.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {
namespace {

// Partial maxima written by the amax kernel, one per CTA.  Every device that
// loads the library holds this array until the process exits.  Each call
// writes every entry it later reads, so nothing has to start at zero.
static __device__ __align__(256) float g_noalloc_partials[MOE_NOALLOC_MAX_PARTIALS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the array's address and the unique id of the CUDA context it
// was looked up in.  A module's device symbols live in one context, so a new
// context on the device (after cudaDeviceReset, or another current driver
// context) gets its address looked up again.
float* g_ptr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};

// Unique id of the calling thread's current context (cuCtxGetId: ids are
// never reused within a process).  0 when it cannot be read.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array in the current device's current context.  It
// is looked up (cudaGetSymbolAddress, with that device current; this also
// binds the runtime's primary context if none is current yet) on the first
// call in a context and cached under the context's id; a context whose id
// cannot be read is looked up on every call.
cudaError_t scratch_address(int dev, float** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = current_context_id();
  if (ctx != 0 && g_ptr[dev] != nullptr && g_ctx_id[dev] == ctx) {
    *out = g_ptr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_partials);
  if (e != cudaSuccess) return checked(e, "cudaGetSymbolAddress");
  ctx = current_context_id();
  g_ptr[dev] = static_cast<float*>(p);
  g_ctx_id[dev] = ctx;
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_quantize_e4m3_noalloc(const void* x, int T, int H, uint8_t* x_q,
                                                  float* scale, moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || H < 16 || H % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !x_q || !scale || (reinterpret_cast<uintptr_t>(x) & 15) ||
      (reinterpret_cast<uintptr_t>(x_q) & 15) || (reinterpret_cast<uintptr_t>(scale) & 3))
    return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
  // one partial per amax CTA; the amax kernel strides over the whole tensor,
  // so any T*H fits, and the count is still checked against the array
  const long long n = static_cast<long long>(T) * H;
  long long parts = std::min<long long>(MOE_NOALLOC_MAX_PARTIALS, std::max(1, sms * 4));
  parts = std::min<long long>(parts, (n / 8 + 255) / 256);
  if (parts < 1) parts = 1;
  if (parts > MOE_NOALLOC_MAX_PARTIALS) return MOE_ERR_UNSUPPORTED;
  float* partials = nullptr;
  if (scratch_address(dev, &partials) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(x), n, x_q, scale, partials,
                              static_cast<int>(parts), stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
