// route_static.cu -- routing for callers that cannot allocate device memory.
//
// moe_route needs a scratch buffer from its caller.  Some callers have no way
// to provide one: code that runs while a CUDA graph is being captured (where
// cudaMalloc is not allowed), code inside a framework whose caching allocator
// already owns the device memory, or a serving loop that must not allocate on
// its hot path.  For them, moe_route_static_scratch runs the same routing
// kernels on a scratch array that lives in this library's own device memory:
// a file-scope __device__ array, loaded with the library and kept by every GPU
// that loads it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

// Room for any configuration with T <= 32768 tokens (k <= 16, E <= 256): per-slot
// ranks (2 MiB at the limit), the per-block expert histogram (256 KiB) and the
// status header, with room to spare -- 2.5 MiB + 4 KiB.
constexpr size_t kStaticRouteScratchBytes = (size_t{5} << 19) + 4096;

static __device__ __align__(256) uint8_t g_route_scratch[kStaticRouteScratchBytes];

// In host code g_route_scratch names a host-side stand-in, not a device address.
// The device address is looked up with the device current and cached per
// device only once a lookup has succeeded; a failed lookup (for example a first
// call made while the stream is being captured) is retried by the next call.
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

cudaError_t static_scratch(int dev, void **out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();  // leave no error behind for the next launcher to report
      return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_static_scratch(const moe_config *cfg, const float *logits,
                                               const moe_routing *routing, int32_t *device_status,
                                               void *stream) {
  size_t need = 0;
  const moe_status q = moe_query_workspace(cfg, &need, nullptr, nullptr, nullptr);
  if (q != MOE_OK) return q;
  if (need > moe::kStaticRouteScratchBytes) return MOE_ERR_WORKSPACE;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return MOE_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= moe::kMaxDevices) return MOE_ERR_CUDA;
  void *scratch = nullptr;
  if (moe::static_scratch(dev, &scratch) != cudaSuccess || !scratch) return MOE_ERR_CUDA;
  // moe_route zeroes the status header itself and rewrites every other byte it
  // reads, so nothing from the previous call leaks into this one.
  const moe_status st =
      moe_route(cfg, logits, routing, scratch, moe::kStaticRouteScratchBytes, stream);
  if (st != MOE_OK || !device_status) return st;
  if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
