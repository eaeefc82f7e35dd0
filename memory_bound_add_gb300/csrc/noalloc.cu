// add_layernorm_bwd_noalloc: the Add+LayerNorm backward for callers that
// cannot allocate device memory.
//
// add_layernorm_bwd needs a workspace for its column partials, which the
// caller normally allocates.  Some callers cannot: a plugin that a framework
// or inference engine hands only tensor pointers (the host owns every byte of
// device memory through its own pool and gives the plugin no allocator), or a
// latency-critical loop where cudaMalloc / cudaFree are off limits because
// they can block and synchronise the device.  For them this entry point takes
// its workspace from a fixed buffer compiled into the library instead.
//
// The buffer is a file-scope device array of ADDLN_NOALLOC_SCRATCH_BYTES
// (32 MiB): every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so on the first call on each device, with that
// device current, its device address is looked up with cudaGetSymbolAddress
// and cached; that first call on a device should therefore come before any
// stream capture.  Nothing here allocates: the call forwards to
// add_layernorm_bwd with the buffer as its workspace, so it runs exactly the
// same kernels.  Every CTA writes all of its [2][H] partial before the
// column-sum kernel reads it, so no part of the buffer has to start at zero;
// the buffer keeps whatever the last call left.  All calls on a device share
// the one buffer: calls that can overlap on the GPU (other streams, other host
// threads) race on it and must be serialised by the caller.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/addln.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ADDLN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ADDLN_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ADDLN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ADDLN_OK;
}

}  // namespace

extern "C" int add_layernorm_bwd_noalloc(const void* dy, const void* a, const float* mean,
                                         const float* rstd, const float* gamma, const void* dres,
                                         void* dx, float* dgamma, float* dbeta, int64_t rows,
                                         int64_t H, int dtype, void* stream) {
  if (dgamma != nullptr && rows > 0) {
    const int64_t need = add_layernorm_bwd_workspace_size(rows, H, dtype);
    if (need < 0) return static_cast<int>(need);
    if (need > static_cast<int64_t>(ADDLN_NOALLOC_SCRATCH_BYTES)) return ADDLN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != ADDLN_OK) return rc;
  return add_layernorm_bwd(dy, a, mean, rstd, gamma, dres, dx, dgamma, dbeta, rows, H, dtype,
                           scratch, static_cast<int64_t>(ADDLN_NOALLOC_SCRATCH_BYTES), stream);
}
