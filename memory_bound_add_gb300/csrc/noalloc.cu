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
// names a stand-in object), so on the first call on each device that needs
// the buffer, with that device current, its device address is looked up with
// cudaGetSymbolAddress and cached for that device's current context (a reset
// device gets a new context and the address is looked up again); that first
// call on a device should therefore come before any stream capture.  Nothing
// here allocates: the call forwards to add_layernorm_bwd with the buffer as
// its workspace, so it runs exactly the same kernels.  Every CTA writes all
// of its [2][H] partial before the column-sum kernel reads it, so no part of
// the buffer has to start at zero; the buffer keeps whatever the last call
// left.  All calls on a device share the one buffer: calls that can overlap
// on the GPU (other streams, other host threads) race on it and must be
// serialised by the caller.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/addln.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ADDLN_NOALLOC_SCRATCH_BYTES];

// The driver's current-context query, reached through the runtime so the
// library needs no link to the driver library.  The scratch array lives in
// the library's module of one context: after cudaDeviceReset the device gets
// a new context, the module is loaded again and the array may sit elsewhere,
// so the cached address is keyed on the context's process-unique ID.
using CtxGetCurrent = int (*)(void**);
using CtxGetId = int (*)(void*, unsigned long long*);

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  unsigned long long ctx_id;
  void* ptr;
};
Cached g_scratch[kMaxDevices] = {};
CtxGetCurrent g_get_current = nullptr;
CtxGetId g_get_id = nullptr;

// ID of the current context, or 0 when it cannot be told (then the address
// is looked up again on every call).
unsigned long long current_context_id() {
  if (g_get_current == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return 0;
    g_get_id = reinterpret_cast<CtxGetId>(f2);
    g_get_current = reinterpret_cast<CtxGetCurrent>(f1);
  }
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (g_get_current(&ctx) != 0 || ctx == nullptr || g_get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of the scratch array in the current device's context,
// looked up once per (device, context) with that device current.
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ADDLN_ERR_CUDA;
  // makes the device's primary context current (initialising it if needed)
  if (cudaSetDevice(dev) != cudaSuccess) return ADDLN_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  const unsigned long long id = current_context_id();
  Cached& c = g_scratch[dev];
  if (c.ptr == nullptr || id == 0 || c.ctx_id != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ADDLN_ERR_CUDA;
    c.ptr = ptr;
    c.ctx_id = id;
  }
  *out = c.ptr;
  return ADDLN_OK;
}

}  // namespace

extern "C" int add_layernorm_bwd_noalloc(const void* dy, const void* a, const float* mean,
                                         const float* rstd, const float* gamma, const void* dres,
                                         void* dx, float* dgamma, float* dbeta, int64_t rows,
                                         int64_t H, int dtype, void* stream) {
  // the argument checks add_layernorm_bwd makes before any CUDA call, in its
  // order, so both entry points return the same codes for the same mistakes
  if (dtype != ADDLN_FP32 && dtype != ADDLN_FP16 && dtype != ADDLN_BF16) return ADDLN_ERR_DTYPE;
  const int64_t max_h = addln_max_hidden(dtype);
  if (rows < 0 || H <= 0 || H > max_h || rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  if ((dgamma == nullptr) != (dbeta == nullptr)) return ADDLN_ERR_NULL;
  // no column sums (or no rows): no workspace is used at all
  if (dgamma == nullptr || rows == 0)
    return add_layernorm_bwd(dy, a, mean, rstd, gamma, dres, dx, dgamma, dbeta, rows, H, dtype,
                             nullptr, 0, stream);
  if (!dy || !a || !mean || !rstd || !gamma || !dx) return ADDLN_ERR_NULL;
  const int64_t need = add_layernorm_bwd_workspace_size(rows, H, dtype);
  if (need < 0) return static_cast<int>(need);
  if (need > static_cast<int64_t>(ADDLN_NOALLOC_SCRATCH_BYTES)) return ADDLN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != ADDLN_OK) return rc;
  return add_layernorm_bwd(dy, a, mean, rstd, gamma, dres, dx, dgamma, dbeta, rows, H, dtype,
                           scratch, static_cast<int64_t>(ADDLN_NOALLOC_SCRATCH_BYTES), stream);
}
