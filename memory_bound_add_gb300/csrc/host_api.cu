// add_layernorm_fwd_host: the fused forward from host buffers to host
// buffers, with the host-device traffic inside the call.
//
// Mapped (zero-copy): when the device can reach host memory and X, R and
// every output are mapped page-locked memory with 16-byte aligned rows, the
// kernel reads and writes them in place over the host link, one pass each
// way with both directions at once; only gamma and beta go to the device
// first (a small kernel when they are mapped too, else two copies).  Rows over 1024 then take the CTA kernel with 16-byte
// loads, so no bulk copy ever reads host memory.
//
// Pipelined, otherwise: the rows are cut into chunks of about 4 MiB of X
// each and pipelined over
// three streams: a copy-in stream (X, R of chunk c into device buffer c % 2),
// the caller's stream (add_layernorm_fwd on the chunk, once its copy has
// landed) and a copy-out stream (Y and the optional outputs of chunk c, once
// its kernel is done).  H2D of chunk c+1, the kernel of chunk c and D2H of
// chunk c-1 then run at the same time, and the two copy directions use
// separate copy engines.  Every copy is one cudaMemcpyAsync.
//
// Dependencies are events: the copy-in stream first waits for the work the
// caller had already queued on `stream`; a buffer is refilled only after the
// copy-out of the chunk that last used it has finished; at the end `stream`
// waits for the last copy-out, so that synchronising `stream` covers the
// whole call.  The streams and events are created once per device (on the
// first call, which should therefore come before any stream capture) and
// shared by all calls on that device; a mutex serialises the enqueueing, so
// concurrent calls are correct (they queue behind one another on the shared
// copy streams).
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/addln.h"
#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBufs = 2;                       // device chunk buffers
constexpr int64_t kChunkBytes = 4ll << 20;     // of X per chunk (about)
constexpr int64_t kAlign = 256;

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t loaded[kBufs] = {}, computed[kBufs] = {}, drained[kBufs] = {};
};

std::mutex g_mu;
Pipe g_pipe[kMaxDevices];
std::atomic<int> g_last_mode{0};

int64_t elem_bytes(int dtype) { return dtype == ADDLN_FP32 ? 4 : 2; }

int64_t round_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device workspace layout of one call.
struct Layout {
  int64_t chunk_rows = 0;
  int64_t gamma = 0, beta = 0;
  int64_t x[kBufs] = {}, r[kBufs] = {}, y[kBufs] = {}, a[kBufs] = {}, mean[kBufs] = {},
          rstd[kBufs] = {};
  int64_t total = 0;
};

Layout layout_of(int64_t rows, int64_t H, int dtype, bool want_a, bool want_stats) {
  Layout L;
  const int64_t row_bytes = H * elem_bytes(dtype);
  int64_t cr = kChunkBytes / row_bytes;
  if (cr < 1) cr = 1;
  if (cr > rows) cr = rows;
  L.chunk_rows = cr;
  const int64_t t = round_up(cr * row_bytes), s = round_up(cr * 4);
  int64_t o = 0;
  L.gamma = o;
  o += round_up(H * 4);
  L.beta = o;
  o += round_up(H * 4);
  for (int b = 0; b < kBufs; ++b) {
    L.x[b] = o;
    o += t;
    L.r[b] = o;
    o += t;
    L.y[b] = o;
    o += t;
    if (want_a) {
      L.a[b] = o;
      o += t;
    }
    if (want_stats) {
      L.mean[b] = o;
      o += s;
      L.rstd[b] = o;
      o += s;
    }
  }
  L.total = o;
  return L;
}

// [p, p + n) of two host buffers: identical or disjoint (true), or partly
// overlapping (false).
bool same_or_apart(const void* a, const void* b, int64_t n) {
  if (a == nullptr || b == nullptr || a == b) return true;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x + static_cast<uintptr_t>(n) <= y || y + static_cast<uintptr_t>(n) <= x;
}

bool apart(const void* a, int64_t na, const void* b, int64_t nb) {
  if (a == nullptr || b == nullptr) return true;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x + static_cast<uintptr_t>(na) <= y || y + static_cast<uintptr_t>(nb) <= x;
}

// Device address of the host range [p, p + n) when the device can reach any
// host address (pageable memory access) and both ends of the range are mapped
// pinned memory at device addresses n - 1 apart; otherwise nullptr.
void* mapped_range(const void* p, int64_t n, bool device_reaches_host) {
  if (!device_reaches_host || p == nullptr || n <= 0) return nullptr;
  cudaPointerAttributes a{}, b{};
  const char* last = static_cast<const char*>(p) + (n - 1);
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess ||
      cudaPointerGetAttributes(&b, last) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer is not an error of this call
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || b.type != cudaMemoryTypeHost || a.devicePointer == nullptr ||
      b.devicePointer == nullptr)
    return nullptr;
  if (static_cast<const char*>(b.devicePointer) - static_cast<const char*>(a.devicePointer) != n - 1)
    return nullptr;
  return a.devicePointer;
}

// gamma and beta from mapped host memory into the workspace: one small
// kernel instead of two copies, chained to the row kernel that reads them by
// programmatic dependent launch (it waits for the work queued before it,
// which may still be reading the workspace, before it writes).
__global__ void k_params_in(const float* g, const float* b, float* gd, float* bd, int H) {
  addln::pdl_trigger();
  addln::pdl_wait();
  const int step = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < H; i += step) {
    if (!ADDLN_IN(701, 4 * i, 4, 4 * static_cast<int64_t>(H))) continue;
    gd[i] = g[i];
    bd[i] = b[i];
  }
}

int check_shape(int64_t rows, int64_t H, int dtype) {
  if (dtype != ADDLN_FP32 && dtype != ADDLN_FP16 && dtype != ADDLN_BF16) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || H > addln_max_hidden(dtype)) return ADDLN_ERR_SHAPE;
  if (rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  return ADDLN_OK;
}

// The calling thread's device's pipe, created on first use.  Caller holds g_mu.
int pipe_of_current_device(Pipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ADDLN_ERR_CUDA;
  Pipe& p = g_pipe[dev];
  if (!p.ready) {
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) != cudaSuccess)
      return ADDLN_ERR_CUDA;
    for (int b = 0; b < kBufs; ++b)
      if (cudaEventCreateWithFlags(&p.loaded[b], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.computed[b], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.drained[b], cudaEventDisableTiming) != cudaSuccess)
        return ADDLN_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return ADDLN_OK;
}

}  // namespace

namespace addln {
ADDLN_BOUNDS_READER(read_bounds_host)
}  // namespace addln

extern "C" int64_t add_layernorm_fwd_host_workspace_size(int64_t rows, int64_t H, int dtype,
                                                        int want_resid, int want_stats) {
  const int rc = check_shape(rows, H, dtype);
  if (rc != ADDLN_OK) return rc;
  if (rows == 0) return 0;
  return layout_of(rows, H, dtype, want_resid != 0, want_stats != 0).total;
}

extern "C" int add_layernorm_fwd_host(const void* x_host, const void* r_host,
                                      const float* gamma_host, const float* beta_host,
                                      void* y_host, void* resid_out_host, float* mean_host,
                                      float* rstd_host, int64_t rows, int64_t H, float eps,
                                      int dtype, void* workspace, int64_t workspace_bytes,
                                      void* stream) {
  int rc = check_shape(rows, H, dtype);
  if (rc != ADDLN_OK) return rc;
  if (!(eps >= 0.f) || eps > 3.4e38f) return ADDLN_ERR_EPS;
  if (rows == 0) return ADDLN_OK;
  if (!x_host || !r_host || !gamma_host || !beta_host || !y_host) return ADDLN_ERR_NULL;
  const bool want_a = resid_out_host != nullptr;
  const bool want_stats = mean_host != nullptr || rstd_host != nullptr;
  {
    // Y and A may be X or R exactly (each chunk is copied in before its
    // outputs are copied out) or lie apart from every other buffer.
    const int64_t tb = rows * H * elem_bytes(dtype);
    const void* ins[2] = {x_host, r_host};
    const void* outs[2] = {y_host, resid_out_host};
    for (const void* o : outs)
      for (const void* i : ins)
        if (!same_or_apart(o, i, tb)) return ADDLN_ERR_ALIAS;
    if (want_a && (y_host == resid_out_host || !apart(y_host, tb, resid_out_host, tb)))
      return ADDLN_ERR_ALIAS;
    const void* small[4] = {gamma_host, beta_host, mean_host, rstd_host};
    const int64_t sn[4] = {H * 4, H * 4, rows * 4, rows * 4};
    for (int k = 2; k < 4; ++k) {
      const void* big[4] = {x_host, r_host, y_host, resid_out_host};
      for (const void* b : big)
        if (!apart(small[k], sn[k], b, tb)) return ADDLN_ERR_ALIAS;
      for (int j = 0; j < 4; ++j)
        if (j != k && !apart(small[k], sn[k], small[j], sn[j])) return ADDLN_ERR_ALIAS;
    }
  }
  const Layout L = layout_of(rows, H, dtype, want_a, want_stats);
  if (workspace == nullptr || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return ADDLN_ERR_WORKSPACE;

  // Zero-copy: when X, R and every output are mapped pinned host memory with
  // 16-byte aligned rows, the kernel reads and writes them in place over the
  // host link (one pass each way, both directions at once, no staging and no
  // pipeline fill or drain); only gamma and beta go to the device first (by
  // k_params_in when they are mapped too, else by two copies).  Rows over
  // 1024 then take the CTA kernel with 16-byte loads: no bulk copy reads host
  // memory.
  {
    int dev = 0, reach = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reach, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess)
      return ADDLN_ERR_CUDA;
    const int64_t tb = rows * H * elem_bytes(dtype);
    void* dx = mapped_range(x_host, tb, reach != 0);
    void* dr = mapped_range(r_host, tb, reach != 0);
    void* dy = mapped_range(y_host, tb, reach != 0);
    void* da = want_a ? mapped_range(resid_out_host, tb, reach != 0) : nullptr;
    void* dm = mean_host ? mapped_range(mean_host, rows * 4, reach != 0) : nullptr;
    void* ds = rstd_host ? mapped_range(rstd_host, rows * 4, reach != 0) : nullptr;
    auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const bool all = dx && dr && dy && (!want_a || da) && (!mean_host || dm) && (!rstd_host || ds);
    if (all && (H * elem_bytes(dtype)) % 16 == 0 && a16(dx) && a16(dr) && a16(dy) &&
        (!da || a16(da))) {
      cudaStream_t s = static_cast<cudaStream_t>(stream);
      char* ws = static_cast<char*>(workspace);
      float* gd = reinterpret_cast<float*>(ws + L.gamma);
      float* bd = reinterpret_cast<float*>(ws + L.beta);
      const void* dg = mapped_range(gamma_host, H * 4, true);
      const void* db = mapped_range(beta_host, H * 4, true);
      if (dg && db) {
        constexpr int kThreads = 256;
        const int blocks = static_cast<int>((H + kThreads - 1) / kThreads);
        if (addln::launch_kernel(k_params_in, dim3(blocks), dim3(kThreads), 0, s,
                                 addln::pdl_enabled(), static_cast<const float*>(dg),
                                 static_cast<const float*>(db), gd, bd,
                                 static_cast<int>(H)) != cudaSuccess)
          return ADDLN_ERR_LAUNCH;
      } else if (cudaMemcpyAsync(gd, gamma_host, H * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                 cudaMemcpyAsync(bd, beta_host, H * 4, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        return ADDLN_ERR_CUDA;
      }
      const int out = addln::fwd_rows_mapped(dx, dr, gd, bd, dy, da, static_cast<float*>(dm),
                                             static_cast<float*>(ds), rows, H, eps, dtype, stream);
      if (out == ADDLN_OK) g_last_mode.store(ADDLN_HOST_MAPPED, std::memory_order_relaxed);
      return out;
    }
  }

  std::lock_guard<std::mutex> guard(g_mu);
  Pipe* pp = nullptr;
  rc = pipe_of_current_device(&pp);
  if (rc != ADDLN_OK) return rc;
  Pipe& P = *pp;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int64_t row_bytes = H * elem_bytes(dtype);
  auto h2d = cudaMemcpyHostToDevice;
  auto d2h = cudaMemcpyDeviceToHost;
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };

  // start after the caller's queued work; gamma, beta first
  chk(cudaEventRecord(P.start, s));
  chk(cudaStreamWaitEvent(P.in, P.start, 0));
  chk(cudaMemcpyAsync(ws + L.gamma, gamma_host, H * 4, h2d, P.in));
  chk(cudaMemcpyAsync(ws + L.beta, beta_host, H * 4, h2d, P.in));

  int last = 0;
  for (int64_t r0 = 0, c = 0; ok && r0 < rows; r0 += L.chunk_rows, ++c) {
    const int b = static_cast<int>(c % kBufs);
    const int64_t n = rows - r0 < L.chunk_rows ? rows - r0 : L.chunk_rows;
    const int64_t off = r0 * row_bytes, bytes = n * row_bytes;
    // refill buffer b only once the copy-out of its previous chunk is done
    chk(cudaStreamWaitEvent(P.in, P.drained[b], 0));
    chk(cudaMemcpyAsync(ws + L.x[b], static_cast<const char*>(x_host) + off, bytes, h2d, P.in));
    chk(cudaMemcpyAsync(ws + L.r[b], static_cast<const char*>(r_host) + off, bytes, h2d, P.in));
    chk(cudaEventRecord(P.loaded[b], P.in));
    if (!ok) break;
    chk(cudaStreamWaitEvent(s, P.loaded[b], 0));
    rc = add_layernorm_fwd(ws + L.x[b], ws + L.r[b], reinterpret_cast<const float*>(ws + L.gamma),
                           reinterpret_cast<const float*>(ws + L.beta), ws + L.y[b],
                           want_a ? ws + L.a[b] : nullptr,
                           mean_host ? reinterpret_cast<float*>(ws + L.mean[b]) : nullptr,
                           rstd_host ? reinterpret_cast<float*>(ws + L.rstd[b]) : nullptr, n, H,
                           eps, dtype, stream);
    if (rc != ADDLN_OK) break;
    chk(cudaEventRecord(P.computed[b], s));
    chk(cudaStreamWaitEvent(P.out, P.computed[b], 0));
    chk(cudaMemcpyAsync(static_cast<char*>(y_host) + off, ws + L.y[b], bytes, d2h, P.out));
    if (want_a)
      chk(cudaMemcpyAsync(static_cast<char*>(resid_out_host) + off, ws + L.a[b], bytes, d2h, P.out));
    if (mean_host) chk(cudaMemcpyAsync(mean_host + r0, ws + L.mean[b], n * 4, d2h, P.out));
    if (rstd_host) chk(cudaMemcpyAsync(rstd_host + r0, ws + L.rstd[b], n * 4, d2h, P.out));
    chk(cudaEventRecord(P.drained[b], P.out));
    last = b;
  }
  // join: `stream` waits for everything queued on the copy streams
  cudaEventRecord(P.loaded[last], P.in);
  cudaStreamWaitEvent(s, P.loaded[last], 0);
  cudaEventRecord(P.drained[last], P.out);
  if (cudaStreamWaitEvent(s, P.drained[last], 0) != cudaSuccess) ok = false;
  if (rc != ADDLN_OK) return rc;
  if (!ok) return ADDLN_ERR_CUDA;
  g_last_mode.store(ADDLN_HOST_PIPELINED, std::memory_order_relaxed);
  return ADDLN_OK;
}

extern "C" int add_layernorm_fwd_host_last_mode(void) {
  return g_last_mode.load(std::memory_order_relaxed);
}
