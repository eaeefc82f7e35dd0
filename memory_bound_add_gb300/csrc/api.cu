// C-ABI entry points declared in include/addln.h: argument checks (all of
// them before the first CUDA call), the alias rules, device facts for grid
// sizing, and the choice of kernel path.
//
// Path choice (a per-call decision from H, dtype, alignment and the device's
// SM count and shared memory, in the spirit of the device-attribute-driven
// tiling of "融合计算范式对比", migration notes item 4):
//   H <= 1024, 16-byte aligned rows        -> one warp per row, vector loads
//   H <= 1024, otherwise                   -> one warp per row, element loads
//   H > 1024,  16-byte aligned rows        -> one CTA per row, TMA bulk staging
//   H > 1024,  otherwise                   -> one CTA per row, element loads
#include <math.h>

#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/addln.h"
#include "launch.h"

using addln::DeviceInfo;
using addln::LaunchCtx;
using addln::RowArgs;

namespace {

std::atomic<int> g_force_path{ADDLN_PATH_AUTO};
std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};
std::atomic<int64_t> g_grid_cap{0};
std::atomic<int> g_pdl{1};
std::atomic<int> g_cta_threads{0};
std::atomic<int> g_stages{0};
std::atomic<int> g_warp_rows{0};
std::atomic<uint64_t> g_bounds_violation{0};
thread_local const char* g_last_path = "none";
thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {};

int elem_bytes(int dtype) { return dtype == ADDLN_FP32 ? 4 : 2; }

bool valid_dtype(int dtype) {
  return dtype == ADDLN_FP32 || dtype == ADDLN_FP16 || dtype == ADDLN_BF16;
}

int64_t max_hidden(int dtype) {
  return dtype == ADDLN_FP32 ? addln::kMaxHidden32 : addln::kMaxHidden16;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
  bool present;
};
Range range_of(const void* p, int64_t bytes) {
  Range r;
  r.present = p != nullptr && bytes > 0;
  r.lo = reinterpret_cast<uintptr_t>(p);
  r.hi = r.lo + static_cast<uintptr_t>(bytes);
  return r;
}
bool overlap(const Range& a, const Range& b) {
  return a.present && b.present && a.lo < b.hi && b.lo < a.hi;
}
// An output may coincide exactly with an input of the same size (in place).
bool bad_pair(const Range& out, const Range& in, bool in_place_ok) {
  if (!overlap(out, in)) return false;
  return !(in_place_ok && out.lo == in.lo && out.hi == in.hi);
}

int check_rows_args(const void* x, const void* r, bool need_r, const float* gamma,
                    const float* beta, void* y, void* a, float* mean, float* rstd, int64_t rows,
                    int64_t H, float eps, int dtype) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || H > max_hidden(dtype)) return ADDLN_ERR_SHAPE;
  if (rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return ADDLN_ERR_EPS;
  if (rows == 0) return ADDLN_OK;
  if (!x || (need_r && !r) || !gamma || !beta || !y) return ADDLN_ERR_NULL;

  const int64_t tb = rows * H * elem_bytes(dtype);
  const Range rx = range_of(x, tb), rr = range_of(need_r ? r : nullptr, tb);
  const Range rg = range_of(gamma, H * 4), rbt = range_of(beta, H * 4);
  const Range ry = range_of(y, tb), ra = range_of(a, tb);
  const Range rm = range_of(mean, rows * 4), rs = range_of(rstd, rows * 4);
  // outputs against inputs
  const Range outs[4] = {ry, ra, rm, rs};
  for (int i = 0; i < 4; ++i) {
    const bool tensor_out = i < 2;
    if (bad_pair(outs[i], rx, tensor_out) || bad_pair(outs[i], rr, tensor_out) ||
        bad_pair(outs[i], rg, false) || bad_pair(outs[i], rbt, false))
      return ADDLN_ERR_ALIAS;
  }
  // outputs against each other
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return ADDLN_ERR_ALIAS;
  return ADDLN_OK;
}

int device_info(DeviceInfo* out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0) return ADDLN_ERR_CUDA;
  if (d < kMaxDevices) {
    std::lock_guard<std::mutex> g(g_dev_mu);
    if (g_dev_ok[d]) {
      *out = g_dev[d];
      return ADDLN_OK;
    }
  }
  DeviceInfo info{};
  info.device = d;
  if (cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
      cudaDeviceGetAttribute(&info.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&info.l2_bytes, cudaDevAttrL2CacheSize, d) != cudaSuccess)
    return ADDLN_ERR_CUDA;
  if (d < kMaxDevices) {
    std::lock_guard<std::mutex> g(g_dev_mu);
    g_dev[d] = info;
    g_dev_ok[d] = true;
  }
  *out = info;
  return ADDLN_OK;
}

// allow_tma false: rows longer than 1024 take the CTA kernel with 16-byte
// loads to registers instead of bulk copies (for rows that live in mapped
// host memory, which only plain loads and stores touch).
int run_rows(const RowArgs& p, int dtype, void* stream, bool allow_tma = true) {
  LaunchCtx c;
  c.stream = stream;
  c.grid_cap = g_grid_cap.load(std::memory_order_relaxed);
  c.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  c.cta_threads = g_cta_threads.load(std::memory_order_relaxed);
  c.stages = g_stages.load(std::memory_order_relaxed);
  c.warp_rows = g_warp_rows.load(std::memory_order_relaxed);
  const int rc = device_info(&c.dev);
  if (rc != ADDLN_OK) return rc;

  const int64_t row_bytes = static_cast<int64_t>(p.H) * elem_bytes(dtype);
  const bool vec_ok = row_bytes % 16 == 0 && aligned16(p.x) && (!p.r || aligned16(p.r)) &&
                      aligned16(p.y) && (!p.a || aligned16(p.a)) && aligned16(p.gamma) &&
                      aligned16(p.beta);
  int path = g_force_path.load(std::memory_order_relaxed);
  if (path == ADDLN_PATH_AUTO) {
    if (p.H <= 1024)
      path = vec_ok ? ADDLN_PATH_WARP_VEC : ADDLN_PATH_SCALAR;
    else
      path = vec_ok ? ADDLN_PATH_CTA_TMA : ADDLN_PATH_SCALAR;
  }
  if (!allow_tma && path == ADDLN_PATH_CTA_TMA) path = ADDLN_PATH_CTA_VEC;
  const char* name = "none";
  int out;
  switch (path) {
    case ADDLN_PATH_WARP_VEC:
      if (!vec_ok || p.H > 1024) return ADDLN_ERR_UNSUPPORTED;
      out = addln::launch_warp_row(dtype, true, p, c, &name);
      break;
    case ADDLN_PATH_CTA_TMA:
    case ADDLN_PATH_CTA_VEC:
      if (!vec_ok) return ADDLN_ERR_UNSUPPORTED;
      out = addln::launch_cta_row(dtype, path == ADDLN_PATH_CTA_TMA, p, c, &name);
      break;
    case ADDLN_PATH_SCALAR:
      out = p.H <= 1024 ? addln::launch_warp_row(dtype, false, p, c, &name)
                        : addln::launch_cta_scalar(dtype, p, c, &name);
      break;
    default:
      return ADDLN_ERR_UNSUPPORTED;
  }
  if (out == ADDLN_OK) g_last_path = name;
  return out;
}

int run_softmax(const RowArgs& p, int dtype, void* stream) {
  LaunchCtx c;
  c.stream = stream;
  c.grid_cap = g_grid_cap.load(std::memory_order_relaxed);
  c.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  c.cta_threads = g_cta_threads.load(std::memory_order_relaxed);
  c.stages = 0;
  const int rc = device_info(&c.dev);
  if (rc != ADDLN_OK) return rc;
  const int64_t row_bytes = static_cast<int64_t>(p.H) * elem_bytes(dtype);
  const bool vec_ok = row_bytes % 16 == 0 && aligned16(p.x) && aligned16(p.y);
  int path = g_force_path.load(std::memory_order_relaxed);
  if (path == ADDLN_PATH_AUTO) {
    if (p.H <= 1024)
      path = vec_ok ? ADDLN_PATH_WARP_VEC : ADDLN_PATH_SCALAR;
    else
      path = vec_ok ? ADDLN_PATH_CTA_TMA : ADDLN_PATH_SCALAR;
  }
  const char* name = "none";
  int out;
  switch (path) {
    case ADDLN_PATH_WARP_VEC:
      if (!vec_ok || p.H > 1024) return ADDLN_ERR_UNSUPPORTED;
      out = addln::launch_softmax_warp(dtype, true, p, c, &name);
      break;
    case ADDLN_PATH_CTA_TMA:
      if (!vec_ok) return ADDLN_ERR_UNSUPPORTED;
      out = addln::launch_softmax_cta(dtype, p, c, &name);
      break;
    case ADDLN_PATH_SCALAR:
      out = p.H <= 1024 ? addln::launch_softmax_warp(dtype, false, p, c, &name)
                        : addln::launch_softmax_scalar(dtype, p, c, &name);
      break;
    default:
      return ADDLN_ERR_UNSUPPORTED;
  }
  if (out == ADDLN_OK) g_last_path = name;
  return out;
}

}  // namespace

void addln::note_cuda_error(int err) { g_last_cuda_error = err; }

extern "C" {

int softmax_fwd(const void* x, void* y, int64_t rows, int64_t H, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || H > max_hidden(dtype)) return ADDLN_ERR_SHAPE;
  if (rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  if (rows == 0) return ADDLN_OK;
  if (!x || !y) return ADDLN_ERR_NULL;
  const int64_t tb = rows * H * elem_bytes(dtype);
  if (bad_pair(range_of(y, tb), range_of(x, tb), true)) return ADDLN_ERR_ALIAS;
  RowArgs p{x, nullptr, nullptr, nullptr, y, nullptr, nullptr, nullptr, rows,
            static_cast<int>(H), 0.f, 0.f, g_wait_limit_ns.load(std::memory_order_relaxed)};
  return run_softmax(p, dtype, stream);
}

int add_layernorm_fwd(const void* x, const void* r, const float* gamma, const float* beta, void* y,
                      void* resid_out, float* mean, float* rstd, int64_t rows, int64_t H,
                      float eps, int dtype, void* stream) {
  int rc = check_rows_args(x, r, true, gamma, beta, y, resid_out, mean, rstd, rows, H, eps, dtype);
  if (rc != ADDLN_OK || rows == 0) return rc;
  RowArgs p{x, r, gamma, beta, y, resid_out, mean, rstd, rows, static_cast<int>(H),
            static_cast<float>(1.0 / static_cast<double>(H)), eps,
            g_wait_limit_ns.load(std::memory_order_relaxed)};
  return run_rows(p, dtype, stream);
}

int layernorm_fwd(const void* a, const float* gamma, const float* beta, void* y, float* mean,
                  float* rstd, int64_t rows, int64_t H, float eps, int dtype, void* stream) {
  int rc = check_rows_args(a, nullptr, false, gamma, beta, y, nullptr, mean, rstd, rows, H, eps,
                           dtype);
  if (rc != ADDLN_OK || rows == 0) return rc;
  RowArgs p{a, nullptr, gamma, beta, y, nullptr, mean, rstd, rows, static_cast<int>(H),
            static_cast<float>(1.0 / static_cast<double>(H)), eps,
            g_wait_limit_ns.load(std::memory_order_relaxed)};
  return run_rows(p, dtype, stream);
}

namespace {
int plain_ctx(void* stream, LaunchCtx* c) {
  c->stream = stream;
  c->grid_cap = 0;
  c->pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  c->cta_threads = 0;
  c->stages = 0;
  return device_info(&c->dev);
}
}  // namespace

int bias_gelu_residual_fwd(const void* x, const void* r, const float* bias, void* y, int64_t rows,
                           int64_t H, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  if (rows == 0) return ADDLN_OK;
  if (!x || !r || !bias || !y) return ADDLN_ERR_NULL;
  const int64_t tb = rows * H * elem_bytes(dtype);
  const Range ry = range_of(y, tb);
  if (bad_pair(ry, range_of(x, tb), true) || bad_pair(ry, range_of(r, tb), true) ||
      bad_pair(ry, range_of(bias, H * 4), false))
    return ADDLN_ERR_ALIAS;
  LaunchCtx c;
  const int rc = plain_ctx(stream, &c);
  if (rc != ADDLN_OK) return rc;
  return addln::launch_bias_gelu_residual(dtype, x, r, bias, y, rows, H, c);
}

int bias_add_fwd(const void* x, const float* bias, void* t, int64_t rows, int64_t H, int dtype,
                 void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || rows > INT64_MAX / (H * 4)) return ADDLN_ERR_SHAPE;
  if (rows == 0) return ADDLN_OK;
  if (!x || !bias || !t) return ADDLN_ERR_NULL;
  const int64_t tb = rows * H * elem_bytes(dtype);
  const Range rt = range_of(t, tb);
  if (bad_pair(rt, range_of(x, tb), true) || bad_pair(rt, range_of(bias, H * 4), false))
    return ADDLN_ERR_ALIAS;
  LaunchCtx c;
  const int rc = plain_ctx(stream, &c);
  if (rc != ADDLN_OK) return rc;
  return addln::launch_bias_add(dtype, x, bias, t, rows, H, c);
}

int gelu_fwd(const void* x, void* u, int64_t n, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (n < 0 || n > INT64_MAX / 4) return ADDLN_ERR_SHAPE;
  if (n == 0) return ADDLN_OK;
  if (!x || !u) return ADDLN_ERR_NULL;
  const int64_t tb = n * elem_bytes(dtype);
  if (bad_pair(range_of(u, tb), range_of(x, tb), true)) return ADDLN_ERR_ALIAS;
  LaunchCtx c;
  const int rc = plain_ctx(stream, &c);
  if (rc != ADDLN_OK) return rc;
  return addln::launch_gelu(dtype, x, u, n, c);
}

int64_t add_layernorm_bwd_workspace_size(int64_t rows, int64_t H, int dtype) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || H > max_hidden(dtype) || rows > INT64_MAX / (H * 4))
    return ADDLN_ERR_SHAPE;
  if (rows == 0) return 0;
  DeviceInfo dev;
  const int rc = device_info(&dev);
  if (rc != ADDLN_OK) return rc;
  // the larger of the vector and the element plan (the pointers decide
  // later); a plan that cannot run these rows at all (the element path above
  // its shared-memory limit) does not count
  const int64_t v = addln::bwd_workspace_bytes(dtype, rows, H, true, dev);
  const int64_t s = addln::bwd_workspace_bytes(dtype, rows, H, false, dev);
  if (v < 0 && v != ADDLN_ERR_UNSUPPORTED) return v;
  if (s < 0 && s != ADDLN_ERR_UNSUPPORTED) return s;
  if (v < 0 && s < 0) return ADDLN_ERR_UNSUPPORTED;
  return v > s ? v : s;
}

int add_layernorm_bwd(const void* dy, const void* a, const float* mean, const float* rstd,
                      const float* gamma, const void* dres, void* dx, float* dgamma, float* dbeta,
                      int64_t rows, int64_t H, int dtype, void* workspace,
                      int64_t workspace_bytes, void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (rows < 0 || H <= 0 || H > max_hidden(dtype) || rows > INT64_MAX / (H * 4))
    return ADDLN_ERR_SHAPE;
  if ((dgamma == nullptr) != (dbeta == nullptr)) return ADDLN_ERR_NULL;
  if (workspace_bytes < 0) return ADDLN_ERR_WORKSPACE;
  if (rows == 0) {
    if (dgamma == nullptr) return ADDLN_OK;
    if (cudaMemsetAsync(dgamma, 0, H * 4, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaMemsetAsync(dbeta, 0, H * 4, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return ADDLN_ERR_CUDA;
    return ADDLN_OK;
  }
  if (!dy || !a || !mean || !rstd || !gamma || !dx) return ADDLN_ERR_NULL;
  const int64_t tb = rows * H * elem_bytes(dtype);
  const Range rdx = range_of(dx, tb);
  const Range ins[6] = {range_of(dy, tb), range_of(a, tb), range_of(dres, tb),
                        range_of(mean, rows * 4), range_of(rstd, rows * 4), range_of(gamma, H * 4)};
  for (int i = 0; i < 6; ++i)
    if (bad_pair(rdx, ins[i], i < 3)) return ADDLN_ERR_ALIAS;
  const Range rg = range_of(dgamma, H * 4), rb = range_of(dbeta, H * 4);
  const Range rw = range_of(dgamma ? workspace : nullptr, workspace_bytes);
  const Range outs[4] = {rdx, rg, rb, rw};
  for (int i = 1; i < 4; ++i) {
    for (int k = 0; k < 6; ++k)
      if (overlap(outs[i], ins[k])) return ADDLN_ERR_ALIAS;
    for (int j = 0; j < i; ++j)
      if (overlap(outs[i], outs[j])) return ADDLN_ERR_ALIAS;
  }
  LaunchCtx c;
  c.stream = stream;
  c.grid_cap = 0;
  c.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  c.cta_threads = 0;
  c.stages = g_stages.load(std::memory_order_relaxed);  // ring depth (tuning knob)
  const int rc = device_info(&c.dev);
  if (rc != ADDLN_OK) return rc;
  const int64_t row_bytes = H * elem_bytes(dtype);
  bool vec_ok = row_bytes % 16 == 0 && aligned16(dy) && aligned16(a) && aligned16(dx) &&
                (!dres || aligned16(dres)) && aligned16(gamma);
  const int force = g_force_path.load(std::memory_order_relaxed);
  if (force == ADDLN_PATH_SCALAR) vec_ok = false;
  const char* name = "none";
  const int out = addln::launch_bwd(dtype, dy, a, mean, rstd, gamma, dres, dx, dgamma, dbeta, rows,
                                    H, vec_ok, workspace, workspace_bytes,
                                    g_wait_limit_ns.load(std::memory_order_relaxed), c, &name);
  if (out == ADDLN_OK) g_last_path = name;
  return out;
}

int add_fwd(const void* x, const void* r, void* a, int64_t n, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return ADDLN_ERR_DTYPE;
  if (n < 0 || n > INT64_MAX / 4) return ADDLN_ERR_SHAPE;
  if (n == 0) return ADDLN_OK;
  if (!x || !r || !a) return ADDLN_ERR_NULL;
  const int64_t bytes = n * elem_bytes(dtype);
  const Range ra = range_of(a, bytes);
  if (bad_pair(ra, range_of(x, bytes), true) || bad_pair(ra, range_of(r, bytes), true))
    return ADDLN_ERR_ALIAS;
  LaunchCtx c;
  c.stream = stream;
  c.grid_cap = 0;
  c.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  c.cta_threads = 0;
  c.stages = 0;
  const int rc = device_info(&c.dev);
  if (rc != ADDLN_OK) return rc;
  return addln::launch_add(dtype, x, r, a, n, c);
}

const char* addln_strerror(int code) {
  switch (code) {
    case ADDLN_OK: return "success";
    case ADDLN_ERR_NULL: return "a required pointer is NULL";
    case ADDLN_ERR_SHAPE: return "invalid shape: rows/n < 0, H <= 0 or H above the maximum";
    case ADDLN_ERR_DTYPE: return "unknown dtype code";
    case ADDLN_ERR_EPS: return "eps must be finite and >= 0";
    case ADDLN_ERR_ALIAS: return "an output partially overlaps an input or another output";
    case ADDLN_ERR_LAUNCH: return "CUDA kernel launch failed";
    case ADDLN_ERR_UNSUPPORTED: return "the forced kernel path cannot run these arguments";
    case ADDLN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait on its own copy ran out";
    case ADDLN_ERR_CUDA: return "a CUDA runtime call failed";
    case ADDLN_ERR_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
    case ADDLN_ERR_BOUNDS: return "a kernel skipped an access outside its buffer (checked build)";
    default: return "unknown error code";
  }
}

int64_t addln_max_hidden(int dtype) {
  return valid_dtype(dtype) ? max_hidden(dtype) : static_cast<int64_t>(ADDLN_ERR_DTYPE);
}

int addln_get_device_error(void* stream) {
  int code = 0, code_sm = 0;
  int rc = addln::read_and_clear_device_error(stream, &code);
  if (rc != ADDLN_OK) return rc;
  rc = addln::read_and_clear_softmax_error(&code_sm);
  if (rc != ADDLN_OK) return rc;
  int code_bw = 0;
  rc = addln::read_and_clear_bwd_error(&code_bw);
  if (rc != ADDLN_OK) return rc;
  // checked build: the first out-of-bounds access any kernel met
  int (*const readers[])(unsigned long long*) = {
      addln::read_bounds_rows_warp, addln::read_bounds_rows_cta, addln::read_bounds_softmax,
      addln::read_bounds_bgr,       addln::read_bounds_add,      addln::read_bounds_bwd,
      addln::read_bounds_host};
  unsigned long long word = 0;
  for (auto f : readers) {
    unsigned long long w = 0;
    rc = f(&w);
    if (rc != ADDLN_OK) return rc;
    if (word == 0) word = w;
  }
  if (word != 0) {
    g_bounds_violation.store(word);
    return ADDLN_ERR_BOUNDS;
  }
  return code != 0 ? code : (code_sm != 0 ? code_sm : code_bw);
}

int addln_bounds_checked(void) {
#ifdef ADDLN_CHECK_BOUNDS
  return 1;
#else
  return 0;
#endif
}

uint64_t addln_bounds_violation(void) { return g_bounds_violation.load(); }

int addln_set_force_path(int path) {
  if (path < ADDLN_PATH_AUTO || path > ADDLN_PATH_SCALAR) return ADDLN_ERR_SHAPE;
  return g_force_path.exchange(path);
}

uint64_t addln_set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }

int64_t addln_set_grid_cap(int64_t ctas) { return g_grid_cap.exchange(ctas < 0 ? 0 : ctas); }

int addln_set_pdl(int on) { return g_pdl.exchange(on != 0 ? 1 : 0); }

int addln_set_cta_shape(int threads, int stages) {
  if (threads != 0 && threads != 128 && threads != 256 && threads != 512) return ADDLN_ERR_SHAPE;
  if (stages < 0 || stages > 4) return ADDLN_ERR_SHAPE;
  const int prev = g_cta_threads.exchange(threads);
  g_stages.exchange(stages);
  return prev;
}

const char* addln_last_path(void) { return g_last_path; }

int addln_set_warp_rows(int rows) {
  if (rows < 0 || rows > 2) return ADDLN_ERR_SHAPE;
  return g_warp_rows.exchange(rows);
}


const char* addln_last_cuda_error(void) {
  return g_last_cuda_error == 0 ? "none"
                                : cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda_error));
}

}  // extern "C"

// The fused forward on rows that live in mapped host memory (zero-copy):
// the same checks and kernels as add_layernorm_fwd, without bulk copies.
int addln::fwd_rows_mapped(const void* x, const void* r, const float* gamma, const float* beta,
                           void* y, void* resid_out, float* mean, float* rstd, int64_t rows,
                           int64_t H, float eps, int dtype, void* stream) {
  int rc = check_rows_args(x, r, true, gamma, beta, y, resid_out, mean, rstd, rows, H, eps, dtype);
  if (rc != ADDLN_OK || rows == 0) return rc;
  RowArgs p{x, r, gamma, beta, y, resid_out, mean, rstd, rows, static_cast<int>(H),
            static_cast<float>(1.0 / static_cast<double>(H)), eps,
            g_wait_limit_ns.load(std::memory_order_relaxed)};
  return run_rows(p, dtype, stream, false);
}

bool addln::pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }
