// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-only types; no CUDA headers needed to include it.
#pragma once

#include <stdint.h>

namespace addln {

enum Dtype : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// Arguments of one row-kernel launch.  x, r, y, a are [rows, H] in the I/O
// dtype; r == nullptr means LayerNorm of x alone; a, mean, rstd optional.
struct RowArgs {
  const void* x;
  const void* r;
  const float* gamma;
  const float* beta;
  void* y;
  void* a;
  float* mean;
  float* rstd;
  int64_t rows;
  int H;
  float inv_h;  // 1/H rounded to fp32
  float eps;
  uint64_t wait_limit_ns;  // bound on mbarrier waits (TMA path)
};

// Per-device facts the dispatcher sizes grids and shared memory with.
struct DeviceInfo {
  int device;
  int sms;
  int smem_optin;  // max dynamic shared memory per block (opt-in)
  int l2_bytes;
};

struct LaunchCtx {
  void* stream;  // cudaStream_t
  DeviceInfo dev;
  int64_t grid_cap;  // 0 = one wave of resident CTAs, else min(grid_cap, rows) CTAs
  bool pdl;          // launch with programmatic stream serialisation
  int cta_threads;   // CTA-per-row kernels: threads per CTA, 0 = by H
  int stages;        // TMA path: rows staged per CTA, 0 = by shared memory
  int warp_rows = 0; // warp-per-row vector path: rows a warp takes, 0 = by shape
};

// Each launcher returns 0, or ADDLN_ERR_UNSUPPORTED when its kernel family
// cannot run these arguments, or ADDLN_ERR_LAUNCH.  `path_name` receives the
// static name of the launched kernel.

// One warp per row (H <= 1024).  vec: 16-byte vector loads (requires every
// row pointer and gamma/beta 16-byte aligned and H a multiple of the vector).
int launch_warp_row(int dtype, bool vec, const RowArgs& p, const LaunchCtx& c,
                    const char** path_name);

// One CTA per row, persistent over rows.  tma: rows staged into shared
// memory by bulk copies; otherwise 16-byte vector loads to registers.
int launch_cta_row(int dtype, bool tma, const RowArgs& p, const LaunchCtx& c,
                   const char** path_name);

// One CTA per row, element-wise loads, any alignment, H <= max.
int launch_cta_scalar(int dtype, const RowArgs& p, const LaunchCtx& c, const char** path_name);

// Whether launches use programmatic dependent launch (knob addln_set_pdl).
bool pdl_enabled();

// add_layernorm_fwd on rows in mapped host memory: plain 16-byte loads and
// stores only (no bulk copies); gamma and beta should be device memory.
int fwd_rows_mapped(const void* x, const void* r, const float* gamma, const float* beta, void* y,
                    void* resid_out, float* mean, float* rstd, int64_t rows, int64_t H, float eps,
                    int dtype, void* stream);

// A = X + R over n elements.
int launch_add(int dtype, const void* x, const void* r, void* a, int64_t n, const LaunchCtx& c);

// Row softmax: one warp per row (vec: 16-byte loads), one CTA per row with
// TMA staging, or one CTA per row with element loads.
int launch_softmax_warp(int dtype, bool vec, const RowArgs& p, const LaunchCtx& c,
                        const char** path_name);
int launch_softmax_cta(int dtype, const RowArgs& p, const LaunchCtx& c, const char** path_name);
int launch_softmax_scalar(int dtype, const RowArgs& p, const LaunchCtx& c, const char** path_name);
int read_and_clear_softmax_error(int* code);

// Bias + GELU + residual (fused) and the two extra steps of its unfused chain.
int launch_bias_gelu_residual(int dtype, const void* x, const void* r, const float* bias, void* y,
                              int64_t rows, int64_t H, const LaunchCtx& c);
int launch_bias_add(int dtype, const void* x, const float* bias, void* y, int64_t rows, int64_t H,
                    const LaunchCtx& c);
int launch_gelu(int dtype, const void* x, void* y, int64_t n, const LaunchCtx& c);

// Backward of add+LayerNorm: bytes of workspace the launch needs (its grid's
// [2][H] fp32 column partials), and the launch (row kernel, then the column
// sums when dgamma/dbeta are wanted).
int64_t bwd_workspace_bytes(int dtype, int64_t rows, int64_t H, bool vec_ok, const DeviceInfo& dev);
int launch_bwd(int dtype, const void* dy, const void* a, const float* mean, const float* rstd,
               const float* gamma, const void* dres, void* dx, float* dgamma, float* dbeta,
               int64_t rows, int64_t H, bool vec_ok, void* ws, int64_t ws_bytes,
               uint64_t wait_limit_ns, const LaunchCtx& c, const char** name);
int read_and_clear_bwd_error(int* code);

// Remembers the CUDA error behind the last ADDLN_ERR_LAUNCH / ADDLN_ERR_CUDA
// on this host thread (an int cudaError_t; 0 = none).
void note_cuda_error(int err);

// Device error word (set by a kernel whose bounded wait ran out).
int read_and_clear_device_error(void* stream, int* code);

// Checked build (-DADDLN_CHECK_BOUNDS): each translation unit's bounds word,
// read and cleared (0: no access was out of bounds; always 0 in the normal
// build, which has no word and makes no CUDA call here).
int read_bounds_rows_warp(unsigned long long* word);
int read_bounds_rows_cta(unsigned long long* word);
int read_bounds_softmax(unsigned long long* word);
int read_bounds_bgr(unsigned long long* word);
int read_bounds_add(unsigned long long* word);
int read_bounds_bwd(unsigned long long* word);
int read_bounds_host(unsigned long long* word);

// Largest H per dtype (shared memory and register budget of the CTA paths).
constexpr int64_t kMaxHidden16 = 32768;
constexpr int64_t kMaxHidden32 = 16384;

}  // namespace addln
