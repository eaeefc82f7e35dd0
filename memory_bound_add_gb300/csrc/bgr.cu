// Bias + GELU + residual, fused: Y = GELU(X + bias) + R, one read of X and R
// and one write of Y -- the single fused kernel of the BiasAdd -> GELU ->
// Residual diagram in "算子融合的收益量化".  GELU is the exact form
// v * Phi(v) = v/2 * (1 + erf(v / sqrt 2)), erf by the published rational
// approximation below (absolute error below 1.5e-7).  bias is fp32 [H],
// broadcast along rows.
//
// Also the two extra steps of the diagram's unfused chain, each its own
// kernel with its own HBM round trip: T = X + bias and U = GELU(T) (the third
// step, Y = U + R, is add_fwd).
//
// All kernels stream 16-byte vectors grid-stride with up to four
// independent vectors in flight per thread (fewer on short tensors, so that
// the whole grid has work); element accesses serve misaligned buffers and
// rows that are not whole vectors.
#include "../../include/addln.h"
#include "common.cuh"

namespace addln {
namespace ew {

constexpr int kThreads = 256;

// GELU(v) = v/2 * (1 + erf(v / sqrt 2)).  erf from Abramowitz and Stegun,
// Handbook of Mathematical Functions (1964), formula 7.1.26 (after Hastings):
// for a >= 0, erfc(a) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^(-a^2)
// with t = 1 / (1 + p a), |error| <= 1.5e-7.  With z = v / sqrt 2 and
// a = |z|, 1 + erf(z) is erfc(a) for z < 0 (no cancellation on the negative
// side) and 2 - erfc(a) for z >= 0.  One fast reciprocal, one hardware
// exponential and a degree-5 Horner polynomial.
__device__ __forceinline__ float gelu(float v) {
  constexpr float p = 0.3275911f;
  constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                  a4 = -1.453152027f, a5 = 1.061405429f;
  const float a = fabsf(v) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(p, a, 1.0f));
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, a5, a4), a3), a2), a1);
  const float erfc_a = poly * __expf(-a * a);
  return 0.5f * v * (v >= 0.f ? 2.0f - erfc_a : erfc_a);
}

// The same GELU on a pair of values, in fp32 pair arithmetic: every step but
// the reciprocal, the exponential and the sign select covers both values in
// one instruction.  exp(-a^2) = 2^(-a^2 log2 e) by the hardware base-2
// exponential (PTX ex2.approx.ftz: results below 2^-126 flush to zero,
// where the GELU term is far below any output's rounding).
__device__ __forceinline__ float ex2_ftz(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

__device__ __forceinline__ float2 gelu2(float2 v) {
  constexpr float p = 0.3275911f;
  constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                  a4 = -1.453152027f, a5 = 1.061405429f;
  constexpr float kNegLog2e = -1.4426950408889634f;
  const float2 a = mul2(make_float2(fabsf(v.x), fabsf(v.y)), dup2(0.70710678118654752f));
  const float2 den = fma2(dup2(p), a, dup2(1.0f));
  const float2 t = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
  float2 q = fma2(t, dup2(a5), dup2(a4));
  q = fma2(t, q, dup2(a3));
  q = fma2(t, q, dup2(a2));
  q = fma2(t, q, dup2(a1));
  const float2 arg = mul2(mul2(a, a), dup2(kNegLog2e));
  const float2 erfc_a = mul2(mul2(t, q), make_float2(ex2_ftz(arg.x), ex2_ftz(arg.y)));
  const float2 two_minus = add2(dup2(2.0f), make_float2(-erfc_a.x, -erfc_a.y));
  const float2 w = make_float2(v.x >= 0.f ? two_minus.x : erfc_a.x, v.y >= 0.f ? two_minus.y : erfc_a.y);
  return mul2(mul2(dup2(0.5f), v), w);
}

// What each element becomes.  kBgr: GELU(x + b) + r; kBias: x + b; kGelu: GELU(x).
enum Kind { kBgr = 0, kBias = 1, kGelu = 2 };

template <int KIND>
__device__ __forceinline__ float2 apply2(float2 x, float2 r, float2 b) {
  if constexpr (KIND == kBgr) return add2(gelu2(add2(x, b)), r);
  if constexpr (KIND == kBias) return add2(x, b);
  return gelu2(x);
}

template <int KIND>
__device__ __forceinline__ float apply(float x, float r, float b) {
  if constexpr (KIND == kBgr) return gelu(x + b) + r;
  if constexpr (KIND == kBias) return x + b;
  return gelu(x);
}

// Vector path: every buffer 16-byte aligned, H a multiple of the vector width
// (so a vector never straddles two rows and its bias slice is aligned).
template <int DT, int KIND, int UNROLL>
__global__ void __launch_bounds__(kThreads) k_ew_vec(const void* x, const void* r, const float* bias,
                                                     void* y, int64_t nvec, int64_t hvec) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr bool HAS_R = KIND == kBgr;
  constexpr bool HAS_B = KIND != kGelu;
  const uint4* xv = static_cast<const uint4*>(x);
  const uint4* rv = static_cast<const uint4*>(r);
  uint4* yv = static_cast<uint4*>(y);
  // while the previous kernel may still be finishing, ask L2 for the 512-byte
  // chunks of X and R this warp reads first (a hint only; nothing is read
  // before the wait below); only for short launches (at most eight steps of
  // the grid-stride loop), as on long ones it measured slower
  if ((threadIdx.x & 31) == 0 &&
      nvec <= 8 * static_cast<int64_t>(gridDim.x) * kThreads * UNROLL) {
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kThreads * UNROLL + threadIdx.x;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = w0 + static_cast<int64_t>(u) * kThreads;
      if (i + 32 <= nvec && ADDLN_IN(401, i * 16, 512, nvec * 16)) {
        prefetch_l2(xv + i, 512u);
        if constexpr (HAS_R) prefetch_l2(rv + i, 512u);
      }
    }
  }
  pdl_trigger();
  pdl_wait();
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads * UNROLL;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kThreads * UNROLL + threadIdx.x;
  // bias column of vector i is i % hvec; advanced incrementally (one add and
  // at most one subtraction a vector) instead of a 64-bit remainder each time
  const int64_t tmod = kThreads % hvec, smod = step % hvec;
  int64_t col0 = HAS_B ? first % hvec : 0;
  for (int64_t i0 = first; i0 < nvec; i0 += step) {
    int64_t cols[UNROLL];
    if constexpr (HAS_B) {
      int64_t cc = col0;
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        cols[u] = cc;
        cc += tmod;
        if (cc >= hvec) cc -= hvec;
      }
      col0 += smod;
      if (col0 >= hvec) col0 -= hvec;
    }
    uint4 xs[UNROLL], rs[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * kThreads;
      if (i < nvec && ADDLN_IN(402, i * 16, 16, nvec * 16)) {
        xs[u] = ld_stream_v4(xv + i);
        if constexpr (HAS_R) rs[u] = ld_stream_v4(rv + i);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * kThreads;
      if (i < nvec) {
        constexpr int P = VEC / 2;
        float2 f[P], g[P], b[P];
        IO::to_pairs(xs[u], f);
        if constexpr (HAS_R) IO::to_pairs(rs[u], g);
        if constexpr (HAS_B) {
          const float* bp = bias + cols[u] * VEC;
#pragma unroll
          for (int q = 0; q < VEC / 4; ++q) {
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ADDLN_IN(403, 4 * (cols[u] * VEC + 4 * q), 16, 4 * hvec * VEC)) t = ld_param_f4(bp + 4 * q);
            b[2 * q] = make_float2(t.x, t.y);
            b[2 * q + 1] = make_float2(t.z, t.w);
          }
        }
#pragma unroll
        for (int q = 0; q < P; ++q)
          f[q] = apply2<KIND>(f[q], HAS_R ? g[q] : dup2(0.f), HAS_B ? b[q] : dup2(0.f));
        if (ADDLN_IN(404, i * 16, 16, nvec * 16)) st_stream_v4(yv + i, IO::from_pairs(f));
      }
    }
  }
}

// Element path: any alignment and any H.
template <int DT, int KIND>
__global__ void __launch_bounds__(kThreads) k_ew_scalar(const void* x, const void* r,
                                                        const float* bias, void* y, int64_t n,
                                                        int64_t H) {
  using IO = Io<DT>;
  pdl_trigger();
  pdl_wait();
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  // the bias column k % H, carried along (step % H < H, so one wrap at most)
  const int64_t smod = KIND != kGelu ? step % H : 0;
  int64_t col = KIND != kGelu ? first % H : 0;
  for (int64_t k = first; k < n; k += step) {
    const bool okk = ADDLN_IN(405, k * IO::kBytes, IO::kBytes, n * IO::kBytes);
    const bool okb = KIND == kGelu || ADDLN_IN(406, 4 * col, 4, 4 * H);
    const float xv = okk ? IO::load1(x, k) : 0.f;
    const float rv = KIND == kBgr && okk ? IO::load1(r, k) : 0.f;
    const float bv = KIND != kGelu && okb ? __ldg(bias + col) : 0.f;
    if (okk) IO::store1(y, k, apply<KIND>(xv, rv, bv));
    if (KIND != kGelu) {
      col += smod;
      if (col >= H) col -= H;
    }
  }
}

template <int DT, int KIND>
int launch_t(const void* x, const void* r, const float* bias, void* y, int64_t rows, int64_t H,
             const LaunchCtx& c) {
  constexpr int VEC = Io<DT>::kVec;
  const int64_t n = rows * H;
  auto al = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const int64_t max_blocks = static_cast<int64_t>(c.dev.sms) * (2048 / kThreads);
  cudaError_t e;
  if (H % VEC == 0 && al(x) && al(r) && al(y) && al(bias)) {
    const int64_t nvec = n / VEC;
    // vectors a thread keeps in flight: 4 for long tensors; fewer when a
    // full grid would give each thread only a few vectors, so that every
    // resident thread has work and its loads, arithmetic and stores are not
    // one serial chain (1 up to 2 vectors a resident thread, 2 up to 32)
    const int64_t resident = max_blocks * kThreads;
    const int U = nvec <= 2 * resident ? 1 : nvec <= 32 * resident ? 2 : 4;
    int64_t blocks = (nvec + kThreads * U - 1) / (kThreads * U);
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    const dim3 grid(static_cast<unsigned>(blocks));
    e = U == 1   ? launch_kernel(k_ew_vec<DT, KIND, 1>, grid, dim3(kThreads), 0, c.stream, c.pdl, x, r,
                                 bias, y, nvec, H / VEC)
        : U == 2 ? launch_kernel(k_ew_vec<DT, KIND, 2>, grid, dim3(kThreads), 0, c.stream, c.pdl, x, r,
                                 bias, y, nvec, H / VEC)
                 : launch_kernel(k_ew_vec<DT, KIND, 4>, grid, dim3(kThreads), 0, c.stream, c.pdl, x, r,
                                 bias, y, nvec, H / VEC);
  } else {
    int64_t blocks = (n + kThreads - 1) / kThreads;
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    e = launch_kernel(k_ew_scalar<DT, KIND>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                      c.stream, c.pdl, x, r, bias, y, n, H);
  }
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

template <int KIND>
int launch_kind(int dtype, const void* x, const void* r, const float* bias, void* y, int64_t rows,
                int64_t H, const LaunchCtx& c) {
  switch (dtype) {
    case kF32: return launch_t<kF32, KIND>(x, r, bias, y, rows, H, c);
    case kF16: return launch_t<kF16, KIND>(x, r, bias, y, rows, H, c);
    case kBF16: return launch_t<kBF16, KIND>(x, r, bias, y, rows, H, c);
    default: return ADDLN_ERR_DTYPE;
  }
}

}  // namespace ew

ADDLN_BOUNDS_READER(read_bounds_bgr)

int launch_bias_gelu_residual(int dtype, const void* x, const void* r, const float* bias, void* y,
                              int64_t rows, int64_t H, const LaunchCtx& c) {
  return ew::launch_kind<ew::kBgr>(dtype, x, r, bias, y, rows, H, c);
}

int launch_bias_add(int dtype, const void* x, const float* bias, void* y, int64_t rows, int64_t H,
                    const LaunchCtx& c) {
  return ew::launch_kind<ew::kBias>(dtype, x, nullptr, bias, y, rows, H, c);
}

int launch_gelu(int dtype, const void* x, void* y, int64_t n, const LaunchCtx& c) {
  return ew::launch_kind<ew::kGelu>(dtype, x, nullptr, nullptr, y, 1, n, c);
}

}  // namespace addln
