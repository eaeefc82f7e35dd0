// Unfused baseline, step 1: the separate residual-add kernel of
// "算子融合的收益量化" section 1 -- read X and R, write A = X + R in the I/O
// dtype (rounded to nearest-even from the fp32 sum).  Grid-stride over
// 16-byte vectors with four independent vectors per thread per step (one on
// short tensors, so that the whole grid has work); the last
// n % VEC elements (and misaligned buffers) take element accesses.
#include "../../include/addln.h"
#include "common.cuh"

namespace addln {

constexpr int kAddThreads = 256;

template <int DT, int UNROLL>
__global__ void __launch_bounds__(kAddThreads) k_add_vec(const void* x, const void* r, void* a,
                                                         int64_t nvec, int64_t n) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  const uint4* xv = static_cast<const uint4*>(x);
  const uint4* rv = static_cast<const uint4*>(r);
  uint4* av = static_cast<uint4*>(a);
  // as the fused kernel does: while the previous kernel may still be
  // finishing, ask L2 for the 512-byte chunks of X and R this warp reads
  // first (a hint only; nothing is read before the wait below), for short
  // launches (at most eight steps of the grid-stride loop)
  if ((threadIdx.x & 31) == 0 &&
      nvec <= 8 * static_cast<int64_t>(gridDim.x) * kAddThreads * UNROLL) {
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * kAddThreads * UNROLL + threadIdx.x;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = w0 + static_cast<int64_t>(u) * kAddThreads;
      if (i + 32 <= nvec && ADDLN_IN(501, i * 16, 512, n * IO::kBytes)) {
        prefetch_l2(xv + i, 512u);
        prefetch_l2(rv + i, 512u);
      }
    }
  }
  pdl_trigger();
  pdl_wait();
  const int64_t step = static_cast<int64_t>(gridDim.x) * kAddThreads * UNROLL;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * kAddThreads * UNROLL + threadIdx.x;
       i0 < nvec; i0 += step) {
    uint4 xs[UNROLL], rs[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * kAddThreads;
      if (i < nvec && ADDLN_IN(502, i * 16, 16, n * IO::kBytes)) {
        xs[u] = ld_stream_v4(xv + i);
        rs[u] = ld_stream_v4(rv + i);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + static_cast<int64_t>(u) * kAddThreads;
      if (i < nvec) {
        float f[VEC], g[VEC];
        IO::unpack(xs[u], f);
        IO::unpack(rs[u], g);
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] += g[e];
        if (ADDLN_IN(503, i * 16, 16, n * IO::kBytes)) st_stream_v4(av + i, IO::pack(f));
      }
    }
  }
  // tail elements past the last whole vector
  if (blockIdx.x == 0) {
    for (int64_t j = nvec * VEC + threadIdx.x; j < n; j += kAddThreads)
      if (ADDLN_IN(504, j * IO::kBytes, IO::kBytes, n * IO::kBytes))
        IO::store1(a, j, IO::load1(x, j) + IO::load1(r, j));
  }
}

template <int DT>
__global__ void __launch_bounds__(kAddThreads) k_add_scalar(const void* x, const void* r, void* a,
                                                            int64_t n) {
  using IO = Io<DT>;
  pdl_trigger();
  pdl_wait();
  const int64_t step = static_cast<int64_t>(gridDim.x) * kAddThreads;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * kAddThreads + threadIdx.x; j < n; j += step)
    if (ADDLN_IN(505, j * IO::kBytes, IO::kBytes, n * IO::kBytes))
      IO::store1(a, j, IO::load1(x, j) + IO::load1(r, j));
}

template <int DT>
static int launch_add_t(const void* x, const void* r, void* a, int64_t n, const LaunchCtx& c) {
  constexpr int VEC = Io<DT>::kVec;
  const int64_t max_blocks = static_cast<int64_t>(c.dev.sms) * (2048 / kAddThreads);
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  cudaError_t e;
  if (al(x) && al(r) && al(a)) {
    const int64_t nvec = n / VEC;
    // vectors a thread keeps in flight: 4, or 1 when a full grid would give
    // each thread at most 2 (then every resident thread has work); the
    // GELU kernels' middle setting, 2, measured slower here
    const int64_t resident = max_blocks * kAddThreads;
    const int U = nvec <= 2 * resident ? 1 : 4;
    int64_t blocks = (nvec + kAddThreads * U - 1) / (kAddThreads * U);
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    const dim3 grid(static_cast<unsigned>(blocks));
    e = U == 1 ? launch_kernel(k_add_vec<DT, 1>, grid, dim3(kAddThreads), 0, c.stream, c.pdl, x, r, a,
                               nvec, n)
               : launch_kernel(k_add_vec<DT, 4>, grid, dim3(kAddThreads), 0, c.stream, c.pdl, x, r, a,
                               nvec, n);
  } else {
    int64_t blocks = (n + kAddThreads - 1) / kAddThreads;
    if (blocks > max_blocks) blocks = max_blocks;
    e = launch_kernel(k_add_scalar<DT>, dim3(static_cast<unsigned>(blocks)), dim3(kAddThreads), 0,
                      c.stream, c.pdl, x, r, a, n);
  }
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

ADDLN_BOUNDS_READER(read_bounds_add)

int launch_add(int dtype, const void* x, const void* r, void* a, int64_t n, const LaunchCtx& c) {
  switch (dtype) {
    case kF32: return launch_add_t<kF32>(x, r, a, n, c);
    case kF16: return launch_add_t<kF16>(x, r, a, n, c);
    case kBF16: return launch_add_t<kBF16>(x, r, a, n, c);
    default: return ADDLN_ERR_DTYPE;
  }
}

}  // namespace addln
