// One warp per row: fused residual add + LayerNorm for short rows (H <= 1024).
//
// Each lane loads its share of the row of X and R with 16-byte streaming
// loads (vector path, values then held as fp32 pairs) or element loads
// (scalar path, any alignment) and adds them in fp32 registers.  A (when requested) is stored straight away.  The
// values are then shifted by the row's first sum a_0, which lane 0 holds and
// broadcasts by shuffle; each lane takes two-pass statistics of its own
// values and the warp merges them with a xor butterfly of Chan updates.  The
// row never leaves registers: X and R are read once, Y (and optionally A,
// mean, rstd) written once -- the fused traffic of "算子融合的收益量化"
// section 1.
#include "../../include/addln.h"
#include "common.cuh"

namespace addln {

constexpr int kWarpCtaThreads = 128;  // 4 rows per CTA
constexpr int kRowsPerCta = kWarpCtaThreads / 32;

// Register cap a lane: 64 while it holds at most 24 values in at most four
// vectors (eight 128-thread CTAs to an SM); 72 for fp32 rows of six vectors,
// whose extra addresses need it (seven); above 24 values 80 for 16-bit rows,
// 96 for fp32 ones.  None of them spills.
template <int DT, int NV>
constexpr int warp_row_max_regs() {
  return NV * Io<DT>::kVec <= 24 ? (NV > 4 ? 72 : 64) : DT == kF32 ? 96 : 80;
}

// Vector path: 16-byte loads, values held as fp32 pairs.  FULL: the row's
// vectors divide evenly over the 32 lanes.
template <int DT, int NV, bool FULL>
__global__ void __launch_bounds__(kWarpCtaThreads) __maxnreg__((warp_row_max_regs<DT, NV>()))
    k_warp_row_vec(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;
  constexpr int S = IO::kBytes;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  // while the previous kernel may still be finishing, ask L2 for this warp's
  // row of X and R (a hint only: nothing is read before the wait below, and
  // a line the previous kernel writes afterwards is updated in L2)
  const int H = p.H;
  const int64_t base = row * static_cast<int64_t>(H);  // element offset of the row
  if (lane == 0 && row < p.rows) {
    const uint32_t bytes = static_cast<uint32_t>(H) * S;  // whole 16-byte vectors
    if (ADDLN_IN(101, base * S, bytes, rows_bytes(p, S)))
      prefetch_l2(static_cast<const char*>(p.x) + base * S, bytes);
    if (p.r != nullptr && ADDLN_IN(102, base * S, bytes, rows_bytes(p, S)))
      prefetch_l2(static_cast<const char*>(p.r) + base * S, bytes);
  }
  pdl_trigger();
  pdl_wait();
  if (row >= p.rows) return;  // whole warp leaves together
  const int nvec = H / VEC;

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (lane + 32 * k) < nvec;

  float2 v[NV][P];
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int q = 0; q < P; ++q) v[k][q] = dup2(0.f);

  // ---- load X and R once, add in fp32
  const char* xrow = static_cast<const char*>(p.x) + base * S;
  uint4 xv[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (ok[k] && ADDLN_IN(103, base * S + (lane + 32 * k) * 16, 16, rows_bytes(p, S)))
      xv[k] = ld_stream_v4(xrow + static_cast<int64_t>(lane + 32 * k) * 16);
  if (p.r != nullptr) {
    const char* rrow = static_cast<const char*>(p.r) + base * S;
    uint4 rv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(104, base * S + (lane + 32 * k) * 16, 16, rows_bytes(p, S)))
        rv[k] = ld_stream_v4(rrow + static_cast<int64_t>(lane + 32 * k) * 16);
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k]) IO::sum_pairs(xv[k], rv[k], v[k]);
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k]) IO::to_pairs(xv[k], v[k]);
  }

  // ---- A = X + R rounded to the dtype; each lane writes only what it read
  if (p.a != nullptr) {
    char* arow = static_cast<char*>(p.a) + base * S;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(105, base * S + (lane + 32 * k) * 16, 16, rows_bytes(p, S)))
        st_stream_v4(arow + static_cast<int64_t>(lane + 32 * k) * 16, IO::from_pairs(v[k]));
  }

  // ---- row statistics on the shifted row: per-lane two-pass, warp butterfly
  const float K = __shfl_sync(0xffffffffu, v[0][0].x, 0);  // a_0, held by lane 0
  const float2 negK = dup2(-K);
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int q = 0; q < P; ++q) v[k][q] = add2(v[k][q], negK);
  Part st = thread_part2<NV, P, FULL, false>(v, ok, negK);
  st = butterfly<FULL, 32>(st);
  const float rstd = row_rstd(st.M2, p.inv_h, p.eps);
  const float2 negm = dup2(-st.m), rstd2 = dup2(rstd);

  // ---- normalise + affine, store
  char* yrow = static_cast<char*>(p.y) + base * S;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (ok[k]) {
      const int c = lane + 32 * k;
      float2 o[P];
#pragma unroll
      for (int q = 0; q < P / 2; ++q) {
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), b = g;
        if (ADDLN_IN(106, 4 * (c * VEC + 4 * q), 16, cols_bytes(p))) {
          g = ld_param_f4(p.gamma + c * VEC + 4 * q);
          b = ld_param_f4(p.beta + c * VEC + 4 * q);
        }
        o[2 * q] = normalise2(v[k][2 * q], negm, rstd2, make_float2(g.x, g.y), make_float2(b.x, b.y));
        o[2 * q + 1] =
            normalise2(v[k][2 * q + 1], negm, rstd2, make_float2(g.z, g.w), make_float2(b.z, b.w));
      }
      if (ADDLN_IN(107, base * S + c * 16, 16, rows_bytes(p, S)))
        st_stream_v4(yrow + static_cast<int64_t>(c) * 16, IO::from_pairs(o));
    }
  }
  if (lane == 0 && ADDLN_IN(108, 4 * row, 4, stat_bytes(p))) {
    if (p.mean != nullptr) p.mean[row] = K + st.m;
    if (p.rstd != nullptr) p.rstd[row] = rstd;
  }
}

// Element path (any alignment): one element per lane per slot.  FULL: the
// row's elements divide evenly over the 32 lanes.
template <int DT, int NV, bool FULL>
__global__ void __launch_bounds__(kWarpCtaThreads, 2) k_warp_row(const RowArgs p) {
  using IO = Io<DT>;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  pdl_trigger();
  pdl_wait();
  if (row >= p.rows) return;  // whole warp leaves together
  const int H = p.H;
  const int64_t base = row * static_cast<int64_t>(H);  // element offset of the row

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (lane + 32 * k) < H;

  float v[NV][1];
#pragma unroll
  for (int k = 0; k < NV; ++k) v[k][0] = 0.f;

  // ---- load X and R once, add in fp32
  float t[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (ok[k] && ADDLN_IN(111, (base + lane + 32 * k) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes)))
      v[k][0] = IO::load1(p.x, base + lane + 32 * k);
  if (p.r != nullptr) {
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(112, (base + lane + 32 * k) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes)))
        t[k] = IO::load1(p.r, base + lane + 32 * k);
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k]) v[k][0] += t[k];
  }

  // ---- A = X + R rounded to the dtype; each lane writes only what it read
  if (p.a != nullptr) {
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(113, (base + lane + 32 * k) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes)))
        IO::store1(p.a, base + lane + 32 * k, v[k][0]);
  }

  // ---- row statistics on the shifted row: per-lane two-pass, warp butterfly
  const float K = __shfl_sync(0xffffffffu, v[0][0], 0);  // a_0, held by lane 0
#pragma unroll
  for (int k = 0; k < NV; ++k) v[k][0] -= K;
  Part st = thread_part<NV, 1, FULL>(v, ok, 0.f);
  st = butterfly<FULL, 32>(st);
  const float m = st.m;
  const float rstd = row_rstd(st.M2, p.inv_h, p.eps);

  // ---- normalise + affine, store
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (ok[k]) {
      const int j = lane + 32 * k;
      float g = 0.f, b = 0.f;
      if (ADDLN_IN(114, 4 * j, 4, cols_bytes(p))) g = __ldg(p.gamma + j), b = __ldg(p.beta + j);
      if (ADDLN_IN(115, (base + j) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes)))
        IO::store1(p.y, base + j, normalise(v[k][0], 0.f, m, rstd, g, b));
    }
  }
  if (lane == 0 && ADDLN_IN(116, 4 * row, 4, stat_bytes(p))) {
    if (p.mean != nullptr) p.mean[row] = K + m;
    if (p.rstd != nullptr) p.rstd[row] = rstd;
  }
}

template <int DT, int NV, bool VECTOR>
static int launch(const RowArgs& p, const LaunchCtx& c) {
  const int64_t blocks = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  if (blocks > 0x7fffffff) return ADDLN_ERR_UNSUPPORTED;
  constexpr int VEC = VECTOR ? Io<DT>::kVec : 1;
  const bool full = (p.H / VEC) == 32 * NV;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if constexpr (VECTOR)
    e = full ? launch_kernel(k_warp_row_vec<DT, NV, true>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p)
             : launch_kernel(k_warp_row_vec<DT, NV, false>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p);
  else
    e = full ? launch_kernel(k_warp_row<DT, NV, true>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p)
             : launch_kernel(k_warp_row<DT, NV, false>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

// Per-lane slot counts instantiated; the dispatcher takes the smallest that
// covers the row.
template <int DT>
static int launch_vec(const RowArgs& p, const LaunchCtx& c, const char** name) {
  constexpr int VEC = Io<DT>::kVec;
  const int nv = (p.H / VEC + 31) / 32;
  if (nv <= 1) { *name = "warp_vec_nv1"; return launch<DT, 1, true>(p, c); }
  if (nv <= 2) { *name = "warp_vec_nv2"; return launch<DT, 2, true>(p, c); }
  if (nv <= 3) { *name = "warp_vec_nv3"; return launch<DT, 3, true>(p, c); }
  if (nv <= 4) { *name = "warp_vec_nv4"; return launch<DT, 4, true>(p, c); }
  if constexpr (VEC == 4) {
    if (nv <= 6) { *name = "warp_vec_nv6"; return launch<DT, 6, true>(p, c); }
    if (nv <= 8) { *name = "warp_vec_nv8"; return launch<DT, 8, true>(p, c); }
  }
  return ADDLN_ERR_UNSUPPORTED;
}

template <int DT>
static int launch_scalar(const RowArgs& p, const LaunchCtx& c, const char** name) {
  const int nv = (p.H + 31) / 32;
  if (nv <= 2) { *name = "warp_scalar_nv2"; return launch<DT, 2, false>(p, c); }
  if (nv <= 4) { *name = "warp_scalar_nv4"; return launch<DT, 4, false>(p, c); }
  if (nv <= 8) { *name = "warp_scalar_nv8"; return launch<DT, 8, false>(p, c); }
  if (nv <= 16) { *name = "warp_scalar_nv16"; return launch<DT, 16, false>(p, c); }
  if (nv <= 32) { *name = "warp_scalar_nv32"; return launch<DT, 32, false>(p, c); }
  return ADDLN_ERR_UNSUPPORTED;
}

ADDLN_BOUNDS_READER(read_bounds_rows_warp)

int launch_warp_row(int dtype, bool vec, const RowArgs& p, const LaunchCtx& c,
                    const char** name) {
  switch (dtype) {
    case kF32: return vec ? launch_vec<kF32>(p, c, name) : launch_scalar<kF32>(p, c, name);
    case kF16: return vec ? launch_vec<kF16>(p, c, name) : launch_scalar<kF16>(p, c, name);
    case kBF16: return vec ? launch_vec<kBF16>(p, c, name) : launch_scalar<kBF16>(p, c, name);
    default: return ADDLN_ERR_DTYPE;
  }
}

}  // namespace addln
