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

// Four warps a CTA; one warp a CTA when four-warp CTAs would leave SMs
// without work (a launch of fewer than 4 x SMs warps' rows): then the rows
// spread over as many SMs as there are warps (64x768 fp32: 2.15 -> 1.95 us a
// step; at 4096x768 fp16 one-warp CTAs measured slower, 4.31 against 4.11,
// and two-warp CTAs level).  The kernels take the warps a CTA from blockDim.
constexpr int kWarpCtaThreads = 128;

// Register cap a lane: 64 while it holds at most 24 values in at most four
// vectors (eight 128-thread CTAs to an SM); 72 for fp32 rows of six vectors,
// whose extra addresses need it (seven); above 24 values 80 for 16-bit rows,
// 96 for fp32 ones.  None of them spills.
template <int DT, int NV>
constexpr int warp_row_max_regs() {
  return NV * Io<DT>::kVec <= 24 ? (NV > 4 ? 72 : 64) : DT == kF32 ? 96 : 80;
}

// Two rows a warp hold twice the values: 112 registers (four 128-thread
// CTAs to an SM) up to 24 values a row, 128 above.
template <int DT, int NV>
constexpr int warp_rows2_max_regs() {
  return NV * Io<DT>::kVec <= 24 ? 112 : 128;
}

// Vector path: 16-byte loads, values held as fp32 pairs.  FULL: the row's
// vectors divide evenly over the 32 lanes.  RPW: consecutive rows a warp
// takes (1 or 2).  With two, both rows' loads go out first and the rows'
// statistics and outputs then run as two independent instruction streams,
// gamma and beta loaded once for both: when every row of a launch lands at
// about the same time, the SM's warps then keep more instructions ready in
// the compute burst that follows (4096 x 768 fp16: 4.62 -> 4.30 us a step).
template <int DT, int NV, bool FULL, int RPW>
__global__ void __launch_bounds__(kWarpCtaThreads)
    __maxnreg__((RPW == 1 ? warp_row_max_regs<DT, NV>() : warp_rows2_max_regs<DT, NV>()))
        k_warp_row_vec(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;
  constexpr int S = IO::kBytes;
  const int lane = threadIdx.x & 31;
  const int64_t row0 =
      (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
  const int H = p.H;
  // while the previous kernel may still be finishing, ask L2 for this warp's
  // rows of X and R (a hint only: nothing is read before the wait below, and
  // a line the previous kernel writes afterwards is updated in L2)
  if (lane == 0 && row0 < p.rows) {
    const int nr = p.rows - row0 < RPW ? static_cast<int>(p.rows - row0) : RPW;
    const int64_t off = row0 * H * S;
    const uint32_t bytes = static_cast<uint32_t>(H) * S * nr;  // whole 16-byte vectors
    if (ADDLN_IN(101, off, bytes, rows_bytes(p, S)))
      prefetch_l2(static_cast<const char*>(p.x) + off, bytes);
    if (p.r != nullptr && ADDLN_IN(102, off, bytes, rows_bytes(p, S)))
      prefetch_l2(static_cast<const char*>(p.r) + off, bytes);
  }
  pdl_trigger();
  pdl_wait();
  if (row0 >= p.rows) return;  // whole warp leaves together
  const int nvec = H / VEC;

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (lane + 32 * k) < nvec;
  bool live[RPW];  // a warp's second row may lie past the last row
#pragma unroll
  for (int i = 0; i < RPW; ++i) live[i] = i == 0 || row0 + i < p.rows;

  // ---- load X and R once (every row's loads in flight together), add in fp32
  float2 v[RPW][NV][P];
  {
    uint4 xv[RPW][NV], rv[RPW][NV];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int64_t boff = (row0 + i) * H * S;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        xv[i][k] = rv[i][k] = make_uint4(0u, 0u, 0u, 0u);
        const int64_t off = boff + static_cast<int64_t>(lane + 32 * k) * 16;
        if (ok[k] && live[i] && ADDLN_IN(103, off, 16, rows_bytes(p, S))) {
          xv[i][k] = ld_stream_v4(static_cast<const char*>(p.x) + off);
          if (p.r != nullptr) rv[i][k] = ld_stream_v4(static_cast<const char*>(p.r) + off);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int k = 0; k < NV; ++k) {
#pragma unroll
        for (int q = 0; q < P; ++q) v[i][k][q] = dup2(0.f);
        if (ok[k]) {
          if (p.r != nullptr)
            IO::sum_pairs(xv[i][k], rv[i][k], v[i][k]);
          else
            IO::to_pairs(xv[i][k], v[i][k]);
        }
      }
  }

  // ---- A = X + R rounded to the dtype; each lane writes only what it read
  if (p.a != nullptr) {
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int64_t off = (row0 + i) * H * S + static_cast<int64_t>(lane + 32 * k) * 16;
        if (ok[k] && live[i] && ADDLN_IN(105, off, 16, rows_bytes(p, S)))
          st_stream_v4(static_cast<char*>(p.a) + off, IO::from_pairs(v[i][k]));
      }
  }

  // ---- row statistics on the shifted rows: per-lane two-pass, warp butterfly
  float K[RPW], rstd[RPW];
  Part st[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    K[i] = __shfl_sync(0xffffffffu, v[i][0][0].x, 0);  // a_0 of the row, held by lane 0
    const float2 negK = dup2(-K[i]);
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int q = 0; q < P; ++q) v[i][k][q] = add2(v[i][k][q], negK);
    st[i] = thread_part2<NV, P, FULL, false>(v[i], ok, negK);
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      Part o;
      o.n = FULL ? st[i].n : __shfl_xor_sync(0xffffffffu, st[i].n, off);
      o.m = __shfl_xor_sync(0xffffffffu, st[i].m, off);
      o.M2 = __shfl_xor_sync(0xffffffffu, st[i].M2, off);
      st[i] = merge<FULL>(st[i], o);
    }
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) rstd[i] = row_rstd(st[i].M2, p.inv_h, p.eps);

  // ---- normalise + affine, store (gamma / beta of a column loaded once for
  // the warp's rows)
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (ok[k]) {
      const int c = lane + 32 * k;
      float2 gg[P], bb[P];
#pragma unroll
      for (int q = 0; q < P / 2; ++q) {
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), b = g;
        if (ADDLN_IN(106, 4 * (c * VEC + 4 * q), 16, cols_bytes(p))) {
          g = ld_param_f4(p.gamma + c * VEC + 4 * q);
          b = ld_param_f4(p.beta + c * VEC + 4 * q);
        }
        gg[2 * q] = make_float2(g.x, g.y);
        gg[2 * q + 1] = make_float2(g.z, g.w);
        bb[2 * q] = make_float2(b.x, b.y);
        bb[2 * q + 1] = make_float2(b.z, b.w);
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        if (!live[i]) continue;
        const float2 negm = dup2(-st[i].m), rstd2 = dup2(rstd[i]);
        float2 o[P];
#pragma unroll
        for (int q = 0; q < P; ++q) o[q] = normalise2(v[i][k][q], negm, rstd2, gg[q], bb[q]);
        const int64_t off = (row0 + i) * H * S + static_cast<int64_t>(c) * 16;
        if (ADDLN_IN(107, off, 16, rows_bytes(p, S)))
          st_stream_v4(static_cast<char*>(p.y) + off, IO::from_pairs(o));
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int64_t row = row0 + i;
      if (!live[i] || !ADDLN_IN(108, 4 * row, 4, stat_bytes(p))) continue;
      if (p.mean != nullptr) p.mean[row] = K[i] + st[i].m;
      if (p.rstd != nullptr) p.rstd[row] = rstd[i];
    }
  }
}

// Element path (any alignment): one element per lane per slot.  FULL: the
// row's elements divide evenly over the 32 lanes.
template <int DT, int NV, bool FULL>
__global__ void __launch_bounds__(kWarpCtaThreads, 2) k_warp_row(const RowArgs p) {
  using IO = Io<DT>;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
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

template <int DT, int NV, bool VECTOR, int RPW = 1>
static int launch(const RowArgs& p, const LaunchCtx& c) {
  const int64_t rows_per_cta4 = static_cast<int64_t>(kWarpCtaThreads / 32) * RPW;
  const int warps = (p.rows + rows_per_cta4 - 1) / rows_per_cta4 < c.dev.sms ? 1 : kWarpCtaThreads / 32;
  const int64_t blocks = (p.rows + warps * RPW - 1) / (warps * RPW);
  if (blocks > 0x7fffffff) return ADDLN_ERR_UNSUPPORTED;
  constexpr int VEC = VECTOR ? Io<DT>::kVec : 1;
  const bool full = (p.H / VEC) == 32 * NV;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if constexpr (VECTOR)
    e = full ? launch_kernel(k_warp_row_vec<DT, NV, true, RPW>, grid, dim3(32 * warps), 0, c.stream, c.pdl, p)
             : launch_kernel(k_warp_row_vec<DT, NV, false, RPW>, grid, dim3(32 * warps), 0, c.stream, c.pdl, p);
  else
    e = full ? launch_kernel(k_warp_row<DT, NV, true>, grid, dim3(32 * warps), 0, c.stream, c.pdl, p)
             : launch_kernel(k_warp_row<DT, NV, false>, grid, dim3(32 * warps), 0, c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

// Rows a warp takes on the vector path: two for rows of 3 or 4 vectors a
// lane when the launch gives every SM at least 16 rows, else one; the
// addln_set_warp_rows knob overrides the choice (tests, benchmarks).
static int warp_rows_per_warp(const RowArgs& p, const LaunchCtx& c) {
  if (c.warp_rows > 0) return c.warp_rows;
  return p.rows >= 16 * static_cast<int64_t>(c.dev.sms) ? 2 : 1;
}

// Per-lane slot counts instantiated; the dispatcher takes the smallest that
// covers the row.
template <int DT>
static int launch_vec(const RowArgs& p, const LaunchCtx& c, const char** name) {
  constexpr int VEC = Io<DT>::kVec;
  const int nv = (p.H / VEC + 31) / 32;
  if (warp_rows_per_warp(p, c) == 2) {
    if (nv == 3) { *name = "warp_vec2_nv3"; return launch<DT, 3, true, 2>(p, c); }
    if (nv == 4) { *name = "warp_vec2_nv4"; return launch<DT, 4, true, 2>(p, c); }
  }
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
