// Backward of the fused residual-Add + LayerNorm (the textbook derivative of
// the forward definition; the pages only name autodiff fusion as a direction).
// Per row, from the stored sum A, the saved mean and rstd, gamma and dY:
//   xhat = (A - mean) * rstd,  g = dY * gamma
//   dA   = rstd * (g - mean_j g - xhat * mean_j(g xhat)) (+ dA_in)
//   dX = dR = dA
// and over all rows dgamma = sum dY xhat, dbeta = sum dY.
//
// Row kernels (persistent grid, rows b, b + G, ... for CTA or warp b): read
// dY and A once, compute the two row sums with warp butterflies (plain sums:
// commutative, so every lane gets the same totals), write dX once.  Each
// thread always handles the same columns, so it accumulates its columns'
// dgamma / dbeta contributions in its own shared-memory slots (no races, no
// atomics); at the end every CTA writes one [2][H] partial to the caller's
// workspace, and a second kernel (k_colsum4 for even H, k_colsum otherwise)
// adds the G partials of each column in a fixed order.  The result is bitwise
// deterministic.
//
// Shapes: one warp per row (4 warps per CTA, 16-byte vectors) for H <= 1024;
// one CTA per row with dY and A staged by TMA bulk copies on a bounded
// mbarrier wait above that; element loads for rows that are not 16-byte
// aligned.
#include <mutex>
#include <unordered_map>

#include "../../include/addln.h"
#include "common.cuh"

namespace addln {
namespace bw {

__device__ int g_bwd_error = 0;

struct BwdArgs {
  const void* dy;
  const void* a;
  const float* mean;
  const float* rstd;
  const float* gamma;
  const void* dres;  // optional gradient reaching A from elsewhere
  void* dx;
  float* ws;         // [G][2][H] column partials, or nullptr (no dgamma / dbeta)
  int64_t rows;
  int H;
  float inv_h;
  uint64_t wait_limit_ns;
};

// Byte extents of a backward launch's buffers (for ADDLN_IN): a [rows, H]
// tensor in the I/O dtype, gamma [H], mean / rstd [rows], and the [G][2][H]
// fp32 workspace partials of a grid of G CTAs.
__device__ __forceinline__ int64_t bw_rows_bytes(const BwdArgs& p, int elem) {
  return p.rows * static_cast<int64_t>(p.H) * elem;
}
__device__ __forceinline__ int64_t bw_ws_bytes(const BwdArgs& p) {
  return static_cast<int64_t>(gridDim.x) * 8 * p.H;
}

template <int VEC>
__device__ __forceinline__ void load_gamma(const float* g, float (&out)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 t = ld_param_f4(g + 4 * q);
    out[4 * q] = t.x; out[4 * q + 1] = t.y; out[4 * q + 2] = t.z; out[4 * q + 3] = t.w;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Two warp sums at once, added as a pair at every step.
__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    v = add2(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, off), __shfl_xor_sync(0xffffffffu, v.y, off)));
  return v;
}

// After a wait of warp w ran out: waits (bounded) for that warp's copies
// still in flight -- the row at ring position `ring` and the stages-1 rows
// after it -- so that none lands in shared memory the next CTA on this SM may
// reuse.
__device__ __noinline__ void drain_res(uint64_t* bars, int stages, int nw, int w, uint32_t ring,
                                       int64_t row, int64_t stride, int64_t rows) {
  for (int j = 0; j < stages; ++j, ring = ring_next(ring, stages))
    if (row + j * stride < rows)
      mbar_wait_bounded(smem_addr(&bars[ring_slot(ring) * nw + w]), ring_phase(ring), 1000000000ull);
}

// ---------------------------------------------------- CTA per row (TMA)
template <int DT, int THREADS, int NV, bool FULL>
__global__ void __launch_bounds__(THREADS) k_bwd_cta(const BwdArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int S = IO::kBytes;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.H;
  const int nvec = H / VEC;
  const bool cols = p.ws != nullptr;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * S;  // multiple of 16
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  // partials, thread-major so a warp's accesses hit 32 distinct banks: column
  // (tid + THREADS k) * VEC + i lives at slot (k * VEC + i) * THREADS + tid of
  // the dgamma half [0, THREADS NV VEC) and of the dbeta half after it
  constexpr int kHalf = THREADS * NV * VEC;
  float* part = reinterpret_cast<float*>(smem + 2 * rb);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * rb + 8 * kHalf);
  float2* red = reinterpret_cast<float2*>(reinterpret_cast<char*>(bar) + 16);  // [2][NW]
  const uint32_t s0 = smem_addr(smem);
  const uint32_t bar_a = smem_addr(bar);

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (tid + THREADS * k) < nvec;
  if (cols)
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        part[(k * VEC + e) * THREADS + tid] = 0.f;
        part[kHalf + (k * VEC + e) * THREADS + tid] = 0.f;
      }
  if (tid == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t policy = policy_evict_first();
  pdl_trigger();
  pdl_wait();

  const int64_t stride = gridDim.x;
  int64_t row = blockIdx.x;
  auto issue = [&](int64_t rr) {
    const int64_t off = rr * static_cast<int64_t>(row_bytes);
    const bool okc = ADDLN_IN(601, off, row_bytes, bw_rows_bytes(p, S));
    mbar_arrive_expect_tx(bar_a, okc ? 2u * row_bytes : 0u);
    if (okc) {
      bulk_g2s(s0, static_cast<const char*>(p.dy) + off, row_bytes, bar_a, policy);
      bulk_g2s(s0 + rb, static_cast<const char*>(p.a) + off, row_bytes, bar_a, policy);
    }
  };
  if (tid == 0 && row < p.rows) issue(row);
  // mean and rstd of the next row are loaded one row ahead, off the row's
  // critical path
  float mu_n = 0.f, rs_n = 0.f;
  if (row < p.rows && ADDLN_IN(602, 4 * row, 4, 4 * p.rows))
    mu_n = __ldg(p.mean + row), rs_n = __ldg(p.rstd + row);

  for (int64_t it = 0; row < p.rows; ++it, row += stride) {
    const int64_t boff = row * static_cast<int64_t>(row_bytes);
    const float mu = mu_n, rs = rs_n;
    if (row + stride < p.rows && ADDLN_IN(603, 4 * (row + stride), 4, 4 * p.rows))
      mu_n = __ldg(p.mean + row + stride), rs_n = __ldg(p.rstd + row + stride);
    const bool timed_out = !mbar_wait_bounded(bar_a, static_cast<uint32_t>(it & 1), p.wait_limit_ns);
    uint4 dv[NV];       // dY kept packed; the stage is refilled after the barrier
    float xh[NV][VEC];
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = tid + THREADS * k;
        float d[VEC], gg[VEC];
        dv[k] = ld_shared_v4(s0 + c * 16);
        IO::unpack(dv[k], d);
        IO::unpack(ld_shared_v4(s0 + rb + c * 16), xh[k]);
        if (ADDLN_IN(604, 4 * c * VEC, 4 * VEC, 4 * static_cast<int64_t>(H)))
          load_gamma<VEC>(p.gamma + c * VEC, gg);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          xh[k][i] = (xh[k][i] - mu) * rs;
          const float g = d[i] * gg[i];
          sg += g;
          sgx = fmaf(g, xh[k][i], sgx);
        }
        if (cols && !timed_out)
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            float* sl = part + (k * VEC + i) * THREADS + tid;
            sl[0] = fmaf(d[i], xh[k][i], sl[0]);
            sl[kHalf] += d[i];
          }
      }
    }
    sg = warp_sum(sg);
    sgx = warp_sum(sgx);
    float2* rbuf = red + (it & 1) * NW;
    if (lane == 0) rbuf[warp] = make_float2(sg, sgx);
    if (__syncthreads_or(timed_out)) {  // also: the staged rows are in registers
      if (tid == 0) {
        atomicExch(&g_bwd_error, ADDLN_ERR_DEVICE_TIMEOUT);
        mbar_wait_bounded(bar_a, static_cast<uint32_t>(it & 1), 1000000000ull);
      }
      return;
    }
    if (tid == 0 && row + stride < p.rows) issue(row + stride);
    float tg = 0.f, tgx = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      tg += rbuf[w].x;
      tgx += rbuf[w].y;
    }
    const float mg = tg * p.inv_h, mgx = tgx * p.inv_h;
    char* drow = static_cast<char*>(p.dx) + boff;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = tid + THREADS * k;
        float d[VEC], gg[VEC], o[VEC], rr[VEC];
        IO::unpack(dv[k], d);
        if (ADDLN_IN(605, 4 * c * VEC, 4 * VEC, 4 * static_cast<int64_t>(H)))
          load_gamma<VEC>(p.gamma + c * VEC, gg);
        if (p.dres != nullptr && ADDLN_IN(606, boff + c * 16, 16, bw_rows_bytes(p, S)))
          IO::unpack(ld_stream_v4(static_cast<const char*>(p.dres) + boff + c * 16), rr);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          o[i] = rs * (d[i] * gg[i] - fmaf(xh[k][i], mgx, mg));
          if (p.dres != nullptr) o[i] += rr[i];
        }
        if (ADDLN_IN(607, boff + c * 16, 16, bw_rows_bytes(p, S))) st_stream_v4(drow + c * 16, IO::pack(o));
      }
    }
  }
  if (cols) {
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k])
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const int j = (tid + THREADS * k) * VEC + i;
          if (ADDLN_IN(608, (static_cast<int64_t>(blockIdx.x) * 2 * H + H + j) * 4, 4, bw_ws_bytes(p))) {
            out[j] = part[(k * VEC + i) * THREADS + tid];
            out[H + j] = part[kHalf + (k * VEC + i) * THREADS + tid];
          }
        }
  }
}

// ------------------------------------- register-resident column sums
// The main backward kernels.  gamma and the thread's dgamma / dbeta
// accumulators stay in registers for the CTA's lifetime (so per row the L1
// data path sees only the staged dY and A and the dX stores; keeping the
// partials in shared memory cost four shared accesses an element and reading
// gamma twice a row another two 16-byte loads per 4 columns, which made L1,
// not HBM, the limit), values are held as fp32 pairs, and dY and A arrive by
// bulk copies into a per-warp ring of `stages` slots (each warp's own
// mbarriers), refilled as soon as the warp is past a slot.
//
// ROWWARP: each warp owns whole rows (lanes take vectors lane + 32 k) and
// reduces with shuffles alone; at the end the CTA adds its warps'
// accumulators in warp order into its [2][H] partial.  Otherwise the CTA owns
// a row and warp w the contiguous chunk of vectors [w CV, (w+1) CV); the two
// row sums go through shared memory and one barrier, and every thread writes
// its own columns of the CTA's partial.
constexpr int kMaxStagesRes = 4;

template <int DT, int THREADS, int NV, bool ROWWARP>
constexpr int bwd_res_regs() {
  return ROWWARP ? 168 : 128;
}

template <int DT, int THREADS, int NV, bool FULL, bool ROWWARP>
__global__ void __launch_bounds__(THREADS) __maxnreg__((bwd_res_regs<DT, THREADS, NV, ROWWARP>()))
    k_bwd_res(const BwdArgs p, const int stages) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;
  constexpr int S = IO::kBytes;
  constexpr int NW = THREADS / 32;
  constexpr int CV = 32 * NV;                 // vectors a warp stages per row
  constexpr uint32_t kRegion = 2u * CV * 16u;  // a warp's slot: dY chunk, then A chunk
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.H;
  const int nvec = H / VEC;
  const bool cols = p.ws != nullptr;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * S;
  const uint32_t ring_bytes = static_cast<uint32_t>(stages) * NW * kRegion;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes);  // [stages][NW]
  float2* red = reinterpret_cast<float2*>(smem + ring_bytes + 8u * kMaxStagesRes * NW);  // [2][NW]
  const uint32_t smem0 = smem_addr(smem);

  const int v0 = ROWWARP ? lane : warp * CV + lane;
  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || v0 + 32 * k < nvec;
  const int cvecs = ROWWARP ? nvec : (FULL ? CV : min(CV, max(0, nvec - warp * CV)));
  const uint32_t chunk_bytes = static_cast<uint32_t>(cvecs) * 16u;
  const uint32_t chunk_off = ROWWARP ? 0u : static_cast<uint32_t>(warp * CV) * 16u;

  const int64_t stride = ROWWARP ? static_cast<int64_t>(gridDim.x) * NW : gridDim.x;
  int64_t row = ROWWARP ? static_cast<int64_t>(blockIdx.x) * NW + warp : blockIdx.x;

  // While the previous kernel may still be finishing, ask L2 for the warp's
  // chunks of dY and A of the rows its ring stages first (a hint only:
  // nothing is read before the wait below, and every SM's writes land in
  // L2); only when each CTA or warp has at most eight rows.
  if (lane == 0 && chunk_bytes != 0 && p.rows <= 8 * stride)
    for (int s = 0; s < stages; ++s) {
      const int64_t rr = row + s * stride;
      if (rr >= p.rows) break;
      const int64_t off = rr * static_cast<int64_t>(row_bytes) + chunk_off;
      if (ADDLN_IN(611, off, chunk_bytes, bw_rows_bytes(p, S))) {
        prefetch_l2(static_cast<const char*>(p.dy) + off, chunk_bytes);
        prefetch_l2(static_cast<const char*>(p.a) + off, chunk_bytes);
      }
    }
  if (tid == 0) {
    for (int i = 0; i < stages * NW; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t policy = policy_evict_first();
  pdl_trigger();
  pdl_wait();

  auto region = [&](int s) { return smem0 + static_cast<uint32_t>(s * NW + warp) * kRegion; };
  auto issue = [&](int s, int64_t rr) {  // lane 0: the warp's chunk of row rr into slot s
    const uint32_t bar = smem_addr(&bars[s * NW + warp]);
    const int64_t off = rr * static_cast<int64_t>(row_bytes) + chunk_off;
    const bool okc = ADDLN_IN(612, off, chunk_bytes, bw_rows_bytes(p, S));
    mbar_arrive_expect_tx(bar, okc ? 2u * chunk_bytes : 0u);
    if (chunk_bytes != 0 && okc) {
      bulk_g2s(region(s), static_cast<const char*>(p.dy) + off, chunk_bytes, bar, policy);
      bulk_g2s(region(s) + CV * 16u, static_cast<const char*>(p.a) + off, chunk_bytes, bar, policy);
    }
  };
  if (lane == 0)
    for (int s = 0; s < stages; ++s)
      if (row + s * stride < p.rows) issue(s, row + s * stride);

  float2 gam[NV][P], dg[NV][P], db[NV][P];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
#pragma unroll
    for (int q = 0; q < P / 2; ++q) {
      float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok[k] && ADDLN_IN(613, 4 * ((v0 + 32 * k) * VEC + 4 * q), 16, 4 * static_cast<int64_t>(H)))
        g = ld_param_f4(p.gamma + (v0 + 32 * k) * VEC + 4 * q);
      gam[k][2 * q] = make_float2(g.x, g.y);
      gam[k][2 * q + 1] = make_float2(g.z, g.w);
    }
#pragma unroll
    for (int q = 0; q < P; ++q) dg[k][q] = db[k][q] = dup2(0.f);
  }

  // mean and rstd of the next row are loaded one row ahead, off the row's
  // critical path
  float mu_n = 0.f, rs_n = 0.f;
  if (row < p.rows && ADDLN_IN(602, 4 * row, 4, 4 * p.rows))
    mu_n = __ldg(p.mean + row), rs_n = __ldg(p.rstd + row);

  bool failed = false;
  uint32_t ring = 0;  // ring position of the row: slot, phase, parity
  for (; row < p.rows; row += stride, ring = ring_next(ring, stages)) {
    const int s = static_cast<int>(ring_slot(ring));
    const float mu = mu_n, rs = rs_n;
    if (row + stride < p.rows && ADDLN_IN(603, 4 * (row + stride), 4, 4 * p.rows))
      mu_n = __ldg(p.mean + row + stride), rs_n = __ldg(p.rstd + row + stride);
    // warp-uniform: every lane polls the warp's barrier with its own clock
    const bool timed_out = __any_sync(
        0xffffffffu, !mbar_wait_bounded(smem_addr(&bars[s * NW + warp]),
                                        ring_phase(ring), p.wait_limit_ns));
    const float2 negmu = dup2(-mu), rs2 = dup2(rs);
    // The CTA form keeps xhat and either g = dY gamma (up to 256 threads) or
    // dY still packed (512 threads, where holding g measured slower) in
    // registers across the row sums; the warp form, holding twice the
    // columns, reads dY and A again from its slot, which it refills only
    // after the row is done.
    // (timed_out is warp-uniform: the whole block is skipped, not selected
    // element by element; a slot that is not ok is never read)
    constexpr int KEEP = ROWWARP ? 1 : NV;
    constexpr bool KEEPG = !ROWWARP && THREADS <= 256;
    float2 gk[KEEPG ? KEEP : 1][P];
    uint4 dv[KEEPG ? 1 : KEEP];
    float2 xh[KEEP][P];
    float2 sg2 = dup2(0.f), sgx2 = dup2(0.f);
    if (!timed_out) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int kk = ROWWARP ? 0 : k;
      if (ok[k]) {
        const uint4 dpk = ld_shared_v4(region(s) + (32 * k + lane) * 16);
        if constexpr (!KEEPG) dv[kk] = dpk;
        IO::to_pairs(ld_shared_v4(region(s) + CV * 16u + (32 * k + lane) * 16), xh[kk]);
        float2 d[P];
        IO::to_pairs(dpk, d);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          xh[kk][q] = mul2(add2(xh[kk][q], negmu), rs2);
          const float2 g = mul2(d[q], gam[k][q]);
          if constexpr (KEEPG) gk[kk][q] = g;
          sg2 = add2(sg2, g);
          sgx2 = fma2(g, xh[kk][q], sgx2);
          if (cols) {
            dg[k][q] = fma2(d[q], xh[kk][q], dg[k][q]);
            db[k][q] = add2(db[k][q], d[q]);
          }
        }
      }
    }
    }
    const float2 ts = warp_sum2(make_float2(sg2.x + sg2.y, sgx2.x + sgx2.y));
    float tg = ts.x, tgx = ts.y;
    if constexpr (ROWWARP) {
      if (timed_out) {
        if (lane == 0) drain_res(bars, stages, NW, warp, ring, row, stride, p.rows);
        failed = true;
        break;
      }
    } else {
      float2* rbuf = red + ring_parity(ring) * NW;
      if (lane == 0) rbuf[warp] = make_float2(tg, tgx);
      if (__syncthreads_or(timed_out)) {
        if (tid == 0)
          for (int w = 0; w < NW; ++w) drain_res(bars, stages, NW, w, ring, row, stride, p.rows);
        failed = true;
        break;
      }
      if (lane == 0 && row + stages * stride < p.rows) issue(s, row + stages * stride);
      // the warps' (sum g, sum g xhat) pairs, two to a 16-byte load, added
      // as pairs in a fixed tree
      float2 t[NW];
#pragma unroll
      for (int w = 0; w < NW; w += 2) {
        const float4 u = *reinterpret_cast<const float4*>(rbuf + w);
        t[w] = make_float2(u.x, u.y);
        t[w + 1] = make_float2(u.z, u.w);
      }
#pragma unroll
      for (int h = NW / 2; h > 0; h >>= 1)
#pragma unroll
        for (int w = 0; w < h; ++w) t[w] = add2(t[w], t[w + h]);
      tg = t[0].x;
      tgx = t[0].y;
    }
    // dA = rstd * (g - (xhat * mean(g xhat) + mean(g))) (+ dA_in)
    const float2 nmgx = dup2(-(tgx * p.inv_h)), nmg = dup2(-(tg * p.inv_h));
    char* drow = static_cast<char*>(p.dx) + row * static_cast<int64_t>(row_bytes);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = v0 + 32 * k;
        float2 g[P], o[P], rr[P], x[P];
        if constexpr (ROWWARP) {
          float2 d[P];
          IO::to_pairs(ld_shared_v4(region(s) + (32 * k + lane) * 16), d);
          IO::to_pairs(ld_shared_v4(region(s) + CV * 16u + (32 * k + lane) * 16), x);
#pragma unroll
          for (int q = 0; q < P; ++q) {
            x[q] = mul2(add2(x[q], negmu), rs2);
            g[q] = mul2(d[q], gam[k][q]);
          }
        } else if constexpr (KEEPG) {
#pragma unroll
          for (int q = 0; q < P; ++q) {
            x[q] = xh[k][q];
            g[q] = gk[k][q];
          }
        } else {
          float2 d[P];
          IO::to_pairs(dv[k], d);
#pragma unroll
          for (int q = 0; q < P; ++q) {
            x[q] = xh[k][q];
            g[q] = mul2(d[q], gam[k][q]);
          }
        }
        if (p.dres != nullptr &&
            ADDLN_IN(614, row * static_cast<int64_t>(row_bytes) + c * 16, 16, bw_rows_bytes(p, S)))
          IO::to_pairs(ld_stream_v4(static_cast<const char*>(p.dres) +
                                    row * static_cast<int64_t>(row_bytes) + c * 16),
                       rr);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          o[q] = mul2(rs2, add2(g[q], fma2(x[q], nmgx, nmg)));
          if (p.dres != nullptr) o[q] = add2(o[q], rr[q]);
        }
        if (ADDLN_IN(615, row * static_cast<int64_t>(row_bytes) + c * 16, 16, bw_rows_bytes(p, S)))
          st_stream_v4(drow + static_cast<int64_t>(c) * 16, IO::from_pairs(o));
      }
    }
    if constexpr (ROWWARP) {
      __syncwarp();  // every lane is past slot s
      if (lane == 0 && row + stages * stride < p.rows) issue(s, row + stages * stride);
    }
  }
  if (failed) atomicExch(&g_bwd_error, ADDLN_ERR_DEVICE_TIMEOUT);
  if (!cols) return;

  if constexpr (ROWWARP) {
    // warps' accumulators into shared memory (the ring is free now), then
    // summed in warp order into the CTA's partial
    __syncthreads();
    float* part = reinterpret_cast<float*>(smem);  // [NW][2][H]
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k])
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const int j = (v0 + 32 * k) * VEC + 2 * q;
          float* w0 = part + static_cast<int64_t>(warp) * 2 * H;
          w0[j] = dg[k][q].x;
          w0[j + 1] = dg[k][q].y;
          w0[H + j] = db[k][q].x;
          w0[H + j + 1] = db[k][q].y;
        }
    __syncthreads();
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
    for (int j = tid; j < 2 * H; j += THREADS) {
      float t = part[j];
#pragma unroll
      for (int w = 1; w < NW; ++w) t += part[static_cast<int64_t>(w) * 2 * H + j];
      if (ADDLN_IN(616, (static_cast<int64_t>(blockIdx.x) * 2 * H + j) * 4, 4, bw_ws_bytes(p)))
        out[j] = t;
    }
  } else {
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k])
#pragma unroll
        for (int q = 0; q < P / 2; ++q) {
          const int j = (v0 + 32 * k) * VEC + 4 * q;
          if (!ADDLN_IN(617, (static_cast<int64_t>(blockIdx.x) * 2 * H + H + j) * 4, 16, bw_ws_bytes(p)))
            continue;
          *reinterpret_cast<float4*>(out + j) =
              make_float4(dg[k][2 * q].x, dg[k][2 * q].y, dg[k][2 * q + 1].x, dg[k][2 * q + 1].y);
          *reinterpret_cast<float4*>(out + H + j) =
              make_float4(db[k][2 * q].x, db[k][2 * q].y, db[k][2 * q + 1].x, db[k][2 * q + 1].y);
        }
  }
}

// ------------------------------------------------ CTA per row, elements
template <int DT, int THREADS>
__global__ void __launch_bounds__(THREADS) k_bwd_scalar(const BwdArgs p) {
  using IO = Io<DT>;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = p.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cols = p.ws != nullptr;
  float* sg_ = reinterpret_cast<float*>(smem);        // g per element [H]
  float* sx_ = sg_ + H;                                // xhat per element [H]
  float* part = sx_ + H;                               // dgamma[H], dbeta[H]
  float2* red = reinterpret_cast<float2*>(part + 2 * H);  // [2][NW]
  if (cols)
    for (int j = tid; j < H; j += THREADS) part[j] = part[H + j] = 0.f;
  pdl_trigger();
  pdl_wait();
  int64_t it = 0;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
    const int64_t base = row * static_cast<int64_t>(H);
    float mu = 0.f, rs = 0.f;
    if (ADDLN_IN(621, 4 * row, 4, 4 * p.rows)) mu = __ldg(p.mean + row), rs = __ldg(p.rstd + row);
    float sg = 0.f, sgx = 0.f;
    for (int j = tid; j < H; j += THREADS) {
      const bool okj = ADDLN_IN(622, (base + j) * IO::kBytes, IO::kBytes, bw_rows_bytes(p, IO::kBytes));
      const float d = okj ? IO::load1(p.dy, base + j) : 0.f;
      const float xh = ((okj ? IO::load1(p.a, base + j) : 0.f) - mu) * rs;
      const float g = d * __ldg(p.gamma + j);
      sg_[j] = g;
      sx_[j] = xh;
      sg += g;
      sgx = fmaf(g, xh, sgx);
      if (cols) {
        part[j] = fmaf(d, xh, part[j]);
        part[H + j] += d;
      }
    }
    sg = warp_sum(sg);
    sgx = warp_sum(sgx);
    float2* rbuf = red + (it & 1) * NW;
    if (lane == 0) rbuf[warp] = make_float2(sg, sgx);
    __syncthreads();
    float tg = 0.f, tgx = 0.f;
    for (int w = 0; w < NW; ++w) {
      tg += rbuf[w].x;
      tgx += rbuf[w].y;
    }
    const float mg = tg * p.inv_h, mgx = tgx * p.inv_h;
    for (int j = tid; j < H; j += THREADS) {
      float o = rs * (sg_[j] - fmaf(sx_[j], mgx, mg));
      if (ADDLN_IN(623, (base + j) * IO::kBytes, IO::kBytes, bw_rows_bytes(p, IO::kBytes))) {
        if (p.dres != nullptr) o += IO::load1(p.dres, base + j);
        IO::store1(p.dx, base + j, o);
      }
    }
  }
  if (cols) {
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
    for (int j = tid; j < H; j += THREADS) {
      if (!ADDLN_IN(624, (static_cast<int64_t>(blockIdx.x) * 2 * H + H + j) * 4, 4, bw_ws_bytes(p)))
        continue;
      out[j] = part[j];
      out[H + j] = part[H + j];
    }
  }
}

// dgamma_j = sum_b ws[b][0][j], dbeta_j = sum_b ws[b][1][j].  A block covers
// 32 columns with SLICES slices of the partials (slice s takes b = s,
// s + SLICES, ...; a warp reads 32 adjacent columns of one partial, 128
// coalesced bytes); each thread keeps eight accumulators over interleaved
// subsequences of its slice, so eight loads are in flight, then adds them in
// a fixed order; the slice sums are added in slice order.  The result does
// not depend on scheduling.  Narrow rows (few 32-column blocks) take 32
// slices, so that each thread has fewer partials to walk.
constexpr int kColCols = 32, kColAcc = 8;

template <int SLICES>
__global__ void __launch_bounds__(kColCols * SLICES, 32 / SLICES) k_colsum(const float* ws, int64_t G,
                                                                            int H, float* dgamma,
                                                                            float* dbeta) {
  __shared__ float part[SLICES][kColCols + 1];
  pdl_trigger();
  pdl_wait();
  const int lc = threadIdx.x % kColCols, sl = threadIdx.x / kColCols;
  const int j = blockIdx.x * kColCols + lc;
  const int64_t ld = 2 * static_cast<int64_t>(H);
  float acc[kColAcc];
#pragma unroll
  for (int u = 0; u < kColAcc; ++u) acc[u] = 0.f;
  if (j < 2 * H) {
    constexpr int64_t kStep = static_cast<int64_t>(SLICES) * kColAcc;
    for (int64_t b = sl; b < G; b += kStep) {
#pragma unroll
      for (int u = 0; u < kColAcc; ++u) {
        const int64_t bu = b + static_cast<int64_t>(u) * SLICES;
        if (bu < G && ADDLN_IN(631, (bu * ld + j) * 4, 4, G * ld * 4)) acc[u] += ws[bu * ld + j];
      }
    }
  }
  part[sl][lc] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  __syncthreads();
  if (sl == 0 && j < 2 * H) {
    float t = part[0][lc];
#pragma unroll 8
    for (int q = 1; q < SLICES; ++q) t += part[q][lc];
    if (j < H)
      dgamma[j] = t;
    else if (ADDLN_IN(632, 4 * (j - H), 4, 4 * static_cast<int64_t>(H)))
      dbeta[j - H] = t;
  }
}

// The same sums for even H, where every partial's columns can be read 16
// bytes at a time.  A block covers 4·QUADS adjacent columns (QUADS column
// quads of every partial); thread t takes quad t % QUADS and the partials
// o, o + T/QUADS, o + 2T/QUADS, ... (o = t / QUADS), issues the loads of up
// to eight of them at once and adds them in that order; the sums of a quad
// are then added by a butterfly over the warp's lanes of that quad (every
// lane ends with the same value) and across the warps in warp order.  The
// order depends only on G, H, QUADS and T, never on scheduling.  Every load
// of a thread is in flight at once: the partials sit in L2, and the
// kernel's time is its latency.
constexpr int kCol4Threads = 256;

// Quads a block: the most (of 2, 4, 8) whose G loads a column quad still
// fit in one round of eight loads a thread.  Wider blocks mean fewer of
// them; a second round of L2 latency costs more than the extra blocks.
// (µs a step, backward with these sums, 2 / 4 / 8 quads: 2048×4096 fp16,
// G = 304: 17.31 / 15.87 / 17.19; 4096×768 fp16, G = 608: 11.67 / 13.40 /
// 16.18; 32768×8192 bf16, G = 152: 273.4 / 271.6 / 271.1.)
inline int colsum_quads(int64_t G) {
  constexpr int64_t kOneRound = 8 * kCol4Threads;  // loads a block issues in one round
  if (8 * G <= kOneRound) return 8;
  if (4 * G <= kOneRound) return 4;
  return 2;
}

template <int QUADS>
__global__ void __launch_bounds__(kCol4Threads) k_colsum4(const float* ws, int64_t G, int H,
                                                         float* dgamma, float* dbeta) {
  static_assert(QUADS >= 1 && QUADS <= 32 && (QUADS & (QUADS - 1)) == 0, "quads: a power of two");
  constexpr int NW = kCol4Threads / 32;
  constexpr int64_t kStep = kCol4Threads / QUADS;  // partials between a thread's loads
  constexpr int kU = 8;                            // loads in flight a thread
  __shared__ float4 wsum[NW][QUADS];
  pdl_trigger();
  pdl_wait();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, q = t % QUADS;
  const int64_t ld = 2 * static_cast<int64_t>(H);
  const int64_t j = (static_cast<int64_t>(blockIdx.x) * QUADS + q) * 4;  // the thread's first column
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (j < ld) {
    for (int64_t b0 = t / QUADS; b0 < G; b0 += kStep * kU) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t b = b0 + u * kStep;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < G && ADDLN_IN(633, (b * ld + j) * 4, 16, G * ld * 4))
          v[u] = __ldcg(reinterpret_cast<const float4*>(ws + b * ld + j));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
      }
    }
  }
#pragma unroll
  for (int off = QUADS; off < 32; off <<= 1) {
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
  }
  if (lane < QUADS) wsum[warp][lane] = acc;
  __syncthreads();
  if (t < QUADS && j < ld) {
    float4 r = wsum[0][t];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      const float4 u = wsum[w][t];
      r.x += u.x; r.y += u.y; r.z += u.z; r.w += u.w;
    }
    const float e[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t c = j + k;
      if (c < H)
        dgamma[c] = e[k];
      else if (c < ld && ADDLN_IN(634, 4 * (c - H), 4, 4 * static_cast<int64_t>(H)))
        dbeta[c - H] = e[k];
    }
  }
}

// ------------------------------------------------------------------ host
namespace {

struct Key {
  const void* f;
  int device, smem;
  bool operator==(const Key& o) const { return f == o.f && device == o.device && smem == o.smem; }
};
struct KeyHash {
  size_t operator()(const Key& k) const {
    return std::hash<const void*>()(k.f) ^ (static_cast<size_t>(k.device) << 20) ^
           (static_cast<size_t>(k.smem) << 28);
  }
};
std::mutex g_mu;
std::unordered_map<Key, int, KeyHash> g_occ;

int resident(const void* f, int threads, int smem, const DeviceInfo& dev) {
  const Key key{f, dev.device, smem};
  {
    std::lock_guard<std::mutex> g(g_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  // per-function limit: raised once to the opt-in maximum, never lowered
  // Raised to the device's opt-in maximum less the kernel's static shared
  // memory (the two together may not exceed the per-block limit).
  if (smem > 48 * 1024) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, f) != cudaSuccess ||
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.smem_optin - static_cast<int>(fa.sharedSizeBytes)) != cudaSuccess)
      return -1;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, threads, smem) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> g(g_mu);
  g_occ[key] = n;
  return n;
}

// A launch the row kernels will make: kernel, threads, shared memory, grid.
struct Plan {
  const void* f = nullptr;
  int threads = 0;
  uint32_t smem = 0;
  int64_t grid = 0;  // also the number of workspace partials
  int kind = 0;      // 0 warp, 1 cta, 2 scalar, 3 register-resident (takes `stages`)
  int stages = 0;
  const char* name = "none";
};

// One wave of resident CTAs (no more than there are rows for).
int64_t grid_of(int64_t rows, int64_t per_cta_rows, int per_sm, const DeviceInfo& dev) {
  const int64_t wave = static_cast<int64_t>(per_sm) * dev.sms;
  const int64_t need = (rows + per_cta_rows - 1) / per_cta_rows;
  const int64_t g = need < wave ? need : wave;
  return g < 1 ? 1 : g;
}

template <int DT, int THREADS, int NV, bool FULL>
int plan_cta(const BwdArgs& p, const DeviceInfo& dev, Plan* pl) {
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * Io<DT>::kBytes;
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  pl->f = reinterpret_cast<const void*>(&k_bwd_cta<DT, THREADS, NV, FULL>);
  pl->threads = THREADS;
  pl->smem = 2u * rb + 8u * THREADS * NV * Io<DT>::kVec + 16u + 2u * (THREADS / 32) * sizeof(float2);
  if (pl->smem > static_cast<uint32_t>(dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const int per_sm = resident(pl->f, THREADS, static_cast<int>(pl->smem), dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  pl->grid = grid_of(p.rows, 1, per_sm, dev);
  pl->kind = 1;
  return ADDLN_OK;
}

// Register-resident kernel: two ring slots a warp by default, three for
// 512-thread CTAs (one to an SM, so fewer rows in flight an SM otherwise).
// Measured, µs a step at 2 / 3 / 4 slots: 4096x768 fp16 (warp per row)
// 11.37 / 11.57 / 12.59; 65536x1000 bf16 (warp per row) 69.9 / 70.5 / 75.5;
// 2048x4096 fp16 (256 threads) 15.97 / 16.08 / 16.28; 32768x8192 bf16
// (512 threads) 270.3 / 267.9 / 268.2.  The slot knob (1..4) changes only
// the launch's slots, never its grid, so the workspace size does not depend
// on it.  The warp-per-row form keeps at least two slots, whose space its
// final per-warp column sums reuse.
template <int DT, int THREADS, int NV, bool FULL, bool ROWWARP>
int plan_res(const BwdArgs& p, const DeviceInfo& dev, int stages_knob, Plan* pl) {
  constexpr int NW = THREADS / 32;
  constexpr uint32_t region = 2u * 32u * NV * 16u;
  constexpr int kDefaultStages = !ROWWARP && THREADS >= 512 ? 3 : 2;
  auto smem_of = [](int st) {
    return static_cast<uint32_t>(st) * NW * region + 8u * kMaxStagesRes * NW + 2u * NW * 8u;
  };
  int st = stages_knob > 0 ? stages_knob : kDefaultStages;
  if (ROWWARP && st < 2) st = 2;
  if (st > kMaxStagesRes) return ADDLN_ERR_UNSUPPORTED;
  pl->f = reinterpret_cast<const void*>(&k_bwd_res<DT, THREADS, NV, FULL, ROWWARP>);
  pl->threads = THREADS;
  pl->stages = st;
  pl->smem = smem_of(st);
  if (pl->smem > static_cast<uint32_t>(dev.smem_optin) ||
      smem_of(kDefaultStages) > static_cast<uint32_t>(dev.smem_optin))
    return ADDLN_ERR_UNSUPPORTED;
  const int per_sm = resident(pl->f, THREADS, static_cast<int>(smem_of(kDefaultStages)), dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  if (st != kDefaultStages && resident(pl->f, THREADS, static_cast<int>(pl->smem), dev) <= 0)
    return ADDLN_ERR_UNSUPPORTED;
  pl->grid = grid_of(p.rows, ROWWARP ? NW : 1, per_sm, dev);
  pl->kind = 3;
  return ADDLN_OK;
}

template <int DT>
int plan_scalar(const BwdArgs& p, const DeviceInfo& dev, Plan* pl) {
  constexpr int THREADS = 512;
  pl->f = reinterpret_cast<const void*>(&k_bwd_scalar<DT, THREADS>);
  pl->threads = THREADS;
  pl->smem = 16u * static_cast<uint32_t>(p.H) + 2u * (THREADS / 32) * sizeof(float2);
  if (pl->smem > static_cast<uint32_t>(dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const int per_sm = resident(pl->f, THREADS, static_cast<int>(pl->smem), dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  pl->grid = grid_of(p.rows, 1, per_sm, dev);
  pl->kind = 2;
  return ADDLN_OK;
}

template <int DT>
int plan_dt(const BwdArgs& p, bool vec_ok, const DeviceInfo& dev, int stages_knob, Plan* pl) {
  constexpr int VEC = Io<DT>::kVec;
  const int nvec = p.H / VEC;
  if (vec_ok && p.H <= 1024) {
    // a warp per row, 128-thread CTAs
    const int nv = (nvec + 31) / 32;
    if (nv <= 1) { pl->name = "bwd_res_warp_nv1"; return nvec == 32 ? plan_res<DT, 128, 1, true, true>(p, dev, stages_knob, pl) : plan_res<DT, 128, 1, false, true>(p, dev, stages_knob, pl); }
    if (nv <= 2) { pl->name = "bwd_res_warp_nv2"; return nvec == 64 ? plan_res<DT, 128, 2, true, true>(p, dev, stages_knob, pl) : plan_res<DT, 128, 2, false, true>(p, dev, stages_knob, pl); }
    if (nv <= 3) { pl->name = "bwd_res_warp_nv3"; return nvec == 96 ? plan_res<DT, 128, 3, true, true>(p, dev, stages_knob, pl) : plan_res<DT, 128, 3, false, true>(p, dev, stages_knob, pl); }
    if (nv <= 4) { pl->name = "bwd_res_warp_nv4"; return nvec == 128 ? plan_res<DT, 128, 4, true, true>(p, dev, stages_knob, pl) : plan_res<DT, 128, 4, false, true>(p, dev, stages_knob, pl); }
    if constexpr (VEC == 4)
      if (nv <= 8) { pl->name = "bwd_res_warp_nv8"; return nvec == 256 ? plan_res<DT, 128, 8, true, true>(p, dev, stages_knob, pl) : plan_res<DT, 128, 8, false, true>(p, dev, stages_knob, pl); }
  }
  if (vec_ok && p.H > 1024) {
    // a CTA per row, 16 columns a thread
    constexpr int NVR = 16 / VEC;
    if (nvec <= 128 * NVR) { pl->name = "bwd_res_cta_t128"; return nvec == 128 * NVR ? plan_res<DT, 128, NVR, true, false>(p, dev, stages_knob, pl) : plan_res<DT, 128, NVR, false, false>(p, dev, stages_knob, pl); }
    if (nvec <= 256 * NVR) { pl->name = "bwd_res_cta_t256"; return nvec == 256 * NVR ? plan_res<DT, 256, NVR, true, false>(p, dev, stages_knob, pl) : plan_res<DT, 256, NVR, false, false>(p, dev, stages_knob, pl); }
    if (nvec <= 512 * NVR) { pl->name = "bwd_res_cta_t512"; return nvec == 512 * NVR ? plan_res<DT, 512, NVR, true, false>(p, dev, stages_knob, pl) : plan_res<DT, 512, NVR, false, false>(p, dev, stages_knob, pl); }
  }
  if (vec_ok && p.H > 1024) {
    // longer 16-bit rows: column partials in shared memory
    if (nvec <= 512 * 4) { pl->name = "bwd_cta_tma_t512_nv4"; return nvec == 2048 ? plan_cta<DT, 512, 4, true>(p, dev, pl) : plan_cta<DT, 512, 4, false>(p, dev, pl); }
  }
  pl->name = "bwd_cta_scalar_t512";
  return plan_scalar<DT>(p, dev, pl);
}

}  // namespace

// Chooses the row kernel; *partials = the number of [2][H] fp32 workspace
// partials its grid writes.
int plan_bwd(int dtype, const BwdArgs& p, bool vec_ok, const DeviceInfo& dev, int stages_knob,
             int64_t* partials, const char** name, Plan* out) {
  int rc;
  switch (dtype) {
    case kF32: rc = plan_dt<kF32>(p, vec_ok, dev, stages_knob, out); break;
    case kF16: rc = plan_dt<kF16>(p, vec_ok, dev, stages_knob, out); break;
    case kBF16: rc = plan_dt<kBF16>(p, vec_ok, dev, stages_knob, out); break;
    default: return ADDLN_ERR_DTYPE;
  }
  if (rc == ADDLN_OK) {
    *partials = out->grid;
    *name = out->name;
  }
  return rc;
}

}  // namespace bw

int64_t bwd_workspace_bytes(int dtype, int64_t rows, int64_t H, bool vec_ok, const DeviceInfo& dev) {
  bw::BwdArgs p{};
  p.rows = rows;
  p.H = static_cast<int>(H);
  bw::Plan pl;
  int64_t partials = 0;
  const char* name = nullptr;
  const int rc = bw::plan_bwd(dtype, p, vec_ok, dev, 0, &partials, &name, &pl);
  if (rc != ADDLN_OK) return rc;
  return partials * 2 * H * 4;
}

int launch_bwd(int dtype, const void* dy, const void* a, const float* mean, const float* rstd,
               const float* gamma, const void* dres, void* dx, float* dgamma, float* dbeta,
               int64_t rows, int64_t H, bool vec_ok, void* ws, int64_t ws_bytes,
               uint64_t wait_limit_ns, const LaunchCtx& c, const char** name) {
  bw::BwdArgs p{dy, a, mean, rstd, gamma, dres, dx, nullptr, rows, static_cast<int>(H),
                static_cast<float>(1.0 / static_cast<double>(H)), wait_limit_ns};
  bw::Plan pl;
  int64_t partials = 0;
  int rc = bw::plan_bwd(dtype, p, vec_ok, c.dev, c.stages, &partials, name, &pl);
  if (rc != ADDLN_OK) return rc;
  const bool want_cols = dgamma != nullptr;
  if (want_cols) {
    if (ws == nullptr || ws_bytes < partials * 2 * H * 4 || (reinterpret_cast<uintptr_t>(ws) & 15u))
      return ADDLN_ERR_WORKSPACE;
    p.ws = static_cast<float*>(ws);
  }
  // the register-resident kernels take (BwdArgs, stages), the others (BwdArgs)
  cudaError_t e;
  if (pl.kind == 3) {
    auto kernel = reinterpret_cast<void (*)(bw::BwdArgs, int)>(const_cast<void*>(pl.f));
    e = launch_kernel(kernel, dim3(static_cast<unsigned>(pl.grid)), dim3(pl.threads), pl.smem,
                      c.stream, c.pdl, p, pl.stages);
  } else {
    auto kernel = reinterpret_cast<void (*)(bw::BwdArgs)>(const_cast<void*>(pl.f));
    e = launch_kernel(kernel, dim3(static_cast<unsigned>(pl.grid)), dim3(pl.threads), pl.smem,
                      c.stream, c.pdl, p);
  }
  if (e != cudaSuccess) {
    note_cuda_error(static_cast<int>(e));
    return ADDLN_ERR_LAUNCH;
  }
  if (want_cols && H % 2 == 0) {
    // 16-byte reads of the partials: 2H is a multiple of 4 and the
    // workspace is 16-byte aligned
    const int quads = bw::colsum_quads(partials);
    const int64_t blocks = (2 * H / 4 + quads - 1) / quads;
    auto k = quads == 2 ? bw::k_colsum4<2> : quads == 4 ? bw::k_colsum4<4> : bw::k_colsum4<8>;
    e = launch_kernel(k, dim3(static_cast<unsigned>(blocks)), dim3(bw::kCol4Threads), 0, c.stream, c.pdl,
                      static_cast<const float*>(ws), partials, static_cast<int>(H), dgamma, dbeta);
    if (e != cudaSuccess) {
      note_cuda_error(static_cast<int>(e));
      return ADDLN_ERR_LAUNCH;
    }
  } else if (want_cols) {
    const int64_t cols = 2 * H;
    const int64_t blocks = (cols + bw::kColCols - 1) / bw::kColCols;
    if (blocks < c.dev.sms)
      e = launch_kernel(bw::k_colsum<32>, dim3(static_cast<unsigned>(blocks)), dim3(bw::kColCols * 32),
                        0, c.stream, c.pdl, static_cast<const float*>(ws), partials,
                        static_cast<int>(H), dgamma, dbeta);
    else
      e = launch_kernel(bw::k_colsum<16>, dim3(static_cast<unsigned>(blocks)), dim3(bw::kColCols * 16),
                        0, c.stream, c.pdl, static_cast<const float*>(ws), partials,
                        static_cast<int>(H), dgamma, dbeta);
    if (e != cudaSuccess) {
      note_cuda_error(static_cast<int>(e));
      return ADDLN_ERR_LAUNCH;
    }
  }
  return ADDLN_OK;
}

ADDLN_BOUNDS_READER(read_bounds_bwd)

int read_and_clear_bwd_error(int* code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, bw::g_bwd_error, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(bw::g_bwd_error, &zero, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  *code = v;
  return ADDLN_OK;
}

}  // namespace addln
