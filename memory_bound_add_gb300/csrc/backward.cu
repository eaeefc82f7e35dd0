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
// workspace, and k_colsum adds the G partials of each column in a fixed
// order.  The result is bitwise deterministic.
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

// --------------------------------------------------------- warp per row
constexpr int kWarps = 4;

template <int DT, int NV, bool FULL>
__global__ void __launch_bounds__(kWarps * 32, 3) k_bwd_warp(const BwdArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int S = IO::kBytes;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.H;
  const int nvec = H / VEC;
  const bool cols = p.ws != nullptr;
  // this warp's partials, lane-major so a warp's accesses hit 32 distinct
  // banks: column (lane + 32 k) * VEC + i lives at slot (k * VEC + i) * 32 + lane
  // of the dgamma half [0, 32 NV VEC) and of the dbeta half after it
  constexpr int kHalf = 32 * NV * VEC;
  float* part = reinterpret_cast<float*>(smem) + warp * 2 * kHalf;

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (lane + 32 * k) < nvec;
  if (cols)
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        part[(k * VEC + e) * 32 + lane] = 0.f;
        part[kHalf + (k * VEC + e) * 32 + lane] = 0.f;
      }
  pdl_trigger();
  pdl_wait();

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < p.rows;
       row += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int64_t boff = row * static_cast<int64_t>(H) * S;
    uint4 dv[NV], av[NV], rv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k]) {
        dv[k] = ld_stream_v4(static_cast<const char*>(p.dy) + boff + (lane + 32 * k) * 16);
        av[k] = ld_stream_v4(static_cast<const char*>(p.a) + boff + (lane + 32 * k) * 16);
      }
    if (p.dres != nullptr)
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (ok[k]) rv[k] = ld_stream_v4(static_cast<const char*>(p.dres) + boff + (lane + 32 * k) * 16);
    const float mu = __ldg(p.mean + row), rs = __ldg(p.rstd + row);
    float xh[NV][VEC];  // dY stays packed in dv; g = dY * gamma is formed twice
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = lane + 32 * k;
        float d[VEC], gg[VEC];
        IO::unpack(dv[k], d);
        IO::unpack(av[k], xh[k]);
        load_gamma<VEC>(p.gamma + c * VEC, gg);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          xh[k][i] = (xh[k][i] - mu) * rs;
          const float g = d[i] * gg[i];
          sg += g;
          sgx = fmaf(g, xh[k][i], sgx);
        }
        if (cols)
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            float* sl = part + (k * VEC + i) * 32 + lane;
            sl[0] = fmaf(d[i], xh[k][i], sl[0]);
            sl[kHalf] += d[i];
          }
      }
    }
    sg = warp_sum(sg);
    sgx = warp_sum(sgx);
    const float mg = sg * p.inv_h, mgx = sgx * p.inv_h;
    char* drow = static_cast<char*>(p.dx) + boff;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = lane + 32 * k;
        float d[VEC], gg[VEC], o[VEC], rr[VEC];
        IO::unpack(dv[k], d);
        load_gamma<VEC>(p.gamma + c * VEC, gg);
        if (p.dres != nullptr) IO::unpack(rv[k], rr);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          o[i] = rs * (d[i] * gg[i] - fmaf(xh[k][i], mgx, mg));
          if (p.dres != nullptr) o[i] += rr[i];
        }
        st_stream_v4(drow + c * 16, IO::pack(o));
      }
    }
  }
  if (cols) {
    __syncthreads();
    const float* all = reinterpret_cast<const float*>(smem);
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
    for (int j = tid; j < 2 * H; j += kWarps * 32) {
      const int half = j < H ? 0 : 1, col = j - half * H;
      const int c = col / VEC, i = col - c * VEC;
      const int slot = half * kHalf + ((c >> 5) * VEC + i) * 32 + (c & 31);
      float s = all[slot];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) s += all[w * 2 * kHalf + slot];
      out[j] = s;
    }
  }
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
    mbar_arrive_expect_tx(bar_a, 2u * row_bytes);
    const int64_t off = rr * static_cast<int64_t>(row_bytes);
    bulk_g2s(s0, static_cast<const char*>(p.dy) + off, row_bytes, bar_a, policy);
    bulk_g2s(s0 + rb, static_cast<const char*>(p.a) + off, row_bytes, bar_a, policy);
  };
  if (tid == 0 && row < p.rows) issue(row);

  for (int64_t it = 0; row < p.rows; ++it, row += stride) {
    const int64_t boff = row * static_cast<int64_t>(row_bytes);
    const bool timed_out = !mbar_wait_bounded(bar_a, static_cast<uint32_t>(it & 1), p.wait_limit_ns);
    const float mu = __ldg(p.mean + row), rs = __ldg(p.rstd + row);
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
        load_gamma<VEC>(p.gamma + c * VEC, gg);
        if (p.dres != nullptr)
          IO::unpack(ld_stream_v4(static_cast<const char*>(p.dres) + boff + c * 16), rr);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          o[i] = rs * (d[i] * gg[i] - fmaf(xh[k][i], mgx, mg));
          if (p.dres != nullptr) o[i] += rr[i];
        }
        st_stream_v4(drow + c * 16, IO::pack(o));
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
          out[j] = part[(k * VEC + i) * THREADS + tid];
          out[H + j] = part[kHalf + (k * VEC + i) * THREADS + tid];
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
    const float mu = __ldg(p.mean + row), rs = __ldg(p.rstd + row);
    float sg = 0.f, sgx = 0.f;
    for (int j = tid; j < H; j += THREADS) {
      const float d = IO::load1(p.dy, base + j);
      const float xh = (IO::load1(p.a, base + j) - mu) * rs;
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
      if (p.dres != nullptr) o += IO::load1(p.dres, base + j);
      IO::store1(p.dx, base + j, o);
    }
  }
  if (cols) {
    float* out = p.ws + static_cast<int64_t>(blockIdx.x) * 2 * H;
    for (int j = tid; j < H; j += THREADS) {
      out[j] = part[j];
      out[H + j] = part[H + j];
    }
  }
}

// dgamma_j = sum_b ws[b][0][j], dbeta_j = sum_b ws[b][1][j].  A block covers
// 32 columns with 8 slices of the partials each (slice s takes b = s, s + 8,
// ...); the 8 slice sums are then added in slice order, so the result does
// not depend on scheduling.
constexpr int kColCols = 32, kColSlices = 8;

__global__ void __launch_bounds__(kColCols * kColSlices) k_colsum(const float* ws, int64_t G, int H,
                                                                  float* dgamma, float* dbeta) {
  __shared__ float part[kColSlices][kColCols];
  pdl_trigger();
  pdl_wait();
  const int lc = threadIdx.x % kColCols, sl = threadIdx.x / kColCols;
  const int j = blockIdx.x * kColCols + lc;
  const int64_t ld = 2 * static_cast<int64_t>(H);
  float s = 0.f;
  if (j < 2 * H) {
#pragma unroll 4
    for (int64_t b = sl; b < G; b += kColSlices) s += ws[b * ld + j];
  }
  part[sl][lc] = s;
  __syncthreads();
  if (sl == 0 && j < 2 * H) {
    float t = part[0][lc];
#pragma unroll
    for (int q = 1; q < kColSlices; ++q) t += part[q][lc];
    if (j < H)
      dgamma[j] = t;
    else
      dbeta[j - H] = t;
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
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin) !=
          cudaSuccess)
    return -1;
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
  int kind = 0;      // 0 warp, 1 cta, 2 scalar
  const char* name = "none";
};

// One wave of resident CTAs, but no more than needed to give every CTA about
// four rows (fewer partials to write and sum) and never fewer than two per SM.
int64_t grid_of(int64_t rows, int64_t per_cta_rows, int per_sm, const DeviceInfo& dev) {
  int64_t wave = static_cast<int64_t>(per_sm) * dev.sms;
  int64_t want = (rows + 4 * per_cta_rows - 1) / (4 * per_cta_rows);
  if (want < 2 * static_cast<int64_t>(dev.sms)) want = 2 * static_cast<int64_t>(dev.sms);
  int64_t g = want < wave ? want : wave;
  const int64_t need = (rows + per_cta_rows - 1) / per_cta_rows;
  if (g > need) g = need;
  return g < 1 ? 1 : g;
}

template <int DT, int NV, bool FULL>
int plan_warp(const BwdArgs& p, const DeviceInfo& dev, Plan* pl) {
  pl->f = reinterpret_cast<const void*>(&k_bwd_warp<DT, NV, FULL>);
  pl->threads = kWarps * 32;
  pl->smem = kWarps * 2u * 32u * NV * Io<DT>::kVec * 4u;
  const int per_sm = resident(pl->f, pl->threads, static_cast<int>(pl->smem), dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  pl->grid = grid_of(p.rows, kWarps, per_sm, dev);
  pl->kind = 0;
  return ADDLN_OK;
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
int plan_dt(const BwdArgs& p, bool vec_ok, const DeviceInfo& dev, Plan* pl) {
  constexpr int VEC = Io<DT>::kVec;
  const int nvec = p.H / VEC;
  if (vec_ok && p.H <= 1024) {
    const int nv = (nvec + 31) / 32;
    if (nv <= 1) { pl->name = "bwd_warp_nv1"; return nvec == 32 ? plan_warp<DT, 1, true>(p, dev, pl) : plan_warp<DT, 1, false>(p, dev, pl); }
    if (nv <= 2) { pl->name = "bwd_warp_nv2"; return nvec == 64 ? plan_warp<DT, 2, true>(p, dev, pl) : plan_warp<DT, 2, false>(p, dev, pl); }
    if (nv <= 4) { pl->name = "bwd_warp_nv4"; return nvec == 128 ? plan_warp<DT, 4, true>(p, dev, pl) : plan_warp<DT, 4, false>(p, dev, pl); }
    if constexpr (VEC == 4)
      if (nv <= 8) { pl->name = "bwd_warp_nv8"; return nvec == 256 ? plan_warp<DT, 8, true>(p, dev, pl) : plan_warp<DT, 8, false>(p, dev, pl); }
  }
  if (vec_ok && p.H > 1024) {
    if (nvec <= 128 * 4) { pl->name = "bwd_cta_tma_t128_nv4"; return nvec == 512 ? plan_cta<DT, 128, 4, true>(p, dev, pl) : plan_cta<DT, 128, 4, false>(p, dev, pl); }
    if (nvec <= 256 * 4) { pl->name = "bwd_cta_tma_t256_nv4"; return nvec == 1024 ? plan_cta<DT, 256, 4, true>(p, dev, pl) : plan_cta<DT, 256, 4, false>(p, dev, pl); }
    if (nvec <= 512 * 4) { pl->name = "bwd_cta_tma_t512_nv4"; return nvec == 2048 ? plan_cta<DT, 512, 4, true>(p, dev, pl) : plan_cta<DT, 512, 4, false>(p, dev, pl); }
  }
  pl->name = "bwd_cta_scalar_t512";
  return plan_scalar<DT>(p, dev, pl);
}

}  // namespace

// Chooses the row kernel; *partials = the number of [2][H] fp32 workspace
// partials its grid writes.
int plan_bwd(int dtype, const BwdArgs& p, bool vec_ok, const DeviceInfo& dev, int64_t* partials,
             const char** name, Plan* out) {
  int rc;
  switch (dtype) {
    case kF32: rc = plan_dt<kF32>(p, vec_ok, dev, out); break;
    case kF16: rc = plan_dt<kF16>(p, vec_ok, dev, out); break;
    case kBF16: rc = plan_dt<kBF16>(p, vec_ok, dev, out); break;
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
  const int rc = bw::plan_bwd(dtype, p, vec_ok, dev, &partials, &name, &pl);
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
  int rc = bw::plan_bwd(dtype, p, vec_ok, c.dev, &partials, name, &pl);
  if (rc != ADDLN_OK) return rc;
  const bool want_cols = dgamma != nullptr;
  if (want_cols) {
    if (ws == nullptr || ws_bytes < partials * 2 * H * 4 || (reinterpret_cast<uintptr_t>(ws) & 15u))
      return ADDLN_ERR_WORKSPACE;
    p.ws = static_cast<float*>(ws);
  }
  // every row kernel has the signature void(BwdArgs)
  auto kernel = reinterpret_cast<void (*)(bw::BwdArgs)>(const_cast<void*>(pl.f));
  cudaError_t e = launch_kernel(kernel, dim3(static_cast<unsigned>(pl.grid)), dim3(pl.threads),
                                pl.smem, c.stream, c.pdl, p);
  if (e != cudaSuccess) {
    note_cuda_error(static_cast<int>(e));
    return ADDLN_ERR_LAUNCH;
  }
  if (want_cols) {
    const int64_t cols = 2 * H;
    e = launch_kernel(bw::k_colsum, dim3(static_cast<unsigned>((cols + bw::kColCols - 1) / bw::kColCols)),
                      dim3(bw::kColCols * bw::kColSlices), 0,
                      c.stream, c.pdl, static_cast<const float*>(ws), partials,
                      static_cast<int>(H), dgamma, dbeta);
    if (e != cudaSuccess) {
      note_cuda_error(static_cast<int>(e));
      return ADDLN_ERR_LAUNCH;
    }
  }
  return ADDLN_OK;
}

int read_and_clear_bwd_error(int* code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, bw::g_bwd_error, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(bw::g_bwd_error, &zero, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  *code = v;
  return ADDLN_OK;
}

}  // namespace addln
