// One CTA per row: fused residual add + LayerNorm for long rows (H > 1024).
//
// The grid is persistent (one wave of resident CTAs, sized from the SM count
// and the occupancy the kernel reaches); CTA b takes rows b, b + grid, ...
//
// TMA variant: each warp stages its own chunk of every row of X and R into
// shared memory with one-dimensional bulk copies (cp.async.bulk, completion
// counted on the warp's mbarrier) into a ring of `stages` slots: the first
// `stages` rows are requested at once, and a slot is refilled with the CTA's
// row `stages` ahead as soon as every thread has moved the slot's row into
// registers.  The reduction and the normalisation both run on those
// registers, and Y / A go straight to global memory with 16-byte streaming
// stores.  When a thread
// holds at most 32 values, it also keeps gamma and beta of its columns in
// registers for the CTA's lifetime: reloading them for every row (8 bytes a
// column, twice the row's own 16-bit X and R) would make the L1 data path,
// not HBM, the limit.
//
// Vector variant: the same kernel with 16-byte loads from global memory in
// place of the staging copies (kept for comparison and for forced runs).
//
// Scalar variant: element loads for rows whose bytes or base addresses are
// not 16-byte aligned; the fp32 row sum is kept in shared memory.
//
// Waits on the staging copies are bounded.  A wait that runs out sets the
// device error word, waits (bounded again) for the CTA's copies still in
// flight so no copy lands in reused shared memory, and the CTA returns.
#include <mutex>
#include <unordered_map>

#include "../../include/addln.h"
#include "common.cuh"

namespace addln {

__device__ int g_device_error = 0;

constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s
constexpr int kMaxStages = 4;  // staging slots a CTA (one mbarrier each)

// CTA-level all-reduce of per-warp partials: lane 0 of each warp has put its
// warp's totals in red[0..NW); every warp reads red[lane % NW] and runs the
// butterfly over NW lanes, so all threads end with identical row totals.
template <bool FULL, int NW>
__device__ __forceinline__ Part cta_totals(const Part* red, int lane) {
  Part q = red[lane % NW];
  return butterfly<FULL, NW>(q);
}

// After a wait ran out: flags the device error and waits (bounded) for the
// copies still in flight -- every warp's chunk of the row at ring position
// `ring` and of the stages-1 rows after it -- so that no copy lands in shared
// memory the next CTA on this SM may reuse.
__device__ __noinline__ void drain_after_timeout(uint64_t* bars, int stages, int nw, uint32_t ring,
                                                 int64_t row, int64_t stride, int64_t rows) {
  atomicExch(&g_device_error, ADDLN_ERR_DEVICE_TIMEOUT);
  for (int j = 0; j < stages; ++j, ring = ring_next(ring, stages)) {
    if (row + j * stride >= rows) continue;
    for (int w = 0; w < nw; ++w)
      mbar_wait_bounded(smem_addr(&bars[ring_slot(ring) * nw + w]), ring_phase(ring), kDrainLimitNs);
  }
}

// gamma / beta stay in registers (TMA path, at most 32 values a thread).
template <int DT, int NV, bool TMA>
__host__ __device__ constexpr bool cta_row_resident() {
  return TMA && NV * Io<DT>::kVec <= 32;
}

// Register cap a thread: 128 with resident gamma / beta (four 128-thread CTAs
// to an SM; 136, three, for the ragged-row variant, which otherwise spills);
// otherwise by the fp32 values held (64 for 16); the vector path also holds
// the loaded vectors.
template <int DT, int THREADS, int NV, bool TMA, bool FULL>
constexpr int cta_row_max_regs() {
  return cta_row_resident<DT, NV, TMA>() ? (FULL || THREADS > 256 ? 128 : 136)
         : !TMA                         ? 128
         : NV * Io<DT>::kVec <= 16      ? 64
                                        : 128;
}

// A warp's partial statistics of a row, with the shift they are taken around.
struct WarpPart {
  float K;  // the warp's shift: the first sum of its chunk
  float n;
  float m;  // mean of (a - K) over the warp's n values
  float M2;
};

// FULL: the row's 16-byte vectors divide evenly over the CTA's threads.
//
// Warp w owns the contiguous chunk of vectors [w*32*NV, (w+1)*32*NV) of every
// row (lane l, slot k: vector w*32*NV + 32*k + l), so on the TMA path each
// warp's share of X and R arrives by its own pair of bulk copies, completing
// its own mbarrier, and the warp starts on it as soon as it lands.  Each warp
// shifts its values by the first sum of its chunk (Chan, Golub and LeVeque's
// shifted data, per warp); the CTA merge first moves every warp's mean to
// warp 0's shift, K_0 - the row's first sum a_0 - and then combines.
template <int DT, int THREADS, int NV, bool TMA, bool FULL>
__global__ void __launch_bounds__(THREADS) __maxnreg__((cta_row_max_regs<DT, THREADS, NV, TMA, FULL>()))
    k_cta_row(const RowArgs p, const int stages) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;  // fp32 pairs per vector
  constexpr int S = IO::kBytes;
  constexpr int NW = THREADS / 32;
  constexpr int CV = 32 * NV;  // vectors in a warp's chunk
  constexpr bool RES = cta_row_resident<DT, NV, TMA>();
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.H;
  const int nvec = H / VEC;
  const bool has_r = p.r != nullptr;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * S;  // multiple of 16
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  const uint32_t slot = has_r ? 2u * rb : rb;
  const uint32_t data_bytes = TMA ? static_cast<uint32_t>(stages) * slot : 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + data_bytes);  // [stages][NW]
  WarpPart* red = reinterpret_cast<WarpPart*>(smem + data_bytes + 8u * kMaxStages * NW);  // [2][NW]
  const uint32_t smem0 = smem_addr(smem);

  const int v0 = warp * CV + lane;  // this thread's first vector
  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || v0 + 32 * k < nvec;

  // bytes of X in this warp's chunk (0 for a warp past the end of a short row)
  const int cvecs = FULL ? CV : min(CV, max(0, nvec - warp * CV));
  const uint32_t chunk_bytes = static_cast<uint32_t>(cvecs) * 16u;
  const uint32_t chunk_off = static_cast<uint32_t>(warp * CV) * 16u;

  const int64_t stride = gridDim.x;
  int64_t row = blockIdx.x;
  uint64_t policy = 0;

  if constexpr (TMA) {
    // While the previous kernel in the stream may still be finishing (this
    // CTA can start in its tail under programmatic dependent launch), ask L2
    // for the warp's chunks of the rows the ring will stage first, so that
    // their DRAM latency overlaps that tail.  Nothing is read into registers
    // or shared memory before the wait below.  Only for short launches (at
    // most eight rows a CTA), whose time that start-up latency is a real
    // part of; on long ones it measured slightly slower.
    if (lane == 0 && chunk_bytes != 0 && p.rows <= 8 * stride)
      for (int s = 0; s < stages; ++s) {
        const int64_t rr = row + s * stride;
        if (rr >= p.rows) break;
        const int64_t off = rr * static_cast<int64_t>(row_bytes) + chunk_off;
        if (ADDLN_IN(201, off, chunk_bytes, rows_bytes(p, S)))
          prefetch_l2(static_cast<const char*>(p.x) + off, chunk_bytes);
        if (has_r && ADDLN_IN(202, off, chunk_bytes, rows_bytes(p, S)))
          prefetch_l2(static_cast<const char*>(p.r) + off, chunk_bytes);
      }
    if (tid == 0) {
      for (int s = 0; s < stages * NW; ++s) mbar_init(smem_addr(&bars[s]), 1);
      fence_mbar_init();
    }
    __syncthreads();
    // Ordinary L2 priority for the staged rows.  Marking them evict-first
    // (they are read once) measured slower back to back: 2048 x 4096 fp16
    // 8.81 us a step against 7.90, 2048 x 8192 bf16 21.9 against 21.0, the
    // same at 32768 x 8192 (DRAM bytes a launch unchanged).
    policy = policy_evict_normal();
  }
  pdl_trigger();
  pdl_wait();  // the previous kernel's writes are visible from here on

  // Lane 0 of each warp: stage the warp's chunk of row `rr` into slot `s`.
  auto issue = [&](int s, int64_t rr) {
    const uint32_t bar = smem_addr(&bars[s * NW + warp]);
    const int64_t off = rr * static_cast<int64_t>(row_bytes) + chunk_off;
    // checked build: a copy that would leave its buffer is not issued, and
    // the barrier is not told to expect its bytes either
    const bool okx = ADDLN_IN(203, off, chunk_bytes, rows_bytes(p, S));
    const bool okr = has_r && ADDLN_IN(204, off, chunk_bytes, rows_bytes(p, S));
    mbar_arrive_expect_tx(bar, (okx ? chunk_bytes : 0u) + (okr ? chunk_bytes : 0u));
    if (chunk_bytes != 0) {
      const uint32_t dst = smem0 + s * slot + chunk_off;
      if (okx) bulk_g2s(dst, static_cast<const char*>(p.x) + off, chunk_bytes, bar, policy);
      if (okr) bulk_g2s(dst + rb, static_cast<const char*>(p.r) + off, chunk_bytes, bar, policy);
    }
  };
  if constexpr (TMA) {
    if (lane == 0)
      for (int s = 0; s < stages; ++s)
        if (row + s * stride < p.rows) issue(s, row + s * stride);
  }

  // gamma / beta of this thread's columns, while the first rows stream in
  float2 gr[RES ? NV : 1][RES ? P : 1], br[RES ? NV : 1][RES ? P : 1];
  if constexpr (RES) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
#pragma unroll
      for (int q = 0; q < P / 2; ++q) {
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), b = g;
        const int c = v0 + 32 * k;
        if (ok[k] && ADDLN_IN(205, 4 * (c * VEC + 4 * q), 16, cols_bytes(p))) {
          g = ld_param_f4(p.gamma + c * VEC + 4 * q);
          b = ld_param_f4(p.beta + c * VEC + 4 * q);
        }
        gr[k][2 * q] = make_float2(g.x, g.y);
        gr[k][2 * q + 1] = make_float2(g.z, g.w);
        br[k][2 * q] = make_float2(b.x, b.y);
        br[k][2 * q + 1] = make_float2(b.z, b.w);
      }
    }
  }

  uint32_t ring = 0;  // ring position of the row: slot, phase, parity
  for (; row < p.rows; row += stride, ring = ring_next(ring, stages)) {
    const int s = static_cast<int>(ring_slot(ring));
    const int64_t base = row * static_cast<int64_t>(H);
    // the row's sums a = x + r as fp32 pairs, each thread's slice in registers
    float2 v[NV][P];
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int q = 0; q < P; ++q) v[k][q] = dup2(0.f);

    bool timed_out = false;
    if constexpr (TMA) {
      // the whole warp waits for its own chunk (one instruction a poll)
      timed_out = !mbar_wait_bounded(smem_addr(&bars[s * NW + warp]),
                                     ring_phase(ring), p.wait_limit_ns);
      if (!timed_out) {
        const uint32_t xs = smem0 + s * slot;
        if (has_r) {
#pragma unroll
          for (int k = 0; k < NV; ++k)
            if (ok[k])
              IO::sum_pairs(ld_shared_v4(xs + (v0 + 32 * k) * 16),
                            ld_shared_v4(xs + rb + (v0 + 32 * k) * 16), v[k]);
        } else {
#pragma unroll
          for (int k = 0; k < NV; ++k)
            if (ok[k]) IO::to_pairs(ld_shared_v4(xs + (v0 + 32 * k) * 16), v[k]);
        }
      }
    } else {
      const char* xrow = static_cast<const char*>(p.x) + base * S;
      uint4 xv[NV], rv[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (ok[k] && ADDLN_IN(206, base * S + (v0 + 32 * k) * 16, 16, rows_bytes(p, S)))
          xv[k] = ld_stream_v4(xrow + static_cast<int64_t>(v0 + 32 * k) * 16);
      if (has_r) {
        const char* rrow = static_cast<const char*>(p.r) + base * S;
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (ok[k] && ADDLN_IN(207, base * S + (v0 + 32 * k) * 16, 16, rows_bytes(p, S)))
            rv[k] = ld_stream_v4(rrow + static_cast<int64_t>(v0 + 32 * k) * 16);
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (ok[k]) IO::sum_pairs(xv[k], rv[k], v[k]);
      } else {
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (ok[k]) IO::to_pairs(xv[k], v[k]);
      }
    }

    // ---- A = X + R rounded to the dtype; each thread writes only what it
    // read itself, and the shift below comes from registers, so A may alias
    // X or R
    if (p.a != nullptr && !timed_out) {
      char* arow = static_cast<char*>(p.a) + base * S;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (ok[k] && ADDLN_IN(208, base * S + (v0 + 32 * k) * 16, 16, rows_bytes(p, S)))
          st_stream_v4(arow + static_cast<int64_t>(v0 + 32 * k) * 16, IO::from_pairs(v[k]));
    }

    // ---- the warp's statistics around its shift K_w (lane 0's first sum)
    const float Kw = __shfl_sync(0xffffffffu, v[0][0].x, 0);
    const float2 negK = dup2(-Kw);
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int q = 0; q < P; ++q) v[k][q] = add2(v[k][q], negK);
    Part st = thread_part2<NV, P, FULL, false>(v, ok, negK);
    st = butterfly<FULL, 32>(st);
    WarpPart* rbuf = red + ring_parity(ring) * NW;
    if (lane == 0) rbuf[warp] = WarpPart{Kw, st.n, st.m, st.M2};

    // ---- all warps' partials in; also the point after which no thread
    // reads slot s any more
    if constexpr (TMA) {
      if (__syncthreads_or(timed_out)) {
        if (tid == 0) drain_after_timeout(bars, stages, NW, ring, row, stride, p.rows);
        return;
      }
      if (lane == 0) {
        const int64_t next = row + stages * stride;
        if (next < p.rows) issue(s, next);
      }
    } else {
      __syncthreads();
    }

    // ---- CTA merge: every warp's mean moved to warp 0's shift K_0, then
    // combined (identical totals in every lane)
    const float K0 = rbuf[0].K;
    const WarpPart wp = rbuf[lane % NW];
    Part q;
    q.n = wp.n;
    q.m = wp.m + (wp.K - K0);
    q.M2 = wp.M2;
    const Part tot = butterfly<FULL, NW>(q);
    const float rstd = row_rstd(tot.M2, p.inv_h, p.eps);
    // this warp's values are a - K_w; the row mean is K_0 + m, so
    // a - mean = (a - K_w) - (m - (K_w - K_0))
    const float2 negm = dup2(-(tot.m - (Kw - K0))), rstd2 = dup2(rstd);

    // ---- normalise + affine from registers, store
    char* yrow = static_cast<char*>(p.y) + base * S;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        const int c = v0 + 32 * k;
        float2 o[P];
        if constexpr (RES) {
#pragma unroll
          for (int qq = 0; qq < P; ++qq) o[qq] = normalise2(v[k][qq], negm, rstd2, gr[k][qq], br[k][qq]);
        } else {
#pragma unroll
          for (int qq = 0; qq < P / 2; ++qq) {
            float4 g = make_float4(0.f, 0.f, 0.f, 0.f), b = g;
            if (ADDLN_IN(209, 4 * (c * VEC + 4 * qq), 16, cols_bytes(p))) {
              g = ld_param_f4(p.gamma + c * VEC + 4 * qq);
              b = ld_param_f4(p.beta + c * VEC + 4 * qq);
            }
            o[2 * qq] =
                normalise2(v[k][2 * qq], negm, rstd2, make_float2(g.x, g.y), make_float2(b.x, b.y));
            o[2 * qq + 1] =
                normalise2(v[k][2 * qq + 1], negm, rstd2, make_float2(g.z, g.w), make_float2(b.z, b.w));
          }
        }
        if (ADDLN_IN(210, base * S + c * 16, 16, rows_bytes(p, S)))
          st_stream_v4(yrow + static_cast<int64_t>(c) * 16, IO::from_pairs(o));
      }
    }
    if (tid == 0 && ADDLN_IN(211, 4 * row, 4, stat_bytes(p))) {
      if (p.mean != nullptr) p.mean[row] = K0 + tot.m;
      if (p.rstd != nullptr) p.rstd[row] = rstd;
    }
  }
}

// Element-wise variant: any alignment, any H up to the maximum.  Each thread
// keeps the fp32 sums of its own elements (j = tid + THREADS*k) in shared
// memory, so no thread reads another's slots and only the statistics need a
// barrier.  All global stores of a row follow that barrier, by which time
// every thread has read a_0, so outputs may alias inputs.
template <int DT, int THREADS>
__global__ void __launch_bounds__(THREADS) k_cta_scalar(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = p.H;
  float* sa = reinterpret_cast<float*>(smem);
  Part* red = reinterpret_cast<Part*>(smem + ((static_cast<uint32_t>(H) * 4u + 127u) & ~127u));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool has_r = p.r != nullptr;
  pdl_trigger();
  pdl_wait();

  int64_t it = 0;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
    const int64_t base = row * static_cast<int64_t>(H);
    [[maybe_unused]] constexpr int S = IO::kBytes;  // used by the checked build's tests
    float K = 0.f;
    if (ADDLN_IN(221, base * S, S, rows_bytes(p, S)))
      K = has_r ? IO::load1(p.x, base) + IO::load1(p.r, base) : IO::load1(p.x, base);
    float sum = 0.f;
    int cnt = 0;
#pragma unroll 8
    for (int j = tid; j < H; j += THREADS) {
      float a = 0.f;
      if (ADDLN_IN(222, (base + j) * S, S, rows_bytes(p, S))) {
        a = IO::load1(p.x, base + j);
        if (has_r) a += IO::load1(p.r, base + j);
      }
      sa[j] = a;
      sum += a - K;
      ++cnt;
    }
    Part st;
    st.n = static_cast<float>(cnt);
    st.m = cnt ? __fdiv_rn(sum, st.n) : 0.f;
    float M2 = 0.f;
    for (int j = tid; j < H; j += THREADS) {
      const float d = (sa[j] - K) - st.m;
      M2 = fmaf(d, d, M2);
    }
    st.M2 = M2;
    st = butterfly<false, 32>(st);
    Part* rbuf = red + (it & 1) * NW;
    if (lane == 0) rbuf[warp] = st;
    __syncthreads();
    const Part tot = cta_totals<false, NW>(rbuf, lane);
    const float rstd = row_rstd(tot.M2, p.inv_h, p.eps);
#pragma unroll 4
    for (int j = tid; j < H; j += THREADS) {
      const float a = sa[j];
      if (ADDLN_IN(223, 4 * j, 4, cols_bytes(p)) && ADDLN_IN(224, (base + j) * S, S, rows_bytes(p, S))) {
        IO::store1(p.y, base + j, normalise(a, K, tot.m, rstd, __ldg(p.gamma + j), __ldg(p.beta + j)));
        if (p.a != nullptr) IO::store1(p.a, base + j, a);
      }
    }
    if (tid == 0 && ADDLN_IN(225, 4 * row, 4, stat_bytes(p))) {
      if (p.mean != nullptr) p.mean[row] = K + tot.m;
      if (p.rstd != nullptr) p.rstd[row] = rstd;
    }
  }
}

// ------------------------------------------------------------------ host
namespace {

struct FuncKey {
  const void* f;
  int device;
  int smem;
  bool operator==(const FuncKey& o) const { return f == o.f && device == o.device && smem == o.smem; }
};
struct FuncKeyHash {
  size_t operator()(const FuncKey& k) const {
    return std::hash<const void*>()(k.f) ^ (static_cast<size_t>(k.device) << 20) ^
           (static_cast<size_t>(k.smem) << 28);
  }
};

std::mutex g_occ_mu;
std::unordered_map<FuncKey, int, FuncKeyHash> g_occ;  // resident CTAs per SM

// Resident CTAs per SM for (kernel, dynamic smem) on this device; raises the
// kernel's dynamic shared memory limit first when needed.  -1 on error.
int resident_ctas(const void* f, int threads, int smem, const DeviceInfo& dev) {
  const FuncKey key{f, dev.device, smem};
  {
    std::lock_guard<std::mutex> g(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  // The limit is per function: raise it once to the device's opt-in maximum
  // (never to this launch's size, which a later, larger launch would exceed).
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
  std::lock_guard<std::mutex> g(g_occ_mu);
  g_occ[key] = n;
  return n;
}

// One wave of resident CTAs by default; a set grid cap replaces it (and may
// exceed one wave, e.g. one CTA per row).
int64_t persistent_grid(int64_t rows, int per_sm, const LaunchCtx& c) {
  int64_t g = static_cast<int64_t>(per_sm) * c.dev.sms;
  if (c.grid_cap > 0) g = c.grid_cap;
  if (g > 0x7fffffff) g = 0x7fffffff;
  if (rows < g) g = rows;
  return g;
}

template <int DT, int THREADS, int NV, bool TMA, bool FULL>
int launch_row_t(const RowArgs& p, const LaunchCtx& c) {
  constexpr int S = Io<DT>::kBytes;
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * S;
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  const uint32_t slot = p.r ? 2u * rb : rb;
  const uint32_t extra = 8u * kMaxStages * (THREADS / 32) + 2u * (THREADS / 32) * sizeof(WarpPart);
  const void* f = reinterpret_cast<const void*>(&k_cta_row<DT, THREADS, NV, TMA, FULL>);
  int stages = 0, per_sm = 0;
  uint32_t smem = extra;
  if (TMA) {
    if (c.stages > 0) {
      if (c.stages > kMaxStages) return ADDLN_ERR_UNSUPPORTED;
      stages = c.stages;
      smem = stages * slot + extra;
      if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
      per_sm = resident_ctas(f, THREADS, static_cast<int>(smem), c.dev);
    } else if (cta_row_resident<DT, NV, TMA>()) {
      // Registers bound the CTAs an SM holds.  Two slots a CTA, unless the
      // second would cost resident CTAs, or the kernel also writes A (writes
      // then weigh as much as reads) and every CTA has more than eight rows
      // to do: there one slot measured faster (32768 x 8192 bf16), two
      // everywhere else (2048 .. 17024 x 4096 fp16, 2048 x 8192 bf16).
      smem = slot + extra;
      if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
      stages = 1;
      per_sm = resident_ctas(f, THREADS, static_cast<int>(smem), c.dev);
      if (per_sm < 0) return ADDLN_ERR_CUDA;
      const bool long_with_a =
          p.a != nullptr && p.rows > 8 * static_cast<int64_t>(per_sm) * c.dev.sms;
      const uint32_t smem2 = 2 * slot + extra;
      if (!long_with_a && smem2 <= static_cast<uint32_t>(c.dev.smem_optin)) {
        const int n2 = resident_ctas(f, THREADS, static_cast<int>(smem2), c.dev);
        if (n2 < 0) return ADDLN_ERR_CUDA;
        if (n2 >= per_sm) {
          stages = 2;
          smem = smem2;
        }
      }
    } else {
      // One slot: a second one costs more resident CTAs (rows reduced in
      // parallel) than its prefetch gains.
      stages = 1;
      smem = slot + extra;
      if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
      per_sm = resident_ctas(f, THREADS, static_cast<int>(smem), c.dev);
    }
  } else {
    per_sm = resident_ctas(f, THREADS, static_cast<int>(smem), c.dev);
  }
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  const int64_t grid = persistent_grid(p.rows, per_sm, c);
  const cudaError_t e = launch_kernel(k_cta_row<DT, THREADS, NV, TMA, FULL>,
                                      dim3(static_cast<unsigned>(grid)), dim3(THREADS), smem,
                                      c.stream, c.pdl, p, stages);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

template <int DT, int THREADS, int NV, bool TMA>
int launch_row(const RowArgs& p, const LaunchCtx& c) {
  const bool full = p.H / Io<DT>::kVec == THREADS * NV;
  return full ? launch_row_t<DT, THREADS, NV, TMA, true>(p, c)
              : launch_row_t<DT, THREADS, NV, TMA, false>(p, c);
}

// (threads, vectors per thread) by the number of 16-byte vectors in a row.
template <int DT, bool TMA>
int launch_row_dispatch(const RowArgs& p, const LaunchCtx& c, const char** name) {
  constexpr int VEC = Io<DT>::kVec;
  const int nvec = p.H / VEC;
  if (c.cta_threads != 0) {
    // Tuning shapes (TMA staging of 16-bit rows only); otherwise by H below.
    if constexpr (TMA && VEC == 8) {
      if (c.cta_threads == 128 && nvec <= 128 * 4) { *name = "cta_tma_t128_nv4"; return launch_row<DT, 128, 4, true>(p, c); }
      if (c.cta_threads == 256 && nvec <= 256 * 2) { *name = "cta_tma_t256_nv2"; return launch_row<DT, 256, 2, true>(p, c); }
      if (c.cta_threads == 512 && nvec <= 512 * 1) { *name = "cta_tma_t512_nv1"; return launch_row<DT, 512, 1, true>(p, c); }
    }
    return ADDLN_ERR_UNSUPPORTED;
  }
  if (nvec <= 128 * 2) { *name = TMA ? "cta_tma_t128_nv2" : "cta_vec_t128_nv2"; return launch_row<DT, 128, 2, TMA>(p, c); }
  if (nvec <= 128 * 4) { *name = TMA ? "cta_tma_t128_nv4" : "cta_vec_t128_nv4"; return launch_row<DT, 128, 4, TMA>(p, c); }
  if (nvec <= 256 * 4) { *name = TMA ? "cta_tma_t256_nv4" : "cta_vec_t256_nv4"; return launch_row<DT, 256, 4, TMA>(p, c); }
  if (nvec <= 512 * 4) { *name = TMA ? "cta_tma_t512_nv4" : "cta_vec_t512_nv4"; return launch_row<DT, 512, 4, TMA>(p, c); }
  // The longest rows: 512 threads with 8 vectors each (a 1024-thread CTA
  // would cap registers at 64 a thread, too few to hold the row).
  if constexpr (TMA) {
    if (nvec <= 512 * 8) { *name = "cta_tma_t512_nv8"; return launch_row<DT, 512, 8, true>(p, c); }
  }
  return ADDLN_ERR_UNSUPPORTED;
}

template <int DT>
int launch_scalar_impl(const RowArgs& p, const LaunchCtx& c) {
  constexpr int THREADS = 512;
  const uint32_t smem = ((static_cast<uint32_t>(p.H) * 4u + 127u) & ~127u) +
                        2u * (THREADS / 32) * sizeof(Part);
  if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const void* f = reinterpret_cast<const void*>(&k_cta_scalar<DT, THREADS>);
  const int per_sm = resident_ctas(f, THREADS, static_cast<int>(smem), c.dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  const int64_t grid = persistent_grid(p.rows, per_sm, c);
  const cudaError_t e = launch_kernel(k_cta_scalar<DT, THREADS>, dim3(static_cast<unsigned>(grid)),
                                      dim3(THREADS), smem, c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

}  // namespace

int launch_cta_row(int dtype, bool tma, const RowArgs& p, const LaunchCtx& c, const char** name) {
  switch (dtype) {
    case kF32: return tma ? launch_row_dispatch<kF32, true>(p, c, name) : launch_row_dispatch<kF32, false>(p, c, name);
    case kF16: return tma ? launch_row_dispatch<kF16, true>(p, c, name) : launch_row_dispatch<kF16, false>(p, c, name);
    case kBF16: return tma ? launch_row_dispatch<kBF16, true>(p, c, name) : launch_row_dispatch<kBF16, false>(p, c, name);
    default: return ADDLN_ERR_DTYPE;
  }
}

int launch_cta_scalar(int dtype, const RowArgs& p, const LaunchCtx& c, const char** name) {
  *name = "cta_scalar_t512";
  switch (dtype) {
    case kF32: return launch_scalar_impl<kF32>(p, c);
    case kF16: return launch_scalar_impl<kF16>(p, c);
    case kBF16: return launch_scalar_impl<kBF16>(p, c);
    default: return ADDLN_ERR_DTYPE;
  }
}

ADDLN_BOUNDS_READER(read_bounds_rows_cta)

int read_and_clear_device_error(void* stream, int* code) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ADDLN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  *code = v;
  return ADDLN_OK;
}

}  // namespace addln
