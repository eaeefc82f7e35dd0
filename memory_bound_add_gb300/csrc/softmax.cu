// Fused row softmax: y_j = exp(x_j - max) / sum_k exp(x_k - max), the
// reduce-elementwise pattern of fused_softmax in "算子融合与Kernel合并" 4.3
// (max reduce, exp-sum reduce, divide), with the three passes fused into one
// read of the row and one write.
//
// Two ways to reach (M, S) = (max, sum exp(x - M)):
// - max first (the 16-byte vector kernels: warp per row, CTA per row, long
//   rows): reduce M, then S = sum exp(x_j - M) and y_j = exp(x_j - M) / S,
//   in fp32 pairs with exp(d) = 2^(d log2 e) on the hardware base-2
//   exponential (relative error about 2^-22; results under 2^-126 flush to
//   zero).
// - one pass (element kernels, for rows that are not 16-byte aligned): each
//   thread takes its own maximum m_t, replaces every value by
//   e_j = exp(x_j - m_t) and sums s_t = sum e_j; partials (m, s) merge with
//   the online-softmax update
//       m = max(m_a, m_b),  s = s_a * exp(m_a - m) + s_b * exp(m_b - m),
//   whose two terms are computed the same way on either side, so the xor
//   butterfly leaves identical totals (M, S) in every lane, and
//   y_j = e_j * (exp(m_t - M) / S).  exp here is CUDA's __expf; its error
//   grows with |x - max| but stays below 1e-5 relative wherever the result
//   is above 1e-30.
//
// Kernels: one warp per row for H <= 1024 (16-byte vector or element loads);
// one CTA per row for longer rows, the row staged into shared memory by a TMA
// bulk copy on a bounded mbarrier wait (persistent grid, one row staged per
// CTA; the row then held in registers, or for the longest rows re-read from
// the staged copy), or element loads into shared memory when rows are not
// 16-byte aligned.
#include <math.h>

#include <mutex>
#include <unordered_map>

#include "../../include/addln.h"
#include "common.cuh"

namespace addln {

namespace sm {

__device__ int g_softmax_error = 0;

struct SPart {
  float m;  // maximum of the covered values (-inf when none)
  float s;  // sum of exp(value - m)
};

// Factor exp(from - to) with to >= from; exactly 1 when equal (which also
// covers two empty partials, both -inf).
__device__ __forceinline__ float rescale(float from, float to) {
  return from == to ? 1.0f : __expf(from - to);
}

__device__ __forceinline__ SPart merge(const SPart& a, const SPart& b) {
  SPart o;
  o.m = fmaxf(a.m, b.m);
  // explicit roundings keep merge(a, b) and merge(b, a) bitwise equal (a
  // contracted multiply-add would round the two sides differently)
  o.s = __fadd_rn(__fmul_rn(a.s, rescale(a.m, o.m)), __fmul_rn(b.s, rescale(b.m, o.m)));
  return o;
}

template <int WIDTH>
__device__ __forceinline__ SPart butterfly(SPart p) {
#pragma unroll
  for (int off = 1; off < WIDTH; off <<= 1) {
    SPart o;
    o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, p.s, off);
    p = merge(p, o);
  }
  return p;
}

// Thread partial: max of its values, then v <- exp(v - max) in place and
// their sum (four accumulators).
template <int NV, int VEC, bool FULL>
__device__ __forceinline__ SPart thread_part(float (&v)[NV][VEC], const bool (&ok)[NV]) {
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (FULL || ok[k])
#pragma unroll
      for (int e = 0; e < VEC; ++e) mx = fmaxf(mx, v[k][e]);
  // a slice that is all -inf contributes exp(-inf) = 0, not exp(NaN)
  const float mb = mx == -INFINITY ? 0.f : mx;
  constexpr int L = VEC >= 4 ? 4 : VEC;
  float acc[L];
#pragma unroll
  for (int l = 0; l < L; ++l) acc[l] = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (FULL || ok[k]) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        v[k][e] = __expf(v[k][e] - mb);
        acc[e % L] += v[k][e];
      }
    }
  }
  float s = acc[0];
#pragma unroll
  for (int l = 1; l < L; ++l) s += acc[l];
  return SPart{mx, s};
}

// Largest value of a 16-byte vector (the non-NaN operand of a pair, as
// fmaxf); 16-bit vectors are compared as packed pairs, without widening.
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& u) {
  if constexpr (DT == kF32) {
    return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                 fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
  } else if constexpr (DT == kF16) {
    const __half2 a = __hmax2(*reinterpret_cast<const __half2*>(&u.x), *reinterpret_cast<const __half2*>(&u.y));
    const __half2 b = __hmax2(*reinterpret_cast<const __half2*>(&u.z), *reinterpret_cast<const __half2*>(&u.w));
    const __half2 c = __hmax2(a, b);
    return __half2float(__hmax(__low2half(c), __high2half(c)));
  } else {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.z),
                                     *reinterpret_cast<const __nv_bfloat162*>(&u.w));
    const __nv_bfloat162 c = __hmax2(a, b);
    return __bfloat162float(__hmax(__low2bfloat16(c), __high2bfloat16(c)));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// exp(d) = 2^(d log2 e), by the hardware base-2 exponential (PTX
// ex2.approx, relative error about 2^-22), on a pair of values.  Results
// below 2^-126 flush to zero (.ftz): far under the 1e-12 absolute floor of
// any softmax output that matters, and one instruction instead of several.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}
__device__ __forceinline__ float2 exp_pair(float2 v, float2 negm, float2 log2e) {
  const float2 t = mul2(add2(v, negm), log2e);
  return make_float2(ex2(t.x), ex2(t.y));
}

// ------------------------------------------------------ warp per row
constexpr int kWarpCtaThreads = 128;
constexpr int kRowsPerCta = kWarpCtaThreads / 32;

// 16-byte rows: the warp's maximum M first (16-bit values compared as packed
// pairs, then a five-step xor butterfly), so every exponential is
// exp(x - M) and the sum needs no rescaling; exponentials, their sum and
// the scaling by 1/S run on fp32 pairs.  Element rows: each thread keeps
// exp(x - m_t) of its own elements and the (m, s) partials merge by the
// online update.
template <int DT, int NV, bool VECTOR, bool FULL>
__global__ void __launch_bounds__(kWarpCtaThreads, 2) k_softmax_warp(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = VECTOR ? IO::kVec : 1;
  constexpr int S = IO::kBytes;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  pdl_trigger();
  pdl_wait();
  if (row >= p.rows) return;
  const int nvec = p.H / VEC;
  const int64_t base = row * static_cast<int64_t>(p.H);

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (lane + 32 * k) < nvec;

  if constexpr (VECTOR) {
    constexpr int P = VEC / 2;
    const char* xrow = static_cast<const char*>(p.x) + base * S;
    uint4 xv[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(301, base * S + (lane + 32 * k) * 16, 16, rows_bytes(p, S)))
        xv[k] = ld_stream_v4(xrow + static_cast<int64_t>(lane + 32 * k) * 16);
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k]) mx = fmaxf(mx, vec_max<DT>(xv[k]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // a row that is all -inf gives exp(-inf) = 0 terms, not exp(NaN)
    const float2 negm = dup2(mx == -INFINITY ? 0.f : -mx);
    const float2 log2e = dup2(kLog2e);
    float2 e[NV][P];
    float2 acc[2] = {dup2(0.f), dup2(0.f)};
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        IO::to_pairs(xv[k], e[k]);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          e[k][q] = exp_pair(e[k][q], negm, log2e);
          acc[q & 1] = add2(acc[q & 1], e[k][q]);
        }
      }
    }
    const float2 inv = dup2(1.0f / warp_sum((acc[0].x + acc[1].x) + (acc[0].y + acc[1].y)));
    char* yrow = static_cast<char*>(p.y) + base * S;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
#pragma unroll
        for (int q = 0; q < P; ++q) e[k][q] = mul2(e[k][q], inv);
        if (ADDLN_IN(302, base * S + (lane + 32 * k) * 16, 16, rows_bytes(p, S)))
          st_stream_v4(yrow + static_cast<int64_t>(lane + 32 * k) * 16, IO::from_pairs(e[k]));
      }
    }
  } else {
    float v[NV][1];
#pragma unroll
    for (int k = 0; k < NV; ++k)
      v[k][0] = ok[k] && ADDLN_IN(303, (base + lane + 32 * k) * S, S, rows_bytes(p, S))
                    ? IO::load1(p.x, base + lane + 32 * k)
                    : 0.f;
    const SPart mine = thread_part<NV, 1, FULL>(v, ok);
    const SPart tot = butterfly<32>(mine);
    const float f = rescale(mine.m, tot.m) / tot.s;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ok[k] && ADDLN_IN(304, (base + lane + 32 * k) * S, S, rows_bytes(p, S)))
        IO::store1(p.y, base + lane + 32 * k, v[k][0] * f);
  }
}

// ------------------------------------------------------ CTA per row (TMA)
// Max first, as in the warp kernel: the row's 16-byte vectors stay packed in
// registers while the CTA agrees on the maximum M (warp maxima through
// shared memory, one barrier, after which the staging slot is refilled);
// then exp(x - M) on fp32 pairs and their sum S (warp sums, a second
// barrier), and y = exp(x - M) / S.  Each buffer of the warps' partials
// alternates with the row's parity, so a warp that runs ahead into the next
// row never overwrites values a slower warp is still reading.
template <int DT, int THREADS, int NV, bool FULL>
__global__ void __launch_bounds__(THREADS) k_softmax_cta(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;
  constexpr int S = IO::kBytes;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = p.H / VEC;
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * S;  // multiple of 16
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + rb);
  SPart* red = reinterpret_cast<SPart*>(smem + rb + 16);  // [2][NW]: warp maxima (m), sums (s)
  const uint32_t xs = smem_addr(smem);
  const uint32_t bar_a = smem_addr(bar);
  const float2 log2e = dup2(kLog2e);

  bool ok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) ok[k] = FULL || (tid + THREADS * k) < nvec;

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
    // checked build: a copy that would leave X is not issued (nor expected)
    const bool okx = ADDLN_IN(305, rr * static_cast<int64_t>(row_bytes), row_bytes, rows_bytes(p, S));
    mbar_arrive_expect_tx(bar_a, okx ? row_bytes : 0u);
    if (okx)
      bulk_g2s(xs, static_cast<const char*>(p.x) + rr * static_cast<int64_t>(row_bytes), row_bytes,
               bar_a, policy);
  };
  if (tid == 0 && row < p.rows) issue(row);

  for (uint32_t par = 0; row < p.rows; par ^= 1u, row += stride) {
    const bool timed_out = !mbar_wait_bounded(bar_a, par, p.wait_limit_ns);
    uint4 raw[NV];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k] && !timed_out) {
        raw[k] = ld_shared_v4(xs + (tid + THREADS * k) * 16);
        mx = fmaxf(mx, vec_max<DT>(raw[k]));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    SPart* rbuf = red + par * NW;
    if (lane == 0) rbuf[warp].m = mx;
    // every thread has its slice in registers: the slot may be refilled
    if (__syncthreads_or(timed_out)) {
      if (tid == 0) {
        atomicExch(&g_softmax_error, ADDLN_ERR_DEVICE_TIMEOUT);
        mbar_wait_bounded(bar_a, par, 1000000000ull);
      }
      return;
    }
    if (tid == 0 && row + stride < p.rows) issue(row + stride);
    mx = rbuf[0].m;
#pragma unroll
    for (int w = 1; w < NW; ++w) mx = fmaxf(mx, rbuf[w].m);
    // a row that is all -inf gives exp(-inf) = 0 terms, not exp(NaN)
    const float2 negm = dup2(mx == -INFINITY ? 0.f : -mx);
    float2 e[NV][P];
    float2 acc[2] = {dup2(0.f), dup2(0.f)};
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
        IO::to_pairs(raw[k], e[k]);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          e[k][q] = exp_pair(e[k][q], negm, log2e);
          acc[q & 1] = add2(acc[q & 1], e[k][q]);
        }
      }
    }
    const float ws = warp_sum((acc[0].x + acc[1].x) + (acc[0].y + acc[1].y));
    if (lane == 0) rbuf[warp].s = ws;
    __syncthreads();
    float sum = rbuf[0].s;
#pragma unroll
    for (int w = 1; w < NW; ++w) sum += rbuf[w].s;
    const float2 inv = dup2(1.0f / sum);
    char* yrow = static_cast<char*>(p.y) + row * static_cast<int64_t>(row_bytes);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (ok[k]) {
#pragma unroll
        for (int q = 0; q < P; ++q) e[k][q] = mul2(e[k][q], inv);
        if (ADDLN_IN(306, row * static_cast<int64_t>(row_bytes) + (tid + THREADS * k) * 16, 16,
                     rows_bytes(p, S)))
          st_stream_v4(yrow + static_cast<int64_t>(tid + THREADS * k) * 16, IO::from_pairs(e[k]));
      }
    }
  }
}

// ------------------------------------------- CTA per row, long rows (TMA)
// Rows too long to sit in the registers of several CTAs per SM (more than
// 2048 16-byte vectors) stay in their staged shared-memory copy (three CTAs,
// rows, per SM) and are read three times: the row maximum M (16-bit values
// compared as packed pairs), then S = sum exp(x - M), then y = exp(x - M) / S
// (fp32 pair arithmetic).  With M known before any exponential is taken the
// sum needs no rescaling, and the passes issue about a third of the
// instructions of a running (max, sum) pass.  Warp w owns the contiguous
// chunk w of every row (ceil(vectors / warps) vectors), staged by its own
// bulk copy onto its own mbarrier: it starts as soon as its chunk lands, and
// once it has written its chunk of y it refills the chunk with the CTA's next
// row while the other warps are still normalising theirs.
template <int DT, int THREADS>
__global__ void __launch_bounds__(THREADS) k_softmax_cta_smem(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int VEC = IO::kVec;
  constexpr int P = VEC / 2;
  constexpr int S = IO::kBytes;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = p.H / VEC;
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * S;  // multiple of 16
  const uint32_t rb = (row_bytes + 127u) & ~127u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + rb);  // [NW]
  float* redm = reinterpret_cast<float*>(smem + rb + 8u * NW);  // [NW] warp maxima
  float* reds = redm + NW;                                       // [NW] warp sums
  const uint32_t xs = smem_addr(smem);
  const uint32_t bar_w = smem_addr(&bars[warp]);
  // this warp's chunk of every row: vectors [c0, c0 + cvecs)
  const int cw = (nvec + NW - 1) / NW;
  const int c0 = min(warp * cw, nvec);
  const int cvecs = min(cw, nvec - c0);
  const uint32_t chunk_off = static_cast<uint32_t>(c0) * 16u;
  const uint32_t chunk_bytes = static_cast<uint32_t>(cvecs) * 16u;
  const float2 log2e = dup2(kLog2e);

  if (tid == 0) {
    for (int w = 0; w < NW; ++w) mbar_init(smem_addr(&bars[w]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t policy = policy_evict_first();
  pdl_trigger();
  pdl_wait();

  const int64_t stride = gridDim.x;
  int64_t row = blockIdx.x;
  auto issue = [&](int64_t rr) {  // lane 0: the warp's chunk of row rr
    const int64_t off = rr * static_cast<int64_t>(row_bytes) + chunk_off;
    const bool okx = ADDLN_IN(307, off, chunk_bytes, rows_bytes(p, S));
    mbar_arrive_expect_tx(bar_w, okx ? chunk_bytes : 0u);
    if (chunk_bytes != 0 && okx)
      bulk_g2s(xs + chunk_off, static_cast<const char*>(p.x) + off, chunk_bytes, bar_w, policy);
  };
  if (lane == 0 && row < p.rows) issue(row);

  for (int64_t it = 0; row < p.rows; ++it, row += stride) {
    const bool timed_out =
        __any_sync(0xffffffffu, !mbar_wait_bounded(bar_w, static_cast<uint32_t>(it & 1), p.wait_limit_ns));
    // pass 1: the row maximum
    float mx = -INFINITY;
    if (!timed_out)
      for (int c = c0 + lane; c < c0 + cvecs; c += 32) mx = fmaxf(mx, vec_max<DT>(ld_shared_v4(xs + c * 16)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) redm[warp] = mx;
    if (__syncthreads_or(timed_out)) {
      if (tid == 0) {
        // each warp's chunk of this row is the only copy in flight
        atomicExch(&g_softmax_error, ADDLN_ERR_DEVICE_TIMEOUT);
        for (int w = 0; w < NW; ++w)
          mbar_wait_bounded(smem_addr(&bars[w]), static_cast<uint32_t>(it & 1), 1000000000ull);
      }
      return;
    }
    mx = redm[lane % NW];
#pragma unroll
    for (int off = 1; off < NW; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float2 negm = dup2(mx == -INFINITY ? 0.f : -mx);
    // pass 2: S = sum exp(x - M)
    float2 acc = dup2(0.f);
    for (int c = c0 + lane; c < c0 + cvecs; c += 32) {
      float2 v[P];
      IO::to_pairs(ld_shared_v4(xs + c * 16), v);
#pragma unroll
      for (int q = 0; q < P; ++q) acc = add2(acc, exp_pair(v[q], negm, log2e));
    }
    float sum = warp_sum(acc.x + acc.y);
    if (lane == 0) reds[warp] = sum;
    __syncthreads();
    sum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) sum += reds[w];
    const float2 inv = dup2(1.0f / sum);
    // pass 3: normalise this warp's chunk from the staged copy
    char* yrow = static_cast<char*>(p.y) + row * static_cast<int64_t>(row_bytes);
    for (int c = c0 + lane; c < c0 + cvecs; c += 32) {
      float2 v[P];
      IO::to_pairs(ld_shared_v4(xs + c * 16), v);
#pragma unroll
      for (int q = 0; q < P; ++q) v[q] = mul2(exp_pair(v[q], negm, log2e), inv);
      if (ADDLN_IN(308, row * static_cast<int64_t>(row_bytes) + c * 16, 16, rows_bytes(p, S)))
        st_stream_v4(yrow + static_cast<int64_t>(c) * 16, IO::from_pairs(v));
    }
    // every lane of the warp is done with its chunk before it is refilled
    __syncwarp();
    if (lane == 0 && row + stride < p.rows) issue(row + stride);
  }
}

// ------------------------------------------------ CTA per row, elements
// Misaligned rows: element loads; each thread keeps exp(x_j - m_t) of its own
// elements (j = tid + THREADS*k) in shared memory.  Every store of a row
// follows the row's barrier, so y may be x.
template <int DT, int THREADS>
__global__ void __launch_bounds__(THREADS) k_softmax_scalar(const RowArgs p) {
  using IO = Io<DT>;
  constexpr int NW = THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = p.H;
  float* se = reinterpret_cast<float*>(smem);
  SPart* red = reinterpret_cast<SPart*>(smem + ((static_cast<uint32_t>(H) * 4u + 127u) & ~127u));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  int64_t it = 0;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x, ++it) {
    const int64_t base = row * static_cast<int64_t>(H);
    float mx = -INFINITY;
#pragma unroll 8
    for (int j = tid; j < H; j += THREADS) {
      const float a = ADDLN_IN(309, (base + j) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes))
                          ? IO::load1(p.x, base + j)
                          : 0.f;
      se[j] = a;
      mx = fmaxf(mx, a);
    }
    const float mb = mx == -INFINITY ? 0.f : mx;
    float s = 0.f;
    for (int j = tid; j < H; j += THREADS) {
      const float e = __expf(se[j] - mb);
      se[j] = e;
      s += e;
    }
    const SPart mine{mx, s};
    const SPart wp = butterfly<32>(mine);
    SPart* rbuf = red + (it & 1) * NW;
    if (lane == 0) rbuf[warp] = wp;
    __syncthreads();
    const SPart tot = butterfly<NW>(rbuf[lane % NW]);
    const float f = rescale(mine.m, tot.m) / tot.s;
#pragma unroll 4
    for (int j = tid; j < H; j += THREADS)
      if (ADDLN_IN(310, (base + j) * IO::kBytes, IO::kBytes, rows_bytes(p, IO::kBytes)))
        IO::store1(p.y, base + j, se[j] * f);
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
  std::lock_guard<std::mutex> g(g_mu);
  g_occ[key] = n;
  return n;
}

int64_t grid_for(int64_t rows, int per_sm, const LaunchCtx& c) {
  int64_t g = static_cast<int64_t>(per_sm) * c.dev.sms;
  if (c.grid_cap > 0) g = c.grid_cap;
  if (g > 0x7fffffff) g = 0x7fffffff;
  return rows < g ? rows : g;
}

template <int DT, int NV, bool VECTOR>
int warp_launch(const RowArgs& p, const LaunchCtx& c) {
  const int64_t blocks = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  if (blocks > 0x7fffffff) return ADDLN_ERR_UNSUPPORTED;
  constexpr int VEC = VECTOR ? Io<DT>::kVec : 1;
  const bool full = p.H / VEC == 32 * NV;
  const dim3 grid(static_cast<unsigned>(blocks));
  const cudaError_t e =
      full ? launch_kernel(k_softmax_warp<DT, NV, VECTOR, true>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p)
           : launch_kernel(k_softmax_warp<DT, NV, VECTOR, false>, grid, dim3(kWarpCtaThreads), 0, c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

template <int DT>
int warp_dispatch(bool vec, const RowArgs& p, const LaunchCtx& c, const char** name) {
  if (vec) {
    constexpr int VEC = Io<DT>::kVec;
    const int nv = (p.H / VEC + 31) / 32;
    if (nv <= 1) { *name = "softmax_warp_vec_nv1"; return warp_launch<DT, 1, true>(p, c); }
    if (nv <= 2) { *name = "softmax_warp_vec_nv2"; return warp_launch<DT, 2, true>(p, c); }
    if (nv <= 4) { *name = "softmax_warp_vec_nv4"; return warp_launch<DT, 4, true>(p, c); }
    if constexpr (VEC == 4)
      if (nv <= 8) { *name = "softmax_warp_vec_nv8"; return warp_launch<DT, 8, true>(p, c); }
    return ADDLN_ERR_UNSUPPORTED;
  }
  const int nv = (p.H + 31) / 32;
  if (nv <= 4) { *name = "softmax_warp_scalar_nv4"; return warp_launch<DT, 4, false>(p, c); }
  if (nv <= 8) { *name = "softmax_warp_scalar_nv8"; return warp_launch<DT, 8, false>(p, c); }
  if (nv <= 16) { *name = "softmax_warp_scalar_nv16"; return warp_launch<DT, 16, false>(p, c); }
  if (nv <= 32) { *name = "softmax_warp_scalar_nv32"; return warp_launch<DT, 32, false>(p, c); }
  return ADDLN_ERR_UNSUPPORTED;
}

template <int DT, int THREADS, int NV, bool FULL>
int cta_launch_t(const RowArgs& p, const LaunchCtx& c) {
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * Io<DT>::kBytes;
  const uint32_t smem = ((row_bytes + 127u) & ~127u) + 16u + 2u * (THREADS / 32) * sizeof(SPart);
  if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const void* f = reinterpret_cast<const void*>(&k_softmax_cta<DT, THREADS, NV, FULL>);
  const int per_sm = resident(f, THREADS, static_cast<int>(smem), c.dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  const int64_t grid = grid_for(p.rows, per_sm, c);
  const cudaError_t e = launch_kernel(k_softmax_cta<DT, THREADS, NV, FULL>,
                                      dim3(static_cast<unsigned>(grid)), dim3(THREADS), smem,
                                      c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

template <int DT, int THREADS, int NV>
int cta_launch(const RowArgs& p, const LaunchCtx& c) {
  return p.H / Io<DT>::kVec == THREADS * NV ? cta_launch_t<DT, THREADS, NV, true>(p, c)
                                            : cta_launch_t<DT, THREADS, NV, false>(p, c);
}

template <int DT>
int smem_launch(const RowArgs& p, const LaunchCtx& c) {
  constexpr int THREADS = 256;
  const uint32_t row_bytes = static_cast<uint32_t>(p.H) * Io<DT>::kBytes;
  const uint32_t smem = ((row_bytes + 127u) & ~127u) + 16u * (THREADS / 32);
  if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const void* f = reinterpret_cast<const void*>(&k_softmax_cta_smem<DT, THREADS>);
  const int per_sm = resident(f, THREADS, static_cast<int>(smem), c.dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  const int64_t grid = grid_for(p.rows, per_sm, c);
  const cudaError_t e = launch_kernel(k_softmax_cta_smem<DT, THREADS>,
                                      dim3(static_cast<unsigned>(grid)), dim3(THREADS), smem,
                                      c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

// Rows up to 2048 vectors: registers hold the row; longer rows: the staged
// copy holds it (k_softmax_cta_smem).  cta_shape threads = 512 forces the
// register variant for the longest rows too (comparison).
template <int DT>
int cta_dispatch(const RowArgs& p, const LaunchCtx& c, const char** name) {
  const int nvec = p.H / Io<DT>::kVec;
  if (nvec <= 128 * 4) { *name = "softmax_cta_tma_t128_nv4"; return cta_launch<DT, 128, 4>(p, c); }
  if (nvec <= 256 * 4) { *name = "softmax_cta_tma_t256_nv4"; return cta_launch<DT, 256, 4>(p, c); }
  if (nvec <= 512 * 4) { *name = "softmax_cta_tma_t512_nv4"; return cta_launch<DT, 512, 4>(p, c); }
  if (c.cta_threads == 512 && nvec <= 512 * 8) {
    *name = "softmax_cta_tma_t512_nv8";
    return cta_launch<DT, 512, 8>(p, c);
  }
  *name = "softmax_cta_tma_smem_t256";
  return smem_launch<DT>(p, c);
}

template <int DT>
int scalar_launch(const RowArgs& p, const LaunchCtx& c) {
  constexpr int THREADS = 512;
  const uint32_t smem = ((static_cast<uint32_t>(p.H) * 4u + 127u) & ~127u) +
                        2u * (THREADS / 32) * sizeof(SPart);
  if (smem > static_cast<uint32_t>(c.dev.smem_optin)) return ADDLN_ERR_UNSUPPORTED;
  const void* f = reinterpret_cast<const void*>(&k_softmax_scalar<DT, THREADS>);
  const int per_sm = resident(f, THREADS, static_cast<int>(smem), c.dev);
  if (per_sm < 0) return ADDLN_ERR_CUDA;
  if (per_sm == 0) return ADDLN_ERR_UNSUPPORTED;
  const int64_t grid = grid_for(p.rows, per_sm, c);
  const cudaError_t e = launch_kernel(k_softmax_scalar<DT, THREADS>, dim3(static_cast<unsigned>(grid)),
                                      dim3(THREADS), smem, c.stream, c.pdl, p);
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e));
  return e == cudaSuccess ? ADDLN_OK : ADDLN_ERR_LAUNCH;
}

}  // namespace
}  // namespace sm

int launch_softmax_warp(int dtype, bool vec, const RowArgs& p, const LaunchCtx& c, const char** name) {
  switch (dtype) {
    case kF32: return sm::warp_dispatch<kF32>(vec, p, c, name);
    case kF16: return sm::warp_dispatch<kF16>(vec, p, c, name);
    case kBF16: return sm::warp_dispatch<kBF16>(vec, p, c, name);
    default: return ADDLN_ERR_DTYPE;
  }
}

int launch_softmax_cta(int dtype, const RowArgs& p, const LaunchCtx& c, const char** name) {
  switch (dtype) {
    case kF32: return sm::cta_dispatch<kF32>(p, c, name);
    case kF16: return sm::cta_dispatch<kF16>(p, c, name);
    case kBF16: return sm::cta_dispatch<kBF16>(p, c, name);
    default: return ADDLN_ERR_DTYPE;
  }
}

int launch_softmax_scalar(int dtype, const RowArgs& p, const LaunchCtx& c, const char** name) {
  *name = "softmax_cta_scalar_t512";
  switch (dtype) {
    case kF32: return sm::scalar_launch<kF32>(p, c);
    case kF16: return sm::scalar_launch<kF16>(p, c);
    case kBF16: return sm::scalar_launch<kBF16>(p, c);
    default: return ADDLN_ERR_DTYPE;
  }
}

ADDLN_BOUNDS_READER(read_bounds_softmax)

int read_and_clear_softmax_error(int* code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, sm::g_softmax_error, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(sm::g_softmax_error, &zero, sizeof(int)) != cudaSuccess) return ADDLN_ERR_CUDA;
  *code = v;
  return ADDLN_OK;
}

}  // namespace addln
