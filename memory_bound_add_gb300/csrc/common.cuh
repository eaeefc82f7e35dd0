// Device-side building blocks shared by the row kernels: I/O dtype traits,
// 16-byte vector (un)packing, inline-PTX memory operations (streaming loads
// and stores, mbarrier, TMA bulk copy) and the Chan combination of partial
// (count, mean, M2) statistics.
//
// The statistics follow the LayerNorm of "算子融合与Kernel合并" 4.2 (mean,
// then the biased variance around it, eps inside the square root) but are
// gathered in one pass over registers: each thread takes the exact two-pass
// mean/M2 of the values it holds (shifted by the row's first value), and
// partial results are merged with Chan, Golub and LeVeque's pairwise update.  The
// page's own one-pass shortcut (sum and sum of squares, same page 4.3) is
// avoided: it cancels when the row mean is large against its spread.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace addln {

// ----------------------------------------------------------- checked build
// Built with -DADDLN_CHECK_BOUNDS, every global access of the kernels is
// first tested against the extent of the buffer it falls in, taken from the
// launch's own arguments (rows, H, element size, grid).  An access that would
// leave its buffer is skipped, and the first one met is recorded in this
// translation unit's bounds word: bit 63 set, the site number in bits 48..62,
// the byte offset in bits 0..47.  addln_get_device_error reports it as
// ADDLN_ERR_BOUNDS.  Skipping rather than trapping keeps the context usable,
// so one process can run the checked library over many shapes.  In the
// normal build ADDLN_IN is the constant true and compiles away.
#ifdef ADDLN_CHECK_BOUNDS
static __device__ unsigned long long g_bounds_error = 0;
__device__ __forceinline__ bool in_bounds(int site, int64_t off, int64_t len, int64_t extent) {
  // an access of no bytes touches nothing (e.g. a warp past a short row's
  // last vector, whose copy is never issued)
  if (len == 0 || (off >= 0 && len > 0 && off + len <= extent)) return true;
  atomicCAS(&g_bounds_error, 0ull,
            (1ull << 63) | (static_cast<unsigned long long>(site & 0x7fff) << 48) |
                (static_cast<unsigned long long>(off) & 0xffffffffffffull));
  return false;
}
#define ADDLN_IN(site, off, len, extent) \
  ::addln::in_bounds((site), static_cast<int64_t>(off), static_cast<int64_t>(len), \
                     static_cast<int64_t>(extent))
// Host: reads and clears this translation unit's bounds word.
#define ADDLN_BOUNDS_READER(fn)                                                              \
  int fn(unsigned long long* out) {                                                          \
    unsigned long long v = 0, zero = 0;                                                      \
    if (cudaMemcpyFromSymbol(&v, ::addln::g_bounds_error, sizeof(v)) != cudaSuccess ||       \
        cudaMemcpyToSymbol(::addln::g_bounds_error, &zero, sizeof(zero)) != cudaSuccess)     \
      return ADDLN_ERR_CUDA;                                                                 \
    *out = v;                                                                                \
    return ADDLN_OK;                                                                         \
  }
#else
#define ADDLN_IN(site, off, len, extent) true
#define ADDLN_BOUNDS_READER(fn)    \
  int fn(unsigned long long* out) { \
    *out = 0;                       \
    return ADDLN_OK;                \
  }
#endif

// Byte extents of a row launch's buffers (for ADDLN_IN): a [rows, H] tensor
// in the I/O dtype, a per-column fp32 [H] vector, a per-row fp32 [rows] one.
__device__ __forceinline__ int64_t rows_bytes(const RowArgs& p, int elem) {
  return p.rows * static_cast<int64_t>(p.H) * elem;
}
__device__ __forceinline__ int64_t cols_bytes(const RowArgs& p) { return 4 * static_cast<int64_t>(p.H); }
__device__ __forceinline__ int64_t stat_bytes(const RowArgs& p) { return 4 * p.rows; }

// ------------------------------------------------------------ fp32 pairs
// sm_100 and later execute an fp32 add, multiply or fma on a pair of values
// as one instruction.  The vector paths of the row kernels keep their fp32
// values as float2 pairs and do their element-wise arithmetic through these;
// each is the correctly rounded scalar operation applied to .x and to .y.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 dup2(float s) { return make_float2(s, s); }

// ------------------------------------------------------------ dtype traits
// unpack / pack: a 16-byte vector to and from fp32 values; to_pairs /
// from_pairs: the same as kVec/2 float2 pairs; sum_pairs: a = x + r for
// each element of two vectors, as pairs (the exact fp32 value of each input,
// one rounding of the sum).
template <int DT>
struct Io;

template <>
struct Io<kF32> {
  static constexpr int kBytes = 4;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ static __forceinline__ void to_pairs(const uint4& u, float2* f) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
  __device__ static __forceinline__ uint4 from_pairs(const float2* f) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
  }
  __device__ static __forceinline__ void sum_pairs(const uint4& x, const uint4& r, float2* a) {
    float2 t[2], u[2];
    to_pairs(x, t);
    to_pairs(r, u);
    a[0] = add2(t[0], u[0]);
    a[1] = add2(t[1], u[1]);
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};

template <>
struct Io<kF16> {
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ float2 w2f(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
  __device__ static __forceinline__ uint32_t f2w(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ void unpack(const uint4& u, float* f) {
    float2 t;
    t = w2f(u.x); f[0] = t.x; f[1] = t.y;
    t = w2f(u.y); f[2] = t.x; f[3] = t.y;
    t = w2f(u.z); f[4] = t.x; f[5] = t.y;
    t = w2f(u.w); f[6] = t.x; f[7] = t.y;
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(f2w(f[0], f[1]), f2w(f[2], f[3]), f2w(f[4], f[5]), f2w(f[6], f[7]));
  }
  __device__ static __forceinline__ void to_pairs(const uint4& u, float2* f) {
    f[0] = w2f(u.x);
    f[1] = w2f(u.y);
    f[2] = w2f(u.z);
    f[3] = w2f(u.w);
  }
  __device__ static __forceinline__ uint4 from_pairs(const float2* f) {
    return make_uint4(f2w(f[0].x, f[0].y), f2w(f[1].x, f[1].y), f2w(f[2].x, f[2].y),
                      f2w(f[3].x, f[3].y));
  }
  // Both halves of a word of X widened, then each added to the matching half
  // of R by the mixed-precision add (f16 operand + f32 operand -> f32).
  __device__ static __forceinline__ float2 word_sum(uint32_t xw, uint32_t rw) {
    float2 o;
    asm("{\n\t.reg .b16 x0, x1, r0, r1;\n\t.reg .f32 f0, f1;\n\t"
        "mov.b32 {x0, x1}, %2;\n\tmov.b32 {r0, r1}, %3;\n\t"
        "cvt.f32.f16 f0, x0;\n\tcvt.f32.f16 f1, x1;\n\t"
        "add.rn.f32.f16 %0, r0, f0;\n\tadd.rn.f32.f16 %1, r1, f1;\n\t}"
        : "=f"(o.x), "=f"(o.y)
        : "r"(xw), "r"(rw));
    return o;
  }
  __device__ static __forceinline__ void sum_pairs(const uint4& x, const uint4& r, float2* a) {
    a[0] = word_sum(x.x, r.x);
    a[1] = word_sum(x.y, r.y);
    a[2] = word_sum(x.z, r.z);
    a[3] = word_sum(x.w, r.w);
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    unsigned short b = __ldg(static_cast<const unsigned short*>(p) + i);
    return __half2float(__ushort_as_half(b));
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  }
};

template <>
struct Io<kBF16> {
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ float2 w2f(uint32_t w) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(h);
  }
  __device__ static __forceinline__ uint32_t f2w(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ void unpack(const uint4& u, float* f) {
    float2 t;
    t = w2f(u.x); f[0] = t.x; f[1] = t.y;
    t = w2f(u.y); f[2] = t.x; f[3] = t.y;
    t = w2f(u.z); f[4] = t.x; f[5] = t.y;
    t = w2f(u.w); f[6] = t.x; f[7] = t.y;
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(f2w(f[0], f[1]), f2w(f[2], f[3]), f2w(f[4], f[5]), f2w(f[6], f[7]));
  }
  __device__ static __forceinline__ void to_pairs(const uint4& u, float2* f) {
    f[0] = w2f(u.x);
    f[1] = w2f(u.y);
    f[2] = w2f(u.z);
    f[3] = w2f(u.w);
  }
  __device__ static __forceinline__ uint4 from_pairs(const float2* f) {
    return make_uint4(f2w(f[0].x, f[0].y), f2w(f[1].x, f[1].y), f2w(f[2].x, f[2].y),
                      f2w(f[3].x, f[3].y));
  }
  __device__ static __forceinline__ float2 word_sum(uint32_t xw, uint32_t rw) {
    float2 o;
    asm("{\n\t.reg .b16 x0, x1, r0, r1;\n\t.reg .f32 f0, f1;\n\t"
        "mov.b32 {x0, x1}, %2;\n\tmov.b32 {r0, r1}, %3;\n\t"
        "cvt.f32.bf16 f0, x0;\n\tcvt.f32.bf16 f1, x1;\n\t"
        "add.rn.f32.bf16 %0, r0, f0;\n\tadd.rn.f32.bf16 %1, r1, f1;\n\t}"
        : "=f"(o.x), "=f"(o.y)
        : "r"(xw), "r"(rw));
    return o;
  }
  __device__ static __forceinline__ void sum_pairs(const uint4& x, const uint4& r, float2* a) {
    a[0] = word_sum(x.x, r.x);
    a[1] = word_sum(x.y, r.y);
    a[2] = word_sum(x.z, r.z);
    a[3] = word_sum(x.w, r.w);
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    unsigned short b = __ldg(static_cast<const unsigned short*>(p) + i);
    return __bfloat162float(__ushort_as_bfloat16(b));
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

// --------------------------------------------------------- global memory
// Streaming 16-byte load of data that is read exactly once: read-only path,
// no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Streaming 16-byte store (evict-first): outputs are not re-read here.
__device__ __forceinline__ void st_stream_v4(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// gamma / beta: re-read by every row, so keep them cached.
__device__ __forceinline__ float4 ld_param_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ------------------------------------------- programmatic dependent launch
// Every kernel here lets the next kernel in the stream start launching as
// soon as all of its CTAs are running, and waits for the previous kernel's
// grid to complete (memory flushed) before its first global access, so a
// dependent chain keeps its order while launch latency and CTA prologues
// overlap the previous kernel's tail.  Both are no-ops without the launch
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches kernel<<<grid, block, smem, stream>>>(args...), with the
// programmatic-stream-serialisation attribute when pdl is set.
template <typename... KArgs, typename... Args>
__host__ cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   void* stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------- shared memory
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// --------------------------------------------------- mbarrier + TMA bulk
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One-dimensional bulk copy global -> shared, completing `bytes` of the
// barrier's transaction count.  src, dst 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Ask L2 for [src, src + bytes) (16-byte aligned, a multiple of 16 bytes).  A
// hint only: it returns nothing and changes no value anyone reads, and since
// writes from every SM land in L2, a line fetched before another kernel
// writes it is updated in place, never read stale.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy of ordinary priority (a bulk copy given no hint gets the same).
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Tests phase `parity`; if it is not complete the thread may be suspended
// (not spinning, so it takes no issue slots) until the phase completes or
// about suspend_ns nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A ring of `stages` staging slots walked one row at a time, held in one
// register: bit 0 the row's parity (alternates every row), bit 1 the slot's
// mbarrier phase, bits 2 and up the slot.  For the it-th row: slot
// it % stages, phase (it / stages) & 1, parity it & 1, advanced without a
// division.
__device__ __forceinline__ uint32_t ring_slot(uint32_t r) { return r >> 2; }
__device__ __forceinline__ uint32_t ring_phase(uint32_t r) { return (r >> 1) & 1u; }
__device__ __forceinline__ uint32_t ring_parity(uint32_t r) { return r & 1u; }
__device__ __forceinline__ uint32_t ring_next(uint32_t r, int stages) {
  const uint32_t par = (r & 1u) ^ 1u;
  const uint32_t slot = (r >> 2) + 1u;
  return slot == static_cast<uint32_t>(stages) ? ((((r >> 1) & 1u) ^ 1u) << 1) | par
                                               : (slot << 2) | (r & 2u) | par;
}

// Waits for phase `parity` of the barrier, giving up after limit_ns
// nanoseconds (limit 0: give up without waiting).  Returns true once the
// phase has completed.  try_wait gives up after a short, hardware-chosen
// time, so a warp waiting on HBM would otherwise re-poll every ~100 ns and
// take issue slots from the warps that are computing; between polls it
// sleeps 64, 128, then 256 ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  constexpr uint32_t kSuspendNs = 20000;
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t sleep_ns = 64;
  for (;;) {
    __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
    if (sleep_ns < 256) sleep_ns <<= 1;
  }
}

// ------------------------------------------------------------- statistics
// Threads work on the row's values shifted by a value K of that row (the
// row's first sum in the warp kernels, the first sum of a warp's chunk in the
// CTA kernel): Chan, Golub and LeVeque's "shifted data".  The sums then run
// at the size of the row's spread, so a row whose mean is large against its
// standard deviation loses nothing to the mean's magnitude, and a constant
// row gives exactly m = 0, M2 = 0.
//
// A partial covers n of the row's values: m = mean of (a - K), M2 = sum of
// squared deviations from that mean.
struct Part {
  float n;
  float m;
  float M2;
};

// Chan et al.'s pairwise update, written so that merge(a, b) and merge(b, a)
// give bitwise the same result (only commutative operations on the two
// sides), so a xor butterfly leaves identical totals in every lane with no
// broadcast.  EQUAL: both sides hold the same count (the case for every level
// when each thread holds the same number of values): no division.
template <bool EQUAL>
__device__ __forceinline__ Part merge(const Part& a, const Part& b) {
  Part o;
  const float d = b.m - a.m;  // squared below, so its sign does not matter
  o.n = a.n + b.n;
  if constexpr (EQUAL) {
    o.m = __fmul_rn(__fadd_rn(a.m, b.m), 0.5f);
    o.M2 = fmaf(__fmul_rn(d, d), __fmul_rn(a.n, 0.5f), __fadd_rn(a.M2, b.M2));
  } else {
    // explicit roundings: a multiply-add the compiler contracted into one
    // fma would round the two sides differently and break the symmetry
    const float inv = __frcp_rn(fmaxf(o.n, 1.0f));
    o.m = __fmul_rn(__fadd_rn(__fmul_rn(a.n, a.m), __fmul_rn(b.n, b.m)), inv);
    o.M2 = fmaf(__fmul_rn(d, d), __fmul_rn(__fmul_rn(a.n, b.n), inv), __fadd_rn(a.M2, b.M2));
  }
  return o;
}

// All-reduce of partials over groups of WIDTH lanes (xor butterfly).
template <bool EQUAL, int WIDTH>
__device__ __forceinline__ Part butterfly(Part p) {
#pragma unroll
  for (int off = 1; off < WIDTH; off <<= 1) {
    Part o;
    o.n = EQUAL ? p.n : __shfl_xor_sync(0xffffffffu, p.n, off);
    o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
    o.M2 = __shfl_xor_sync(0xffffffffu, p.M2, off);
    p = merge<EQUAL>(p, o);
  }
  return p;
}

// Two-pass statistics of the values one thread holds, relative to the row
// shift K (pass K = 0.f for values already shifted): the mean of its own
// values, then the sum of squared deviations around it.  FULL: every slot
// holds a value (the row divides evenly over the threads).
template <int NV, int VEC, bool FULL>
__device__ __forceinline__ Part thread_part(const float (&v)[NV][VEC], const bool (&ok)[NV],
                                            float K) {
  // four independent partial sums shorten the dependent-add chain
  constexpr int L = VEC >= 4 ? 4 : VEC;
  float acc[L];
#pragma unroll
  for (int l = 0; l < L; ++l) acc[l] = 0.f;
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (FULL || ok[k]) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e % L] += v[k][e] - K;
      cnt += VEC;
    }
  }
  float sum = acc[0];
#pragma unroll
  for (int l = 1; l < L; ++l) sum += acc[l];
  Part p;
  p.n = static_cast<float>(cnt);
  constexpr int kN = NV * VEC;
  if constexpr (FULL && (kN & (kN - 1)) == 0)
    p.m = sum * (1.0f / kN);  // exact: a power of two
  else
    p.m = cnt ? __fdiv_rn(sum, p.n) : 0.f;
  float sq[L];
#pragma unroll
  for (int l = 0; l < L; ++l) sq[l] = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (FULL || ok[k]) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float d = (v[k][e] - K) - p.m;
        sq[e % L] = fmaf(d, d, sq[e % L]);
      }
    }
  }
  float M2 = sq[0];
#pragma unroll
  for (int l = 1; l < L; ++l) M2 += sq[l];
  p.M2 = M2;
  return p;
}

// thread_part on values held as fp32 pairs.  SHIFT: subtract negK's
// negation on the fly (the values are the unshifted sums); otherwise the
// values are already shifted.  Pairs alternate between two accumulators, four
// independent sums in all.
template <int NV, int P, bool FULL, bool SHIFT>
__device__ __forceinline__ Part thread_part2(const float2 (&v)[NV][P], const bool (&ok)[NV],
                                             float2 negK) {
  float2 acc[2] = {dup2(0.f), dup2(0.f)};
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (FULL || ok[k]) {
#pragma unroll
      for (int q = 0; q < P; ++q)
        acc[q & 1] = add2(acc[q & 1], SHIFT ? add2(v[k][q], negK) : v[k][q]);
      cnt += 2 * P;
    }
  }
  const float sum = (acc[0].x + acc[1].x) + (acc[0].y + acc[1].y);
  Part p;
  p.n = static_cast<float>(cnt);
  constexpr int kN = NV * P * 2;
  if constexpr (FULL && (kN & (kN - 1)) == 0)
    p.m = sum * (1.0f / kN);  // exact: a power of two
  else
    p.m = cnt ? __fdiv_rn(sum, p.n) : 0.f;
  const float2 negm = dup2(-p.m);
  float2 sq[2] = {dup2(0.f), dup2(0.f)};
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (FULL || ok[k]) {
#pragma unroll
      for (int q = 0; q < P; ++q) {
        const float2 d = add2(SHIFT ? add2(v[k][q], negK) : v[k][q], negm);
        sq[q & 1] = fma2(d, d, sq[q & 1]);
      }
    }
  }
  p.M2 = (sq[0].x + sq[1].x) + (sq[0].y + sq[1].y);
  return p;
}

// normalise() on a pair of shifted values: ((v - m) * rstd) * g + b, the
// same three roundings per element; negm = (-m, -m), rstd2 = (rstd, rstd).
__device__ __forceinline__ float2 normalise2(float2 v, float2 negm, float2 rstd2, float2 g,
                                             float2 b) {
  return fma2(mul2(add2(v, negm), rstd2), g, b);
}

// y = gamma * (a - mean) * rstd + beta with mean = K + m; the deviation is
// taken as (a - K) - m so it never passes through the rounded absolute mean.
__device__ __forceinline__ float normalise(float a, float K, float m, float rstd, float g, float b) {
  return fmaf(((a - K) - m) * rstd, g, b);
}

// rstd = 1 / sqrt(M2 / H + eps); inv_h = 1/H rounded to fp32.
__device__ __forceinline__ float row_rstd(float M2, float inv_h, float eps) {
  return rsqrtf(fmaf(M2, inv_h, eps));
}

}  // namespace addln
