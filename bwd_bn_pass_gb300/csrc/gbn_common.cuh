// Device-side building blocks shared by the normalization kernels.
//
// - storage <-> fp32 conversion and 2..16-byte vector loads/stores;
// - double-fp32 ("DF") accumulation: Knuth's TwoSum keeps the exact rounding
//   error of every addition, and an FMA recovers the exact error of a
//   product, so fp32 outputs that are sums of 10^5..10^6 terms stay within a
//   few fp32 ulps of the exact sum even when the sum nearly cancels;
// - warp / block reductions with a fixed shuffle tree (deterministic);
// - programmatic dependent launch (griddepcontrol), mbarrier and 1-D bulk
//   copy (cp.async.bulk, the non-tensor TMA form) wrappers, with waits that
//   give up after about a second instead of spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbn {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------ conversion --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round-to-nearest-even
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// n / d for 0 <= n < 2^31 by a precomputed multiplier (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994,
// unsigned division with a 33-bit multiplier): q = (t + ((n - t) >> 1)) >>
// (l - 1) with t = mulhi(m, n), l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1.  For d = 1, m = 0 and both shifts are
// 0, so q = n.  A few integer instructions instead of the division routine.
struct FastDiv {
  uint32_t d, m, sh1, sh2;
};
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.sh1)) >> f.sh2;
}

// Multiplier and shifts of FastDiv for a divisor d >= 1.
inline FastDiv make_fast_div(uint32_t d) {
  FastDiv f{d, 0u, 0u, 0u};
  if (d <= 1) return f;  // n / 1: t = 0, (0 + n) >> 0 >> 0
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
  f.sh1 = 1;
  f.sh2 = l - 1;
  return f;
}

// VEC elements of T moved as one raw word group (VEC*sizeof(T) bytes, a
// power of two <= 16) and converted to fp32 only when used, so a thread can
// keep several vectors in flight in few registers.  bf16 element 0 sits in
// the low half of a 32-bit word.
template <typename T, int VEC> struct Vec;

template <> struct Vec<float, 1> {
  using raw = uint32_t;
  __device__ static raw ld(const float* p) { return __float_as_uint(*p); }
  __device__ static void cvt(raw r, float (&v)[1]) { v[0] = __uint_as_float(r); }
  __device__ static void store(float* p, const float (&v)[1]) { *p = v[0]; }
};
template <> struct Vec<float, 2> {
  using raw = uint2;
  __device__ static raw ld(const float* p) { return *reinterpret_cast<const uint2*>(p); }
  __device__ static void cvt(raw r, float (&v)[2]) {
    v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
  }
  __device__ static void store(float* p, const float (&v)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
};
template <> struct Vec<float, 4> {
  using raw = uint4;
  __device__ static raw ld(const float* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static void cvt(raw r, float (&v)[4]) {
    v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
    v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct Vec<bf16, 1> {
  using raw = uint32_t;
  __device__ static raw ld(const bf16* p) { return *reinterpret_cast<const uint16_t*>(p); }
  __device__ static void cvt(raw r, float (&v)[1]) { v[0] = bf16_lo(r); }
  __device__ static void store(bf16* p, const float (&v)[1]) { *p = __float2bfloat16_rn(v[0]); }
};
template <> struct Vec<bf16, 2> {
  using raw = uint32_t;
  __device__ static raw ld(const bf16* p) { return *reinterpret_cast<const uint32_t*>(p); }
  __device__ static void cvt(raw r, float (&v)[2]) { v[0] = bf16_lo(r); v[1] = bf16_hi(r); }
  __device__ static void store(bf16* p, const float (&v)[2]) {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(v[0], v[1]);
  }
};
template <> struct Vec<bf16, 4> {
  using raw = uint2;
  __device__ static raw ld(const bf16* p) { return *reinterpret_cast<const uint2*>(p); }
  __device__ static void cvt(raw r, float (&v)[4]) {
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
  }
  __device__ static void store(bf16* p, const float (&v)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
  }
};
template <> struct Vec<bf16, 8> {
  using raw = uint4;
  __device__ static raw ld(const bf16* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static void cvt(raw r, float (&v)[8]) {
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
  }
  __device__ static void store(bf16* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  }
};

// 16-byte shared-memory vector of T (VE = 16 / sizeof(T) elements).
template <typename T> struct Vec16 {
  static constexpr int VE = 16 / sizeof(T);
  __device__ static void load(const void* p, float (&v)[VE]) {
    Vec<T, VE>::cvt(Vec<T, VE>::ld(reinterpret_cast<const T*>(p)), v);
  }
  __device__ static void store(void* p, const float (&v)[VE]) {
    Vec<T, VE>::store(reinterpret_cast<T*>(p), v);
  }
};

// ------------------------------------------------- double-fp32 arithmetic --

struct DF {
  float hi, lo;
};

// The error-free transformations below use __fadd_rn / __fsub_rn /
// __fmul_rn: the compiler never contracts those into an FMA, which would
// silently break TwoSum (e.g. fusing q = p*r into s = hi + q).

// a += v with the rounding error of the addition kept in a.lo (TwoSum).
__device__ __forceinline__ void df_add(DF& a, float v) {
  const float s = __fadd_rn(a.hi, v);
  const float bb = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(v, bb));
  a.hi = s;
  a.lo = __fadd_rn(a.lo, err);
}

// a += p*q with the product's rounding error kept (FMA residual).
__device__ __forceinline__ void df_add_prod(DF& a, float p, float q) {
  const float m = __fmul_rn(p, q);
  const float e = fmaf(p, q, -m);
  df_add(a, m);
  a.lo = __fadd_rn(a.lo, e);
}

__device__ __forceinline__ double df_value(const DF& a) { return (double)a.hi + (double)a.lo; }

// Error-free building blocks: exact a + b and a * b as (hi, lo) pairs.
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return DF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return DF{p, fmaf(a, b, -p)};
}
// (hi, lo) * b, keeping the exact error of hi*b (lo*b is rounded; it is
// already ~2^-24 of the result).
__device__ __forceinline__ DF df_mul(DF a, float b) {
  DF p = two_prod(a.hi, b);
  p.lo = fmaf(a.lo, b, p.lo);
  return p;
}
// (hi, lo) + b
__device__ __forceinline__ DF df_plus(DF a, float b) {
  DF s = two_sum(a.hi, b);
  s.lo = __fadd_rn(s.lo, a.lo);
  return s;
}
// acc += t for a (hi, lo) term
__device__ __forceinline__ void df_acc(DF& acc, DF t) {
  df_add(acc, t.hi);
  acc.lo = __fadd_rn(acc.lo, t.lo);
}
__device__ __forceinline__ float df_round(DF a) { return __fadd_rn(a.hi, a.lo); }

// a + b for two (hi, lo) pairs.  Symmetric in a and b (the TwoSum error of
// hi + hi is exact, and lo + lo is commutative), so an xor-shuffle tree gives
// every lane the same bits.
__device__ __forceinline__ DF df_sum(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  return DF{s.hi, __fadd_rn(__fadd_rn(a.lo, b.lo), s.lo)};
}
// Renormalise so that hi = fl(hi + lo).
__device__ __forceinline__ DF df_norm(DF a) { return two_sum(a.hi, a.lo); }
// (hi, lo) * (hi, lo), first-order terms
__device__ __forceinline__ DF df_mul_df(DF a, DF b) {
  DF p = two_prod(a.hi, b.hi);
  p.lo = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, p.lo));
  return p;
}
// (hi, lo) / d for a positive fp32 d: q = hi/d, then the exact remainder
// hi - q*d (FMA) plus lo gives the low part.
__device__ __forceinline__ DF df_div(DF a, float d) {
  const float q = a.hi / d;
  const float r = __fadd_rn(fmaf(-q, d, a.hi), a.lo);
  return DF{q, r / d};
}
__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }

__device__ __forceinline__ DF shfl_xor_df(DF v, int o) {
  return DF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_sum(v, shfl_xor_df(v, o));
  return v;
}

// Sum two (hi, lo) pairs over the block in a fixed tree; every thread gets
// the result.  `red` must hold 2*32 float2.  Contains __syncthreads.
__device__ __forceinline__ void block_sum2_df(DF& a, DF& b, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  a = warp_sum_df(a);
  b = warp_sum_df(b);
  if (lane == 0) {
    red[warp] = make_float2(a.hi, a.lo);
    red[32 + warp] = make_float2(b.hi, b.lo);
  }
  __syncthreads();
  const float2 x = lane < nwarps ? red[lane] : make_float2(0.f, 0.f);
  const float2 y = lane < nwarps ? red[32 + lane] : make_float2(0.f, 0.f);
  a = warp_sum_df(DF{x.x, x.y});
  b = warp_sum_df(DF{y.x, y.y});
}

// -------------------------------------------- packed fp32x2 (sm_100+) --
//
// Two fp32 lanes in one 64-bit register, operated on by the paired FP32
// instructions (add/sub/mul/fma .rn.f32x2): every lane is an ordinary IEEE
// fp32 operation, two per instruction.

using f2 = unsigned long long;

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(f2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return make_float2(lo, hi);
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// 16 bytes of T as NP packed pairs (lane 0 = the lower-addressed element),
// and back (bf16 rounding is round-to-nearest-even).
template <typename T> struct Pairs16;
template <> struct Pairs16<float> {
  static constexpr int NP = 2;
  __device__ static void get(uint4 r, f2 (&p)[NP]) {
    p[0] = f2_pack(__uint_as_float(r.x), __uint_as_float(r.y));
    p[1] = f2_pack(__uint_as_float(r.z), __uint_as_float(r.w));
  }
  __device__ static uint4 put(const f2 (&p)[NP]) {
    const float2 a = f2_unpack(p[0]), b = f2_unpack(p[1]);
    return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x),
                      __float_as_uint(b.y));
  }
};
template <> struct Pairs16<bf16> {
  static constexpr int NP = 4;
  __device__ static f2 word(uint32_t w) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static void get(uint4 r, f2 (&p)[NP]) {
    p[0] = word(r.x);
    p[1] = word(r.y);
    p[2] = word(r.z);
    p[3] = word(r.w);
  }
  __device__ static uint32_t bf2(f2 v) {
    const float2 t = f2_unpack(v);
    return pack_bf16x2(t.x, t.y);
  }
  __device__ static uint4 put(const f2 (&p)[NP]) {
    return make_uint4(bf2(p[0]), bf2(p[1]), bf2(p[2]), bf2(p[3]));
  }
};

__device__ __forceinline__ f2 f2_splat(float v) { return f2_pack(v, v); }
__device__ __forceinline__ float f2_hsum(f2 v) {
  const float2 t = f2_unpack(v);
  return t.x + t.y;
}

// a*b rounded once, as an FMA with a +0 addend.  A packed mul.rn.f32x2 that
// feeds a packed add may be fused into an FMA by the assembler, which breaks
// TwoSum (s = hi + q must be the rounded sum of the rounded product); an
// FMA's result is never fused again.  Use this for every product that enters
// an error-free sum.
__device__ __forceinline__ f2 f2_mul_rounded(f2 a, f2 b) { return f2_fma(a, b, 0ull); }

// Two independent double-fp32 accumulators, one per lane.
struct DF2 {
  f2 hi, lo;
};

// a += v lane-wise, keeping each addition's exact error (TwoSum).
__device__ __forceinline__ void df2_add(DF2& a, f2 v) {
  const f2 s = f2_add(a.hi, v);
  const f2 bb = f2_sub(s, a.hi);
  const f2 err = f2_add(f2_sub(a.hi, f2_sub(s, bb)), f2_sub(v, bb));
  a.hi = s;
  a.lo = f2_add(a.lo, err);
}

// The two lanes folded into one (hi, lo) pair.
__device__ __forceinline__ DF df2_fold(const DF2& a) {
  const float2 h = f2_unpack(a.hi), l = f2_unpack(a.lo);
  const DF s = two_sum(h.x, h.y);
  return DF{s.hi, __fadd_rn(__fadd_rn(l.x, l.y), s.lo)};
}

// --------------------------------------------------------------- reduce --

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum two doubles over the block; every thread gets the result.  `red` must
// hold 2*32 doubles.  Contains __syncthreads (all threads must call it).
__device__ __forceinline__ void block_sum2(double& a, double& b, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) { red[warp] = a; red[32 + warp] = b; }
  __syncthreads();
  double x = lane < nwarps ? red[lane] : 0.0;
  double y = lane < nwarps ? red[32 + lane] : 0.0;
  a = warp_sum(x);
  b = warp_sum(y);
}

// ------------------------------------------- programmatic dependent launch --

// Let the next kernel on the stream (launched with the programmatic stream
// serialization attribute) be scheduled; it must still wait before reading
// anything this grid writes.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the preceding grid has completed and its writes are visible.
// A no-op when the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------- mbarrier / bulk copy --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Plain arrival (count 1) on a shared-memory mbarrier (release, CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction-priority policies for cache-hinted loads (createpolicy).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Wait for phase `parity` of `bar` to complete; false if it has not after
// about `limit_ns` nanoseconds (the caller records an error and stops).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void report_status(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// ------------------------------------------- flags between resident CTAs --
//
// Kernels whose CTAs are all resident (cooperative launch) hand results to
// each other through a workspace of 64-bit words: an epoch pair (e, ~e) at
// the start, then one flag pair per CTA.  A CTA publishes by storing
// (t, ~t) with t = e + 1 (release); a reader acquires the pair and checks
// both halves.  The epoch comes from the workspace when its pair is
// self-consistent, else from a host nonce, and one CTA advances it after it
// has seen every flag, so a reused or replayed workspace never matches a
// stale flag.  No memset and no atomics.

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ float2 ld_relaxed_f2(const float2* p) {
  float a, b;
  asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(a), "=f"(b) : "l"(p) : "memory");
  return make_float2(a, b);
}

// Flag pair of CTA k: word 0 is stored last, with release semantics.
__device__ __forceinline__ bool flag_ready(const unsigned long long* f, unsigned long long t) {
  return ld_acquire_u64(f) == t && ld_relaxed_u64(f + 1) == ~t;
}
// Polls back to back for the first few hundred tries (a flag is usually
// published within microseconds), then with short sleeps.
__device__ __forceinline__ bool wait_flag(const unsigned long long* f, unsigned long long t) {
  if (flag_ready(f, t)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (it > 256) __nanosleep(64);
    if (flag_ready(f, t)) return true;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// The flag value of this launch: (epoch of the workspace's pair, or the
// nonce when the pair is not self-consistent) + 1.
__device__ __forceinline__ unsigned long long flag_target(const unsigned long long* sync,
                                                          unsigned long long nonce) {
  const unsigned long long ea = ld_relaxed_u64(sync), eb = ld_relaxed_u64(sync + 1);
  return (eb == ~ea ? ea : nonce) + 1ull;
}

// Publish CTA k's flag after its earlier global writes (the caller makes
// the writes of the other threads of the CTA visible to this one first,
// e.g. with a barrier).
__device__ __forceinline__ void flag_publish(unsigned long long* sync, int k,
                                             unsigned long long t) {
  unsigned long long* f = sync + 2 + 2 * (int64_t)k;
  __threadfence();
  st_relaxed_u64(f + 1, ~t);
  st_release_u64(f, t);
}

// Store the next epoch (after every flag of this launch was seen).  After a
// failure one epoch is skipped so that no flag of this launch can match the
// next launch's target.
__device__ __forceinline__ void epoch_advance(unsigned long long* sync, unsigned long long t,
                                              bool all_seen) {
  const unsigned long long next = all_seen ? t : t + 1ull;
  st_relaxed_u64(sync + 1, ~next);
  st_relaxed_u64(sync, next);
}


}  // namespace gbn
