// BatchNorm2d training forward / backward kernels (NCHW).
//
// Method: Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
// statistics, finalize kernels".
//   * "Reduction grid": a grid of (C, grid_y) 256-thread blocks that fills
//     every resident block slot once; block (c, j) owns a contiguous slice of
//     channel c's M = B*HW elements.
//   * "One-pass statistics": each block sums d = x - x[0,c,0] and d*d and
//     writes its pair to partials[2, grid_y, C] -- no atomics, no zero-init.
//     The finalize reduces the partials into stats (mean, var, inv_std,
//     gamma*inv_std) and updates the running statistics; the apply is the
//     centred form (x - mean)*scale + beta.
//   * "Backward finalize": grad_sums partials (sum dy, sum dy*(x - mean)),
//     finalize to grads (dgamma, dbeta, k1, k2), dx = dy*scale + (x-mean)*k1
//     + k2.
//
// GB300 design (differs from the three launches per direction of Aether-ML
// PR #18, "Reduction grid" and "Backward finalize"):
//   * Two launches per direction.  The finalize is the prologue of the
//     consuming kernel: every block of channel c reduces that channel's
//     partials in the same fixed order (so all blocks hold bit-identical
//     values), and block j = 0 writes stats/grads and the running update.
//     The consumer is launched with programmatic dependent launch: it loads
//     its first vectors of x (and dy) before griddepcontrol.wait.
//   * Partials are double-fp32 (hi, lo) pairs.  Per thread, sums are
//     double-fp32 (TwoSum); the backward also keeps each product's FMA
//     residual and, for fp32 inputs, the rounding error of x - shift, so
//     sum dy*(x - mean) is accurate even when it nearly cancels.  The
//     backward forms S = sum dy*(x - shift) - (mean - shift)*sum dy in
//     double-fp32 from the forward's (mean - shift) pair.
//   * The consumer walks its slice in reverse, so the tail that the producer
//     read last (still in L2) is read first.
#include <atomic>

#include "bn_finalize.cuh"
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

// Geometry of one launch.  Vector offsets are in units of VEC elements from
// the tensor base; I is uint32_t unless the tensor has >= 2^32 vectors.
struct BnGeom {
  uint64_t step;   // offset change for +blockDim vectors of a channel, no wrap
  uint64_t wrap;   // extra change when the in-plane index wraps: C*Pv - Pv
  int64_t P;       // plane size in elements (x[0, c, 0] is element c*P)
  float Mh, Ml;    // per-channel count M = Mh + Ml exactly
  int32_t C;
  int32_t Pv;      // vectors per plane
  int32_t Mv;      // vectors per channel
  int32_t grid_y;
  int32_t tmod;    // blockDim % Pv
};

template <typename I>
struct Cursor {
  I vo;       // vector offset from the tensor base
  int32_t p;  // vector index inside the (b, c) plane
};

template <typename I>
__device__ __forceinline__ Cursor<I> cursor_at(const BnGeom& g, int c, int32_t v) {
  const int32_t b = v / g.Pv;
  Cursor<I> q;
  q.p = v - b * g.Pv;
  q.vo = ((I)b * (I)g.C + (I)c) * (I)g.Pv + (I)q.p;
  return q;
}
template <typename I>
__device__ __forceinline__ void cursor_fwd(Cursor<I>& q, const BnGeom& g) {
  q.p += g.tmod;
  q.vo += (I)g.step;
  if (q.p >= g.Pv) { q.p -= g.Pv; q.vo += (I)g.wrap; }
}
template <typename I>
__device__ __forceinline__ void cursor_back(Cursor<I>& q, const BnGeom& g) {
  q.p -= g.tmod;
  q.vo -= (I)g.step;
  if (q.p < 0) { q.p += g.Pv; q.vo -= (I)g.wrap; }
}

// Block j's slice [v0, v1) of the channel's vectors and this thread's count
// of vectors in it (stride blockDim).
__device__ __forceinline__ void slice(const BnGeom& g, int j, int32_t& v0, int32_t& cnt) {
  v0 = (int32_t)((int64_t)g.Mv * j / g.grid_y);
  const int32_t v1 = (int32_t)((int64_t)g.Mv * (j + 1) / g.grid_y);
  const int32_t n = v1 - v0 - (int32_t)threadIdx.x;
  cnt = n > 0 ? (n + kBnThreads - 1) / kBnThreads : 0;
}

// Channel c's partials summed over j in a fixed order by warp 0, in
// double-fp32 (GB300's fp64 rate is too low to spend in every block).  All
// lanes end with the same bits: the xor-shuffle tree of df_sum is symmetric.
__device__ __forceinline__ void reduce_partials(const float2* part, const BnGeom& g, int c,
                                                DF& s0, DF& s1) {
  const int lane = threadIdx.x & 31;
  DF a{0.f, 0.f}, b{0.f, 0.f};
  for (int jj = lane; jj < g.grid_y; jj += 32) {
    const float2 p0 = part[(int64_t)jj * g.C + c];
    const float2 p1 = part[((int64_t)g.grid_y + jj) * g.C + c];
    a = df_sum(a, DF{p0.x, p0.y});
    b = df_sum(b, DF{p1.x, p1.y});
  }
  s0 = warp_sum_df(a);
  s1 = warp_sum_df(b);
}

template <typename T>
__device__ __forceinline__ void x_minus_shift(float e, float shift, float& d, float& d_lo) {
  d = __fsub_rn(e, shift);
  if constexpr (sizeof(T) == 4) {
    // rounding error of the subtraction (TwoSum); zero when exact
    const float bb = __fsub_rn(d, e);
    d_lo = __fadd_rn(__fsub_rn(e, __fsub_rn(d, bb)), __fsub_rn(-shift, bb));
  } else {
    // bf16 operands: the fp32 difference is exact unless x and shift differ
    // in magnitude by more than 2^16; then d carries one fp32 rounding, a
    // per-term relative error of 2^-24 that does not grow with the sum.
    d_lo = 0.f;
  }
}

// ------------------------------------------------------------- stats --

// Blocks of 256 threads sized for kBnBlocksPerSm (4) resident blocks per SM
// (<= 64 registers/thread); vectors stay raw until used.  16-byte vectors in
// flight per thread: stats 8, apply 4, grad_sums 4 of each input, dx 2 of
// each input -- 128 KB of loads in flight per SM for the read passes.
constexpr int kUStats = 8;
constexpr int kUApply = 4;
constexpr int kUSums = 4;
constexpr int kUDx = 2;

template <typename T, int VEC, typename I>
__global__ void __launch_bounds__(kBnThreads, kBnBlocksPerSm)
    bn_stats_kernel(const T* __restrict__ x, BnGeom g, float2* __restrict__ part) {
  using V = Vec<T, VEC>;
  __shared__ float2 red[64];
  pdl_launch_dependents();
  const int c = blockIdx.x, j = blockIdx.y;
  int32_t v0, cnt;
  slice(g, j, v0, cnt);
  const float shift = to_f32(x[(int64_t)c * g.P]);

  DF s1, s2;
  Cursor<I> q = cursor_at<I>(g, c, v0 + (int32_t)threadIdx.x);
  if constexpr (VEC >= 2) {
    // Two packed lanes: pairs of elements per fp32x2 instruction.  sum d per
    // element in double-fp32 (plus, for fp32 input, the rounding error of
    // x - shift); sum d^2 per vector in fp32, then double-fp32.
    const f2 sh2 = f2_pack(shift, shift);
    const f2 nsh2 = f2_pack(-shift, -shift);
    DF2 a1{0ull, 0ull}, a2{0ull, 0ull};
    for (int32_t i = 0; i < cnt; i += kUStats) {
      typename V::raw r[kUStats];
#pragma unroll
      for (int u = 0; u < kUStats; ++u) {
        if (i + u < cnt) r[u] = V::ld(x + (size_t)q.vo * VEC);
        cursor_fwd(q, g);
      }
#pragma unroll
      for (int u = 0; u < kUStats; ++u) {
        if (i + u < cnt) {
          float e[VEC];
          V::cvt(r[u], e);
          f2 l2 = 0ull;  // +0.0f in both lanes
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            const f2 x2 = f2_pack(e[2 * k], e[2 * k + 1]);
            const f2 d = f2_sub(x2, sh2);
            df2_add(a1, d);
            if constexpr (sizeof(T) == 4) {
              const f2 bb = f2_sub(d, x2);
              a1.lo = f2_add(a1.lo, f2_add(f2_sub(x2, f2_sub(d, bb)), f2_sub(nsh2, bb)));
            }
            l2 = f2_fma(d, d, l2);
          }
          df2_add(a2, l2);
        }
      }
    }
    s1 = df2_fold(a1);
    s2 = df2_fold(a2);
  } else {
    s1 = DF{0.f, 0.f};
    s2 = DF{0.f, 0.f};
    for (int32_t i = 0; i < cnt; i += kUStats) {
      typename V::raw r[kUStats];
#pragma unroll
      for (int u = 0; u < kUStats; ++u) {
        if (i + u < cnt) r[u] = V::ld(x + (size_t)q.vo * VEC);
        cursor_fwd(q, g);
      }
#pragma unroll
      for (int u = 0; u < kUStats; ++u) {
        if (i + u < cnt) {
          float e[VEC];
          V::cvt(r[u], e);
          float d, d_lo;
          x_minus_shift<T>(e[0], shift, d, d_lo);
          df_add(s1, d);
          if constexpr (sizeof(T) == 4) s1.lo = __fadd_rn(s1.lo, d_lo);
          df_add(s2, d * d);
        }
      }
    }
  }
  block_sum2_df(s1, s2, red);
  if (threadIdx.x == 0) {
    part[(int64_t)j * g.C + c] = make_float2(s1.hi, s1.lo);
    part[((int64_t)g.grid_y + j) * g.C + c] = make_float2(s2.hi, s2.lo);
  }
}

// ------------------------------------------------- finalize + apply --

struct ApplyArgs {
  int mode;
  const float2* part;
  const float* gamma;
  const float* beta;
  float* stats;
  float* running_mean;
  float* running_var;
  float momentum;
  float eps;
  const float* mean;
  const float* scale;
  int act;      // GBN_ACT_*
  float slope;
};

// Warp 0 computes (shift, mean - shift, scale, beta) for channel c; in
// training mode this is the forward finalize, returned so that block j = 0
// can write the stats rows and the running-statistics update after its
// outputs (nothing in this launch reads them).  shift_x, gamma and beta are
// the channel's inputs that the stats grid does not write: the caller loads
// them before it waits for that grid, so that only the partials are read
// after the wait.
__device__ __noinline__ BnFwdFinal apply_prologue(const BnGeom& g, const ApplyArgs& a, int c,
                                                  float shift_x, float gamma, float beta,
                                                  float* fin) {
  float shift, mean_d, scale;
  BnFwdFinal f{};
  if (a.mode == kApplyTrain) {
    DF s1, s2;
    reduce_partials(a.part, g, c, s1, s2);
    f = bn_fwd_final(s1, s2, g.Mh, g.Ml, gamma, a.eps);
    shift = shift_x;
    mean_d = f.md.hi;
    scale = f.scale;
  } else if (a.mode == kApplyStats) {
    const int64_t C = g.C;
    shift = a.stats[4 * C + c];
    mean_d = a.stats[5 * C + c];
    scale = a.stats[3 * C + c];
  } else {
    shift = a.mean[c];
    mean_d = 0.f;
    scale = a.scale[c];
  }
  if (threadIdx.x == 0) { fin[0] = shift; fin[1] = mean_d; fin[2] = scale; fin[3] = beta; }
  return f;
}

template <typename T, int VEC, typename I>
__global__ void __launch_bounds__(kBnThreads, kBnBlocksPerSm)
    bn_apply_kernel(const T* __restrict__ x, T* y, BnGeom g, ApplyArgs a) {
  using V = Vec<T, VEC>;
  __shared__ float fin[4];  // shift, mean_d, scale, beta
  const int c = blockIdx.x, j = blockIdx.y;
  int32_t v0, cnt;
  slice(g, j, v0, cnt);

  // The channel's own inputs first (ahead of the vector loads below): the
  // finalize then waits on nothing but the stats grid's partials.
  float shift_x = 0.f, gam = 1.f, bet = 0.f, rm_old = 0.f, rv_old = 0.f;
  if (threadIdx.x < 32) {
    shift_x = to_f32(x[(int64_t)c * g.P]);
    if (a.gamma) gam = a.gamma[c];
    if (a.beta) bet = a.beta[c];
    if (a.mode == kApplyTrain && j == 0 && threadIdx.x == 0) {
      if (a.running_mean) rm_old = a.running_mean[c];
      if (a.running_var) rv_old = a.running_var[c];
    }
  }
  // Walk this thread's vectors backwards (the stats pass read the slice
  // tails last, so they are the likeliest to be in L2); load the first batch
  // before waiting on the stats grid (x is never written by it).
  const int32_t vlast = v0 + (int32_t)threadIdx.x + (cnt > 0 ? cnt - 1 : 0) * kBnThreads;
  Cursor<I> q = cursor_at<I>(g, c, vlast);
  typename V::raw r[kUApply];
  I off[kUApply];
#pragma unroll
  for (int u = 0; u < kUApply; ++u) {
    off[u] = q.vo;
    if (u < cnt) r[u] = V::ld(x + (size_t)q.vo * VEC);
    cursor_back(q, g);
  }

  if (a.mode == kApplyTrain) pdl_wait();
  BnFwdFinal fin_f{};
  if (threadIdx.x < 32) fin_f = apply_prologue(g, a, c, shift_x, gam, bet, fin);
  __syncthreads();
  const float shift = fin[0], mean_d = fin[1], scale = fin[2], beta = fin[3];
  // 16-byte vectors without an activation: two elements per instruction
  // (fp32x2), the same operations and rounding as the scalar form
  constexpr bool kPacked = sizeof(typename V::raw) == 16;
  const bool packed = kPacked && a.act == GBN_ACT_NONE;
  const f2 sh2 = f2_splat(shift), md2 = f2_splat(mean_d), sc2 = f2_splat(scale),
           be2 = f2_splat(beta);

  for (int32_t i = 0; i < cnt; i += kUApply) {
#pragma unroll
    for (int u = 0; u < kUApply; ++u) {
      if (i + u < cnt) {
        if constexpr (kPacked) {
          if (packed) {
            using PK = Pairs16<T>;
            f2 p[PK::NP];
            PK::get(r[u], p);
#pragma unroll
            for (int k = 0; k < PK::NP; ++k) p[k] = f2_fma(f2_sub(f2_sub(p[k], sh2), md2), sc2, be2);
            *reinterpret_cast<uint4*>(y + (size_t)off[u] * VEC) = PK::put(p);
            continue;
          }
        }
        float e[VEC];
        V::cvt(r[u], e);
#pragma unroll
        for (int k = 0; k < VEC; ++k)
          e[k] = act_out(fmaf((e[k] - shift) - mean_d, scale, beta), a.act, a.slope);
        V::store(y + (size_t)off[u] * VEC, e);
      }
    }
#pragma unroll
    for (int u = 0; u < kUApply; ++u) {
      off[u] = q.vo;
      if (i + kUApply + u < cnt) r[u] = V::ld(x + (size_t)q.vo * VEC);
      cursor_back(q, g);
    }
  }
  if (a.mode == kApplyTrain && j == 0 && threadIdx.x == 0)
    bn_fwd_write_from(fin_f, shift, g.C, c, g.Mh + g.Ml, a.stats, a.running_mean,
                      a.running_var, a.momentum, rm_old, rv_old);
}

// --------------------------------------------------------- grad_sums --

template <typename T, int VEC, typename I, bool GATE>
__global__ void __launch_bounds__(kBnThreads, kBnBlocksPerSm)
    bn_grad_sums_kernel(const T* __restrict__ x, const T* __restrict__ dy, BnGeom g,
                        const float* __restrict__ stats, float2* __restrict__ part,
                        const float* __restrict__ beta, int act, float slope) {
  using V = Vec<T, VEC>;
  __shared__ float2 red[64];
  pdl_launch_dependents();
  const int c = blockIdx.x, j = blockIdx.y;
  int32_t v0, cnt;
  slice(g, j, v0, cnt);
  const float shift = stats[4 * (int64_t)g.C + c];
  // With an activation, dy is gated by d act / d pre, pre recomputed as in
  // the forward apply.
  float mean_d = 0.f, scale = 0.f, bta = 0.f;
  if constexpr (GATE) {
    mean_d = stats[5 * (int64_t)g.C + c];
    scale = stats[3 * (int64_t)g.C + c];
    bta = beta ? beta[c] : 0.f;
  }
  auto gate = [&](const float (&ex)[VEC], float (&ed)[VEC]) {
    if constexpr (GATE) {
#pragma unroll
      for (int k = 0; k < VEC; ++k)
        ed[k] = __fmul_rn(ed[k], act_gate(fmaf((ex[k] - shift) - mean_d, scale, bta), act, slope));
    }
  };

  DF s0, s1;
  Cursor<I> q = cursor_at<I>(g, c, v0 + (int32_t)threadIdx.x);
  if constexpr (VEC >= 2) {
    // Packed lanes.  sum dy and sum dy*d with d = x - shift; every product's
    // exact residual (FMA against the negated product) and, for fp32 input,
    // the rounding error of x - shift are kept in the low parts.
    const f2 sh2 = f2_pack(shift, shift);
    const f2 nsh2 = f2_pack(-shift, -shift);
    DF2 a0{0ull, 0ull}, a1{0ull, 0ull};
    for (int32_t i = 0; i < cnt; i += kUSums) {
      typename V::raw rx[kUSums], rd[kUSums];
#pragma unroll
      for (int u = 0; u < kUSums; ++u) {
        if (i + u < cnt) {
          rx[u] = V::ld(x + (size_t)q.vo * VEC);
          rd[u] = V::ld(dy + (size_t)q.vo * VEC);
        }
        cursor_fwd(q, g);
      }
#pragma unroll
      for (int u = 0; u < kUSums; ++u) {
        if (i + u < cnt) {
          float ex[VEC], ed[VEC];
          V::cvt(rx[u], ex);
          V::cvt(rd[u], ed);
          gate(ex, ed);
#pragma unroll
          for (int k = 0; k < VEC / 2; ++k) {
            const f2 x2 = f2_pack(ex[2 * k], ex[2 * k + 1]);
            const f2 dy2 = f2_pack(ed[2 * k], ed[2 * k + 1]);
            const f2 d = f2_sub(x2, sh2);
            const f2 nd = f2_sub(sh2, x2);  // exactly -d
            df2_add(a0, dy2);
            const f2 prod = f2_mul_rounded(dy2, d);
            df2_add(a1, prod);
            a1.lo = f2_add(a1.lo, f2_fma(dy2, d, f2_mul_rounded(dy2, nd)));
            if constexpr (sizeof(T) == 4) {
              const f2 bb = f2_sub(d, x2);
              const f2 d_lo = f2_add(f2_sub(x2, f2_sub(d, bb)), f2_sub(nsh2, bb));
              a1.lo = f2_fma(dy2, d_lo, a1.lo);
            }
          }
        }
      }
    }
    s0 = df2_fold(a0);
    s1 = df2_fold(a1);
  } else {
    s0 = DF{0.f, 0.f};
    s1 = DF{0.f, 0.f};
    for (int32_t i = 0; i < cnt; i += kUSums) {
      typename V::raw rx[kUSums], rd[kUSums];
#pragma unroll
      for (int u = 0; u < kUSums; ++u) {
        if (i + u < cnt) {
          rx[u] = V::ld(x + (size_t)q.vo * VEC);
          rd[u] = V::ld(dy + (size_t)q.vo * VEC);
        }
        cursor_fwd(q, g);
      }
#pragma unroll
      for (int u = 0; u < kUSums; ++u) {
        if (i + u < cnt) {
          float ex[VEC], ed[VEC];
          V::cvt(rx[u], ex);
          V::cvt(rd[u], ed);
          gate(ex, ed);
          float d, d_lo;
          x_minus_shift<T>(ex[0], shift, d, d_lo);
          df_add(s0, ed[0]);
          df_add_prod(s1, ed[0], d);
          if constexpr (sizeof(T) == 4) s1.lo = fmaf(ed[0], d_lo, s1.lo);
        }
      }
    }
  }
  block_sum2_df(s0, s1, red);
  if (threadIdx.x == 0) {
    part[(int64_t)j * g.C + c] = make_float2(s0.hi, s0.lo);
    part[((int64_t)g.grid_y + j) * g.C + c] = make_float2(s1.hi, s1.lo);
  }
}

// ---------------------------------------------------- finalize + dx --

// The forward's per-channel values the backward finalize and dx need,
// read from stats (written by the forward, before the grad-sums grid).
struct DxChan {
  float shift, mean_d, inv_std, scale, md_hi, md_lo, beta;
};

// Warp 0: the backward finalize for channel c (block j = 0 writes grads).
// S = sum dy*(x - mean) = sum dy*(x - shift) - (mean - shift)*sum dy, in
// double-fp32 with the forward's (mean - shift) pair.  ch was loaded before
// the wait for the grad-sums grid, so only its partials are read after it.
__device__ __noinline__ void dx_prologue(const BnGeom& g, const float2* part, float* grads,
                                         int c, int j, const DxChan ch, float* fin) {
  DF p0, p1;
  reduce_partials(part, g, c, p0, p1);
  const int64_t C = g.C;
  const DF md{ch.md_hi, ch.md_lo};
  const BnBwdFinal f = bn_bwd_final(p0, p1, md, ch.inv_std, ch.scale, g.Mh + g.Ml);
  const float k1 = f.k1, k2 = f.k2;
  if (j == 0 && threadIdx.x == 0) {
    grads[c] = f.dgamma;
    grads[C + c] = f.dbeta;
    grads[2 * C + c] = k1;
    grads[3 * C + c] = k2;
  }
  if (threadIdx.x == 0) {
    fin[0] = ch.shift;
    fin[1] = ch.mean_d;
    fin[2] = ch.scale;
    fin[3] = k1;
    fin[4] = k2;
    fin[5] = ch.beta;
  }
}

template <typename T, int VEC, typename I>
__global__ void __launch_bounds__(kBnThreads, kBnBlocksPerSm)
    bn_dx_kernel(const T* __restrict__ x, const T* dy, T* dx, BnGeom g,
                 const float* __restrict__ stats, const float2* __restrict__ part,
                 float* __restrict__ grads, const float* __restrict__ beta, int act,
                 float slope) {
  using V = Vec<T, VEC>;
  __shared__ float fin[6];  // shift, mean_d, scale, k1, k2, beta
  const int c = blockIdx.x, j = blockIdx.y;
  int32_t v0, cnt;
  slice(g, j, v0, cnt);

  // The forward's values of this channel first (stats rows 2-7; beta for
  // the activation gate), ahead of the vector loads below.
  DxChan ch{0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (threadIdx.x < 32) {
    const int64_t C = g.C;
    ch.inv_std = stats[2 * C + c];
    ch.scale = stats[3 * C + c];
    ch.shift = stats[4 * C + c];
    ch.mean_d = stats[5 * C + c];
    ch.md_hi = stats[6 * C + c];
    ch.md_lo = stats[7 * C + c];
    ch.beta = beta ? beta[c] : 0.f;
  }
  const int32_t vlast = v0 + (int32_t)threadIdx.x + (cnt > 0 ? cnt - 1 : 0) * kBnThreads;
  Cursor<I> q = cursor_at<I>(g, c, vlast);
  typename V::raw rx[kUDx], rd[kUDx];
  I off[kUDx];
#pragma unroll
  for (int u = 0; u < kUDx; ++u) {
    off[u] = q.vo;
    if (u < cnt) {
      rx[u] = V::ld(x + (size_t)q.vo * VEC);
      rd[u] = V::ld(dy + (size_t)q.vo * VEC);
    }
    cursor_back(q, g);
  }

  pdl_wait();
  if (threadIdx.x < 32) dx_prologue(g, part, grads, c, j, ch, fin);
  __syncthreads();
  const float shift = fin[0], mean_d = fin[1], scale = fin[2], k1 = fin[3], k2 = fin[4];
  const float bta = fin[5];
  // 16-byte vectors without an activation: two elements per instruction
  // (fp32x2), the same operations and rounding as the scalar form
  constexpr bool kPacked = sizeof(typename V::raw) == 16;
  const bool packed = kPacked && act == GBN_ACT_NONE;
  const f2 sh2 = f2_splat(shift), md2 = f2_splat(mean_d), sc2 = f2_splat(scale),
           k12 = f2_splat(k1), k22 = f2_splat(k2);

  for (int32_t i = 0; i < cnt; i += kUDx) {
#pragma unroll
    for (int u = 0; u < kUDx; ++u) {
      if (i + u < cnt) {
        if constexpr (kPacked) {
          if (packed) {
            using PK = Pairs16<T>;
            f2 px[PK::NP], pd[PK::NP];
            PK::get(rx[u], px);
            PK::get(rd[u], pd);
#pragma unroll
            for (int k = 0; k < PK::NP; ++k)
              px[k] = f2_fma(pd[k], sc2, f2_fma(f2_sub(f2_sub(px[k], sh2), md2), k12, k22));
            *reinterpret_cast<uint4*>(dx + (size_t)off[u] * VEC) = PK::put(px);
            continue;
          }
        }
        float ex[VEC], ed[VEC];
        V::cvt(rx[u], ex);
        V::cvt(rd[u], ed);
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const float xc = (ex[k] - shift) - mean_d;
          const float gk = act == GBN_ACT_NONE
                               ? ed[k]
                               : __fmul_rn(ed[k], act_gate(fmaf(xc, scale, bta), act, slope));
          ex[k] = fmaf(gk, scale, fmaf(xc, k1, k2));
        }
        V::store(dx + (size_t)off[u] * VEC, ex);
      }
    }
#pragma unroll
    for (int u = 0; u < kUDx; ++u) {
      off[u] = q.vo;
      if (i + kUDx + u < cnt) {
        rx[u] = V::ld(x + (size_t)q.vo * VEC);
        rd[u] = V::ld(dy + (size_t)q.vo * VEC);
      }
      cursor_back(q, g);
    }
  }
}

BnGeom make_geom(const BnPlan& p) {
  BnGeom g;
  const int64_t Pv = p.P / p.vec;
  g.P = p.P;
  g.C = (int32_t)p.C;
  g.Pv = (int32_t)Pv;
  g.Mv = (int32_t)(p.B * Pv);
  g.grid_y = p.grid_y;
  g.tmod = (int32_t)(kBnThreads % Pv);
  g.step = (uint64_t)(kBnThreads / Pv) * (uint64_t)p.C * (uint64_t)Pv + (uint64_t)g.tmod;
  g.wrap = (uint64_t)p.C * (uint64_t)Pv - (uint64_t)Pv;
  g.Mh = (float)p.M;
  g.Ml = (float)(p.M - (int64_t)g.Mh);
  return g;
}

dim3 bn_grid(const BnPlan& p) { return dim3((unsigned)p.C, (unsigned)p.grid_y, 1); }

// Dispatch on (dtype, vec, offset width) to a template instance.
template <template <typename, int, typename> class F, typename I, typename... A>
cudaError_t dispatch_t(int dtype, int vec, A&&... args) {
  if (dtype == GBN_F32) {
    switch (vec) {
      case 4: return F<float, 4, I>::run(args...);
      case 2: return F<float, 2, I>::run(args...);
      default: return F<float, 1, I>::run(args...);
    }
  }
  switch (vec) {
    case 8: return F<bf16, 8, I>::run(args...);
    case 4: return F<bf16, 4, I>::run(args...);
    case 2: return F<bf16, 2, I>::run(args...);
    default: return F<bf16, 1, I>::run(args...);
  }
}

std::atomic<int> g_force_wide{0};

template <template <typename, int, typename> class F, typename... A>
cudaError_t dispatch(const BnPlan& p, int dtype, A&&... args) {
  const uint64_t vectors = (uint64_t)p.B * (uint64_t)p.C * (uint64_t)(p.P / p.vec);
  if (vectors < (1ull << 32) && g_force_wide.load(std::memory_order_relaxed) == 0)
    return dispatch_t<F, uint32_t>(dtype, p.vec, args...);
  return dispatch_t<F, uint64_t>(dtype, p.vec, args...);
}

template <typename T, int VEC, typename I> struct StatsL {
  static cudaError_t run(const void* x, const BnPlan& p, float2* part, cudaStream_t st) {
    return launch(bn_stats_kernel<T, VEC, I>, bn_grid(p), dim3(kBnThreads), 0, st, false,
                  static_cast<const T*>(x), make_geom(p), part);
  }
};
template <typename T, int VEC, typename I> struct ApplyL {
  static cudaError_t run(const void* x, void* y, const BnPlan& p, const ApplyArgs& a,
                         cudaStream_t st, bool pdl) {
    return launch(bn_apply_kernel<T, VEC, I>, bn_grid(p), dim3(kBnThreads), 0, st, pdl,
                  static_cast<const T*>(x), static_cast<T*>(y), make_geom(p), a);
  }
};
template <typename T, int VEC, typename I> struct GradSumsL {
  static cudaError_t run(const void* x, const void* dy, const BnPlan& p, const float* stats,
                         float2* part, const float* beta, int act, float slope,
                         cudaStream_t st) {
    // The gate is a template switch: the ungated kernel keeps the register
    // budget it has without an activation.
    return act == GBN_ACT_NONE
               ? launch(bn_grad_sums_kernel<T, VEC, I, false>, bn_grid(p), dim3(kBnThreads), 0,
                        st, false, static_cast<const T*>(x), static_cast<const T*>(dy),
                        make_geom(p), stats, part, beta, act, slope)
               : launch(bn_grad_sums_kernel<T, VEC, I, true>, bn_grid(p), dim3(kBnThreads), 0,
                        st, false, static_cast<const T*>(x), static_cast<const T*>(dy),
                        make_geom(p), stats, part, beta, act, slope);
  }
};
template <typename T, int VEC, typename I> struct DxL {
  static cudaError_t run(const void* x, const void* dy, void* dx, const BnPlan& p,
                         const float* stats, const float2* part, float* grads, const float* beta,
                         int act, float slope, cudaStream_t st, bool pdl) {
    return launch(bn_dx_kernel<T, VEC, I>, bn_grid(p), dim3(kBnThreads), 0, st, pdl,
                  static_cast<const T*>(x), static_cast<const T*>(dy), static_cast<T*>(dx),
                  make_geom(p), stats, part, grads, beta, act, slope);
  }
};

}  // namespace

int bn_set_wide_offsets(int force) { return g_force_wide.exchange(force != 0 ? 1 : 0); }

bool bn_plan(int64_t B, int64_t C, int64_t HW, const DevInfo& dev, BnPlan* plan) {
  if (B < 0 || C < 0 || HW < 0) return false;
  plan->B = B;
  plan->C = C;
  plan->P = HW;
  plan->M = B * HW;
  // Fill every resident block slot once (Aether-ML PR #18, "Reduction grid",
  // counts mp_count * max_threads_per_mp / 256 slots; these kernels hold 64
  // registers per thread, so kBnBlocksPerSm 256-thread blocks are resident
  // per SM), but give each block at least kBnMinElemsPerBlock elements.
  const int64_t slots = (int64_t)dev.sms * kBnBlocksPerSm;
  int64_t gy = C > 0 ? slots / C : 1;
  const int64_t by_work = (plan->M + kBnMinElemsPerBlock - 1) / kBnMinElemsPerBlock;
  if (by_work < gy) gy = by_work;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  plan->grid_y = (int)gy;
  const size_t bytes = (size_t)2 * (size_t)gy * (size_t)(C > 0 ? C : 1) * sizeof(float2);
  plan->ws_partials = (bytes + 255) & ~(size_t)255;
  plan->ws_bytes = plan->ws_partials;
  // The same workspace also serves the persistent path of either dtype.
  BnFusedPlan fp;
  for (int dtype : {GBN_F32, GBN_BF16})
    for (bool backward : {false, true})
      if (bn_fused_plan(dtype, backward, B, C, HW, dev, &fp) && fp.ws_bytes > plan->ws_bytes)
        plan->ws_bytes = fp.ws_bytes;
  return true;
}

int bn_vec_width(int dtype, int64_t P, const void* const* ptrs, int nptrs) {
  const int esize = dtype == GBN_F32 ? 4 : 2;
  int vec = 16 / esize;
  while (vec > 1) {
    bool ok = (P % vec) == 0;
    for (int i = 0; i < nptrs && ok; ++i)
      if (ptrs[i] != nullptr && (reinterpret_cast<uintptr_t>(ptrs[i]) % (uintptr_t)(vec * esize)) != 0)
        ok = false;
    if (ok) break;
    vec >>= 1;
  }
  return vec;
}

cudaError_t bn_launch_stats(const void* x, int dtype, const BnPlan& p, float2* part,
                            cudaStream_t st) {
  return dispatch<StatsL>(p, dtype, x, p, part, st);
}

cudaError_t bn_launch_apply(const void* x, void* y, int dtype, const BnPlan& p, int mode,
                            const float2* part, const float* gamma, const float* beta,
                            float* stats, float* running_mean, float* running_var,
                            float momentum, float eps, const float* mean, const float* scale,
                            int act, float slope, cudaStream_t st, bool pdl) {
  ApplyArgs a;
  a.act = act;
  a.slope = slope;
  a.mode = mode;
  a.part = part;
  a.gamma = gamma;
  a.beta = beta;
  a.stats = stats;
  a.running_mean = running_mean;
  a.running_var = running_var;
  a.momentum = momentum;
  a.eps = eps;
  a.mean = mean;
  a.scale = scale;
  return dispatch<ApplyL>(p, dtype, x, y, p, a, st, pdl);
}

cudaError_t bn_launch_grad_sums(const void* x, const void* dy, int dtype, const BnPlan& p,
                                const float* stats, float2* part, const float* beta, int act,
                                float slope, cudaStream_t st) {
  return dispatch<GradSumsL>(p, dtype, x, dy, p, stats, part, beta, act, slope, st);
}

cudaError_t bn_launch_dx(const void* x, const void* dy, void* dx, int dtype, const BnPlan& p,
                         const float* stats, const float2* part, float* grads, const float* beta,
                         int act, float slope, cudaStream_t st, bool pdl) {
  return dispatch<DxL>(p, dtype, x, dy, dx, p, stats, part, grads, beta, act, slope, st, pdl);
}

}  // namespace gbn
