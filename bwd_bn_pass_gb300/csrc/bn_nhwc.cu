// BatchNorm2d training forward / backward for channels-last (NHWC) tensors.
//
// Method: Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
// statistics, finalize kernels" -- the same statistics, finalize and
// centred apply as the NCHW path, and "Part 2" for the fused activation.
//
// Layout: x, y, dy, dx are [M, C] row-major (M = N*H*W, the channel
// innermost); a channel is a column with stride C.  The channel reductions
// are column sums, so the kernels stream rows:
//   * a 256-thread block is TX x TY threads; TX threads cover TX vectors of
//     VEC adjacent channels (a warp reads 32 * 16 contiguous bytes of a
//     row), the TY thread rows stride down the block's slice of rows;
//   * every thread keeps double-fp32 sums for its VEC channels (two channels
//     per packed fp32x2 register): sum d per element with TwoSum (and, for
//     fp32, the rounding error of x - shift) so that sum d is exact; sum d^2
//     over eight rows in fp32 before its double-fp32 add; backward sum dy*d
//     per element with each product's FMA residual, and sum dy per element
//     (fp32) or over four rows first (bf16, exact for 8-bit significands);
//   * the TY thread rows are added in a fixed tree in shared memory and
//     the block writes one (hi, lo) pair per channel and sum to
//     partials[2][grid_y][C] -- no atomics;
//   * a finalize kernel (one warp per channel, programmatic dependent
//     launch) adds the grid_y partials in a fixed order and writes stats /
//     grads and the running statistics with the NCHW path's formulas;
//   * the apply / dx kernel (programmatic dependent launch) reads the
//     per-channel parameters once per thread and streams the rows again,
//     each slice from its end (the part the sum kernel read last).
// Three launches per direction; x (and dy) are read twice.
#include "bn_finalize.cuh"
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

constexpr int kNThreads = 256;
constexpr int kNSumBlocksPerSm = 2;  // the sum kernels hold ~100 registers
// Rows each thread loads before using them: 8 for the one-input kernels, 4
// for the two-input ones (more ran slower there: register pressure).
constexpr int kNRowsUnroll1 = 8;
constexpr int kNRowsUnroll2 = 4;

struct NhwcGeom {
  int64_t M;       // rows
  int32_t C;       // channels
  int32_t Cv;      // vectors per row (C / VEC)
  int32_t TX, TY;  // block shape: TX vectors x TY rows
  int32_t grid_y;  // row slices
  float Mh, Ml;    // M = Mh + Ml exactly
};

template <int VEC> struct Pk {
  static constexpr int NP = (VEC + 1) / 2;  // packed pairs; VEC = 1 pads with 0
};

template <int VEC>
__device__ __forceinline__ f2 pair_of(const float (&e)[VEC], int k) {
  return f2_pack(e[2 * k], 2 * k + 1 < VEC ? e[2 * k + 1] : 0.f);
}

// Rows [r0, r1) of block row-slice j.
__device__ __forceinline__ void row_slice(const NhwcGeom& g, int j, int64_t& r0, int64_t& r1) {
  r0 = g.M * j / g.grid_y;
  r1 = g.M * (j + 1) / g.grid_y;
}

// Adds the TY thread rows of each column in a fixed tree; thread row 0 ends
// with the block's sums.  red holds kNThreads * NP float4 (hi/lo of two
// packed sums per pair).
template <int NP>
__device__ __forceinline__ void column_tree(DF2 (&a)[NP], DF2 (&b)[NP], float4* red,
                                            const NhwcGeom& g) {
  const int tx = threadIdx.x % g.TX, ty = threadIdx.x / g.TX;
  for (int step = g.TY / 2; step >= 1; step /= 2) {
    if (ty >= step && ty < 2 * step) {
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const float2 ah = f2_unpack(a[k].hi), al = f2_unpack(a[k].lo);
        const float2 bh = f2_unpack(b[k].hi), bl = f2_unpack(b[k].lo);
        red[((ty - step) * g.TX + tx) * 2 * NP + 2 * k] = make_float4(ah.x, al.x, ah.y, al.y);
        red[((ty - step) * g.TX + tx) * 2 * NP + 2 * k + 1] = make_float4(bh.x, bl.x, bh.y, bl.y);
      }
    }
    __syncthreads();
    if (ty < step) {
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const float4 u = red[(ty * g.TX + tx) * 2 * NP + 2 * k];
        const float4 w = red[(ty * g.TX + tx) * 2 * NP + 2 * k + 1];
        const float2 ah = f2_unpack(a[k].hi), al = f2_unpack(a[k].lo);
        const float2 bh = f2_unpack(b[k].hi), bl = f2_unpack(b[k].lo);
        const DF a0 = df_sum(DF{ah.x, al.x}, DF{u.x, u.y});
        const DF a1 = df_sum(DF{ah.y, al.y}, DF{u.z, u.w});
        const DF b0 = df_sum(DF{bh.x, bl.x}, DF{w.x, w.y});
        const DF b1 = df_sum(DF{bh.y, bl.y}, DF{w.z, w.w});
        a[k].hi = f2_pack(a0.hi, a1.hi);
        a[k].lo = f2_pack(a0.lo, a1.lo);
        b[k].hi = f2_pack(b0.hi, b1.hi);
        b[k].lo = f2_pack(b0.lo, b1.lo);
      }
    }
    __syncthreads();
  }
}

template <int VEC>
__device__ __forceinline__ void write_partials(const DF2 (&a)[Pk<VEC>::NP],
                                               const DF2 (&b)[Pk<VEC>::NP], const NhwcGeom& g,
                                               int cv, float2* part) {
  const int64_t base = (int64_t)blockIdx.y * g.C + (int64_t)cv * VEC;
  const int64_t off = (int64_t)g.grid_y * g.C;
#pragma unroll
  for (int k = 0; k < Pk<VEC>::NP; ++k) {
    const float2 ah = f2_unpack(a[k].hi), al = f2_unpack(a[k].lo);
    const float2 bh = f2_unpack(b[k].hi), bl = f2_unpack(b[k].lo);
    part[base + 2 * k] = make_float2(ah.x, al.x);
    part[off + base + 2 * k] = make_float2(bh.x, bl.x);
    if (2 * k + 1 < VEC) {
      part[base + 2 * k + 1] = make_float2(ah.y, al.y);
      part[off + base + 2 * k + 1] = make_float2(bh.y, bl.y);
    }
  }
}

// ---------------------------------------------------------------- stats --

template <typename T, int VEC>
__global__ void __launch_bounds__(kNThreads, kNSumBlocksPerSm)
    nhwc_stats_kernel(const T* __restrict__ x, NhwcGeom g, float2* __restrict__ part) {
  constexpr int NP = Pk<VEC>::NP;
  using V = Vec<T, VEC>;
  __shared__ float4 red[kNThreads * 2 * NP];
  pdl_launch_dependents();
  const int tx = threadIdx.x % g.TX, ty = threadIdx.x / g.TX;
  const int cv = blockIdx.x * g.TX + tx;
  const bool active = cv < g.Cv;
  int64_t r0, r1;
  row_slice(g, blockIdx.y, r0, r1);
  DF2 s1[NP], s2[NP];
  f2 sh2[NP], nsh2[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) s1[k] = s2[k] = DF2{0ull, 0ull};
  if (active) {
    float sh[VEC];
    V::cvt(V::ld(x + (int64_t)cv * VEC), sh);  // row 0: shift = x[0, c]
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      sh2[k] = pair_of<VEC>(sh, k);
      nsh2[k] = f2_sub(0ull, sh2[k]);
    }
    for (int64_t r = r0 + ty; r < r1; r += (int64_t)kNRowsUnroll1 * g.TY) {
      typename V::raw raw[kNRowsUnroll1];
#pragma unroll
      for (int u = 0; u < kNRowsUnroll1; ++u) {
        const int64_t ru = r + (int64_t)u * g.TY;
        if (ru < r1) raw[u] = V::ld(x + ru * g.C + (int64_t)cv * VEC);
      }
      f2 l2[NP];
#pragma unroll
      for (int k = 0; k < NP; ++k) l2[k] = 0ull;
#pragma unroll
      for (int u = 0; u < kNRowsUnroll1; ++u) {
        if (r + (int64_t)u * g.TY < r1) {
          float e[VEC];
          V::cvt(raw[u], e);
#pragma unroll
          for (int k = 0; k < NP; ++k) {
            const f2 x2 = pair_of<VEC>(e, k);
            const f2 d = f2_sub(x2, sh2[k]);
            df2_add(s1[k], d);
            if constexpr (sizeof(T) == 4) {
              const f2 bb = f2_sub(d, x2);
              s1[k].lo = f2_add(s1[k].lo, f2_add(f2_sub(x2, f2_sub(d, bb)), f2_sub(nsh2[k], bb)));
            }
            l2[k] = f2_fma(d, d, l2[k]);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < NP; ++k) df2_add(s2[k], l2[k]);
    }
  }
  column_tree<NP>(s1, s2, red, g);
  if (ty == 0 && active) write_partials<VEC>(s1, s2, g, cv, part);
}

// ------------------------------------------------------------ grad sums --

template <typename T, int VEC, int ACT>
__global__ void __launch_bounds__(kNThreads, kNSumBlocksPerSm)
    nhwc_grad_sums_kernel(const T* __restrict__ x, const T* __restrict__ dy, NhwcGeom g,
                          const float* __restrict__ stats, const float* __restrict__ beta,
                          float slope, float2* __restrict__ part) {
  constexpr int NP = Pk<VEC>::NP;
  using V = Vec<T, VEC>;
  __shared__ float4 red[kNThreads * 2 * NP];
  pdl_launch_dependents();
  const int tx = threadIdx.x % g.TX, ty = threadIdx.x / g.TX;
  const int cv = blockIdx.x * g.TX + tx;
  const bool active = cv < g.Cv;
  int64_t r0, r1;
  row_slice(g, blockIdx.y, r0, r1);
  DF2 p0[NP], p1[NP];
  f2 sh2[NP], nsh2[NP], md2[NP], sc2[NP], be2[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) p0[k] = p1[k] = DF2{0ull, 0ull};
  if (active) {
    float sh[VEC], md[VEC], sc[VEC], be[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const int64_t c = (int64_t)cv * VEC + k;
      sh[k] = stats[4 * (int64_t)g.C + c];
      md[k] = stats[5 * (int64_t)g.C + c];
      sc[k] = stats[3 * (int64_t)g.C + c];
      be[k] = beta ? beta[c] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      sh2[k] = pair_of<VEC>(sh, k);
      nsh2[k] = f2_sub(0ull, sh2[k]);
      md2[k] = pair_of<VEC>(md, k);
      sc2[k] = pair_of<VEC>(sc, k);
      be2[k] = pair_of<VEC>(be, k);
    }
    for (int64_t r = r0 + ty; r < r1; r += (int64_t)kNRowsUnroll2 * g.TY) {
      typename V::raw rx[kNRowsUnroll2], rd[kNRowsUnroll2];
#pragma unroll
      for (int u = 0; u < kNRowsUnroll2; ++u) {
        const int64_t ru = r + (int64_t)u * g.TY;
        if (ru < r1) {
          rx[u] = V::ld(x + ru * g.C + (int64_t)cv * VEC);
          rd[u] = V::ld(dy + ru * g.C + (int64_t)cv * VEC);
        }
      }
      // bf16 dy (plain or ReLU-gated, so still bf16 values) is summed over
      // the row group in fp32 first: exact for 8-bit significands within
      // 2^14 of each other.
      constexpr bool kLocalDy = sizeof(T) == 2 && ACT != GBN_ACT_LEAKY_RELU;
      f2 l0[NP];
#pragma unroll
      for (int k = 0; k < NP; ++k) l0[k] = 0ull;
#pragma unroll
      for (int u = 0; u < kNRowsUnroll2; ++u) {
        if (r + (int64_t)u * g.TY < r1) {
          float ex[VEC], ed[VEC];
          V::cvt(rx[u], ex);
          V::cvt(rd[u], ed);
#pragma unroll
          for (int k = 0; k < NP; ++k) {
            const f2 x2 = pair_of<VEC>(ex, k);
            f2 dy2 = pair_of<VEC>(ed, k);
            const f2 d = f2_sub(x2, sh2[k]);
            if constexpr (ACT != GBN_ACT_NONE) {
              // gate: d act / d pre with pre as the forward computed it
              const float2 pre = f2_unpack(f2_fma(f2_sub(d, md2[k]), sc2[k], be2[k]));
              dy2 = f2_mul_rounded(dy2, f2_pack(act_gate(pre.x, ACT, slope),
                                                act_gate(pre.y, ACT, slope)));
            }
            if constexpr (kLocalDy)
              l0[k] = f2_add(l0[k], dy2);
            else
              df2_add(p0[k], dy2);
            const f2 prod = f2_mul_rounded(dy2, d);
            df2_add(p1[k], prod);
            p1[k].lo = f2_add(p1[k].lo, f2_fma(dy2, d, prod ^ 0x8000000080000000ull));
            if constexpr (sizeof(T) == 4) {
              const f2 bb = f2_sub(d, x2);
              const f2 d_lo = f2_add(f2_sub(x2, f2_sub(d, bb)), f2_sub(nsh2[k], bb));
              p1[k].lo = f2_fma(dy2, d_lo, p1[k].lo);
            }
          }
        }
      }
      if constexpr (kLocalDy) {
#pragma unroll
        for (int k = 0; k < NP; ++k) df2_add(p0[k], l0[k]);
      }
    }
  }
  column_tree<NP>(p0, p1, red, g);
  if (ty == 0 && active) write_partials<VEC>(p0, p1, g, cv, part);
}

// ------------------------------------------------------------ finalize --

// One warp per channel: the grid_y partials added in a fixed order.
__device__ __forceinline__ void nhwc_reduce(const float2* part, const NhwcGeom& g, int64_t c,
                                            DF& s0, DF& s1) {
  const int lane = threadIdx.x & 31;
  DF a{0.f, 0.f}, b{0.f, 0.f};
  for (int jj = lane; jj < g.grid_y; jj += 32) {
    const float2 u = part[(int64_t)jj * g.C + c];
    const float2 w = part[((int64_t)g.grid_y + jj) * g.C + c];
    a = df_sum(a, DF{u.x, u.y});
    b = df_sum(b, DF{w.x, w.y});
  }
  s0 = warp_sum_df(a);
  s1 = warp_sum_df(b);
}

template <typename T>
__global__ void __launch_bounds__(kNThreads)
    nhwc_fwd_finalize_kernel(const T* __restrict__ x, NhwcGeom g,
                             const float2* __restrict__ part, const float* __restrict__ gamma,
                             float* __restrict__ stats, float* running_mean, float* running_var,
                             float momentum, float eps) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t c = (int64_t)blockIdx.x * (kNThreads / 32) + (threadIdx.x >> 5);
  if (c >= g.C) return;
  DF s1, s2;
  nhwc_reduce(part, g, c, s1, s2);
  const BnFwdFinal f = bn_fwd_final(s1, s2, g.Mh, g.Ml, gamma ? gamma[c] : 1.f, eps);
  if ((threadIdx.x & 31) == 0)  // shift = x[0, c]
    bn_fwd_write(f, to_f32(x[c]), g.C, (int)c, g.Mh + g.Ml, stats, running_mean, running_var,
                 momentum);
}

__global__ void __launch_bounds__(kNThreads)
    nhwc_bwd_finalize_kernel(NhwcGeom g, const float2* __restrict__ part,
                             const float* __restrict__ stats, float* __restrict__ grads) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t c = (int64_t)blockIdx.x * (kNThreads / 32) + (threadIdx.x >> 5);
  if (c >= g.C) return;
  DF p0, p1;
  nhwc_reduce(part, g, c, p0, p1);
  const int64_t C = g.C;
  const DF md{stats[6 * C + c], stats[7 * C + c]};
  const BnBwdFinal f = bn_bwd_final(p0, p1, md, stats[2 * C + c], stats[3 * C + c], g.Mh + g.Ml);
  if ((threadIdx.x & 31) == 0) {
    grads[c] = f.dgamma;
    grads[C + c] = f.dbeta;
    grads[2 * C + c] = f.k1;
    grads[3 * C + c] = f.k2;
  }
}

// ---------------------------------------------------------- apply / dx --

template <typename T, int VEC, int ACT, bool BWD>
__global__ void __launch_bounds__(kNThreads)
    nhwc_out_kernel(const T* __restrict__ x, const T* dy, T* out, NhwcGeom g,
                    const float* __restrict__ stats, const float* __restrict__ grads,
                    const float* __restrict__ beta, float slope, const float* __restrict__ imean,
                    const float* __restrict__ iscale) {
  using V = Vec<T, VEC>;
  constexpr int U = BWD ? kNRowsUnroll2 : kNRowsUnroll1;
  const int tx = threadIdx.x % g.TX, ty = threadIdx.x / g.TX;
  const int cv = blockIdx.x * g.TX + tx;
  if (cv >= g.Cv) return;
  int64_t r0, r1;
  row_slice(g, blockIdx.y, r0, r1);
  pdl_wait();
  float sh[VEC], md[VEC], sc[VEC], be[VEC], k1[VEC], k2[VEC];
  const int64_t C = g.C;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int64_t c = (int64_t)cv * VEC + k;
    if (stats != nullptr) {
      sh[k] = stats[4 * C + c];
      md[k] = stats[5 * C + c];
      sc[k] = stats[3 * C + c];
    } else {  // inference: (x - mean)*scale + beta from the given vectors
      sh[k] = imean[c];
      md[k] = 0.f;
      sc[k] = iscale[c];
    }
    be[k] = beta ? beta[c] : 0.f;
    if constexpr (BWD) {
      k1[k] = grads[2 * C + c];
      k2[k] = grads[3 * C + c];
    }
  }
  // This thread's rows r0 + ty + j*TY, j < n, walked from the last: the
  // sum kernel read every slice front to back, so the slice tails are the
  // likeliest to still be in L2.
  const int64_t n = r1 - r0 > ty ? (r1 - r0 - ty + g.TY - 1) / g.TY : 0;
  for (int64_t jb = n - 1; jb >= 0; jb -= U) {
    typename V::raw rx[U], rd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t ru = r0 + ty + (jb - u) * g.TY;
      if (jb - u >= 0) {
        rx[u] = V::ld(x + ru * C + (int64_t)cv * VEC);
        if constexpr (BWD) rd[u] = V::ld(dy + ru * C + (int64_t)cv * VEC);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t ru = r0 + ty + (jb - u) * g.TY;
      if (jb - u >= 0) {
        float e[VEC];
        V::cvt(rx[u], e);
        if constexpr (!BWD) {
#pragma unroll
          for (int k = 0; k < VEC; ++k)
            e[k] = act_out(fmaf((e[k] - sh[k]) - md[k], sc[k], be[k]), ACT, slope);
        } else {
          float gd[VEC];
          V::cvt(rd[u], gd);
#pragma unroll
          for (int k = 0; k < VEC; ++k) {
            const float xc = (e[k] - sh[k]) - md[k];
            const float gk = ACT == GBN_ACT_NONE
                                 ? gd[k]
                                 : __fmul_rn(gd[k], act_gate(fmaf(xc, sc[k], be[k]), ACT, slope));
            e[k] = fmaf(gk, sc[k], fmaf(xc, k1[k], k2[k]));
          }
        }
        V::store(out + ru * C + (int64_t)cv * VEC, e);
      }
    }
  }
}

// ---------------------------------------------------------------- host --

NhwcGeom make_geom(const NhwcPlan& p) {
  NhwcGeom g;
  g.M = p.M;
  g.C = (int32_t)p.C;
  g.Cv = (int32_t)(p.C / p.vec);  // p.vec divides C
  g.TX = p.TX;
  g.TY = kNThreads / p.TX;
  g.grid_y = p.grid_y;
  g.Mh = (float)p.M;
  g.Ml = (float)(p.M - (int64_t)g.Mh);
  return g;
}

dim3 sum_grid(const NhwcPlan& p) {
  return dim3((unsigned)((p.C / p.vec + p.TX - 1) / p.TX), (unsigned)p.grid_y, 1);
}

template <typename T, int VEC> struct NStats {
  static cudaError_t run(const NhwcPlan& p, const void* x, float2* part, cudaStream_t st) {
    return launch(nhwc_stats_kernel<T, VEC>, sum_grid(p), dim3(kNThreads), 0, st, false,
                  static_cast<const T*>(x), make_geom(p), part);
  }
};

template <typename T, int VEC> struct NGrad {
  static cudaError_t run(const NhwcPlan& p, const void* x, const void* dy, const float* stats,
                         const float* beta, int act, float slope, float2* part,
                         cudaStream_t st) {
    const T* xt = static_cast<const T*>(x);
    const T* dt = static_cast<const T*>(dy);
    if (act == GBN_ACT_RELU)
      return launch(nhwc_grad_sums_kernel<T, VEC, GBN_ACT_RELU>, sum_grid(p), dim3(kNThreads),
                    0, st, false, xt, dt, make_geom(p), stats, beta, slope, part);
    if (act == GBN_ACT_LEAKY_RELU)
      return launch(nhwc_grad_sums_kernel<T, VEC, GBN_ACT_LEAKY_RELU>, sum_grid(p),
                    dim3(kNThreads), 0, st, false, xt, dt, make_geom(p), stats, beta, slope,
                    part);
    return launch(nhwc_grad_sums_kernel<T, VEC, GBN_ACT_NONE>, sum_grid(p), dim3(kNThreads), 0,
                  st, false, xt, dt, make_geom(p), stats, beta, slope, part);
  }
};

template <typename T, int VEC> struct NOut {
  template <bool BWD>
  static cudaError_t go(const NhwcPlan& p, const void* x, const void* dy, void* out,
                        const float* stats, const float* grads, const float* beta, int act,
                        float slope, const float* imean, const float* iscale, cudaStream_t st) {
    const T* xt = static_cast<const T*>(x);
    const T* dt = static_cast<const T*>(dy);
    T* ot = static_cast<T*>(out);
    if (act == GBN_ACT_RELU)
      return launch(nhwc_out_kernel<T, VEC, GBN_ACT_RELU, BWD>, sum_grid(p), dim3(kNThreads), 0,
                    st, true, xt, dt, ot, make_geom(p), stats, grads, beta, slope, imean,
                    iscale);
    if (act == GBN_ACT_LEAKY_RELU)
      return launch(nhwc_out_kernel<T, VEC, GBN_ACT_LEAKY_RELU, BWD>, sum_grid(p),
                    dim3(kNThreads), 0, st, true, xt, dt, ot, make_geom(p), stats, grads, beta,
                    slope, imean, iscale);
    return launch(nhwc_out_kernel<T, VEC, GBN_ACT_NONE, BWD>, sum_grid(p), dim3(kNThreads), 0,
                  st, true, xt, dt, ot, make_geom(p), stats, grads, beta, slope, imean, iscale);
  }
  static cudaError_t run(const NhwcPlan& p, bool bwd, const void* x, const void* dy, void* out,
                         const float* stats, const float* grads, const float* beta, int act,
                         float slope, const float* imean, const float* iscale, cudaStream_t st) {
    return bwd ? go<true>(p, x, dy, out, stats, grads, beta, act, slope, imean, iscale, st)
               : go<false>(p, x, dy, out, stats, grads, beta, act, slope, imean, iscale, st);
  }
};

template <template <typename, int> class F, typename... A>
cudaError_t ndispatch(const NhwcPlan& p, int dtype, A&&... args) {
  if (dtype == GBN_F32) {
    switch (p.vec) {
      case 4: return F<float, 4>::run(p, args...);
      case 2: return F<float, 2>::run(p, args...);
      default: return F<float, 1>::run(p, args...);
    }
  }
  switch (p.vec) {
    case 8: return F<bf16, 8>::run(p, args...);
    case 4: return F<bf16, 4>::run(p, args...);
    case 2: return F<bf16, 2>::run(p, args...);
    default: return F<bf16, 1>::run(p, args...);
  }
}

}  // namespace

// Block shape and row slices for vectors of `vec` channels: TX = the power
// of two >= the vectors per row (at most 32), grid_y fills the resident
// block slots of the sum kernels with at least 8 rows per thread.
bool nhwc_plan(int64_t M, int64_t C, int vec, const DevInfo& dev, NhwcPlan* p) {
  if (M < 0 || C <= 0 || C > INT32_MAX || vec < 1) return false;
  p->M = M;
  p->C = C;
  p->vec = vec;
  const int64_t Cv = (C + vec - 1) / vec;
  int tx = 1;
  while (tx < 32 && tx < Cv) tx *= 2;
  p->TX = tx;
  const int64_t gx = (Cv + tx - 1) / tx;
  const int64_t slots = (int64_t)dev.sms * kNSumBlocksPerSm;
  const int64_t ty = kNThreads / tx;
  int64_t gy = slots / gx;
  const int64_t by_rows = (M + ty * 8 - 1) / (ty * 8);
  if (by_rows < gy) gy = by_rows;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  p->grid_y = (int)gy;
  p->ws_bytes = ((size_t)2 * (size_t)gy * (size_t)C * sizeof(float2) + 255) & ~(size_t)255;
  return true;
}

// Workspace for any vector width the call may pick (grid_y depends on it).
size_t nhwc_ws_bound(int64_t M, int64_t C, const DevInfo& dev) {
  size_t most = 0;
  for (int vec : {1, 2, 4, 8}) {
    NhwcPlan p;
    if (C % vec == 0 && nhwc_plan(M, C, vec, dev, &p) && p.ws_bytes > most) most = p.ws_bytes;
  }
  return most;
}

cudaError_t nhwc_forward(const NhwcPlan& p, int dtype, const void* x, void* y,
                         const float* gamma, const float* beta, float* stats,
                         float* running_mean, float* running_var, float momentum, float eps,
                         int act, float slope, void* ws, cudaStream_t st) {
  float2* part = static_cast<float2*>(ws);
  const NhwcGeom g = make_geom(p);
  cudaError_t e = ndispatch<NStats>(p, dtype, x, part, st);
  if (e != cudaSuccess) return e;
  const unsigned fb = (unsigned)((p.C + kNThreads / 32 - 1) / (kNThreads / 32));
  e = dtype == GBN_F32
          ? launch(nhwc_fwd_finalize_kernel<float>, dim3(fb), dim3(kNThreads), 0, st, true,
                   static_cast<const float*>(x), g, static_cast<const float2*>(part), gamma,
                   stats, running_mean, running_var, momentum, eps)
          : launch(nhwc_fwd_finalize_kernel<bf16>, dim3(fb), dim3(kNThreads), 0, st, true,
                   static_cast<const bf16*>(x), g, static_cast<const float2*>(part), gamma,
                   stats, running_mean, running_var, momentum, eps);
  if (e != cudaSuccess) return e;
  return ndispatch<NOut>(p, dtype, false, x, static_cast<const void*>(nullptr), y,
                         static_cast<const float*>(stats), static_cast<const float*>(nullptr),
                         beta, act, slope, static_cast<const float*>(nullptr),
                         static_cast<const float*>(nullptr), st);
}

cudaError_t nhwc_apply(const NhwcPlan& p, int dtype, const void* x, void* y, const float* stats,
                       const float* mean, const float* scale, const float* beta, int act,
                       float slope, cudaStream_t st) {
  return ndispatch<NOut>(p, dtype, false, x, static_cast<const void*>(nullptr), y, stats,
                         static_cast<const float*>(nullptr), beta, act, slope, mean, scale, st);
}

cudaError_t nhwc_backward(const NhwcPlan& p, int dtype, const void* x, const void* dy, void* dx,
                          const float* stats, const float* beta, int act, float slope,
                          float* grads, void* ws, cudaStream_t st) {
  float2* part = static_cast<float2*>(ws);
  const NhwcGeom g = make_geom(p);
  cudaError_t e = ndispatch<NGrad>(p, dtype, x, dy, stats, beta, act, slope, part, st);
  if (e != cudaSuccess) return e;
  const unsigned fb = (unsigned)((p.C + kNThreads / 32 - 1) / (kNThreads / 32));
  e = launch(nhwc_bwd_finalize_kernel, dim3(fb), dim3(kNThreads), 0, st, true, g,
             static_cast<const float2*>(part), stats, grads);
  if (e != cudaSuccess) return e;
  return ndispatch<NOut>(p, dtype, true, x, dy, dx, stats, static_cast<const float*>(grads),
                         beta, act, slope, static_cast<const float*>(nullptr),
                         static_cast<const float*>(nullptr), st);
}

}  // namespace gbn
