// Single-launch BatchNorm2d training forward and backward (NCHW) for small
// channels: the latency-bound shapes (a few thousand elements per channel)
// that the two-launch kernels would spend two launches on.
//
// Method: Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
// statistics, finalize kernels" -- per channel the shifted one-pass sums
// (d = x - x[0,c]), the forward finalize (mean, biased variance, inv_std,
// scale, running statistics) and the centred apply; backward the sums of dy
// and dy*(x - shift), the backward finalize (dgamma, dbeta, k1, k2) and
// dx = dy*scale + (x - mean)*k1 + k2.  The arithmetic is that of the other
// BatchNorm kernels (the same finalize helpers, exact per-element sums).
//
// GB300 design: one 256-thread block per channel stages the whole channel
// (at most 2048 elements, 8 KB of fp32; 16 KB backward) in shared memory as
// it reads it once -- every load of a thread in flight at once, so a channel
// costs one memory round trip -- reduces in a fixed tree, finalizes, and
// writes the outputs from shared memory.  One launch, no workspace, no
// second read from global memory.
//
// Channels of up to eight times that size take a thread-block cluster of K
// blocks (K = 2, 4 or 8) per channel: each block stages its contiguous share
// of at most 2048 elements the same way (again one memory round trip), puts
// its two double-fp32 partial sums in its shared memory, and after the
// cluster barrier every block reads the K partials through distributed
// shared memory and adds them in rank order -- the same bits in every block
// -- so each finalizes on its own and writes its share.  Still one launch
// and no workspace; the hand-off is the hardware cluster barrier, not a
// global-memory round trip or a second launch.  (One block per channel at
// 4920 elements, three load rounds per thread, measured slower than the
// two-launch kernels; larger channels take those.)
#include <cooperative_groups.h>

#include "bn_finalize.cuh"
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

constexpr int kSmallThreads = 256;

// x - shift and, for fp32 input, the rounding error of the subtraction
// (TwoSum); bf16 differences are exact unless the magnitudes differ by more
// than 2^16 (then one fp32 rounding per term).
template <typename T>
__device__ __forceinline__ void shifted(float e, float shift, float& d, float& d_lo) {
  d = __fsub_rn(e, shift);
  if constexpr (sizeof(T) == 4) {
    const float bb = __fsub_rn(d, e);
    d_lo = __fadd_rn(__fsub_rn(e, __fsub_rn(d, bb)), __fsub_rn(-shift, bb));
  } else {
    d_lo = 0.f;
  }
}

// Loads per thread issued together: a whole channel (kBnSmallMaxM / 256).
constexpr int kSmallBatch = (int)(kBnSmallMaxM / kSmallThreads);

__device__ __forceinline__ int64_t elem_offset(int m, int C, int c, int P, const FastDiv& pd) {
  const int n = (int)fast_div((uint32_t)m, pd);
  return ((int64_t)n * C + c) * P + (m - n * P);
}

// Dynamic shared memory: the channel's M values in (b, h, w) order, fp32
// (forward: x; backward: x, then the gated dy).
template <typename T>
__global__ void __launch_bounds__(kSmallThreads, 1)
    bn_small_fwd_kernel(const T* __restrict__ x, T* __restrict__ y, int B, int C, int P,
                        const float* __restrict__ gamma, const float* __restrict__ beta,
                        float* __restrict__ stats, float* running_mean, float* running_var,
                        float momentum, float eps, float Mh, float Ml, int act, float slope,
                        FastDiv pd) {
  extern __shared__ float vals[];
  __shared__ float2 red[64];
  const int c = blockIdx.x, t = threadIdx.x, M = B * P;
  const float shift = to_f32(x[(int64_t)c * P]);  // x[0, c, 0, 0]
  // The channel's parameters and running statistics are read now, with x:
  // after the block's reduction each would be one more memory round trip.
  const float gam = gamma ? gamma[c] : 1.f, b = beta ? beta[c] : 0.f;
  float rm = 0.f, rv = 0.f;
  if (t == 0) {
    rm = running_mean ? running_mean[c] : 0.f;
    rv = running_var ? running_var[c] : 0.f;
  }
  DF s1{0.f, 0.f}, s2{0.f, 0.f};
  for (int m0 = t; m0 < M; m0 += kSmallBatch * kSmallThreads) {
    float v[kSmallBatch];
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int m = m0 + u * kSmallThreads;
      v[u] = m < M ? to_f32(x[elem_offset(m, C, c, P, pd)]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int m = m0 + u * kSmallThreads;
      if (m < M) {
        vals[m] = v[u];
        float d, d_lo;
        shifted<T>(v[u], shift, d, d_lo);
        df_add(s1, d);
        if constexpr (sizeof(T) == 4) s1.lo = __fadd_rn(s1.lo, d_lo);
        df_add(s2, d * d);
      }
    }
  }
  block_sum2_df(s1, s2, red);  // contains __syncthreads: vals is complete
  const BnFwdFinal f = bn_fwd_final(s1, s2, Mh, Ml, gam, eps);
  const float mean_d = f.md.hi, scale = f.scale;
  for (int m = t; m < M; m += kSmallThreads)
    y[elem_offset(m, C, c, P, pd)] =
        from_f32<T>(act_out(fmaf((vals[m] - shift) - mean_d, scale, b), act, slope));
  if (t == 0)
    bn_fwd_write_from(f, shift, C, c, Mh + Ml, stats, running_mean, running_var, momentum, rm,
                      rv);
}

template <typename T>
__global__ void __launch_bounds__(kSmallThreads, 1)
    bn_small_bwd_kernel(const T* __restrict__ x, const T* __restrict__ dy, T* __restrict__ dx,
                        int B, int C, int P, const float* __restrict__ stats,
                        const float* __restrict__ beta, float* __restrict__ grads, float Mf,
                        int act, float slope, FastDiv pd) {
  extern __shared__ float vals[];  // [2][M]: x, then the gated dy
  __shared__ float2 red[64];
  const int c = blockIdx.x, t = threadIdx.x, M = B * P;
  const float inv_std = stats[2 * C + c], scale = stats[3 * C + c];
  const float shift = stats[4 * C + c], mean_d = stats[5 * C + c];
  const DF md{stats[6 * C + c], stats[7 * C + c]};
  const float bta = beta ? beta[c] : 0.f;
  DF p0{0.f, 0.f}, p1{0.f, 0.f};
  for (int m0 = t; m0 < M; m0 += kSmallBatch * kSmallThreads) {
    float xv[kSmallBatch], gv[kSmallBatch];
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int m = m0 + u * kSmallThreads;
      const int64_t o = m < M ? elem_offset(m, C, c, P, pd) : 0;
      xv[u] = m < M ? to_f32(x[o]) : 0.f;
      gv[u] = m < M ? to_f32(dy[o]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int m = m0 + u * kSmallThreads;
      if (m < M) {
        float g = gv[u];
        // with an activation, dy gated by d act / d pre (pre as in the forward)
        if (act != GBN_ACT_NONE)
          g = __fmul_rn(g, act_gate(fmaf((xv[u] - shift) - mean_d, scale, bta), act, slope));
        vals[m] = xv[u];
        vals[M + m] = g;
        float d, d_lo;
        shifted<T>(xv[u], shift, d, d_lo);
        df_add(p0, g);
        df_add_prod(p1, g, d);
        if constexpr (sizeof(T) == 4) p1.lo = fmaf(g, d_lo, p1.lo);
      }
    }
  }
  block_sum2_df(p0, p1, red);  // contains __syncthreads: vals is complete
  const BnBwdFinal f = bn_bwd_final(p0, p1, md, inv_std, scale, Mf);
  if (t == 0) {
    grads[c] = f.dgamma;
    grads[C + c] = f.dbeta;
    grads[2 * C + c] = f.k1;
    grads[3 * C + c] = f.k2;
  }
  for (int m = t; m < M; m += kSmallThreads) {
    const float xc = (vals[m] - shift) - mean_d;
    dx[elem_offset(m, C, c, P, pd)] = from_f32<T>(fmaf(vals[M + m], scale, fmaf(xc, f.k1, f.k2)));
  }
}

// ------------------------------------------------ one cluster per channel

namespace cg = cooperative_groups;

// Blocks of a cluster are consecutive in x: channel blockIdx.x / K, rank
// blockIdx.x % K, share [M r / K, M (r + 1) / K) of the channel's (b, h, w)
// order.
__device__ __forceinline__ void cluster_share(int M, int K, int r, int& lo, int& n) {
  lo = (int)((int64_t)M * r / K);
  n = (int)((int64_t)M * (r + 1) / K) - lo;
}

// The cluster's sums: the K blocks' (a, b) partials, read from each block's
// shared memory and added in rank order (every block gets the same bits).
__device__ __forceinline__ void cluster_sum2(cg::cluster_group& cl, float4* part, int K, DF& a,
                                             DF& b) {
  const float4 p0 = *cl.map_shared_rank(part, 0);
  a = DF{p0.x, p0.y};
  b = DF{p0.z, p0.w};
  for (int q = 1; q < K; ++q) {
    const float4 p = *cl.map_shared_rank(part, q);
    a = df_sum(a, DF{p.x, p.y});
    b = df_sum(b, DF{p.z, p.w});
  }
}

// Split cluster barrier: arrive once this block is done reading the others'
// shared memory, wait before exiting (no block leaves while another may
// still read its partials).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(kSmallThreads, 1)
    bn_cluster_fwd_kernel(const T* __restrict__ x, T* __restrict__ y, int B, int C, int P, int K,
                          const float* __restrict__ gamma, const float* __restrict__ beta,
                          float* __restrict__ stats, float* running_mean, float* running_var,
                          float momentum, float eps, float Mh, float Ml, int act, float slope,
                          FastDiv pd) {
  extern __shared__ float vals[];  // this block's share, fp32
  __shared__ float2 red[64];
  __shared__ float4 part;  // this block's (sum d, sum d^2) as (hi, lo) pairs
  cg::cluster_group cl = cg::this_cluster();
  const int r = (int)cl.block_rank();
  const int c = blockIdx.x / K, t = threadIdx.x, M = B * P;
  int lo, n;
  cluster_share(M, K, r, lo, n);
  const float shift = to_f32(x[(int64_t)c * P]);  // x[0, c, 0, 0]
  const float gam = gamma ? gamma[c] : 1.f, b = beta ? beta[c] : 0.f;
  float rm = 0.f, rv = 0.f;
  if (r == 0 && t == 0) {
    rm = running_mean ? running_mean[c] : 0.f;
    rv = running_var ? running_var[c] : 0.f;
  }
  DF s1{0.f, 0.f}, s2{0.f, 0.f};
  for (int i0 = t; i0 < n; i0 += kSmallBatch * kSmallThreads) {
    float v[kSmallBatch];
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int i = i0 + u * kSmallThreads;
      v[u] = i < n ? to_f32(x[elem_offset(lo + i, C, c, P, pd)]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int i = i0 + u * kSmallThreads;
      if (i < n) {
        vals[i] = v[u];
        float d, d_lo;
        shifted<T>(v[u], shift, d, d_lo);
        df_add(s1, d);
        if constexpr (sizeof(T) == 4) s1.lo = __fadd_rn(s1.lo, d_lo);
        df_add(s2, d * d);
      }
    }
  }
  block_sum2_df(s1, s2, red);  // contains __syncthreads: vals is complete
  if (t == 0) part = make_float4(s1.hi, s1.lo, s2.hi, s2.lo);
  cl.sync();  // every block's partials are visible cluster-wide
  cluster_sum2(cl, &part, K, s1, s2);
  cluster_arrive_relaxed();
  const BnFwdFinal f = bn_fwd_final(s1, s2, Mh, Ml, gam, eps);
  const float mean_d = f.md.hi, scale = f.scale;
  for (int i = t; i < n; i += kSmallThreads)
    y[elem_offset(lo + i, C, c, P, pd)] =
        from_f32<T>(act_out(fmaf((vals[i] - shift) - mean_d, scale, b), act, slope));
  if (r == 0 && t == 0)
    bn_fwd_write_from(f, shift, C, c, Mh + Ml, stats, running_mean, running_var, momentum, rm,
                      rv);
  cluster_wait();
}

template <typename T>
__global__ void __launch_bounds__(kSmallThreads, 1)
    bn_cluster_bwd_kernel(const T* __restrict__ x, const T* __restrict__ dy, T* __restrict__ dx,
                          int B, int C, int P, int K, const float* __restrict__ stats,
                          const float* __restrict__ beta, float* __restrict__ grads, float Mf,
                          int act, float slope, FastDiv pd) {
  extern __shared__ float vals[];  // [2][share]: x, then the gated dy
  __shared__ float2 red[64];
  __shared__ float4 part;  // this block's (sum dy, sum dy*(x - shift)) as (hi, lo) pairs
  cg::cluster_group cl = cg::this_cluster();
  const int r = (int)cl.block_rank();
  const int c = blockIdx.x / K, t = threadIdx.x, M = B * P;
  int lo, n;
  cluster_share(M, K, r, lo, n);
  const int S = (int)((M + K - 1) / K);  // the largest share: the dy half's offset
  const float inv_std = stats[2 * C + c], scale = stats[3 * C + c];
  const float shift = stats[4 * C + c], mean_d = stats[5 * C + c];
  const DF md{stats[6 * C + c], stats[7 * C + c]};
  const float bta = beta ? beta[c] : 0.f;
  DF p0{0.f, 0.f}, p1{0.f, 0.f};
  for (int i0 = t; i0 < n; i0 += kSmallBatch * kSmallThreads) {
    float xv[kSmallBatch], gv[kSmallBatch];
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int i = i0 + u * kSmallThreads;
      const int64_t o = i < n ? elem_offset(lo + i, C, c, P, pd) : 0;
      xv[u] = i < n ? to_f32(x[o]) : 0.f;
      gv[u] = i < n ? to_f32(dy[o]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kSmallBatch; ++u) {
      const int i = i0 + u * kSmallThreads;
      if (i < n) {
        float g = gv[u];
        // with an activation, dy gated by d act / d pre (pre as in the forward)
        if (act != GBN_ACT_NONE)
          g = __fmul_rn(g, act_gate(fmaf((xv[u] - shift) - mean_d, scale, bta), act, slope));
        vals[i] = xv[u];
        vals[S + i] = g;
        float d, d_lo;
        shifted<T>(xv[u], shift, d, d_lo);
        df_add(p0, g);
        df_add_prod(p1, g, d);
        if constexpr (sizeof(T) == 4) p1.lo = fmaf(g, d_lo, p1.lo);
      }
    }
  }
  block_sum2_df(p0, p1, red);  // contains __syncthreads: vals is complete
  if (t == 0) part = make_float4(p0.hi, p0.lo, p1.hi, p1.lo);
  cl.sync();
  cluster_sum2(cl, &part, K, p0, p1);
  cluster_arrive_relaxed();
  const BnBwdFinal f = bn_bwd_final(p0, p1, md, inv_std, scale, Mf);
  for (int i = t; i < n; i += kSmallThreads) {
    const float xc = (vals[i] - shift) - mean_d;
    dx[elem_offset(lo + i, C, c, P, pd)] =
        from_f32<T>(fmaf(vals[S + i], scale, fmaf(xc, f.k1, f.k2)));
  }
  if (r == 0 && t == 0) {
    grads[c] = f.dgamma;
    grads[C + c] = f.dbeta;
    grads[2 * C + c] = f.k1;
    grads[3 * C + c] = f.k2;
  }
  cluster_wait();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_clusters(void (*kern)(KArgs...), int K, unsigned grid, size_t smem,
                            cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <typename T>
cudaError_t small_fwd(const void* x, void* y, int64_t B, int64_t C, int64_t HW, const float* gamma,
                      const float* beta, float* stats, float* running_mean, float* running_var,
                      float momentum, float eps, int act, float slope, int K,
                      cudaStream_t st) {
  const int64_t M = B * HW;
  const float Mh = (float)M, Ml = (float)(M - (int64_t)Mh);
  if (K > 1)
    return launch_clusters(bn_cluster_fwd_kernel<T>, K, (unsigned)(C * K),
                           (size_t)((M + K - 1) / K) * sizeof(float), st,
                           static_cast<const T*>(x), static_cast<T*>(y), (int)B, (int)C, (int)HW,
                           K, gamma, beta, stats, running_mean, running_var, momentum, eps, Mh,
                           Ml, act, slope, make_fast_div((uint32_t)HW));
  return launch(bn_small_fwd_kernel<T>, dim3((unsigned)C), dim3(kSmallThreads),
                (size_t)M * sizeof(float), st, false, static_cast<const T*>(x),
                static_cast<T*>(y), (int)B, (int)C, (int)HW, gamma, beta, stats, running_mean,
                running_var, momentum, eps, Mh, Ml, act, slope, make_fast_div((uint32_t)HW));
}

template <typename T>
cudaError_t small_bwd(const void* x, const void* dy, void* dx, int64_t B, int64_t C, int64_t HW,
                      const float* stats, const float* beta, int act, float slope, float* grads,
                      int K, cudaStream_t st) {
  const int64_t M = B * HW;
  if (K > 1)
    return launch_clusters(bn_cluster_bwd_kernel<T>, K, (unsigned)(C * K),
                           2 * (size_t)((M + K - 1) / K) * sizeof(float), st,
                           static_cast<const T*>(x), static_cast<const T*>(dy),
                           static_cast<T*>(dx), (int)B, (int)C, (int)HW, K, stats, beta, grads,
                           (float)M, act, slope, make_fast_div((uint32_t)HW));
  return launch(bn_small_bwd_kernel<T>, dim3((unsigned)C), dim3(kSmallThreads),
                2 * (size_t)M * sizeof(float), st, false, static_cast<const T*>(x),
                static_cast<const T*>(dy), static_cast<T*>(dx), (int)B, (int)C, (int)HW, stats,
                beta, grads, (float)M, act, slope, make_fast_div((uint32_t)HW));
}

}  // namespace

int bn_small_blocks(int64_t M, int64_t C, int64_t lim, const DevInfo& dev) {
  if (lim <= 0 || lim > kBnSmallMaxM) return 0;
  for (int K = 1; K <= kBnClusterMax; K *= 2)
    if ((M + K - 1) / K <= lim)
      return C * K <= (int64_t)dev.sms * (K == 1 ? kBnSmallBlocksPerSm : 1) ? K : 0;
  return 0;
}

cudaError_t bn_small_forward(int dtype, const void* x, void* y, int64_t B, int64_t C,
                             int64_t HW, const float* gamma, const float* beta, float* stats,
                             float* running_mean, float* running_var, float momentum, float eps,
                             int act, float slope, int K, cudaStream_t st) {
  if (K < 1 || K > kBnClusterMax || (K & (K - 1)) != 0) return cudaErrorInvalidValue;
  if (dtype == GBN_F32)
    return small_fwd<float>(x, y, B, C, HW, gamma, beta, stats, running_mean, running_var,
                            momentum, eps, act, slope, K, st);
  return small_fwd<bf16>(x, y, B, C, HW, gamma, beta, stats, running_mean, running_var, momentum,
                         eps, act, slope, K, st);
}

cudaError_t bn_small_backward(int dtype, const void* x, const void* dy, void* dx, int64_t B,
                              int64_t C, int64_t HW, const float* stats, const float* beta,
                              int act, float slope, float* grads, int K, cudaStream_t st) {
  if (K < 1 || K > kBnClusterMax || (K & (K - 1)) != 0) return cudaErrorInvalidValue;
  if (dtype == GBN_F32)
    return small_bwd<float>(x, dy, dx, B, C, HW, stats, beta, act, slope, grads, K, st);
  return small_bwd<bf16>(x, dy, dx, B, C, HW, stats, beta, act, slope, grads, K, st);
}

}  // namespace gbn
