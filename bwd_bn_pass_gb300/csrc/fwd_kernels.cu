// LayerNorm and RMSNorm training forward (rows [R, H]).
//
// Method: nvFuser issue #3629 "Performance gap between manual nvfuser
// definition and thunder.jit for rmsnorm" -- the forward of the
// `rmsnorm_prims` / F.rms_norm section: y = w*x*rstd with
// rstd = 1/sqrt(mean(x^2) + eps), the statistic the backward takes.
// nvFuser issue #1473 "Why is LayerNorm Backward Segmenting?" -- the forward
// whose saved statistics (the fp32 per-row mean and rstd) the backward
// repros take:
// y = (z - mean)*rstd*gamma + beta with the biased variance, and in the fused
// form z = residual + mask*scale*(input + bias), the residual-stream output
// (written when requested).
//
// GB300 design: no reduction crosses rows, so each row belongs to one team of
// threads that loads it once into registers (16-byte vectors; every load of
// the row is issued before any is used), reduces with warp shuffles, and
// writes y (and z) from the registers:
//   * rows of at most 256 vectors: the team is one warp (no block barrier),
//     which keeps the row's fp32 values in shared memory;
//   * rows of at most 2048 vectors: the team is a 256-thread block (one
//     shared-memory exchange per reduction);
//   * otherwise, or without 16-byte alignment: a block per row streams the
//     row from global memory once per pass (the later passes hit L2).
// LayerNorm centres every row on its first element (shift = z_r0): it sums
// d = z - shift, takes mean_d = mean(d), the variance as a second pass
// sum (d - mean_d)^2 (never E[z^2] - mean^2), and y from (d - mean_d), so a
// row whose mean is large next to its spread loses nothing to the rounding
// of the mean (the same shifted form as the BatchNorm kernels).  Reductions
// are fixed trees, so results are bit-deterministic.
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

struct FwdArgs {
  const void* x;         // RMSNorm x; LayerNorm input (fused: the dropout input)
  const void* res;       // fused: residual
  const void* bias;      // fused: bias or null
  const uint8_t* mask;   // fused: mask (nonzero = kept) or null
  const void* w;         // RMSNorm weight / LayerNorm gamma, or null (ones)
  const void* beta;      // LayerNorm beta or null (zeros)
  void* y;
  void* z;               // fused: z output or null
  float* mean;           // LayerNorm
  float* rstd;
  int64_t R;
  int32_t H;
  int32_t Hv;            // 16-byte vectors per row (vector kernels)
  float eps;
  float scale;           // dropout scale
};

constexpr int kThreads = 256;

// Sum over the team (a warp, or the whole block in a fixed order).
template <bool WARP>
__device__ __forceinline__ float team_sum(float v, float* red) {
  v = warp_sum(v);
  if constexpr (WARP) {
    return v;
  } else {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();  // the previous use of red is finished
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
  }
}

// Mask bytes of one vector of VE elements (8 or 4 bytes).
template <int VE>
__device__ __forceinline__ uint2 load_mask(const uint8_t* p) {
  if constexpr (VE == 8) return *reinterpret_cast<const uint2*>(p);
  return make_uint2(*reinterpret_cast<const uint32_t*>(p), 0u);
}
__device__ __forceinline__ bool mask_byte(uint2 m, int e) {
  const uint32_t w = e < 4 ? m.x : m.y;
  return ((w >> (8 * (e & 3))) & 0xffu) != 0u;
}

// Rows of at most 8*256 vectors: a 256-thread block per row, KV vectors per
// thread in registers.
template <typename T, int KIND, int KV>
__global__ void __launch_bounds__(kThreads) row_fwd_kernel(FwdArgs a) {
  constexpr bool WARP = false;
  constexpr int VE = 16 / sizeof(T);
  constexpr bool FUSED = KIND == GBN_ROW_LN_FUSED;
  using V = Vec<T, VE>;
  __shared__ float red[32];
  const int lane = threadIdx.x & 31;
  const int tt = WARP ? lane : (int)threadIdx.x;    // index in the team
  const int TS = WARP ? 32 : (int)blockDim.x;       // team size
  const int64_t team =
      WARP ? (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5) : (int64_t)blockIdx.x;
  const int64_t nteams = WARP ? (int64_t)gridDim.x * (blockDim.x >> 5) : (int64_t)gridDim.x;
  const T* x = static_cast<const T*>(a.x);
  const T* res = static_cast<const T*>(a.res);
  const T* bias = static_cast<const T*>(a.bias);
  const T* w = static_cast<const T*>(a.w);
  const T* beta = static_cast<const T*>(a.beta);
  const float invH = 1.f / (float)a.H;

  for (int64_t r = team; r < a.R; r += nteams) {
    const int64_t ro = r * (int64_t)a.H;
    typename V::raw rx[KV], rr[KV];
    uint2 mk[KV];
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = tt + k * TS;
      if (vi < a.Hv) {
        rx[k] = V::ld(x + ro + (int64_t)vi * VE);
        if constexpr (FUSED) {
          rr[k] = V::ld(res + ro + (int64_t)vi * VE);
          mk[k] = a.mask ? load_mask<VE>(a.mask + ro + (int64_t)vi * VE)
                         : make_uint2(0x01010101u, 0x01010101u);
        }
      }
    }
    float z[KV][VE];
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = tt + k * TS;
      if (vi < a.Hv) {
        V::cvt(rx[k], z[k]);
        if constexpr (FUSED) {
          float rv[VE], bv[VE];
          V::cvt(rr[k], rv);
          if (bias) {
            V::cvt(V::ld(bias + (int64_t)vi * VE), bv);
          } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) bv[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float keep = mask_byte(mk[k], e) ? a.scale : 0.f;
            z[k][e] = fmaf(keep, z[k][e] + bv[e], rv[e]);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) z[k][e] = 0.f;
      }
    }
    // shift = z of the row's first element (team thread 0, vector 0).  In a
    // block team it goes through red[31] (team_sum uses red[0..7]); the
    // previous row's reads of red[31] precede that row's later barriers.
    float shift = 0.f;
    if constexpr (KIND != GBN_ROW_RMS) {
      if constexpr (WARP) {
        shift = __shfl_sync(0xffffffffu, z[0][0], 0);
      } else {
        if (tt == 0) red[31] = z[0][0];
        __syncthreads();
        shift = red[31];
      }
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < KV; ++k)
      if (tt + k * TS < a.Hv) {
#pragma unroll
        for (int e = 0; e < VE; ++e)
          s += KIND == GBN_ROW_RMS ? z[k][e] * z[k][e] : z[k][e] - shift;
      }
    float md = 0.f, rs;
    if constexpr (KIND == GBN_ROW_RMS) {
      rs = 1.f / sqrtf(team_sum<WARP>(s, red) * invH + a.eps);
    } else {
      md = team_sum<WARP>(s, red) * invH;
      float s2 = 0.f;
#pragma unroll
      for (int k = 0; k < KV; ++k)
        if (tt + k * TS < a.Hv) {
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float c = (z[k][e] - shift) - md;
            s2 = fmaf(c, c, s2);
          }
        }
      rs = 1.f / sqrtf(team_sum<WARP>(s2, red) * invH + a.eps);
    }
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = tt + k * TS;
      if (vi >= a.Hv) continue;
      float g[VE], b[VE], o[VE];
      if (w) {
        V::cvt(V::ld(w + (int64_t)vi * VE), g);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) g[e] = 1.f;
      }
      if (KIND != GBN_ROW_RMS && beta) {
        V::cvt(V::ld(beta + (int64_t)vi * VE), b);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) b[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < VE; ++e)
        o[e] = KIND == GBN_ROW_RMS ? (z[k][e] * rs) * g[e]
                                   : fmaf(((z[k][e] - shift) - md) * rs, g[e], b[e]);
      V::store(static_cast<T*>(a.y) + ro + (int64_t)vi * VE, o);
      if (FUSED && a.z != nullptr) V::store(static_cast<T*>(a.z) + ro + (int64_t)vi * VE, z[k]);
    }
    if (tt == 0) {
      if (KIND != GBN_ROW_RMS) a.mean[r] = shift + md;
      a.rstd[r] = rs;
    }
  }
}

// Rows of at most 256 vectors: one warp per row.  Lane l owns vectors
// l, l+32, ... of the row; it keeps their fp32 z values in its own slice of
// shared memory (no other lane reads them, so no barrier is needed) rather
// than in registers, which keeps the kernel within 64 registers and four
// 8-warp blocks per SM; UNR vectors per lane are loaded before any is
// converted.  (Loading all of a lane's vectors at once, eight for a
// 1600-wide bf16 row, needs ~125 registers and halves the resident warps; it
// measured slower.)
template <typename T, int KIND, int UNR>
__global__ void __launch_bounds__(kThreads, 4) row_fwd_warp_kernel(FwdArgs a) {
  constexpr int VE = 16 / sizeof(T);
  constexpr bool FUSED = KIND == GBN_ROW_LN_FUSED;
  using V = Vec<T, VE>;
  extern __shared__ __align__(16) float zsm[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  float* zw = zsm + (size_t)wib * a.Hv * VE;  // this warp's row of z
  const int64_t team = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
  const int64_t nteams = (int64_t)gridDim.x * (blockDim.x >> 5);
  const T* x = static_cast<const T*>(a.x);
  const T* res = static_cast<const T*>(a.res);
  const T* bias = static_cast<const T*>(a.bias);
  const T* w = static_cast<const T*>(a.w);
  const T* beta = static_cast<const T*>(a.beta);
  const float invH = 1.f / (float)a.H;

  auto zvec = [&](int64_t ro, int vi, float (&z)[VE]) {
    V::cvt(V::ld(x + ro + (int64_t)vi * VE), z);
    if constexpr (FUSED) {
      float rv[VE], bv[VE];
      V::cvt(V::ld(res + ro + (int64_t)vi * VE), rv);
      const uint2 mk = a.mask ? load_mask<VE>(a.mask + ro + (int64_t)vi * VE)
                              : make_uint2(0x01010101u, 0x01010101u);
      if (bias) {
        V::cvt(V::ld(bias + (int64_t)vi * VE), bv);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) bv[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const float keep = mask_byte(mk, e) ? a.scale : 0.f;
        z[e] = fmaf(keep, z[e] + bv[e], rv[e]);
      }
    }
  };

  for (int64_t r = team; r < a.R; r += nteams) {
    const int64_t ro = r * (int64_t)a.H;
    float shift = 0.f;
    if constexpr (KIND != GBN_ROW_RMS) {
      float z0[VE];
      if (lane == 0) zvec(ro, 0, z0);
      shift = __shfl_sync(0xffffffffu, lane == 0 ? z0[0] : 0.f, 0);
    }
    float s = 0.f;
    for (int v0 = lane; v0 < a.Hv; v0 += 32 * UNR) {
      float z[UNR][VE];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        if (v0 + 32 * u < a.Hv) zvec(ro, v0 + 32 * u, z[u]);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int vi = v0 + 32 * u;
        if (vi >= a.Hv) continue;
        float4* d = reinterpret_cast<float4*>(zw + (size_t)vi * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) d[e / 4] = make_float4(z[u][e], z[u][e + 1], z[u][e + 2], z[u][e + 3]);
#pragma unroll
        for (int e = 0; e < VE; ++e)
          s += KIND == GBN_ROW_RMS ? z[u][e] * z[u][e] : z[u][e] - shift;
      }
    }
    float md = 0.f, rs;
    if constexpr (KIND == GBN_ROW_RMS) {
      rs = 1.f / sqrtf(warp_sum(s) * invH + a.eps);
    } else {
      md = warp_sum(s) * invH;
      float s2 = 0.f;
      for (int vi = lane; vi < a.Hv; vi += 32) {
        const float4* d = reinterpret_cast<const float4*>(zw + (size_t)vi * VE);
#pragma unroll
        for (int e = 0; e < VE; e += 4) {
          const float4 q = d[e / 4];
          const float c0 = (q.x - shift) - md, c1 = (q.y - shift) - md;
          const float c2 = (q.z - shift) - md, c3 = (q.w - shift) - md;
          s2 = fmaf(c0, c0, s2);
          s2 = fmaf(c1, c1, s2);
          s2 = fmaf(c2, c2, s2);
          s2 = fmaf(c3, c3, s2);
        }
      }
      rs = 1.f / sqrtf(warp_sum(s2) * invH + a.eps);
    }
    for (int vi = lane; vi < a.Hv; vi += 32) {
      float z[VE], g[VE], b[VE], o[VE];
      const float4* d = reinterpret_cast<const float4*>(zw + (size_t)vi * VE);
#pragma unroll
      for (int e = 0; e < VE; e += 4) {
        const float4 q = d[e / 4];
        z[e] = q.x; z[e + 1] = q.y; z[e + 2] = q.z; z[e + 3] = q.w;
      }
      if (w) {
        V::cvt(V::ld(w + (int64_t)vi * VE), g);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) g[e] = 1.f;
      }
      if (KIND != GBN_ROW_RMS && beta) {
        V::cvt(V::ld(beta + (int64_t)vi * VE), b);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) b[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < VE; ++e)
        o[e] = KIND == GBN_ROW_RMS ? (z[e] * rs) * g[e] : fmaf(((z[e] - shift) - md) * rs, g[e], b[e]);
      V::store(static_cast<T*>(a.y) + ro + (int64_t)vi * VE, o);
      if (FUSED && a.z != nullptr) V::store(static_cast<T*>(a.z) + ro + (int64_t)vi * VE, z);
    }
    if (lane == 0) {
      if (KIND != GBN_ROW_RMS) a.mean[r] = shift + md;
      a.rstd[r] = rs;
    }
    __syncwarp();  // the next row's z stores follow this row's reads
  }
}

// Any H and alignment: block g owns rows g, g+G, ...; each pass walks the
// row with stride blockDim (z is recomputed, the row is re-read from L2).
template <typename T, int KIND>
__global__ void __launch_bounds__(kThreads) row_fwd_generic_kernel(FwdArgs a) {
  constexpr bool FUSED = KIND == GBN_ROW_LN_FUSED;
  __shared__ float red[32];
  const int64_t H = a.H;
  const T* x = static_cast<const T*>(a.x);
  const T* res = static_cast<const T*>(a.res);
  const T* bias = static_cast<const T*>(a.bias);
  const T* w = static_cast<const T*>(a.w);
  const T* beta = static_cast<const T*>(a.beta);
  const float invH = 1.f / (float)a.H;
  auto zval = [&](int64_t o, int64_t j) {
    float v = to_f32(x[o + j]);
    if constexpr (FUSED) {
      const float keep = (a.mask == nullptr || a.mask[o + j] != 0) ? a.scale : 0.f;
      v = fmaf(keep, v + (bias ? to_f32(bias[j]) : 0.f), to_f32(res[o + j]));
    }
    return v;
  };
  for (int64_t r = blockIdx.x; r < a.R; r += gridDim.x) {
    const int64_t o = r * H;
    const float shift = KIND == GBN_ROW_RMS ? 0.f : zval(o, 0);
    float s = 0.f;
    for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
      const float v = zval(o, j);
      s += KIND == GBN_ROW_RMS ? v * v : v - shift;
    }
    float md = 0.f, rs;
    if constexpr (KIND == GBN_ROW_RMS) {
      rs = 1.f / sqrtf(team_sum<false>(s, red) * invH + a.eps);
    } else {
      md = team_sum<false>(s, red) * invH;
      float s2 = 0.f;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float c = (zval(o, j) - shift) - md;
        s2 = fmaf(c, c, s2);
      }
      rs = 1.f / sqrtf(team_sum<false>(s2, red) * invH + a.eps);
    }
    for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
      const float v = zval(o, j);
      const float g = w ? to_f32(w[j]) : 1.f;
      const float b = (KIND != GBN_ROW_RMS && beta) ? to_f32(beta[j]) : 0.f;
      const float out =
          KIND == GBN_ROW_RMS ? (v * rs) * g : fmaf(((v - shift) - md) * rs, g, b);
      static_cast<T*>(a.y)[o + j] = from_f32<T>(out);
      if (FUSED && a.z != nullptr) static_cast<T*>(a.z)[o + j] = from_f32<T>(v);
    }
    if (threadIdx.x == 0) {
      if (KIND != GBN_ROW_RMS) a.mean[r] = shift + md;
      a.rstd[r] = rs;
    }
  }
}

template <typename T, int KIND>
cudaError_t launch_kind(const FwdArgs& a, bool vec_ok, const DevInfo& dev, cudaStream_t st) {
  const int64_t R = a.R;
  if (vec_ok && a.Hv <= 256) {
    // one warp per row, 8 per block; z of each row in shared memory
    constexpr int VE = 16 / sizeof(T);
    const size_t smem = (size_t)(kThreads / 32) * a.Hv * VE * sizeof(float);
    int64_t G = (R + 7) / 8;
    const int64_t cap = (int64_t)dev.sms * 4;
    if (G > cap) G = cap;
    return launch(row_fwd_warp_kernel<T, KIND, 4>, dim3((unsigned)G), dim3(kThreads), smem, st,
                  false, a);
  }
  int64_t G = R;
  const int64_t cap = (int64_t)dev.sms * 8;
  if (G > cap) G = cap;
  const dim3 grid((unsigned)G), block(kThreads);
  if (vec_ok && a.Hv <= 4 * kThreads)
    return launch(row_fwd_kernel<T, KIND, 4>, grid, block, 0, st, false, a);
  if (vec_ok && a.Hv <= 8 * kThreads)
    return launch(row_fwd_kernel<T, KIND, 8>, grid, block, 0, st, false, a);
  return launch(row_fwd_generic_kernel<T, KIND>, grid, block, 0, st, false, a);
}

template <typename T>
cudaError_t launch_typed(int kind, const FwdArgs& a, bool vec_ok, const DevInfo& dev,
                         cudaStream_t st) {
  if (kind == GBN_ROW_RMS) return launch_kind<T, GBN_ROW_RMS>(a, vec_ok, dev, st);
  if (kind == GBN_ROW_LN) return launch_kind<T, GBN_ROW_LN>(a, vec_ok, dev, st);
  return launch_kind<T, GBN_ROW_LN_FUSED>(a, vec_ok, dev, st);
}

template <typename T, int UNR>
cudaError_t configure_unr(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = cudaFuncSetAttribute(row_fwd_warp_kernel<T, GBN_ROW_RMS, UNR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  if ((r = cudaFuncSetAttribute(row_fwd_warp_kernel<T, GBN_ROW_LN, UNR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  if ((r = cudaFuncSetAttribute(row_fwd_warp_kernel<T, GBN_ROW_LN_FUSED, UNR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
    e = r;
  return e;
}

template <typename T>
cudaError_t configure_typed(int bytes) {
  return configure_unr<T, 4>(bytes);
}

}  // namespace

// The warp kernels hold at most 8 warps x 256 vectors x 8 fp32 values (64 KB).
cudaError_t row_fwd_configure() {
  const int bytes = (kThreads / 32) * 256 * 8 * (int)sizeof(float);
  cudaError_t e1 = configure_typed<float>(bytes);
  cudaError_t e2 = configure_typed<bf16>(bytes);
  return e1 != cudaSuccess ? e1 : e2;
}

cudaError_t row_fwd_launch(int kind, int dtype, const RowFwdPtrs& p, int64_t R, int64_t H,
                           float eps, float scale, bool vec_ok, const DevInfo& dev,
                           cudaStream_t st) {
  if (R == 0 || H == 0) return cudaSuccess;
  FwdArgs a;
  a.x = p.x;
  a.res = p.residual;
  a.bias = p.bias;
  a.mask = p.mask;
  a.w = p.w;
  a.beta = p.beta;
  a.y = p.y;
  a.z = p.z;
  a.mean = p.mean;
  a.rstd = p.rstd;
  a.R = R;
  a.H = (int32_t)H;
  a.Hv = (int32_t)(H * (dtype == GBN_F32 ? 4 : 2) / 16);
  a.eps = eps;
  a.scale = scale;
  return dtype == GBN_F32 ? launch_typed<float>(kind, a, vec_ok, dev, st)
                          : launch_typed<bf16>(kind, a, vec_ok, dev, st);
}

}  // namespace gbn
