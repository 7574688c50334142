// RMSNorm backward.
//
// Method: nvFuser issue #3629 "Performance gap between manual nvfuser
// definition and thunder.jit for rmsnorm", section "nvfuser pre-generated
// definition" (rmsnorm_bwd_fusion), with the saved statistic taken as
// rstd = 1/rms like the Thunder definition on the same page:
//   S_r   = sum_j w_j * dy_rj * x_rj
//   dx_rj = rstd_r * w_j * dy_rj - x_rj * rstd_r^3 * S_r / H
//   dw_j  = sum_r dy_rj * x_rj * rstd_r
// The page's lessons are kept: rstd^3 is two multiplies (never pow), and
// rstd and the row sum stay fp32 (no bf16 round trip).
//
// GB300 design.  A persistent grid (one block per SM) owns rows r = g, g+G,
// ...; a single thread streams each block's next rows of x and dy into a
// shared-memory ring with 1-D bulk copies (cp.async.bulk + mbarrier), so the
// loads of several rows are always in flight without occupying threads.  Each
// thread owns fixed 16-byte column vectors: it keeps their weights and its
// dweight accumulators in registers for the whole kernel, reads x and dy once
// from shared memory, reduces S_r across the block with warp shuffles, and
// writes dx.  At the end every block stores its dweight partial row; a second
// small kernel (colsum.cu) adds the G rows in a fixed order.  fp32 outputs
// accumulate dweight in double-fp32 with exact product residuals.
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

constexpr int kMaxStages = 8;
constexpr uint32_t kRmsHeader = 64 + 2 * 32 * 4;  // mbarriers + row-sum slots

struct RmsArgs {
  const void* dy;
  const void* x;
  const void* w;
  const float* rstd;
  void* dx;
  float* part;
  int* status;
  int64_t R;
  int32_t H;
  int32_t Hv;      // 16-byte vectors per row (fast path)
  int32_t nstage;
  uint32_t row_bytes;
};

template <typename T, int KV, bool COMP>
__global__ void __launch_bounds__(512, 1) rms_bwd_fast_kernel(RmsArgs a) {
  constexpr int VE = 16 / sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 64);
  unsigned char* data = smem + kRmsHeader;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t nrows = (a.R - g + G - 1) / G;
  const int nst = a.nstage;
  const uint32_t rb = a.row_bytes;
  const char* gx = static_cast<const char*>(a.x);
  const char* gdy = static_cast<const char*>(a.dy);

  auto issue = [&](int64_t i) {
    const int s = (int)(i % nst);
    const int64_t r = g + i * G;
    mbar_arrive_expect_tx(&bar[s], 2u * rb);
    bulk_g2s(data + (size_t)(2 * s) * rb, gx + r * rb, rb, &bar[s]);
    bulk_g2s(data + (size_t)(2 * s + 1) * rb, gdy + r * rb, rb, &bar[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < nrows && i < nst; ++i) issue(i);

  float wv[KV][VE];
  const T* w = static_cast<const T*>(a.w);
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int vi = tid + k * blockDim.x;
    if (vi < a.Hv) Vec16<T>::load(w + (int64_t)vi * VE, wv[k]);
    else
#pragma unroll
      for (int e = 0; e < VE; ++e) wv[k][e] = 0.f;
  }
  DF acc[KV][VE];
#pragma unroll
  for (int k = 0; k < KV; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[k][e] = DF{0.f, 0.f};

  const float Hf = (float)a.H;
  bool failed = false;
  int64_t i = 0;
  for (; i < nrows; ++i) {
    const int s = (int)(i % nst);
    const uint32_t par = (uint32_t)((i / nst) & 1);
    const int64_t r = g + i * G;
    const float rho = a.rstd[r];
    const bool ok = mbar_wait_bounded(&bar[s], par);

    float xv[KV][VE], dv[KV][VE];
    float part = 0.f;
    const unsigned char* sx = data + (size_t)(2 * s) * rb;
    const unsigned char* sdy = data + (size_t)(2 * s + 1) * rb;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = tid + k * blockDim.x;
      if (ok && vi < a.Hv) {
        Vec16<T>::load(sx + (size_t)vi * 16, xv[k]);
        Vec16<T>::load(sdy + (size_t)vi * 16, dv[k]);
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) { xv[k][e] = 0.f; dv[k][e] = 0.f; }
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) part = fmaf(wv[k][e] * dv[k][e], xv[k][e], part);
    }
    part = warp_sum(part);
    float* slot = red + (i & 1) * 32;
    if (lane == 0) slot[warp] = part;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    // Every thread holds its part of row i in registers: refill the stage.
    if (tid == 0 && i + nst < nrows) {
      fence_proxy_async_smem();
      issue(i + nst);
    }
    float S = 0.f;
    for (int wi = 0; wi < nwarps; ++wi) S += slot[wi];
    const float coef = rho * rho * rho * S / Hf;

    T* dxr = static_cast<T*>(a.dx) + r * (int64_t)a.H;
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = tid + k * blockDim.x;
      if (vi < a.Hv) {
        float o[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          o[e] = fmaf(-xv[k][e], coef, rho * wv[k][e] * dv[k][e]);
          if constexpr (COMP) {
            const float p = dv[k][e] * xv[k][e];
            const float pe = fmaf(dv[k][e], xv[k][e], -p);
            const float q = p * rho;
            const float qe = fmaf(p, rho, -q);
            df_add(acc[k][e], q);
            acc[k][e].lo += fmaf(pe, rho, qe);
          } else {
            acc[k][e].hi = fmaf(dv[k][e] * xv[k][e], rho, acc[k][e].hi);
          }
        }
        Vec16<T>::store(dxr + (int64_t)vi * VE, o);
      }
    }
  }

  if (failed) {
    report_status(a.status, GBN_DEV_WAIT_TIMEOUT);
    if (tid == 0) {
      // Let the copies still in flight land before the block exits.
      for (int64_t k = i; k < nrows && k < i + nst; ++k)
        mbar_wait_bounded(&bar[k % nst], (uint32_t)((k / nst) & 1), kWaitLimitNs / 8);
    }
    __syncthreads();
    return;
  }

  float* hi = a.part + (int64_t)g * a.H;
  float* lo = a.part + ((int64_t)G + g) * a.H;
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int vi = tid + k * blockDim.x;
    if (vi < a.Hv) {
#pragma unroll
      for (int e = 0; e < VE; e += 4) {
        *reinterpret_cast<float4*>(hi + (int64_t)vi * VE + e) =
            make_float4(acc[k][e].hi, acc[k][e + 1].hi, acc[k][e + 2].hi, acc[k][e + 3].hi);
        if constexpr (COMP)
          *reinterpret_cast<float4*>(lo + (int64_t)vi * VE + e) =
              make_float4(acc[k][e].lo, acc[k][e + 1].lo, acc[k][e + 2].lo, acc[k][e + 3].lo);
      }
    }
  }
  pdl_launch_dependents();
}

// Any H and alignment: block g owns rows g, g+G, ...; thread t owns columns
// t, t+256, ... and accumulates them straight into this block's partial row.
template <typename T, bool COMP>
__global__ void __launch_bounds__(256) rms_bwd_generic_kernel(RmsArgs a) {
  __shared__ float red[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t H = a.H;
  const T* x = static_cast<const T*>(a.x);
  const T* dy = static_cast<const T*>(a.dy);
  const T* w = static_cast<const T*>(a.w);
  T* dx = static_cast<T*>(a.dx);
  float* hi = a.part + (int64_t)g * H;
  float* lo = a.part + ((int64_t)G + g) * H;
  for (int64_t j = tid; j < H; j += blockDim.x) {
    hi[j] = 0.f;
    if constexpr (COMP) lo[j] = 0.f;
  }
  int it = 0;
  for (int64_t r = g; r < a.R; r += G, ++it) {
    const float rho = a.rstd[r];
    const T* xr = x + r * H;
    const T* dyr = dy + r * H;
    float part = 0.f;
    for (int64_t j = tid; j < H; j += blockDim.x)
      part = fmaf(to_f32(w[j]) * to_f32(dyr[j]), to_f32(xr[j]), part);
    part = warp_sum(part);
    if (lane == 0) red[it & 1][warp] = part;
    __syncthreads();
    float S = 0.f;
    for (int wi = 0; wi < nwarps; ++wi) S += red[it & 1][wi];
    const float coef = rho * rho * rho * S / (float)H;
    for (int64_t j = tid; j < H; j += blockDim.x) {
      const float xv = to_f32(xr[j]), dv = to_f32(dyr[j]);
      dx[r * H + j] = from_f32<T>(fmaf(-xv, coef, rho * to_f32(w[j]) * dv));
      if constexpr (COMP) {
        DF acc{hi[j], lo[j]};
        const float p = dv * xv;
        const float pe = fmaf(dv, xv, -p);
        const float q = p * rho;
        const float qe = fmaf(p, rho, -q);
        df_add(acc, q);
        acc.lo += fmaf(pe, rho, qe);
        hi[j] = acc.hi;
        lo[j] = acc.lo;
      } else {
        hi[j] = fmaf(dv * xv, rho, hi[j]);
      }
    }
  }
  pdl_launch_dependents();
}

template <typename T, int KV>
cudaError_t launch_fast(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  constexpr bool COMP = sizeof(T) == 4;
  return launch(rms_bwd_fast_kernel<T, KV, COMP>, dim3(p.G), dim3(p.threads), p.smem, st, false, a);
}

template <typename T>
cudaError_t launch_typed(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  if (!p.fast) {
    constexpr bool COMP = sizeof(T) == 4;
    return launch(rms_bwd_generic_kernel<T, COMP>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  }
  switch (p.kv) {
    case 1: return launch_fast<T, 1>(p, a, st);
    case 2: return launch_fast<T, 2>(p, a, st);
    case 3: return launch_fast<T, 3>(p, a, st);
    default: return launch_fast<T, 4>(p, a, st);
  }
}

template <typename T, int KV>
cudaError_t set_smem(int bytes) {
  constexpr bool COMP = sizeof(T) == 4;
  return cudaFuncSetAttribute(rms_bwd_fast_kernel<T, KV, COMP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

uint32_t rms_smem_header() { return kRmsHeader; }

cudaError_t rms_configure(int smem_optin) {
  cudaError_t e = cudaSuccess;
  cudaError_t r;
  if ((r = set_smem<float, 1>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<float, 2>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<float, 3>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<float, 4>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<bf16, 1>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<bf16, 2>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<bf16, 3>(smem_optin)) != cudaSuccess) e = r;
  if ((r = set_smem<bf16, 4>(smem_optin)) != cudaSuccess) e = r;
  return e;
}

cudaError_t rms_launch(const RowPlan& p, const void* dy, const void* x, const void* w,
                       const float* rstd, void* dx, void* dw, float* part, int* status,
                       cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (p.R > 0 && p.H > 0) {
    RmsArgs a;
    a.dy = dy;
    a.x = x;
    a.w = w;
    a.rstd = rstd;
    a.dx = dx;
    a.part = part;
    a.status = status;
    a.R = p.R;
    a.H = (int32_t)p.H;
    a.Hv = (int32_t)(p.H * (p.dtype == GBN_F32 ? 4 : 2) / 16);
    a.nstage = p.nstage;
    a.row_bytes = (uint32_t)(p.H * (p.dtype == GBN_F32 ? 4 : 2));
    e = p.dtype == GBN_F32 ? launch_typed<float>(p, a, st) : launch_typed<bf16>(p, a, st);
    if (e != cudaSuccess) return e;
  }
  void* outs[3] = {dw, nullptr, nullptr};
  return colsum_launch(part, 1, p.nplanes, p.R > 0 ? p.G : 0, p.H, p.dtype, outs, st,
                       p.R > 0 && p.H > 0);
}

}  // namespace gbn
