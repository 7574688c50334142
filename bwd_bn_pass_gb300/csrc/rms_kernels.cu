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

// Shared memory: 8 mbarriers, then [2][RB][32] row-sum slots, then stages.
__host__ __device__ constexpr uint32_t rms_header(int rb) { return 64 + 2 * rb * 32 * 4; }

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

// Sum of the nwarps per-warp partials in slot[0..nwarps) as a fixed
// pairwise tree (every thread computes the same bits).
__device__ __forceinline__ float sum_warp_slots(const float* slot, int nwarps) {
  float v[16];
#pragma unroll
  for (int w = 0; w < 16; ++w) v[w] = w < nwarps ? slot[w] : 0.f;
#pragma unroll
  for (int step = 1; step < 16; step *= 2)
#pragma unroll
    for (int w = 0; w < 16; w += 2 * step) v[w] += v[w + step];
  return v[0];
}

template <typename T, int KV, int RB, bool COMP, int MINB>
__global__ void __launch_bounds__(512, MINB) rms_bwd_fast_kernel(RmsArgs a) {
  using PK = Pairs16<T>;
  constexpr int NP = PK::NP;  // packed pairs per 16-byte vector
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 64);  // [2][RB][32]
  unsigned char* data = smem + rms_header(RB);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t nblk = (a.R + RB - 1) / RB;
  const int64_t nmine = (nblk - g + G - 1) / G;
  const int nst = a.nstage;
  const uint32_t rb = a.row_bytes;
  const uint32_t xoff = RB * rb;  // dy rows follow the x rows in a stage
  const char* gx = static_cast<const char*>(a.x);
  const char* gdy = static_cast<const char*>(a.dy);

  auto issue = [&](int64_t i) {
    const int s = (int)(i % nst);
    const int64_t r0 = (g + i * G) * RB;
    const int64_t nr = a.R - r0 < RB ? a.R - r0 : RB;
    const uint32_t bytes = (uint32_t)nr * rb;
    unsigned char* st = data + (size_t)s * 2 * xoff;
    mbar_arrive_expect_tx(&bar[s], 2u * bytes);
    bulk_g2s(st, gx + r0 * rb, bytes, &bar[s]);
    bulk_g2s(st + xoff, gdy + r0 * rb, bytes, &bar[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < nmine && i < nst; ++i) issue(i);

  // Weights and the dweight accumulators of this thread's columns, packed.
  f2 w2[KV][NP], acc[KV][NP], acc_lo[KV][NP];
  const T* w = static_cast<const T*>(a.w);
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int vi = tid + k * blockDim.x;
    const uint4 rw = vi < a.Hv ? *reinterpret_cast<const uint4*>(w + (int64_t)vi * (2 * NP))
                               : make_uint4(0u, 0u, 0u, 0u);
    PK::get(rw, w2[k]);
#pragma unroll
    for (int p = 0; p < NP; ++p) { acc[k][p] = 0ull; acc_lo[k][p] = 0ull; }
  }

  const float Hf = (float)a.H;
  bool failed = false;
  int64_t i = 0;
  for (; i < nmine; ++i) {
    const int s = (int)(i % nst);
    const uint32_t par = (uint32_t)((i / nst) & 1);
    const int64_t r0 = (g + i * G) * RB;
    const int nr = (int)(a.R - r0 < RB ? a.R - r0 : RB);
    float rho[RB];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) rho[rr] = rr < nr ? a.rstd[r0 + rr] : 0.f;
    const bool ok = mbar_wait_bounded(&bar[s], par);
    const unsigned char* sx = data + (size_t)s * 2 * xoff;
    const unsigned char* sdy = sx + xoff;

    // Row sums S = sum_j w_j dy_j x_j (two lanes per instruction).
    float* slot = red + (i & 1) * (RB * 32);
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      f2 part = 0ull;
      if (ok && rr < nr) {
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          const int vi = tid + k * blockDim.x;
          if (vi < a.Hv) {
            f2 x2[NP], d2[NP];
            PK::get(*reinterpret_cast<const uint4*>(sx + (size_t)rr * rb + (size_t)vi * 16), x2);
            PK::get(*reinterpret_cast<const uint4*>(sdy + (size_t)rr * rb + (size_t)vi * 16), d2);
#pragma unroll
            for (int p = 0; p < NP; ++p) part = f2_fma(f2_mul(w2[k][p], d2[p]), x2[p], part);
          }
        }
      }
      const float v = warp_sum(f2_hsum(part));
      if (lane == 0) slot[rr * 32 + warp] = v;
    }
    if (__syncthreads_or(!ok)) { failed = true; break; }
    // Every thread is past iteration i-1: its stage can be refilled.
    if (tid == 0 && i >= 1 && i - 1 + nst < nmine) {
      fence_proxy_async_smem();
      issue(i - 1 + nst);
    }

#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      if (rr >= nr) break;
      const float S = sum_warp_slots(slot + rr * 32, nwarps);
      const float coef = rho[rr] * rho[rr] * rho[rr] * S / Hf;
      const f2 rho2 = f2_splat(rho[rr]);
      const f2 ncoef2 = f2_splat(-coef);
      T* dxr = static_cast<T*>(a.dx) + (r0 + rr) * (int64_t)a.H;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int vi = tid + k * blockDim.x;
        if (vi >= a.Hv) continue;
        f2 x2[NP], d2[NP], o2[NP];
        PK::get(*reinterpret_cast<const uint4*>(sx + (size_t)rr * rb + (size_t)vi * 16), x2);
        PK::get(*reinterpret_cast<const uint4*>(sdy + (size_t)rr * rb + (size_t)vi * 16), d2);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          // dx = rstd*w*dy - x*rstd^3*S/H
          o2[p] = f2_fma(x2[p], ncoef2, f2_mul(rho2, f2_mul(w2[k][p], d2[p])));
          if constexpr (COMP) {
            // dweight += dy*x*rstd with both products' exact residuals
            const f2 prod = f2_mul_rounded(d2[p], x2[p]);
            const f2 pe = f2_fma(d2[p], x2[p], f2_sub(0ull, prod));
            const f2 q = f2_mul_rounded(prod, rho2);
            const f2 qe = f2_fma(prod, rho2, f2_sub(0ull, q));
            DF2 t{acc[k][p], acc_lo[k][p]};
            df2_add(t, q);
            acc[k][p] = t.hi;
            acc_lo[k][p] = f2_add(t.lo, f2_fma(pe, rho2, qe));
          } else {
            acc[k][p] = f2_fma(f2_mul(d2[p], x2[p]), rho2, acc[k][p]);
          }
        }
        *reinterpret_cast<uint4*>(dxr + (int64_t)vi * (2 * NP)) = PK::put(o2);
      }
    }
  }

  if (failed) {
    report_status(a.status, GBN_DEV_WAIT_TIMEOUT);
    if (tid == 0) {
      // Blocks issued and not consumed: i .. i + nst - 2 (lagged refill).
      for (int64_t k = i; k < nmine && k < i + nst - 1; ++k)
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
      float4* h4 = reinterpret_cast<float4*>(hi + (int64_t)vi * (2 * NP));
      float4* l4 = reinterpret_cast<float4*>(lo + (int64_t)vi * (2 * NP));
#pragma unroll
      for (int p = 0; p < NP; p += 2) {
        const float2 a0 = f2_unpack(acc[k][p]), a1 = f2_unpack(acc[k][p + 1]);
        h4[p / 2] = make_float4(a0.x, a0.y, a1.x, a1.y);
        if constexpr (COMP) {
          const float2 b0 = f2_unpack(acc_lo[k][p]), b1 = f2_unpack(acc_lo[k][p + 1]);
          l4[p / 2] = make_float4(b0.x, b0.y, b1.x, b1.y);
        }
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
        const DF p = two_prod(dv, xv);
        const DF q = two_prod(p.hi, rho);
        df_add(acc, q.hi);
        acc.lo = __fadd_rn(acc.lo, fmaf(p.lo, rho, q.lo));
        hi[j] = acc.hi;
        lo[j] = acc.lo;
      } else {
        hi[j] = fmaf(dv * xv, rho, hi[j]);
      }
    }
  }
  pdl_launch_dependents();
}

template <typename T, int KV, int RB, int MINB>
cudaError_t launch_fast(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  constexpr bool COMP = sizeof(T) == 4;
  return launch(rms_bwd_fast_kernel<T, KV, RB, COMP, MINB>, dim3(p.G), dim3(p.threads), p.smem,
                st, false, a);
}

// Instances: (KV, RB, min blocks per SM).  The plan picks RB = 2 for short
// rows and for two-vector rows (then one block per SM), and 2 blocks per SM
// whenever the columns a thread owns fit.
template <typename T>
cudaError_t launch_typed(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  if (!p.fast) {
    constexpr bool COMP = sizeof(T) == 4;
    return launch(rms_bwd_generic_kernel<T, COMP>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  }
  if (p.rb == 2 && p.kv == 2) return launch_fast<T, 2, 2, 1>(p, a, st);
  if (p.rb == 2) return launch_fast<T, 1, 2, 2>(p, a, st);
  switch (p.kv) {
    case 1: return launch_fast<T, 1, 1, 2>(p, a, st);
    case 2: return launch_fast<T, 2, 1, 2>(p, a, st);
    case 3: return launch_fast<T, 3, 1, 1>(p, a, st);
    default: return launch_fast<T, 4, 1, 1>(p, a, st);
  }
}

template <typename T, int KV, int RB, int MINB>
cudaError_t set_smem(int bytes) {
  constexpr bool COMP = sizeof(T) == 4;
  return cudaFuncSetAttribute(rms_bwd_fast_kernel<T, KV, RB, COMP, MINB>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T>
cudaError_t set_smem_all(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_smem<T, 1, 2, 2>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 2, 2, 1>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 1, 1, 2>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 2, 1, 2>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 3, 1, 1>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 4, 1, 1>(bytes)) != cudaSuccess) e = r;
  return e;
}

}  // namespace

uint32_t rms_smem_header(int rb) { return rms_header(rb); }

cudaError_t rms_configure(int smem_optin) {
  cudaError_t e1 = set_smem_all<float>(smem_optin);
  cudaError_t e2 = set_smem_all<bf16>(smem_optin);
  return e1 != cudaSuccess ? e1 : e2;
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
