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
// GB300 design.  One launch.  A persistent grid (one CTA per SM, all
// resident: cooperative launch) owns row blocks b = g, g+G, ... of RB rows.
// Warp 0 streams each block's x and dy rows into a ring of shared-memory
// stages with 1-D bulk copies (cp.async.bulk + mbarrier); the consumer warps
// own fixed 16-byte column vectors: they keep their weights and dweight
// accumulators in registers for the whole kernel, copy their vectors of the
// stage into registers and release the stage at once (so the next copy into
// that slot starts while they compute), reduce S_r over the consumer warps
// (one barrier per stage) and write dx.  Then every CTA stores its dweight
// partial row, publishes a flag, waits for every other CTA's flag and sums a
// slice of the columns over all G partial rows in a fixed order (no second
// launch, no atomics; bit-identical from run to run).  fp32 outputs
// accumulate dweight in double-fp32 with exact product residuals.  Shapes the
// ring does not take (rows that are not whole 16-byte vectors, unaligned
// tensors, rows too long for the registers) run a plain kernel followed by a
// separate fixed-order column-sum launch.
#include "gbn_common.cuh"
#include "gbn_internal.h"
#include "row_engine.cuh"

namespace gbn {

namespace {

struct RmsArgs {
  const void* dy;
  const void* x;
  const void* w;
  const float* rstd;
  void* dx;
  void* dw;
  float* part;               // column partials [nplanes][G][H]
  unsigned long long* sync;  // epoch pair, then one flag pair per CTA
  unsigned long long nonce;
  int* status;
  int64_t R;
  int32_t H;
  int32_t Hv;      // 16-byte vectors per row (ring kernel)
  int32_t nstage;
  uint32_t row_bytes;
};

// Sum of the NW per-warp partials in slot[0..NW) as a fixed pairwise tree
// (every thread computes the same bits).
template <int NW>
__device__ __forceinline__ float sum_slots(const float* slot) {
  float v[NW];
#pragma unroll
  for (int w = 0; w < NW; w += 4) {
    const float4 q = *reinterpret_cast<const float4*>(slot + w);
    v[w] = q.x; v[w + 1] = q.y; v[w + 2] = q.z; v[w + 3] = q.w;
  }
#pragma unroll
  for (int step = 1; step < NW; step *= 2)
#pragma unroll
    for (int w = 0; w < NW; w += 2 * step) v[w] += v[w + step];
  return v[0];
}

// KV: 16-byte vectors per consumer thread and row; RB: rows per stage;
// NCW: consumer warps (a multiple of 4).  EARLY: the thread's vectors of a
// stage are copied into registers and the stage is released before the row
// sums (the next copy into the slot overlaps the arithmetic); otherwise they
// are read from shared memory twice and the stage is released at its end
// (fewer registers, for threads that own many columns).
template <typename T, int KV, int RB, int NCW, bool COMP, bool EARLY>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) rms_bwd_ring_kernel(RmsArgs a) {
  static_assert(sizeof(RowShared) + sizeof(float) * 2 * RB * NCW <= kRowStaticSmem,
                "static shared memory bound");
  using PK = Pairs16<T>;
  constexpr int NP = PK::NP;  // packed pairs per 16-byte vector
  constexpr int NC = NCW * 32;
  extern __shared__ __align__(128) unsigned char data[];
  __shared__ RowShared sh;
  __shared__ __align__(16) float red[2][RB][NCW];

  const int tid = threadIdx.x;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t nblk = (a.R + RB - 1) / RB;
  const int64_t nmine = (nblk - g + G - 1) / G;
  const int NS = a.nstage;
  const uint32_t rb = a.row_bytes;
  const uint32_t xoff = RB * rb;  // dy rows follow the x rows in a stage

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], NCW);
      sh.issued[s] = 0;
    }
    sh.abort = 0;
    fence_mbarrier_init();
    GBN_RING_TRACE(0);
  }
  __syncthreads();

  if (tid < 32) {
    if (tid == 0) {
      const char* gx = static_cast<const char*>(a.x);
      const char* gdy = static_cast<const char*>(a.dy);
      ring_produce(sh, NS, nmine, a.status, [&](int64_t i, int s) {
        const int64_t r0 = (g + i * G) * RB;
        const int64_t nr = a.R - r0 < RB ? a.R - r0 : RB;
        const uint32_t bytes = (uint32_t)nr * rb;
        unsigned char* st = data + (size_t)s * 2 * xoff;
        mbar_arrive_expect_tx(&sh.full[s], 2u * bytes);
        bulk_g2s(st, gx + r0 * rb, bytes, &sh.full[s]);
        bulk_g2s(st + xoff, gdy + r0 * rb, bytes, &sh.full[s]);
      });
    }
  } else {
    const int ct = tid - 32, lane = ct & 31, cw = ct >> 5;
    epoch_read(sh, a.sync, ct);
    // Weights and the dweight accumulators of this thread's columns, packed.
    f2 w2[KV][NP], acc[KV][NP], acc_lo[KV][NP];
    const T* w = static_cast<const T*>(a.w);
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = ct + k * NC;
      const uint4 rw = vi < a.Hv ? *reinterpret_cast<const uint4*>(w + (int64_t)vi * (2 * NP))
                                 : make_uint4(0u, 0u, 0u, 0u);
      PK::get(rw, w2[k]);
#pragma unroll
      for (int p = 0; p < NP; ++p) { acc[k][p] = 0ull; acc_lo[k][p] = 0ull; }
    }
    const float invH = 1.f / (float)a.H;  // one rounding more than / H, no division per row
    bool failed = false;
    int64_t i = 0;
    // ring slot s = i mod NS and lap = i / NS, advanced per stage (no
    // 64-bit division in the loop); the slot's phase parity is lap & 1
    int s = 0;
    uint32_t lap = 0;
    for (; i < nmine; ++i, ring_advance(s, lap, NS)) {
      const uint32_t par = lap & 1u;
      const int64_t r0 = (g + i * G) * RB;
      const int nr = (int)(a.R - r0 < RB ? a.R - r0 : RB);
      float rho[RB];
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) rho[rr] = rr < nr ? __ldg(a.rstd + r0 + rr) : 0.f;
      bool ok = __all_sync(0xffffffffu, ring_wait(&sh.full[s], par, &sh.abort));
      if (i == 0 && ct == 0) GBN_RING_TRACE(1);
      // This thread's vectors of the stage (EARLY: copied into registers,
      // then the slot is released so that the producer can refill it while
      // we compute).
      const unsigned char* sx = data + (size_t)s * 2 * xoff;
      auto vec = [&](int rr, int k, bool dyv) {
        const int vi = ct + k * NC;
        return (ok && rr < nr && vi < a.Hv)
                   ? *reinterpret_cast<const uint4*>(sx + (dyv ? xoff : 0u) + (size_t)rr * rb +
                                                     (size_t)vi * 16)
                   : make_uint4(0u, 0u, 0u, 0u);
      };
      uint4 xr[EARLY ? RB : 1][KV], dr[EARLY ? RB : 1][KV];
      if constexpr (EARLY) {
#pragma unroll
        for (int rr = 0; rr < RB; ++rr)
#pragma unroll
          for (int k = 0; k < KV; ++k) {
            xr[rr][k] = vec(rr, k, false);
            dr[rr][k] = vec(rr, k, true);
          }
        if (ok) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.empty[s]);
        }
      }
      auto getx = [&](int rr, int k) {
        if constexpr (EARLY) return xr[rr][k];
        else return vec(rr, k, false);
      };
      auto getd = [&](int rr, int k) {
        if constexpr (EARLY) return dr[rr][k];
        else return vec(rr, k, true);
      };
      // Row sums S = sum_j w_j dy_j x_j (two lanes per instruction); with
      // EARLY the unpacked pairs stay in registers for the second pass
      // (the other instances would spill and unpack again).
      float* slot = &red[i & 1][0][0];
      f2 xs[EARLY ? RB : 1][KV][NP], ds[EARLY ? RB : 1][KV][NP];
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        f2 part = 0ull;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          f2 (&x2)[NP] = xs[EARLY ? rr : 0][k];
          f2 (&d2)[NP] = ds[EARLY ? rr : 0][k];
          PK::get(getx(rr, k), x2);
          PK::get(getd(rr, k), d2);
#pragma unroll
          for (int p = 0; p < NP; ++p) part = f2_fma(f2_mul(w2[k][p], d2[p]), x2[p], part);
        }
        const float v = warp_sum(f2_hsum(part));
        if (lane == 0) slot[rr * NCW + cw] = v;
      }
      if (consumers_bar_or(!ok, NC)) {
        failed = true;
        break;
      }
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        if (rr >= nr) break;
        const float S = sum_slots<NCW>(slot + rr * NCW);
        const float coef = rho[rr] * rho[rr] * rho[rr] * S * invH;
        const f2 rho2 = f2_splat(rho[rr]);
        const f2 ncoef2 = f2_splat(-coef);
        T* dxr = static_cast<T*>(a.dx) + (r0 + rr) * (int64_t)a.H;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          const int vi = ct + k * NC;
          if (vi >= a.Hv) continue;
          f2 (&x2)[NP] = xs[EARLY ? rr : 0][k];
          f2 (&d2)[NP] = ds[EARLY ? rr : 0][k];
          if constexpr (!EARLY) {
            PK::get(getx(rr, k), x2);
            PK::get(getd(rr, k), d2);
          }
          f2 o2[NP];
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
      if constexpr (!EARLY) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
      }
    }
    if (ct == 0) GBN_RING_TRACE(2);

    if (!failed) {
      // This CTA's dweight partial row (and its low part), then the
      // hand-off and this CTA's slice of the column sums.
      float* hi = a.part + (int64_t)g * a.H;
      float* lo = a.part + ((int64_t)G + g) * a.H;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int vi = ct + k * NC;
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
      if (ct == 0) GBN_RING_TRACE(3);
      if (ring_exchange(sh, a.sync, G, ct, NC, a.status, a.nonce)) {
        if (ct == 0) GBN_RING_TRACE(4);
        T* outs[1] = {static_cast<T*>(a.dw)};
        colsum_warps<T, COMP>(a.part, 1, G, a.H, outs, g, G, cw, NCW, lane);
        if (ct == 0) GBN_RING_TRACE(5);
      }
    } else if (ct == 0) {
      ring_abort(sh, a.status);
    }
  }
  __syncthreads();
  if (tid == 0 && sh.abort) ring_drain(sh, NS);
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

// Rows of at most two vectors per thread keep them in registers (EARLY).
template <int KV> constexpr bool kEarly = KV <= 2;

template <typename T, int KV, int RB, int NCW>
cudaError_t launch_ring(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  constexpr bool COMP = sizeof(T) == 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.G);
  cfg.blockDim = dim3((unsigned)p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rms_bwd_ring_kernel<T, KV, RB, NCW, COMP, kEarly<KV>>, a);
}

// Ring instances: (KV, RB) with 16 consumer warps.  The plan picks KV =
// ceil(vectors per row / 512) and RB = 2 for rows of at most one vector per
// thread (two rows per barrier), else 1 (RB = 2 with KV = 2 would spill).
template <typename T>
cudaError_t launch_typed(const RowPlan& p, const RmsArgs& a, cudaStream_t st) {
  if (!p.fast) {
    constexpr bool COMP = sizeof(T) == 4;
    return launch(rms_bwd_generic_kernel<T, COMP>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  }
  switch (p.kv * 8 + p.rb) {
    case 1 * 8 + 2: return launch_ring<T, 1, 2, 16>(p, a, st);
    case 1 * 8 + 1: return launch_ring<T, 1, 1, 16>(p, a, st);
    case 2 * 8 + 1: return launch_ring<T, 2, 1, 16>(p, a, st);
    case 3 * 8 + 1: return launch_ring<T, 3, 1, 16>(p, a, st);
    default: return launch_ring<T, 4, 1, 16>(p, a, st);
  }
}

template <typename T, int KV, int RB, int NCW>
cudaError_t set_smem(int bytes) {
  constexpr bool COMP = sizeof(T) == 4;
  return cudaFuncSetAttribute(rms_bwd_ring_kernel<T, KV, RB, NCW, COMP, kEarly<KV>>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename T>
cudaError_t set_smem_all(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_smem<T, 1, 2, 16>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 1, 1, 16>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 2, 1, 16>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 3, 1, 16>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 4, 1, 16>(bytes)) != cudaSuccess) e = r;
  return e;
}

}  // namespace

cudaError_t rms_configure(int smem_optin) {
  const int dyn = smem_optin - kRowStaticSmem;
  cudaError_t e1 = set_smem_all<float>(dyn);
  cudaError_t e2 = set_smem_all<bf16>(dyn);
  return e1 != cudaSuccess ? e1 : e2;
}

cudaError_t rms_launch(const RowPlan& p, const void* dy, const void* x, const void* w,
                       const float* rstd, void* dx, void* dw, void* ws, int* status,
                       cudaStream_t st) {
  if (p.R == 0 || p.H == 0) {
    // no rows: dweight is a sum of nothing
    void* outs[3] = {dw, nullptr, nullptr};
    return colsum_launch(nullptr, 1, p.nplanes, 0, p.H, p.dtype, outs, st, false);
  }
  RmsArgs a;
  a.dy = dy;
  a.x = x;
  a.w = w;
  a.rstd = rstd;
  a.dx = dx;
  a.dw = dw;
  a.sync = static_cast<unsigned long long*>(ws);
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + p.part_offset);
  a.nonce = next_nonce();
  a.status = status;
  a.R = p.R;
  a.H = (int32_t)p.H;
  a.Hv = (int32_t)(p.H * (p.dtype == GBN_F32 ? 4 : 2) / 16);
  a.nstage = p.nstage;
  a.row_bytes = (uint32_t)(p.H * (p.dtype == GBN_F32 ? 4 : 2));
  cudaError_t e = p.dtype == GBN_F32 ? launch_typed<float>(p, a, st) : launch_typed<bf16>(p, a, st);
  if (e != cudaSuccess || p.fast) return e;
  // the plain kernel leaves its column partials for a second launch
  void* outs[3] = {dw, nullptr, nullptr};
  return colsum_launch(a.part, 1, p.nplanes, p.G, p.H, p.dtype, outs, st, true);
}

}  // namespace gbn
