// LayerNorm backward, plain or fused with bias + dropout + add.
//
// Method: nvFuser issue #1473 "Why is LayerNorm Backward Segmenting?" --
// the repro of the 1-kernel bias+dropout+add+layer_norm backward
// (nvfuser_fusion_id9) and of the 3-kernel layer_norm backward
// (nvfuser_fusion_id14).  Per row with saved mean mu and rstd rho:
//   xhat = (z - mu)*rho, g = dy*gamma,
//   dz   = rho*(g - mean_j g - xhat*mean_j(g*xhat))   (+ dz_extra)
//   dgamma = sum_rows dy*xhat, dbeta = sum_rows dy
// and in the fused form, where z = residual + mask*scale*(input + bias) is
// recomputed in fp32 from the stored operands:
//   dresidual = dz, dinput = dz*scale*mask, dbias = sum_rows dinput.
// The page's point -- the column reductions must not split the backward into
// separate passes over the [R, H] tensors -- is met by accumulating the
// column sums while the rows stream through.
//
// GB300 design: the same persistent, bulk-copy-fed skeleton as the RMSNorm
// kernel.  A pipeline stage holds RB consecutive rows of dy, input,
// residual and mask (one bulk copy per tensor); each thread owns fixed
// 16-byte column vectors (gamma, bias and the three column accumulators stay
// in registers), computes both row sums for all RB rows of the stage before a
// single block barrier, then writes dx / dresidual with 16-byte stores.
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

namespace {

struct LnArgs {
  const void* dy;
  const void* x;
  const void* res;
  const void* bias;
  const uint8_t* mask;
  const float* dzx;
  const float* mean;
  const float* rstd;
  const void* gamma;
  void* dx;
  void* dres;
  float* part;
  int* status;
  int64_t R;
  float scale;
  int32_t H;
  int32_t Hv;
  int32_t nstage;
  int32_t nplanes;
  uint32_t stage_bytes;
  uint32_t off_dy, off_x, off_res, off_mask;
};

__host__ __device__ constexpr uint32_t ln_header(int rb) { return 64 + 2 * 2 * rb * 32 * 4; }

template <typename T>
__device__ __forceinline__ void ldg16(const T* p, float (&v)[16 / sizeof(T)]) {
  Vec16<T>::load(p, v);
}

// Mask bits of VE consecutive bytes (nonzero = kept).
template <int VE>
__device__ __forceinline__ uint32_t mask_bits(const uint8_t* p) {
  uint32_t bits = 0;
  if constexpr (VE == 8) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      bits |= (((w.x >> (8 * e)) & 0xffu) != 0u) << e;
      bits |= (((w.y >> (8 * e)) & 0xffu) != 0u) << (e + 4);
    }
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
#pragma unroll
    for (int e = 0; e < 4; ++e) bits |= (((w >> (8 * e)) & 0xffu) != 0u) << e;
  }
  return bits;
}

template <typename T, int KV, int RB, bool FUSED>
__global__ void __launch_bounds__(512, 1) ln_bwd_fast_kernel(LnArgs a) {
  constexpr int VE = 16 / sizeof(T);
  constexpr bool COMP = sizeof(T) == 4;
  constexpr uint32_t HDR = ln_header(RB);
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 64);  // [2][2*RB][32]
  unsigned char* data = smem + HDR;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t nblk = (a.R + RB - 1) / RB;
  const int64_t nmine = (nblk - g + G - 1) / G;
  const int nst = a.nstage;
  const int64_t H = a.H;
  const uint32_t rowb = (uint32_t)(H * sizeof(T));
  const bool has_mask = FUSED && a.mask != nullptr;

  auto issue = [&](int64_t i) {
    const int s = (int)(i % nst);
    const int64_t r0 = (g + i * G) * RB;
    const int64_t nr = a.R - r0 < RB ? a.R - r0 : RB;
    const uint32_t bt = (uint32_t)nr * rowb;
    const uint32_t bm = (uint32_t)(nr * H);
    unsigned char* st = data + (size_t)s * a.stage_bytes;
    mbar_arrive_expect_tx(&bar[s], bt * (FUSED ? 3u : 2u) + (has_mask ? bm : 0u));
    bulk_g2s(st + a.off_dy, static_cast<const char*>(a.dy) + r0 * rowb, bt, &bar[s]);
    bulk_g2s(st + a.off_x, static_cast<const char*>(a.x) + r0 * rowb, bt, &bar[s]);
    if (FUSED) bulk_g2s(st + a.off_res, static_cast<const char*>(a.res) + r0 * rowb, bt, &bar[s]);
    if (has_mask) bulk_g2s(st + a.off_mask, a.mask + r0 * H, bm, &bar[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < nmine && i < nst; ++i) issue(i);

  float gam[KV][VE], bia[KV][VE];
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int vi = tid + k * blockDim.x;
#pragma unroll
    for (int e = 0; e < VE; ++e) { gam[k][e] = 0.f; bia[k][e] = 0.f; }
    if (vi < a.Hv) {
      ldg16<T>(static_cast<const T*>(a.gamma) + (int64_t)vi * VE, gam[k]);
      if (FUSED && a.bias != nullptr) ldg16<T>(static_cast<const T*>(a.bias) + (int64_t)vi * VE, bia[k]);
    }
  }
  DF acc_g[KV][VE], acc_b[KV][VE], acc_x[KV][VE];  // dgamma, dbeta, dbias
#pragma unroll
  for (int k = 0; k < KV; ++k)
#pragma unroll
    for (int e = 0; e < VE; ++e) { acc_g[k][e] = acc_b[k][e] = acc_x[k][e] = DF{0.f, 0.f}; }

  const float inv_H = 1.f / (float)H;
  bool failed = false;
  int64_t i = 0;
  for (; i < nmine; ++i) {
    const int s = (int)(i % nst);
    const uint32_t par = (uint32_t)((i / nst) & 1);
    const int64_t r0 = (g + i * G) * RB;
    const int nr = (int)(a.R - r0 < RB ? a.R - r0 : RB);
    float mu[RB], rho[RB];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      mu[rr] = rr < nr ? a.mean[r0 + rr] : 0.f;
      rho[rr] = rr < nr ? a.rstd[r0 + rr] : 0.f;
    }
    const bool ok = mbar_wait_bounded(&bar[s], par);
    const unsigned char* st = data + (size_t)s * a.stage_bytes;

    // Phase 1: load the stage into registers, row sums of g and g*xhat.
    float dyv[RB][KV][VE], zv[RB][KV][VE];
    float zlo[RB][KV][VE];  // exact-z residual (fp32 outputs only)
    uint32_t mk[RB][KV];
    float sg[RB], sgx[RB];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      sg[rr] = 0.f;
      sgx[rr] = 0.f;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int vi = tid + k * blockDim.x;
        mk[rr][k] = 0xffu;
        if (ok && rr < nr && vi < a.Hv) {
          const size_t o = (size_t)rr * rowb + (size_t)vi * 16;
          Vec16<T>::load(st + a.off_dy + o, dyv[rr][k]);
          Vec16<T>::load(st + a.off_x + o, zv[rr][k]);
          if constexpr (FUSED) {
            float rv[VE];
            Vec16<T>::load(st + a.off_res + o, rv);
            if (has_mask) mk[rr][k] = mask_bits<VE>(st + a.off_mask + (size_t)rr * H + (size_t)vi * VE);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              const float keep = ((mk[rr][k] >> e) & 1u) ? a.scale : 0.f;
              if constexpr (COMP) {
                const DF kt = df_mul(two_sum(zv[rr][k][e], bia[k][e]), keep);
                const DF z = df_plus(two_sum(rv[e], kt.hi), kt.lo);
                zv[rr][k][e] = z.hi;
                zlo[rr][k][e] = z.lo;
              } else {
                zv[rr][k][e] = fmaf(keep, zv[rr][k][e] + bia[k][e], rv[e]);
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) zlo[rr][k][e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float xh = (zv[rr][k][e] - mu[rr]) * rho[rr];
            const float gg = dyv[rr][k][e] * gam[k][e];
            sg[rr] += gg;
            sgx[rr] = fmaf(gg, xh, sgx[rr]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            dyv[rr][k][e] = 0.f;
            zv[rr][k][e] = 0.f;
            zlo[rr][k][e] = 0.f;
          }
        }
      }
    }
    float* slot = red + (i & 1) * (2 * RB * 32);
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      const float a0 = warp_sum(sg[rr]);
      const float a1 = warp_sum(sgx[rr]);
      if (lane == 0) { slot[(2 * rr) * 32 + warp] = a0; slot[(2 * rr + 1) * 32 + warp] = a1; }
    }
    if (__syncthreads_or(!ok)) { failed = true; break; }
    if (tid == 0 && i + nst < nmine) {
      fence_proxy_async_smem();
      issue(i + nst);
    }

    // Phase 2: dz, outputs, column sums.
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      if (rr >= nr) break;
      float SG = 0.f, SGX = 0.f;
      for (int wi = 0; wi < nwarps; ++wi) {
        SG += slot[(2 * rr) * 32 + wi];
        SGX += slot[(2 * rr + 1) * 32 + wi];
      }
      const float mg = SG * inv_H, mgx = SGX * inv_H;
      const int64_t r = r0 + rr;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int vi = tid + k * blockDim.x;
        if (vi >= a.Hv) continue;
        const int64_t go = r * H + (int64_t)vi * VE;
        float dzx[VE];
        if (a.dzx != nullptr) {
#pragma unroll
          for (int e = 0; e < VE; e += 4) {
            const float4 t = *reinterpret_cast<const float4*>(a.dzx + go + e);
            dzx[e] = t.x; dzx[e + 1] = t.y; dzx[e + 2] = t.z; dzx[e + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) dzx[e] = 0.f;
        }
        float o_dz[VE], o_dx[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float dyy = dyv[rr][k][e];
          const float keep = FUSED ? (((mk[rr][k] >> e) & 1u) ? a.scale : 0.f) : 1.f;
          if constexpr (COMP) {
            // fp32 outputs: column sums of exactly evaluated terms
            const DF xh = df_mul(df_plus(two_sum(zv[rr][k][e], -mu[rr]), zlo[rr][k][e]), rho[rr]);
            DF inner = df_plus(two_prod(dyy, gam[k][e]), -mg);
            const DF xm = df_mul(xh, mgx);
            inner = df_plus(DF{inner.hi, inner.lo - xm.lo}, -xm.hi);
            const DF dz = df_plus(df_mul(inner, rho[rr]), dzx[e]);
            const DF dxd = df_mul(dz, keep);
            o_dz[e] = df_round(dz);
            o_dx[e] = df_round(dxd);
            df_acc(acc_g[k][e], df_mul(xh, dyy));
            df_add(acc_b[k][e], dyy);
            if (FUSED) df_acc(acc_x[k][e], dxd);
          } else {
            const float xh = (zv[rr][k][e] - mu[rr]) * rho[rr];
            const float gg = dyy * gam[k][e];
            const float dz = fmaf(rho[rr], gg - mg - xh * mgx, dzx[e]);
            o_dz[e] = dz;
            o_dx[e] = FUSED ? dz * keep : dz;
            acc_g[k][e].hi = fmaf(dyy, xh, acc_g[k][e].hi);
            acc_b[k][e].hi += dyy;
            if (FUSED) acc_x[k][e].hi += o_dx[e];
          }
        }
        Vec16<T>::store(static_cast<T*>(a.dx) + go, o_dx);
        if (FUSED && a.dres != nullptr) Vec16<T>::store(static_cast<T*>(a.dres) + go, o_dz);
      }
    }
  }

  if (failed) {
    report_status(a.status, GBN_DEV_WAIT_TIMEOUT);
    if (tid == 0) {
      for (int64_t k = i; k < nmine && k < i + nst; ++k)
        mbar_wait_bounded(&bar[k % nst], (uint32_t)((k / nst) & 1), kWaitLimitNs / 8);
    }
    __syncthreads();
    return;
  }

  // Column partials [nout][nplanes][G][H]: 0 = dgamma, 1 = dbeta, 2 = dbias.
  auto store_part = [&](int o, int k, const DF (&acc)[VE]) {
    const int vi = tid + k * blockDim.x;
    float* hi = a.part + (((int64_t)o * a.nplanes + 0) * G + g) * H + (int64_t)vi * VE;
    float* lo = a.part + (((int64_t)o * a.nplanes + 1) * G + g) * H + (int64_t)vi * VE;
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      *reinterpret_cast<float4*>(hi + e) =
          make_float4(acc[e].hi, acc[e + 1].hi, acc[e + 2].hi, acc[e + 3].hi);
      if constexpr (COMP)
        *reinterpret_cast<float4*>(lo + e) =
            make_float4(acc[e].lo, acc[e + 1].lo, acc[e + 2].lo, acc[e + 3].lo);
    }
  };
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    if (tid + k * (int)blockDim.x >= a.Hv) continue;
    store_part(0, k, acc_g[k]);
    store_part(1, k, acc_b[k]);
    if (FUSED) store_part(2, k, acc_x[k]);
  }
  pdl_launch_dependents();
}

// Any H and alignment.  Block g owns rows g, g+G, ...; thread t owns columns
// t, t+256, ...; column sums go straight into this block's partial rows.
template <typename T, bool FUSED>
__global__ void __launch_bounds__(256) ln_bwd_generic_kernel(LnArgs a) {
  constexpr bool COMP = sizeof(T) == 4;
  __shared__ float red[2][2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int g = blockIdx.x, G = gridDim.x;
  const int64_t H = a.H;
  const T* dy = static_cast<const T*>(a.dy);
  const T* x = static_cast<const T*>(a.x);
  const T* res = static_cast<const T*>(a.res);
  const T* bias = static_cast<const T*>(a.bias);
  const T* gamma = static_cast<const T*>(a.gamma);
  const int nout = FUSED ? 3 : 2;
  auto P = [&](int o, int plane) { return a.part + (((int64_t)o * a.nplanes + plane) * G + g) * H; };
  for (int o = 0; o < nout; ++o)
    for (int64_t j = tid; j < H; j += blockDim.x) {
      P(o, 0)[j] = 0.f;
      if constexpr (COMP) P(o, 1)[j] = 0.f;
    }
  // z (hi, lo): exact for fp32 outputs, plain fp32 otherwise
  auto zval = [&](int64_t r, int64_t j, float& keep) {
    const float xv = to_f32(x[r * H + j]);
    DF z{xv, 0.f};
    keep = 1.f;
    if constexpr (FUSED) {
      keep = (a.mask == nullptr || a.mask[r * H + j] != 0) ? a.scale : 0.f;
      const float b = bias ? to_f32(bias[j]) : 0.f;
      const float rv = to_f32(res[r * H + j]);
      if constexpr (COMP) {
        const DF kt = df_mul(two_sum(xv, b), keep);
        z = df_plus(two_sum(rv, kt.hi), kt.lo);
      } else {
        z = DF{fmaf(keep, xv + b, rv), 0.f};
      }
    }
    return z;
  };
  auto acc_add = [&](int o, int64_t j, float v) {
    if constexpr (COMP) {
      DF d{P(o, 0)[j], P(o, 1)[j]};
      df_add(d, v);
      P(o, 0)[j] = d.hi;
      P(o, 1)[j] = d.lo;
    } else {
      P(o, 0)[j] += v;
    }
  };
  int it = 0;
  for (int64_t r = g; r < a.R; r += G, ++it) {
    const float mu = a.mean[r], rho = a.rstd[r];
    float sg = 0.f, sgx = 0.f;
    for (int64_t j = tid; j < H; j += blockDim.x) {
      float keep;
      const float z = zval(r, j, keep).hi;
      const float xh = (z - mu) * rho;
      const float gg = to_f32(dy[r * H + j]) * to_f32(gamma[j]);
      sg += gg;
      sgx = fmaf(gg, xh, sgx);
    }
    sg = warp_sum(sg);
    sgx = warp_sum(sgx);
    if (lane == 0) { red[it & 1][0][warp] = sg; red[it & 1][1][warp] = sgx; }
    __syncthreads();
    float SG = 0.f, SGX = 0.f;
    for (int wi = 0; wi < nwarps; ++wi) { SG += red[it & 1][0][wi]; SGX += red[it & 1][1][wi]; }
    const float mg = SG / (float)H, mgx = SGX / (float)H;
    for (int64_t j = tid; j < H; j += blockDim.x) {
      float keep;
      const DF z = zval(r, j, keep);
      const float dyy = to_f32(dy[r * H + j]);
      const float gm = to_f32(gamma[j]);
      const float zx = a.dzx ? a.dzx[r * H + j] : 0.f;
      if constexpr (COMP) {
        const DF xh = df_mul(df_plus(two_sum(z.hi, -mu), z.lo), rho);
        DF inner = df_plus(two_prod(dyy, gm), -mg);
        const DF xm = df_mul(xh, mgx);
        inner = df_plus(DF{inner.hi, inner.lo - xm.lo}, -xm.hi);
        const DF dz = df_plus(df_mul(inner, rho), zx);
        const DF dxd = df_mul(dz, FUSED ? keep : 1.f);
        static_cast<T*>(a.dx)[r * H + j] = from_f32<T>(df_round(dxd));
        if (FUSED && a.dres != nullptr) static_cast<T*>(a.dres)[r * H + j] = from_f32<T>(df_round(dz));
        DF d{P(0, 0)[j], P(0, 1)[j]};
        df_acc(d, df_mul(xh, dyy));
        P(0, 0)[j] = d.hi;
        P(0, 1)[j] = d.lo;
        acc_add(1, j, dyy);
        if (FUSED) {
          DF e{P(2, 0)[j], P(2, 1)[j]};
          df_acc(e, dxd);
          P(2, 0)[j] = e.hi;
          P(2, 1)[j] = e.lo;
        }
      } else {
        const float xh = (z.hi - mu) * rho;
        const float dz = fmaf(rho, dyy * gm - mg - xh * mgx, zx);
        const float dxv = FUSED ? dz * keep : dz;
        static_cast<T*>(a.dx)[r * H + j] = from_f32<T>(dxv);
        if (FUSED && a.dres != nullptr) static_cast<T*>(a.dres)[r * H + j] = from_f32<T>(dz);
        P(0, 0)[j] = fmaf(dyy, xh, P(0, 0)[j]);
        acc_add(1, j, dyy);
        if (FUSED) acc_add(2, j, dxv);
      }
    }
  }
  pdl_launch_dependents();
}

template <typename T, int KV, int RB, bool FUSED>
cudaError_t launch_fast(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
  return launch(ln_bwd_fast_kernel<T, KV, RB, FUSED>, dim3(p.G), dim3(p.threads), p.smem, st,
                false, a);
}

template <typename T, bool FUSED>
cudaError_t launch_typed(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
  if (!p.fast)
    return launch(ln_bwd_generic_kernel<T, FUSED>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  // The plan keeps at most 16 owned columns per thread: kv is 1 or 2.
  if (p.rb == 2) return launch_fast<T, 1, 2, FUSED>(p, a, st);
  if (p.kv == 1) return launch_fast<T, 1, 1, FUSED>(p, a, st);
  return launch_fast<T, 2, 1, FUSED>(p, a, st);
}

template <typename T, int KV, int RB>
cudaError_t set_smem(int bytes) {
  cudaError_t e1 = cudaFuncSetAttribute(ln_bwd_fast_kernel<T, KV, RB, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  cudaError_t e2 = cudaFuncSetAttribute(ln_bwd_fast_kernel<T, KV, RB, false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e1 != cudaSuccess ? e1 : e2;
}

template <typename T>
cudaError_t set_smem_all(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_smem<T, 1, 2>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 1, 1>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 2, 1>(bytes)) != cudaSuccess) e = r;
  return e;
}

}  // namespace

uint32_t ln_smem_header(int rb) { return ln_header(rb); }

cudaError_t ln_configure(int smem_optin) {
  cudaError_t e1 = set_smem_all<float>(smem_optin);
  cudaError_t e2 = set_smem_all<bf16>(smem_optin);
  return e1 != cudaSuccess ? e1 : e2;
}

cudaError_t ln_launch(const RowPlan& p, const LnPtrs& q, float* part, int* status,
                      cudaStream_t st) {
  const bool fused = p.kind == GBN_ROW_LN_FUSED;
  cudaError_t e = cudaSuccess;
  if (p.R > 0 && p.H > 0) {
    LnArgs a;
    a.dy = q.dy;
    a.x = q.x;
    a.res = q.residual;
    a.bias = q.bias;
    a.mask = q.mask;
    a.dzx = q.dz_extra;
    a.mean = q.mean;
    a.rstd = q.rstd;
    a.gamma = q.gamma;
    a.dx = q.dx;
    a.dres = q.dres;
    a.part = part;
    a.status = status;
    a.R = p.R;
    a.scale = q.scale;
    a.H = (int32_t)p.H;
    a.Hv = (int32_t)(p.H * (p.dtype == GBN_F32 ? 4 : 2) / 16);
    a.nstage = p.nstage;
    a.nplanes = p.nplanes;
    a.stage_bytes = p.stage_bytes;
    a.off_dy = p.off[0];
    a.off_x = p.off[1];
    a.off_res = p.off[2];
    a.off_mask = p.off[3];
    if (p.dtype == GBN_F32)
      e = fused ? launch_typed<float, true>(p, a, st) : launch_typed<float, false>(p, a, st);
    else
      e = fused ? launch_typed<bf16, true>(p, a, st) : launch_typed<bf16, false>(p, a, st);
    if (e != cudaSuccess) return e;
  }
  void* outs[3] = {q.dgamma, q.dbeta, fused ? q.dbias : nullptr};
  return colsum_launch(part, fused ? 3 : 2, p.nplanes, p.R > 0 ? p.G : 0, p.H, p.dtype, outs, st,
                       p.R > 0 && p.H > 0);
}

}  // namespace gbn
