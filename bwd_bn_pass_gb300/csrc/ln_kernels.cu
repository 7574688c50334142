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
  int32_t zin;       // fused outputs from a saved z (x is z; no residual / bias)
  int32_t dres_f32;  // dresidual written as fp32
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

// Sum of the nwarps per-warp partials in slot[0..nwarps) as a fixed
// pairwise tree (every thread computes the same bits).  Blocks of at most 8
// warps read the 8 slots as two 16-byte words (slot is 16-byte aligned) and
// add the same tree without its all-zero upper half.
template <int MAXW>
__device__ __forceinline__ float sum_warp_slots(const float* slot, int nwarps) {
  if constexpr (MAXW <= 8) {
    const float4 p = reinterpret_cast<const float4*>(slot)[0];
    const float4 q = reinterpret_cast<const float4*>(slot)[1];
    const float v0 = p.x, v1 = nwarps > 1 ? p.y : 0.f, v2 = nwarps > 2 ? p.z : 0.f;
    const float v3 = nwarps > 3 ? p.w : 0.f, v4 = nwarps > 4 ? q.x : 0.f;
    const float v5 = nwarps > 5 ? q.y : 0.f, v6 = nwarps > 6 ? q.z : 0.f;
    const float v7 = nwarps > 7 ? q.w : 0.f;
    return ((v0 + v1) + (v2 + v3)) + ((v4 + v5) + (v6 + v7));
  } else {
    float v[16];
#pragma unroll
    for (int w = 0; w < 16; ++w) v[w] = w < nwarps ? slot[w] : 0.f;
#pragma unroll
    for (int step = 1; step < 16; step *= 2)
#pragma unroll
      for (int w = 0; w < 16; w += 2 * step) v[w] += v[w + step];
    return v[0];
  }
}

// One element's LayerNorm input z from the stage (fused: residual +
// keep*(input + bias), exact (hi, lo) for fp32 outputs).
template <bool FUSED, bool COMP>
__device__ __forceinline__ DF ln_z(float xin, float res, float b, float keep) {
  if constexpr (!FUSED) {
    return DF{xin, 0.f};
  } else if constexpr (COMP) {
    const DF kt = df_mul(two_sum(xin, b), keep);
    return df_plus(two_sum(res, kt.hi), kt.lo);
  } else {
    return DF{fmaf(keep, xin + b, res), 0.f};
  }
}

// keep factors (scale where the mask byte is nonzero, else 0) of the two
// elements of pair p of a 16-byte vector; the vector's mask bytes are in m
// (two words for bf16, one for fp32).
__device__ __forceinline__ f2 keep_pair(uint2 m, int p, float s) {
  const uint32_t w = (p < 2) ? m.x : m.y;
  const int sh = (p & 1) * 16;
  const float lo = ((w >> sh) & 0xffu) ? s : 0.f;
  const float hi = ((w >> (sh + 8)) & 0xffu) ? s : 0.f;
  return f2_pack(lo, hi);
}

template <typename T, int KV, int RB, bool FUSED, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) ln_bwd_fast_kernel(LnArgs a) {
  constexpr int VE = 16 / sizeof(T);
  constexpr bool COMP = sizeof(T) == 4;
  using PK = Pairs16<T>;
  constexpr int NP = PK::NP;
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
    const bool with_res = FUSED && !a.zin;
    mbar_arrive_expect_tx(&bar[s], bt * (with_res ? 3u : 2u) + (has_mask ? bm : 0u));
    bulk_g2s(st + a.off_dy, static_cast<const char*>(a.dy) + r0 * rowb, bt, &bar[s]);
    bulk_g2s(st + a.off_x, static_cast<const char*>(a.x) + r0 * rowb, bt, &bar[s]);
    if (with_res) bulk_g2s(st + a.off_res, static_cast<const char*>(a.res) + r0 * rowb, bt, &bar[s]);
    if (has_mask) bulk_g2s(st + a.off_mask, a.mask + r0 * H, bm, &bar[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < nmine && i < nst; ++i) issue(i);

  // Per-column constants and accumulators of this thread's columns.  fp32
  // outputs use scalar double-fp32 sums; bf16 outputs packed fp32x2 sums.
  float gam[KV][VE], bia[KV][VE];
  f2 gam2[KV][NP], bia2[KV][NP];
  DF acc_g[KV][VE], acc_b[KV][VE], acc_x[KV][VE];  // dgamma, dbeta, dbias (fp32 outputs)
  f2 sg_g[KV][NP], sg_b[KV][NP], sg_x[KV][NP];     // the same, packed (bf16 outputs)
#pragma unroll
  for (int k = 0; k < KV; ++k) {
    const int vi = tid + k * blockDim.x;
    uint4 rg = make_uint4(0u, 0u, 0u, 0u), rbias = make_uint4(0u, 0u, 0u, 0u);
    if (vi < a.Hv) {
      rg = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.gamma) + (int64_t)vi * VE);
      if (FUSED && a.bias != nullptr)
        rbias = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.bias) + (int64_t)vi * VE);
    }
    PK::get(rg, gam2[k]);
    PK::get(rbias, bia2[k]);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const float2 gg = f2_unpack(gam2[k][p]), bb = f2_unpack(bia2[k][p]);
      gam[k][2 * p] = gg.x;
      gam[k][2 * p + 1] = gg.y;
      bia[k][2 * p] = bb.x;
      bia[k][2 * p + 1] = bb.y;
      sg_g[k][p] = sg_b[k][p] = sg_x[k][p] = 0ull;
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) { acc_g[k][e] = acc_b[k][e] = acc_x[k][e] = DF{0.f, 0.f}; }
  }

  // One 16-byte column vector of row rr of the stage as packed pairs: dy, z
  // (fused: residual + keep*(input + bias)) and keep.
  auto load_pairs = [&](const unsigned char* st, int rr, int k, f2 (&dy2)[NP], f2 (&z2)[NP],
                        f2 (&keep2)[NP]) {
    const int vi = tid + k * blockDim.x;
    const size_t o = (size_t)rr * rowb + (size_t)vi * 16;
    PK::get(*reinterpret_cast<const uint4*>(st + a.off_dy + o), dy2);
    f2 x2[NP];
    PK::get(*reinterpret_cast<const uint4*>(st + a.off_x + o), x2);
    if constexpr (FUSED) {
      f2 r2[NP];
      if (!a.zin) PK::get(*reinterpret_cast<const uint4*>(st + a.off_res + o), r2);
      uint2 m = make_uint2(0x01010101u, 0x01010101u);
      if (has_mask) {
        const unsigned char* mp = st + a.off_mask + (size_t)rr * H + (size_t)vi * VE;
        if constexpr (VE == 8) m = *reinterpret_cast<const uint2*>(mp);
        else m.x = *reinterpret_cast<const uint32_t*>(mp);
      }
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        keep2[p] = keep_pair(m, p, a.scale);
        z2[p] = a.zin ? x2[p] : f2_fma(keep2[p], f2_add(x2[p], bia2[k][p]), r2[p]);
      }
    } else {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        keep2[p] = f2_splat(1.f);
        z2[p] = x2[p];
      }
    }
  };

  // Scalar form for fp32 outputs: dy, exact z (hi, lo), keep.
  auto load_elem = [&](const unsigned char* st, int rr, int k, float (&dyv)[VE],
                       DF (&z)[VE], float (&keep)[VE]) {
    const int vi = tid + k * blockDim.x;
    const size_t o = (size_t)rr * rowb + (size_t)vi * 16;
    float xv[VE];
    Vec16<T>::load(st + a.off_dy + o, dyv);
    Vec16<T>::load(st + a.off_x + o, xv);
    if constexpr (FUSED) {
      float rv[VE];
      if (!a.zin) Vec16<T>::load(st + a.off_res + o, rv);
      const uint32_t mk =
          has_mask ? mask_bits<VE>(st + a.off_mask + (size_t)rr * H + (size_t)vi * VE) : 0xffu;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        keep[e] = ((mk >> e) & 1u) ? a.scale : 0.f;
        z[e] = a.zin ? DF{xv[e], 0.f} : ln_z<FUSED, COMP>(xv[e], rv[e], bia[k][e], keep[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        keep[e] = 1.f;
        z[e] = DF{xv[e], 0.f};
      }
    }
  };

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

    // Pass 1 over the stage: row sums of g and g*xhat.
    float* slot = red + (i & 1) * (2 * RB * 32);
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      float sg = 0.f, sgx = 0.f;
      if (ok && rr < nr) {
        const f2 mu2 = f2_splat(mu[rr]), rho2 = f2_splat(rho[rr]);
        f2 sg2 = 0ull, sgx2 = 0ull;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          if (tid + k * (int)blockDim.x >= a.Hv) continue;
          f2 dy2[NP], z2[NP], keep2[NP];
          load_pairs(st, rr, k, dy2, z2, keep2);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const f2 xh2 = f2_mul(f2_sub(z2[p], mu2), rho2);
            const f2 g2 = f2_mul(dy2[p], gam2[k][p]);
            sg2 = f2_add(sg2, g2);
            sgx2 = f2_fma(g2, xh2, sgx2);
          }
        }
        sg = f2_hsum(sg2);
        sgx = f2_hsum(sgx2);
      }
      sg = warp_sum(sg);
      sgx = warp_sum(sgx);
      if (lane == 0) { slot[(2 * rr) * 32 + warp] = sg; slot[(2 * rr + 1) * 32 + warp] = sgx; }
    }
    if (__syncthreads_or(!ok)) { failed = true; break; }
    if (tid == 0 && i >= 1 && i - 1 + nst < nmine) {
      fence_proxy_async_smem();
      issue(i - 1 + nst);
    }

    // Pass 2 over the stage: dz, outputs, column sums.
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      if (rr >= nr) break;
      const float mg = sum_warp_slots<MAXT / 32>(slot + (2 * rr) * 32, nwarps) * inv_H;
      const float mgx = sum_warp_slots<MAXT / 32>(slot + (2 * rr + 1) * 32, nwarps) * inv_H;
      const int64_t r = r0 + rr;
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int vi = tid + k * blockDim.x;
        if (vi >= a.Hv) continue;
        const int64_t go = r * H + (int64_t)vi * VE;
        if constexpr (COMP) {
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
          float dyv[VE], keep[VE];
          DF z[VE];
          load_elem(st, rr, k, dyv, z, keep);
          float o_dz[VE], o_dx[VE];
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            // fp32 outputs: column sums of exactly evaluated terms
            const float dyy = dyv[e];
            const DF xh = df_mul(df_plus(two_sum(z[e].hi, -mu[rr]), z[e].lo), rho[rr]);
            DF inner = df_plus(two_prod(dyy, gam[k][e]), -mg);
            const DF xm = df_mul(xh, mgx);
            inner = df_plus(DF{inner.hi, inner.lo - xm.lo}, -xm.hi);
            const DF dz = df_plus(df_mul(inner, rho[rr]), dzx[e]);
            const DF dxd = df_mul(dz, keep[e]);
            o_dz[e] = df_round(dz);
            o_dx[e] = df_round(dxd);
            df_acc(acc_g[k][e], df_mul(xh, dyy));
            df_add(acc_b[k][e], dyy);
            if (FUSED) df_acc(acc_x[k][e], dxd);
          }
          Vec16<T>::store(static_cast<T*>(a.dx) + go, o_dx);
          if (FUSED && a.dres != nullptr) Vec16<T>::store(static_cast<T*>(a.dres) + go, o_dz);
        } else {
          f2 dy2[NP], z2[NP], keep2[NP], dz2[NP], dx2[NP];
          load_pairs(st, rr, k, dy2, z2, keep2);
          const f2 mu2 = f2_splat(mu[rr]), rho2 = f2_splat(rho[rr]);
          const f2 mg2 = f2_splat(mg), nmgx2 = f2_splat(-mgx);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const f2 xh2 = f2_mul(f2_sub(z2[p], mu2), rho2);
            const f2 g2 = f2_mul(dy2[p], gam2[k][p]);
            const f2 inner = f2_fma(xh2, nmgx2, f2_sub(g2, mg2));
            f2 extra = 0ull;
            if (a.dzx != nullptr) {
              const float2 t = *reinterpret_cast<const float2*>(a.dzx + go + 2 * p);
              extra = f2_pack(t.x, t.y);
            }
            dz2[p] = f2_fma(inner, rho2, extra);
            dx2[p] = FUSED ? f2_mul(dz2[p], keep2[p]) : dz2[p];
            sg_g[k][p] = f2_fma(dy2[p], xh2, sg_g[k][p]);
            sg_b[k][p] = f2_add(sg_b[k][p], dy2[p]);
            if (FUSED) sg_x[k][p] = f2_add(sg_x[k][p], dx2[p]);
          }
          *reinterpret_cast<uint4*>(static_cast<T*>(a.dx) + go) = PK::put(dx2);
          if (FUSED && a.dres != nullptr) {
            if (a.dres_f32) {
              float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(a.dres) + go);
#pragma unroll
              for (int p = 0; p < NP; p += 2) {
                const float2 u = f2_unpack(dz2[p]), w = f2_unpack(dz2[p + 1]);
                d4[p / 2] = make_float4(u.x, u.y, w.x, w.y);
              }
            } else {
              *reinterpret_cast<uint4*>(static_cast<T*>(a.dres) + go) = PK::put(dz2);
            }
          }
        }
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

  if constexpr (!COMP) {
#pragma unroll
    for (int k = 0; k < KV; ++k)
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const float2 a0 = f2_unpack(sg_g[k][p]), a1 = f2_unpack(sg_b[k][p]),
                     a2 = f2_unpack(sg_x[k][p]);
        acc_g[k][2 * p].hi = a0.x;
        acc_g[k][2 * p + 1].hi = a0.y;
        acc_b[k][2 * p].hi = a1.x;
        acc_b[k][2 * p + 1].hi = a1.y;
        acc_x[k][2 * p].hi = a2.x;
        acc_x[k][2 * p + 1].hi = a2.y;
      }
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
      if (a.zin) return z;
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
        if (FUSED && a.dres != nullptr) {
          if (a.dres_f32) static_cast<float*>(a.dres)[r * H + j] = dz;
          else static_cast<T*>(a.dres)[r * H + j] = from_f32<T>(dz);
        }
        P(0, 0)[j] = fmaf(dyy, xh, P(0, 0)[j]);
        acc_add(1, j, dyy);
        if (FUSED) acc_add(2, j, dxv);
      }
    }
  }
  pdl_launch_dependents();
}

template <typename T, int KV, int RB, bool FUSED, int MAXT, int MINB>
cudaError_t launch_fast(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
  return launch(ln_bwd_fast_kernel<T, KV, RB, FUSED, MAXT, MINB>, dim3(p.G), dim3(p.threads),
                p.smem, st, false, a);
}

// Instances (KV, RB, max threads, min blocks per SM).  Rows of at most 256
// 16-byte vectors: four rows per stage and two blocks per SM (measured 6 %
// faster than two rows and three blocks, which remains for smaller shared
// memory); one block per SM otherwise (128 registers).  The plan keeps at
// most 16 owned columns per thread, so kv is 1 or 2.
template <typename T, bool FUSED>
cudaError_t launch_typed(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
  if (!p.fast)
    return launch(ln_bwd_generic_kernel<T, FUSED>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  if (p.rb == 4) return launch_fast<T, 1, 4, FUSED, 256, 2>(p, a, st);
  if (p.rb == 2) return launch_fast<T, 1, 2, FUSED, 256, 3>(p, a, st);
  if (p.kv == 1) return launch_fast<T, 1, 1, FUSED, 512, 1>(p, a, st);
  return launch_fast<T, 2, 1, FUSED, 512, 1>(p, a, st);
}

template <typename T, int KV, int RB, int MAXT, int MINB>
cudaError_t set_smem(int bytes) {
  cudaError_t e1 = cudaFuncSetAttribute(ln_bwd_fast_kernel<T, KV, RB, true, MAXT, MINB>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  cudaError_t e2 = cudaFuncSetAttribute(ln_bwd_fast_kernel<T, KV, RB, false, MAXT, MINB>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e1 != cudaSuccess ? e1 : e2;
}

template <typename T>
cudaError_t set_smem_all(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_smem<T, 1, 4, 256, 2>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 1, 2, 256, 3>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 1, 1, 512, 1>(bytes)) != cudaSuccess) e = r;
  if ((r = set_smem<T, 2, 1, 512, 1>(bytes)) != cudaSuccess) e = r;
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
    a.zin = q.saved_z ? 1 : 0;
    a.dres_f32 = q.dres_f32 ? 1 : 0;
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
