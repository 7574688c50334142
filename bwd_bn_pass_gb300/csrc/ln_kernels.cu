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
// GB300 design: one launch, the ring engine of the RMSNorm kernel
// (row_engine.cuh).  A stage holds RB consecutive rows of dy, input,
// residual and mask (one bulk copy per tensor), filled by the producer warp.
// The consumer warps form NGRP groups of TPRW warps each; group q takes
// stages q, q + NGRP, ... and has its own named barrier, so that one group
// computes while another waits (the producer warp serves them all).  Each
// thread owns fixed 16-byte column vectors of a row (gamma, bias and the
// three column accumulators stay in registers); it copies its vectors of the
// stage's rows into registers and releases the stage at once, computes both
// row sums, meets its group at one barrier per stage, then writes dx /
// dresidual with 16-byte stores.  At the end the groups' column accumulators are added
// in shared memory into one partial row per CTA, the CTAs hand the partials
// to each other through the workspace's arrival counter, and every CTA sums
// its share of the dgamma / dbeta / dbias columns over all partial rows in a
// fixed order -- no second launch.  Shapes the ring does not take (rows that
// are not whole 16-byte vectors, masks of rows that are not whole 16-byte
// words, unaligned tensors, rows longer than the registers hold) run a plain
// kernel followed by a separate fixed-order column-sum launch.
#include <type_traits>

#include "gbn_common.cuh"
#include "gbn_internal.h"
#include "row_engine.cuh"

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
  void* dgamma;
  void* dbeta;
  void* dbias;
  unsigned long long* sync;  // ring kernel: epoch pair, counter, flags
  unsigned long long nonce;
  int32_t tprw;              // ring kernel: consumer warps per row slot
  int32_t rs;                // ring kernel: row slots
};

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

// Row-sum slots [group][buffer][row][warp][sum], the warp run padded to a
// multiple of 4 warps (read as float4: two warps' pairs of sums, added as
// packed pairs).  The plan keeps groups x warps per group within 14, so
// groups x padded warps is at most 56 (14 one-warp groups) and the slots
// take at most 56 x 2 buffers x 2 rows x 2 sums = 448 floats.
constexpr int kLnMaxRedFloats = 512;

// Bit 7 of every byte of the result is set iff that byte of w is nonzero.
__device__ __forceinline__ uint32_t bytes_nonzero(uint32_t w) {
  return (((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u;
}
// All ones if byte E of nz has bit 7 set, else zero (a byte permute that
// replicates the selected byte's top bit).
template <int E>
__device__ __forceinline__ uint32_t byte_select_mask(uint32_t nz) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(nz), "n"(0x8888 | (E * 0x1111)));
  return r;
}
// keep factors (scale where the mask byte is nonzero, else 0) of the NP
// pairs of a 16-byte vector whose mask bytes are in m (bf16: 8 bytes; fp32:
// the 4 bytes of m.x).
template <int NP>
__device__ __forceinline__ void keep_pairs(uint2 m, float s, f2 (&keep2)[NP]) {
  const uint32_t sb = __float_as_uint(s);
  const uint32_t n0 = bytes_nonzero(m.x);
  keep2[0] = f2_pack(__uint_as_float(sb & byte_select_mask<0>(n0)),
                     __uint_as_float(sb & byte_select_mask<1>(n0)));
  keep2[1] = f2_pack(__uint_as_float(sb & byte_select_mask<2>(n0)),
                     __uint_as_float(sb & byte_select_mask<3>(n0)));
  if constexpr (NP == 4) {
    const uint32_t n1 = bytes_nonzero(m.y);
    keep2[2] = f2_pack(__uint_as_float(sb & byte_select_mask<0>(n1)),
                       __uint_as_float(sb & byte_select_mask<1>(n1)));
    keep2[3] = f2_pack(__uint_as_float(sb & byte_select_mask<2>(n1)),
                       __uint_as_float(sb & byte_select_mask<3>(n1)));
  }
}

// Warp sums of four values at once (a transposed butterfly: 6 shuffles
// instead of 20).  Lane l ends with the full sum of value ((l >> 4) & 1) * 2
// + ((l >> 3) & 1); the addition order is fixed, so every lane holding a
// value holds the same bits.
__device__ __forceinline__ float warp_sum4_transposed(float v0, float v1, float v2, float v3) {
  const int lane = threadIdx.x & 31;
  const bool b = (lane & 16) != 0;
  float a0 = b ? v2 : v0, a1 = b ? v3 : v1;
  const float s0 = b ? v0 : v2, s1 = b ? v1 : v3;
  a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool c = (lane & 8) != 0;
  float m = c ? a1 : a0;
  const float o = c ? a0 : a1;
  m += __shfl_xor_sync(0xffffffffu, o, 8);
  m += __shfl_xor_sync(0xffffffffu, m, 4);
  m += __shfl_xor_sync(0xffffffffu, m, 2);
  m += __shfl_xor_sync(0xffffffffu, m, 1);
  return m;
}
// consumer warps of the ring instances, by KV (the plan's choices)
constexpr int kLnRingWarps[3] = {0, kLnRingWarpsKV1, kLnRingWarpsKVn};

// KV: 16-byte vectors per consumer thread and row; a stage holds RPS rows
// (two for one-vector rows, else one).  MAXW: consumer warps at most (the
// register budget of a thread follows from it).
template <typename T, int KV, bool FUSED, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32, 1) ln_bwd_ring_kernel(LnArgs a) {
  constexpr int VE = 16 / sizeof(T);
  constexpr bool COMP = sizeof(T) == 4;
  using PK = Pairs16<T>;
  constexpr int NP = PK::NP;
  constexpr int RPS = KV == 1 ? 2 : 1;
  using MaskRaw = typename std::conditional<VE == 8, uint2, uint32_t>::type;
  extern __shared__ __align__(128) unsigned char data[];
  __shared__ RowShared sh;
  __shared__ __align__(16) float red[kLnMaxRedFloats];
  static_assert(sizeof(RowShared) + sizeof(red) + 16 <= kRowStaticSmem, "static shared memory");

  const int tid = threadIdx.x;
  const int g = blockIdx.x, G = gridDim.x;
  const int TPRW = a.tprw, NGRP = a.rs, NCW = NGRP * TPRW, NC = NCW * 32, TPR = TPRW * 32;
  constexpr int RB = RPS;
  const int64_t nblk = (a.R + RB - 1) / RB;
  const int64_t nmine = (nblk - g + G - 1) / G;
  const int NS = a.nstage;
  const int64_t H = a.H;
  const uint32_t rowb = (uint32_t)(H * sizeof(T));
  const bool has_mask = FUSED && a.mask != nullptr;
  const bool with_res = FUSED && !a.zin;

  const int P = (TPRW + 3) & ~3;  // padded warp run of a slot
  for (int k = tid; k < kLnMaxRedFloats; k += blockDim.x) red[k] = 0.f;  // padding stays 0
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], TPRW);  // the warps of the stage's group
      sh.issued[s] = 0;
    }
    sh.abort = 0;
    fence_mbarrier_init();
    GBN_RING_TRACE(0);
  }
  __syncthreads();

  if (tid < 32) {
    if (tid == 0)
      ring_produce(sh, NS, nmine, a.status, [&](int64_t i, int s) {
        const int64_t r0 = (g + i * G) * RB;
        const int64_t nr = a.R - r0 < RB ? a.R - r0 : RB;
        const uint32_t bt = (uint32_t)nr * rowb;
        const uint32_t bm = (uint32_t)(nr * H);
        unsigned char* st = data + (size_t)s * a.stage_bytes;
        mbar_arrive_expect_tx(&sh.full[s], bt * (with_res ? 3u : 2u) + (has_mask ? bm : 0u));
        bulk_g2s(st + a.off_dy, static_cast<const char*>(a.dy) + r0 * rowb, bt, &sh.full[s]);
        bulk_g2s(st + a.off_x, static_cast<const char*>(a.x) + r0 * rowb, bt, &sh.full[s]);
        if (with_res)
          bulk_g2s(st + a.off_res, static_cast<const char*>(a.res) + r0 * rowb, bt, &sh.full[s]);
        if (has_mask) bulk_g2s(st + a.off_mask, a.mask + r0 * H, bm, &sh.full[s]);
      });
  } else if (tid - 32 < NC) {
    const int ct = tid - 32, lane = ct & 31, cw = ct >> 5;
    const int grp = cw / TPRW, wis = cw - grp * TPRW, lr = ct - grp * TPR;
    epoch_read(sh, a.sync, ct);
    const int gbar = 2 + grp;  // the group's named barrier

    // Per-column constants and accumulators of this thread's columns.  fp32
    // outputs use scalar double-fp32 sums; bf16 outputs packed fp32x2 sums.
    float gam[KV][VE], bia[KV][VE];
    f2 gam2[KV][NP], bia2[KV][NP];
    DF acc_g[KV][VE], acc_b[KV][VE], acc_x[KV][VE];  // dgamma, dbeta, dbias (fp32 outputs)
    f2 sg_g[KV][NP], sg_b[KV][NP], sg_x[KV][NP];     // the same, packed (bf16 outputs)
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int vi = lr + k * TPR;
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

    // One 16-byte column vector as packed pairs: dy, z (fused: residual +
    // keep*(input + bias)) and keep, from the raw words.
    auto pairs = [&](int k, uint4 rdy, uint4 rx, uint4 rres, MaskRaw rm, f2 (&dy2)[NP],
                     f2 (&z2)[NP], f2 (&keep2)[NP]) {
      PK::get(rdy, dy2);
      f2 x2[NP];
      PK::get(rx, x2);
      if constexpr (FUSED) {
        f2 r2[NP];
        PK::get(rres, r2);
        if (has_mask) {
          uint2 m;
          if constexpr (VE == 8) m = rm;
          else m = make_uint2(rm, 0u);
          keep_pairs<NP>(m, a.scale, keep2);
        } else {
#pragma unroll
          for (int p = 0; p < NP; ++p) keep2[p] = f2_splat(a.scale);
        }
#pragma unroll
        for (int p = 0; p < NP; ++p)
          z2[p] = a.zin ? x2[p] : f2_fma(keep2[p], f2_add(x2[p], bia2[k][p]), r2[p]);
      } else {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          keep2[p] = f2_splat(1.f);
          z2[p] = x2[p];
        }
      }
    };
    // Scalar form for fp32 outputs: dy, exact z (hi, lo), keep.
    auto elems = [&](int k, uint4 rdy, uint4 rx, uint4 rres, MaskRaw rm, float (&dyv)[VE],
                     DF (&z)[VE], float (&keep)[VE]) {
      float xv[VE];
      Vec<T, VE>::cvt(rdy, dyv);
      Vec<T, VE>::cvt(rx, xv);
      if constexpr (FUSED) {
        float rv[VE];
        Vec<T, VE>::cvt(rres, rv);
        uint32_t mk = 0xffu;
        if (has_mask) {
          uint32_t bits = 0;
          if constexpr (VE == 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              bits |= (((rm.x >> (8 * e)) & 0xffu) != 0u) << e;
              bits |= (((rm.y >> (8 * e)) & 0xffu) != 0u) << (e + 4);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) bits |= (((rm >> (8 * e)) & 0xffu) != 0u) << e;
          }
          mk = bits;
        }
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
    const bool plain_out = a.dzx == nullptr && !a.dres_f32;
    bool failed = false;

    // ring slot s = i mod NS, its phase parity and this group's slot buffer
    // (i / NGRP) & 1, advanced per stage (no 64-bit division in the loop)
    int s = grp % NS;
    uint32_t par = (uint32_t)((grp / NS) & 1);
    int buf = 0;
    for (int64_t i = grp; i < nmine; i += NGRP, buf ^= 1) {
      if (i != grp) {
        s += NGRP;
        while (s >= NS) {
          s -= NS;
          par ^= 1u;
        }
      }
      const int64_t r0 = (g + i * G) * RB;
      const int nr = (int)(a.R - r0 < RB ? a.R - r0 : RB);
      float mu[RPS], rho[RPS];
#pragma unroll
      for (int q = 0; q < RPS; ++q) {
        const int rr = q;
        mu[q] = rr < nr ? __ldg(a.mean + r0 + rr) : 0.f;
        rho[q] = rr < nr ? __ldg(a.rstd + r0 + rr) : 0.f;
      }
      const bool ok = __all_sync(0xffffffffu, ring_wait(&sh.full[s], par, &sh.abort));
      if (i == 0 && ct == 0) GBN_RING_TRACE(1);
      // This thread's vectors of its rows, into registers; then the stage is
      // released so that the producer can refill it while we compute.
      const unsigned char* st = data + (size_t)s * a.stage_bytes;
      // Loads without a select: a lane past the row's end reads the row's
      // last vector (its gamma and bias are 0, so it adds nothing to the row
      // sums and it stores nothing), and a row past the stage's last
      // (rr >= nr) reads the slot's stale bytes, which no output uses.
      uint4 rdy[RPS][KV], rx[RPS][KV], rres[RPS][KV];
      MaskRaw rmk[RPS][KV];
#pragma unroll
      for (int q = 0; q < RPS; ++q)
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          const int rr = q, vi = min(lr + k * TPR, a.Hv - 1);  // clamped to the row
          const size_t o = (size_t)rr * rowb + (size_t)vi * 16;
          rdy[q][k] = *reinterpret_cast<const uint4*>(st + a.off_dy + o);
          rx[q][k] = *reinterpret_cast<const uint4*>(st + a.off_x + o);
          rres[q][k] = with_res ? *reinterpret_cast<const uint4*>(st + a.off_res + o)
                                : make_uint4(0u, 0u, 0u, 0u);
          if (has_mask)
            rmk[q][k] = *reinterpret_cast<const MaskRaw*>(st + a.off_mask + (size_t)rr * H +
                                                          (size_t)vi * VE);
          else
            rmk[q][k] = MaskRaw{};
        }
      if (ok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
      }

      // Row sums of g and g*xhat of the stage's rows: per warp into the
      // group's slots [buffer][row][sum][warp], double-buffered by stage.
      // bf16 outputs keep xhat and the keep factors for the second pass.
      float* slot = red + ((grp * 2 + buf) * RB) * 2 * P;
      f2 xhs[COMP ? 1 : RPS][KV][NP], kps[COMP ? 1 : RPS][KV][NP];
      float rsum[RPS][2];
#pragma unroll
      for (int q = 0; q < RPS; ++q) {
        const f2 mu2 = f2_splat(mu[q]), rho2 = f2_splat(rho[q]);
        f2 sg2 = 0ull, sgx2 = 0ull;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          f2 dy2[NP], z2[NP], keep2[NP];
          pairs(k, rdy[q][k], rx[q][k], rres[q][k], rmk[q][k], dy2, z2, keep2);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const f2 xh2 = f2_mul(f2_sub(z2[p], mu2), rho2);
            const f2 g2 = f2_mul(dy2[p], gam2[k][p]);
            sg2 = f2_add(sg2, g2);
            sgx2 = f2_fma(g2, xh2, sgx2);
            if constexpr (!COMP) {
              xhs[q][k][p] = xh2;
              kps[q][k][p] = keep2[p];
            }
          }
        }
        rsum[q][0] = f2_hsum(sg2);
        rsum[q][1] = f2_hsum(sgx2);
      }
      if constexpr (RPS == 2) {
        const float v = warp_sum4_transposed(rsum[0][0], rsum[0][1], rsum[1][0], rsum[1][1]);
        // lane / 8 = 2 row + sum
        if ((lane & 7) == 0) slot[((lane >> 4) * P + wis) * 2 + ((lane >> 3) & 1)] = v;
      } else {
#pragma unroll
        for (int q = 0; q < RPS; ++q) {
          const float sg = warp_sum(rsum[q][0]), sgx = warp_sum(rsum[q][1]);
          if (lane == 0) {
            slot[(q * P + wis) * 2 + 0] = sg;
            slot[(q * P + wis) * 2 + 1] = sgx;
          }
        }
      }
      if (consumers_bar_or(!ok, TPR, gbar)) {
        failed = true;
        if (lr == 0) ring_abort(sh, a.status);
        break;
      }

      // dz, outputs and column sums for the stage's rows.  GEN: the form
      // with dz_extra and fp32 dresidual tested at run time; the common form
      // (neither) carries no test in its loops.
      auto rows_out = [&](auto gen) {
      constexpr bool GEN = decltype(gen)::value;
#pragma unroll
      for (int q = 0; q < RPS; ++q) {
        const int rr = q;
        if (rr >= nr) break;
        // both sums at once: (sum g, sum g*xhat) pairs of four warps per step
        const float4* sp = reinterpret_cast<const float4*>(slot + rr * 2 * P);
        f2 acc = 0ull;
        for (int j = 0; j < P / 2; j += 2) {
          const float4 u = sp[j], w = sp[j + 1];
          acc = f2_add(acc, f2_add(f2_add(f2_pack(u.x, u.y), f2_pack(u.z, u.w)),
                                   f2_add(f2_pack(w.x, w.y), f2_pack(w.z, w.w))));
        }
        const float2 sums = f2_unpack(acc);
        const float mg = sums.x * inv_H, mgx = sums.y * inv_H;
        const int64_t r = r0 + rr;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
          const int vi = lr + k * TPR;
          if (vi >= a.Hv) continue;
          const int64_t go = r * H + (int64_t)vi * VE;
          if constexpr (COMP) {
            float dzx[VE];
            if (GEN && a.dzx != nullptr) {
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
            elems(k, rdy[q][k], rx[q][k], rres[q][k], rmk[q][k], dyv, z, keep);
            float o_dz[VE], o_dx[VE];
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              // fp32 outputs: column sums of exactly evaluated terms
              const float dyy = dyv[e];
              const DF xh = df_mul(df_plus(two_sum(z[e].hi, -mu[q]), z[e].lo), rho[q]);
              DF inner = df_plus(two_prod(dyy, gam[k][e]), -mg);
              const DF xm = df_mul(xh, mgx);
              inner = df_plus(DF{inner.hi, inner.lo - xm.lo}, -xm.hi);
              const DF dz = df_plus(df_mul(inner, rho[q]), dzx[e]);
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
            f2 dy2[NP], dz2[NP], dx2[NP];
            PK::get(rdy[q][k], dy2);
            const f2 rho2 = f2_splat(rho[q]);
            const f2 mg2 = f2_splat(mg), nmgx2 = f2_splat(-mgx);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
              const f2 xh2 = xhs[q][k][p];
              const f2 g2 = f2_mul(dy2[p], gam2[k][p]);
              const f2 inner = f2_fma(xh2, nmgx2, f2_sub(g2, mg2));
              f2 extra = 0ull;
              if (GEN && a.dzx != nullptr) {
                const float2 t = *reinterpret_cast<const float2*>(a.dzx + go + 2 * p);
                extra = f2_pack(t.x, t.y);
              }
              dz2[p] = f2_fma(inner, rho2, extra);
              dx2[p] = FUSED ? f2_mul(dz2[p], kps[q][k][p]) : dz2[p];
              sg_g[k][p] = f2_fma(dy2[p], xh2, sg_g[k][p]);
              sg_b[k][p] = f2_add(sg_b[k][p], dy2[p]);
              if (FUSED) sg_x[k][p] = f2_add(sg_x[k][p], dx2[p]);
            }
            *reinterpret_cast<uint4*>(static_cast<T*>(a.dx) + go) = PK::put(dx2);
            if (FUSED && a.dres != nullptr) {
              if (GEN && a.dres_f32) {
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
      };
      if (plain_out) rows_out(std::false_type{});
      else rows_out(std::true_type{});
    }
    // every group has left its loop (a failed group has set the abort flag,
    // which ends the others' waits): one decision for all consumers
    failed = consumers_bar_or(failed, NC);
    if (ct == 0) GBN_RING_TRACE(2);
    if (!failed) {
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
      // The groups' column sums, added in group order in shared memory
      // (the ring is idle now: every stage has been consumed), then written
      // as this CTA's partial row of each output:
      // part[o][plane][g][h], o = 0 dgamma, 1 dbeta, 2 dbias.
      const int nout = FUSED ? 3 : 2;
      const int nplanes = COMP ? 2 : 1;
      float* sm = reinterpret_cast<float*>(data);  // [nout][nplanes][H]
      consumers_bar(NC);
      for (int q = 0; q < NGRP; ++q) {
        if (grp == q) {
#pragma unroll
          for (int k = 0; k < KV; ++k) {
            const int vi = lr + k * TPR;
            if (vi >= a.Hv) continue;
            auto put = [&](int o, const DF (&acc)[VE]) {
              float4* hi = reinterpret_cast<float4*>(sm + ((int64_t)o * nplanes) * H + (int64_t)vi * VE);
              float4* lo = reinterpret_cast<float4*>(reinterpret_cast<float*>(hi) + H);
#pragma unroll
              for (int e = 0; e < VE; e += 4) {
                float4 h = make_float4(acc[e].hi, acc[e + 1].hi, acc[e + 2].hi, acc[e + 3].hi);
                if (q == 0) {
                  hi[e / 4] = h;
                  if constexpr (COMP)
                    lo[e / 4] = make_float4(acc[e].lo, acc[e + 1].lo, acc[e + 2].lo, acc[e + 3].lo);
                } else if constexpr (COMP) {
                  const float4 ph = hi[e / 4], pl = lo[e / 4];
                  const DF t0 = df_sum(DF{ph.x, pl.x}, acc[e]), t1 = df_sum(DF{ph.y, pl.y}, acc[e + 1]);
                  const DF t2 = df_sum(DF{ph.z, pl.z}, acc[e + 2]), t3 = df_sum(DF{ph.w, pl.w}, acc[e + 3]);
                  hi[e / 4] = make_float4(t0.hi, t1.hi, t2.hi, t3.hi);
                  lo[e / 4] = make_float4(t0.lo, t1.lo, t2.lo, t3.lo);
                } else {
                  const float4 ph = hi[e / 4];
                  hi[e / 4] = make_float4(ph.x + h.x, ph.y + h.y, ph.z + h.z, ph.w + h.w);
                }
              }
            };
            put(0, acc_g[k]);
            put(1, acc_b[k]);
            if (FUSED) put(2, acc_x[k]);
          }
        }
        consumers_bar(NC);
      }
      const int64_t H4 = H / 4;  // H is a multiple of 8
      for (int op = 0; op < nout * nplanes; ++op)  // op = o * nplanes + plane
        for (int64_t v = ct; v < H4; v += NC)
          *reinterpret_cast<float4*>(a.part + ((int64_t)op * G + g) * H + v * 4) =
              *reinterpret_cast<const float4*>(sm + (int64_t)op * H + v * 4);
      if (ct == 0) GBN_RING_TRACE(3);
      if (ring_exchange(sh, a.sync, G, ct, NC, a.status, a.nonce)) {
        if (ct == 0) GBN_RING_TRACE(4);
        T* outs[3] = {static_cast<T*>(a.dgamma), static_cast<T*>(a.dbeta),
                      FUSED ? static_cast<T*>(a.dbias) : nullptr};
        colsum_warps<T, COMP>(a.part, nout, G, H, outs, g, G, cw, NCW, lane);
        if (ct == 0) GBN_RING_TRACE(5);
      }
    } else if (ct == 0) {
      ring_abort(sh, a.status);
    }
  }
  __syncthreads();
  if (tid == 0 && sh.abort) ring_drain(sh, NS);
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

template <typename T, int KV, bool FUSED>
cudaError_t launch_ring(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
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
  return cudaLaunchKernelEx(&cfg, ln_bwd_ring_kernel<T, KV, FUSED, kLnRingWarps[KV]>, a);
}

// Ring instances: KV = 1 (at most 14 consumer warps) and, for bf16, KV = 2
// (at most 8), the counts the plan uses.
template <typename T, bool FUSED>
cudaError_t launch_typed(const RowPlan& p, const LnArgs& a, cudaStream_t st) {
  if (!p.fast)
    return launch(ln_bwd_generic_kernel<T, FUSED>, dim3(p.G), dim3(p.threads), 0, st, false, a);
  if constexpr (sizeof(T) == 2)
    if (p.kv == 2) return launch_ring<T, 2, FUSED>(p, a, st);
  return launch_ring<T, 1, FUSED>(p, a, st);
}

template <typename T, int KV>
cudaError_t set_smem(int bytes) {
  cudaError_t e1 = cudaFuncSetAttribute(ln_bwd_ring_kernel<T, KV, true, kLnRingWarps[KV]>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  cudaError_t e2 = cudaFuncSetAttribute(ln_bwd_ring_kernel<T, KV, false, kLnRingWarps[KV]>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e1 != cudaSuccess ? e1 : e2;
}

template <typename T>
cudaError_t set_smem_all(int bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_smem<T, 1>(bytes)) != cudaSuccess) e = r;
  if constexpr (sizeof(T) == 2)
    if ((r = set_smem<T, 2>(bytes)) != cudaSuccess) e = r;
  return e;
}

}  // namespace

cudaError_t ln_configure(int smem_optin) {
  const int dyn = smem_optin - kRowStaticSmem;
  cudaError_t e1 = set_smem_all<float>(dyn);
  cudaError_t e2 = set_smem_all<bf16>(dyn);
  return e1 != cudaSuccess ? e1 : e2;
}

cudaError_t ln_launch(const RowPlan& p, const LnPtrs& q, void* ws, int* status,
                      cudaStream_t st) {
  const bool fused = p.kind == GBN_ROW_LN_FUSED;
  void* outs[3] = {q.dgamma, q.dbeta, fused ? q.dbias : nullptr};
  if (p.R == 0 || p.H == 0)  // no rows: the column outputs are sums of nothing
    return colsum_launch(nullptr, fused ? 3 : 2, p.nplanes, 0, p.H, p.dtype, outs, st, false);
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
  a.dgamma = q.dgamma;
  a.dbeta = q.dbeta;
  a.dbias = fused ? q.dbias : nullptr;
  a.sync = static_cast<unsigned long long*>(ws);
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + p.part_offset);
  a.nonce = next_nonce();
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
  a.tprw = p.tprw;
  a.rs = p.rs;
  cudaError_t e;
  if (p.dtype == GBN_F32)
    e = fused ? launch_typed<float, true>(p, a, st) : launch_typed<float, false>(p, a, st);
  else
    e = fused ? launch_typed<bf16, true>(p, a, st) : launch_typed<bf16, false>(p, a, st);
  if (e != cudaSuccess || p.fast) return e;
  // the plain kernel leaves its column partials for a second launch
  return colsum_launch(a.part, fused ? 3 : 2, p.nplanes, p.G, p.H, p.dtype, outs, st, true);
}

}  // namespace gbn
