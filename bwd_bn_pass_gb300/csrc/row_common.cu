// Launch planning for the row-wise backward kernels and the fixed-order
// column-partials reduction that follows them.
//
// The row kernels leave one partial row per block: part[o][plane][g][h] with
// o the column output (dweight; or dgamma, dbeta, dbias), plane 0 the fp32
// sum and plane 1 its double-fp32 low part (fp32 outputs only).  colsum adds
// the G rows of each output in a fixed order (32 strided groups, then the 32
// group sums in order), so the result is deterministic for a given G.  Each
// thread has at most ceil(G/32) independent loads, all in flight at once.
#include "gbn_common.cuh"
#include "gbn_internal.h"

namespace gbn {

cudaError_t rms_configure(int smem_optin);
cudaError_t ln_configure(int smem_optin);

namespace {

constexpr int kColTile = 32;
constexpr int kColGroups = 32;
constexpr int kMaxStages = 8;
constexpr int kRmsConsumers = 512;       // consumer threads of the RMSNorm ring kernel
constexpr int kRowRingStatic = 4096;     // static shared memory of a ring kernel, at most
constexpr int64_t kRingBytesPerSm = 128 << 10;  // ring bytes in flight per SM, about
constexpr int kLnMaxGroups = 14;         // consumer groups (named barriers 2..15) of the LayerNorm ring kernel

// Epoch pair, arrival counter and one flag pair per CTA, rounded to 256
// bytes (the layout of row_engine.cuh).
size_t ring_sync_bytes(int G) { return ((size_t)32 + (size_t)16 * G + 255) & ~(size_t)255; }

struct ColOuts {
  void* p[3];
};

template <typename T, bool COMP>
__global__ void __launch_bounds__(kColTile* kColGroups)
    colsum_kernel(const float* __restrict__ part, int nplanes, int G, int64_t H, ColOuts outs) {
  __shared__ DF sm[kColGroups][kColTile];
  pdl_wait();
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int o = blockIdx.y;
  const int64_t h = (int64_t)blockIdx.x * kColTile + tx;
  DF acc{0.f, 0.f};
  if (h < H) {
    const float* hi = part + ((int64_t)o * nplanes) * G * H + h;
    const float* lo = hi + (int64_t)G * H;
#pragma unroll 8
    for (int g = ty; g < G; g += kColGroups) {
      df_add(acc, hi[(int64_t)g * H]);
      if (COMP) acc.lo += lo[(int64_t)g * H];
    }
  }
  sm[ty][tx] = acc;
  __syncthreads();
  if (ty == 0 && h < H && outs.p[o] != nullptr) {
    DF t{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kColGroups; ++k) {
      df_add(t, sm[k][tx].hi);
      t.lo += sm[k][tx].lo;
    }
    static_cast<T*>(outs.p[o])[h] = from_f32<T>(df_round(t));
  }
}

uint32_t round16(uint64_t v) { return (uint32_t)((v + 15) & ~(uint64_t)15); }

}  // namespace

cudaError_t colsum_launch(const float* part, int nout, int nplanes, int G, int64_t H, int dtype,
                          void* const* outs, cudaStream_t st, bool pdl) {
  if (H <= 0 || nout <= 0) return cudaSuccess;
  ColOuts o;
  for (int i = 0; i < 3; ++i) o.p[i] = i < nout ? outs[i] : nullptr;
  const dim3 grid((unsigned)((H + kColTile - 1) / kColTile), (unsigned)nout);
  const dim3 block(kColTile, kColGroups);
  if (dtype == GBN_F32)
    return launch(colsum_kernel<float, true>, grid, block, 0, st, pdl, part, nplanes, G, H, o);
  return launch(colsum_kernel<bf16, false>, grid, block, 0, st, pdl, part, nplanes, G, H, o);
}

cudaError_t row_kernels_configure(int smem_optin) {
  cudaError_t e1 = rms_configure(smem_optin);
  cudaError_t e2 = ln_configure(smem_optin);
  return e1 != cudaSuccess ? e1 : e2;
}

bool row_plan(int64_t R, int64_t H, int kind, int dtype, bool fast_ok, bool has_mask,
              bool has_dzx, const DevInfo& dev, RowPlan* p) {
  (void)has_dzx;
  if (R < 0 || H < 0) return false;
  if (kind != GBN_ROW_RMS && kind != GBN_ROW_LN && kind != GBN_ROW_LN_FUSED) return false;
  if (dtype != GBN_F32 && dtype != GBN_BF16) return false;
  *p = RowPlan();
  p->R = R;
  p->H = H;
  p->kind = kind;
  p->dtype = dtype;
  p->nout = kind == GBN_ROW_RMS ? 1 : (kind == GBN_ROW_LN ? 2 : 3);
  p->nplanes = dtype == GBN_F32 ? 2 : 1;
  const int64_t esize = dtype == GBN_F32 ? 4 : 2;
  const bool fused = kind == GBN_ROW_LN_FUSED;

  bool fast = fast_ok && R > 0 && H > 0 && (H * esize) % 16 == 0 && (!has_mask || H % 16 == 0);
  if (fast && kind == GBN_ROW_RMS && H % 8 != 0) fast = false;  // column sums take 8 at a time
  if (fast && kind == GBN_ROW_RMS) {
    // Ring kernel: 16 consumer warps + the producer warp, one CTA per SM;
    // each consumer thread owns kv 16-byte vectors of a row.
    const int64_t Hv = H * esize / 16;
    const int64_t kv = (Hv + kRmsConsumers - 1) / kRmsConsumers;
    const int rb = kv == 1 ? 2 : 1;
    const uint64_t stage = 2ull * rb * (uint64_t)H * esize;
    const int64_t dyn = (int64_t)dev.smem_optin - kRowRingStatic;
    int64_t nst = dyn / (int64_t)stage;
    if (nst > kMaxStages) nst = kMaxStages;
    // about 128 KB in flight per SM: deeper rings measured slower (RMSNorm
    // bf16 [2048, 8192]: 26.3 us at 2-5 stages of 32 KB, 28.0 us at 6)
    int64_t cap = (kRingBytesPerSm + (int64_t)stage - 1) / (int64_t)stage;
    // the instances that hold a stage until the end of their second pass
    // (kv > 2) keep a third stage in flight (fp32 [2048, 8192]: 34.6 ->
    // 33.1 us per launch)
    if (kv > 2 && cap < 3) cap = 3;
    if (nst > cap && cap >= 2) nst = cap;
    if (kv <= 4 && nst >= 2) {
      const int64_t nblk = (R + rb - 1) / rb;
      p->fast = true;
      p->threads = kRmsConsumers + 32;
      p->kv = (int)kv;
      p->rb = rb;
      p->cps = 1;
      p->nstage = (int)nst;
      p->stage_bytes = (uint32_t)stage;
      p->G = (int)(nblk < dev.sms ? nblk : dev.sms);
      p->smem = (size_t)nst * stage;
      p->part_offset = ring_sync_bytes(p->G);
    } else {
      fast = false;
    }
  } else if (fast) {
    // LayerNorm ring kernel: NGRP groups of TPRW consumer warps (at most 14
    // or 8 warps in all) + the producer warp, one CTA per SM; each consumer
    // thread owns kv 16-byte vectors of a row; a stage holds two rows for
    // one-vector rows, else one, and goes to one group.
    const int64_t Hv = H * esize / 16;
    int64_t kv = 1, maxw = kLnRingWarpsKV1;
    if (Hv > 32 * kLnRingWarpsKV1) {  // two vectors per thread (bf16 rows up to 4096)
      kv = 2;
      maxw = kLnRingWarpsKVn;
    }
    const int64_t tprw = (Hv + 32 * kv - 1) / (32 * kv);
    // fp32 keeps three double-fp32 column sums per element: one vector per
    // thread at most; the column sums take 8 columns at a time.
    if (tprw > maxw || (dtype == GBN_F32 && kv > 1) || H % 8 != 0) {
      fast = false;
    } else {
      const int rb = kv == 1 ? 2 : 1;
      int64_t rs = maxw / tprw;  // groups
      if (rs > kLnMaxGroups) rs = kLnMaxGroups;
      const uint64_t rowb = (uint64_t)H * esize;
      uint32_t off = 0;
      p->off[0] = 0;  // dy
      off = round16(rb * rowb);
      p->off[1] = off;  // x / input
      off = round16(off + rb * rowb);
      if (fused) {
        p->off[2] = off;  // residual
        off = round16(off + rb * rowb);
        if (has_mask) {
          p->off[3] = off;  // mask
          off = round16(off + (uint64_t)rb * H);
        }
      }
      const int64_t dyn = (int64_t)dev.smem_optin - kRowRingStatic;
      int64_t nst = dyn / (int64_t)off;
      if (nst > kMaxStages) nst = kMaxStages;
      // the slots' column sums are added in the idle ring at the end
      const uint64_t combine = (uint64_t)p->nout * p->nplanes * (uint64_t)H * 4;
      if (nst < 2 || combine > (uint64_t)dyn) {
        fast = false;
      } else {
        const int64_t nblk = (R + rb - 1) / rb;
        const uint64_t ring = (uint64_t)nst * off;
        p->fast = true;
        p->threads = (int)(32 + rs * tprw * 32);
        p->kv = (int)kv;
        p->rb = rb;
        p->tprw = (int)tprw;
        p->rs = (int)rs;
        p->cps = 1;
        p->nstage = (int)nst;
        p->stage_bytes = off;
        p->smem = (size_t)(ring > combine ? ring : combine);
        p->G = (int)(nblk < dev.sms ? nblk : dev.sms);
        p->part_offset = ring_sync_bytes(p->G);
      }
    }
  }
  if (!fast) {
    p->fast = false;
    p->threads = 256;
    p->part_offset = 0;
    const int64_t cap = 2 * (int64_t)dev.sms;
    p->G = (int)(R < cap ? R : cap);
  }
  const uint64_t g = p->G > 0 ? (uint64_t)p->G : 1;
  const uint64_t bytes =
      p->part_offset + (uint64_t)p->nout * p->nplanes * g * (uint64_t)(H > 0 ? H : 1) * 4;
  p->ws_bytes = (size_t)((bytes + 255) & ~(uint64_t)255);
  return true;
}

}  // namespace gbn
