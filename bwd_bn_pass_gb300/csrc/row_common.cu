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

uint32_t rms_smem_header(int rb);
uint32_t ln_smem_header(int rb);
cudaError_t rms_configure(int smem_optin);
cudaError_t ln_configure(int smem_optin);

namespace {

constexpr int kColTile = 32;
constexpr int kColGroups = 32;
constexpr int kMaxStages = 8;

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
  const int64_t VE = 16 / esize;
  const bool fused = kind == GBN_ROW_LN_FUSED;

  bool fast = fast_ok && R > 0 && H > 0 && (H * esize) % 16 == 0 && (!has_mask || H % 16 == 0);
  if (fast) {
    const int64_t Hv = H * esize / 16;
    const int64_t kv = (Hv + 511) / 512;
    const int64_t threads = ((Hv + kv - 1) / kv + 31) / 32 * 32;
    // Registers: at most 16 owned columns per thread (8 for the fp32
    // LayerNorm, whose three column sums are double-fp32).
    const int64_t max_cols = (kind != GBN_ROW_RMS && dtype == GBN_F32) ? 8 : 16;
    if (kv * VE > max_cols || kv > 4 || (kind != GBN_ROW_RMS && kv > 2)) fast = false;
    // (rows per stage, blocks per SM) in order of preference; these match
    // the compiled kernel instances.
    int cand[3][2];
    int ncand = 0;
    if (kind == GBN_ROW_RMS) {
      // Two-vector rows (e.g. 8192 bf16): two rows per stage at one block
      // per SM amortise the per-row barrier and bookkeeping over twice the
      // elements (29.3 vs 32.4 us at [2048, 8192] bf16).
      if (kv == 2) cand[ncand][0] = 2, cand[ncand++][1] = 1;
      cand[ncand][0] = kv == 1 ? 2 : 1;
      cand[ncand++][1] = kv <= 2 ? 2 : 1;
    } else if (kv == 1 && threads <= 256) {
      cand[ncand][0] = 4, cand[ncand++][1] = 2;
      cand[ncand][0] = 2, cand[ncand++][1] = 3;
    } else if (kv == 1) {
      cand[ncand][0] = 1, cand[ncand++][1] = 1;
    } else {
      cand[ncand][0] = 1, cand[ncand++][1] = 1;
    }
    bool placed = false;
    for (int ci = 0; fast && ci < ncand && !placed; ++ci) {
      const int rb = cand[ci][0], cps = cand[ci][1];
      const uint64_t rowb = (uint64_t)H * esize;
      uint32_t off = 0;
      p->off[0] = 0;  // dy (LayerNorm) / x (RMSNorm: x rows then dy rows)
      off = round16(rb * rowb);
      p->off[1] = off;  // x / input (LayerNorm)
      off = round16(off + rb * rowb);
      if (fused) {
        p->off[2] = off;  // residual
        off = round16(off + rb * rowb);
        if (has_mask) {
          p->off[3] = off;  // mask
          off = round16(off + (uint64_t)rb * H);
        }
      }
      const uint32_t header = kind == GBN_ROW_RMS ? rms_smem_header(rb) : ln_smem_header(rb);
      int64_t per_block = (int64_t)dev.smem_per_sm / cps - dev.smem_reserved;
      if (per_block > dev.smem_optin) per_block = dev.smem_optin;
      int64_t nst = (per_block - header) / off;
      if (nst > kMaxStages) nst = kMaxStages;
      if (nst < 2) continue;
      const int64_t nblk = (R + rb - 1) / rb;
      const int64_t slots = (int64_t)dev.sms * cps;
      p->fast = true;
      p->threads = (int)threads;
      p->kv = (int)kv;
      p->rb = rb;
      p->cps = cps;
      p->nstage = (int)nst;
      p->stage_bytes = off;
      p->smem = header + (size_t)nst * off;
      p->G = (int)(nblk < slots ? nblk : slots);
      placed = true;
    }
    if (!placed) fast = false;
  }
  if (!fast) {
    p->fast = false;
    p->threads = 256;
    const int64_t cap = 2 * (int64_t)dev.sms;
    p->G = (int)(R < cap ? R : cap);
  }
  const uint64_t g = p->G > 0 ? (uint64_t)p->G : 1;
  const uint64_t bytes = (uint64_t)p->nout * p->nplanes * g * (uint64_t)(H > 0 ? H : 1) * 4;
  p->ws_bytes = (size_t)((bytes + 255) & ~(uint64_t)255);
  return true;
}

}  // namespace gbn
