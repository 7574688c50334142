// Per-channel BatchNorm finalize arithmetic, shared by the two-launch kernels
// (bn_kernels.cu) and the persistent kernel (bn_fused.cu) so that both paths
// evaluate the same formulas in the same double-fp32 steps.
//
// Method: Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
// statistics, finalize kernels" -- the finalize step: mean and biased
// variance from the shifted sums, inv_std = 1/sqrt(var + eps), scale =
// gamma*inv_std, running_mean/var momentum update with the unbiased factor
// M/(M-1); and the backward finalize dgamma = S*inv_std, dbeta = sum dy,
// k1 = -scale*inv_std^2*S/M, k2 = -scale*dbeta/M.
#pragma once

#include "gbn_common.cuh"
#include "gbnorm.h"

namespace gbn {

// (hi, lo) / M for the per-channel count M (held exactly as mh + ml).
__device__ __forceinline__ DF div_count(DF a, float mh, float ml) {
  const float q = a.hi / mh;
  const DF p = two_prod(q, mh);
  const float r = __fsub_rn(__fadd_rn(__fsub_rn(__fsub_rn(a.hi, p.hi), p.lo), a.lo), __fmul_rn(q, ml));
  return DF{q, r / mh};
}

struct BnFwdFinal {
  DF md;          // mean - shift
  float var;      // biased batch variance
  float inv_std;  // 1 / sqrt(var + eps)
  float scale;    // gamma * inv_std
};

// From s1 = sum d and s2 = sum d^2 over the channel (d = x - shift).
__device__ __forceinline__ BnFwdFinal bn_fwd_final(DF s1, DF s2, float mh, float ml, float gamma,
                                                   float eps) {
  BnFwdFinal f;
  f.md = df_norm(div_count(s1, mh, ml));
  const DF e2 = div_count(s2, mh, ml);  // E[(x - shift)^2]
  float var = df_round(df_sum(e2, df_neg(df_mul_df(f.md, f.md))));
  if (!(var > 0.f)) var = 0.f;
  f.var = var;
  f.inv_std = 1.f / sqrtf(var + eps);
  f.scale = gamma * f.inv_std;
  return f;
}

// Stats rows 0-7 of channel c (mean, var, inv_std, scale, shift, mean - shift
// rounded, and mean - shift as a (hi, lo) pair) and the running update, from
// the running statistics' previous values rm, rv (read by the caller, which
// may read them early: nothing else in a call writes them).
__device__ __forceinline__ void bn_fwd_write_from(const BnFwdFinal& f, float shift, int64_t C,
                                                  int c, float M, float* stats,
                                                  float* running_mean, float* running_var,
                                                  float momentum, float rm, float rv) {
  const float mean = df_round(df_plus(f.md, shift));
  stats[c] = mean;
  stats[C + c] = f.var;
  stats[2 * C + c] = f.inv_std;
  stats[3 * C + c] = f.scale;
  stats[4 * C + c] = shift;
  stats[5 * C + c] = f.md.hi;
  stats[6 * C + c] = f.md.hi;
  stats[7 * C + c] = f.md.lo;
  const float m = momentum;
  if (running_mean) running_mean[c] = (1.f - m) * rm + m * mean;
  if (running_var) running_var[c] = (1.f - m) * rv + m * f.var * (M / (M - 1.f));
}
__device__ __forceinline__ void bn_fwd_write(const BnFwdFinal& f, float shift, int64_t C, int c,
                                             float M, float* stats, float* running_mean,
                                             float* running_var, float momentum) {
  bn_fwd_write_from(f, shift, C, c, M, stats, running_mean, running_var, momentum,
                    running_mean ? running_mean[c] : 0.f, running_var ? running_var[c] : 0.f);
}

struct BnBwdFinal {
  float dgamma, dbeta, k1, k2;
};

// From p0 = sum dy and p1 = sum dy*(x - shift); S = sum dy*(x - mean) =
// p1 - (mean - shift)*p0 in double-fp32 with the forward's (mean - shift),
// whose channel sum is exact, so a constant dy gives S = 0 to that precision.
__device__ __forceinline__ BnBwdFinal bn_bwd_final(DF p0, DF p1, DF md, float inv_std,
                                                   float scale, float M) {
  const float S = df_round(df_sum(p1, df_neg(df_mul_df(md, p0))));
  BnBwdFinal f;
  f.dbeta = df_round(p0);
  f.k1 = -(scale * inv_std) * inv_std * S / M;
  f.k2 = -scale * f.dbeta / M;
  f.dgamma = S * inv_std;
  return f;
}

// Fused activation of the BatchNorm output pre (Aether-ML PR #18, "Part 2":
// ReLU / LeakyReLU fused into BatchNorm): the output act(pre) and the gate
// d act / d pre applied to the incoming gradient -- 1 where pre > 0, else 0
// (ReLU) or the negative slope (LeakyReLU).  pre is always
// fmaf((x - shift) - mean_d, scale, beta), in the forward and when the
// backward recomputes it, so both take the same decision.
__device__ __forceinline__ float act_out(float pre, int act, float slope) {
  if (act == GBN_ACT_NONE || pre > 0.f) return pre;
  return act == GBN_ACT_RELU ? 0.f : pre * slope;
}
__device__ __forceinline__ float act_gate(float pre, int act, float slope) {
  return pre > 0.f ? 1.f : (act == GBN_ACT_RELU ? 0.f : slope);
}

}  // namespace gbn
