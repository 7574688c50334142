// Shared pieces of the persistent row-wise backward kernels (RMSNorm,
// LayerNorm): the ring of shared-memory stages that a producer warp fills
// with 1-D bulk copies, the consumer-group barriers, and the fixed-order
// column reduction that finishes dweight / dgamma / dbeta / dbias inside the
// same launch once every CTA has published its column partials.
//
// Launch shape: one CTA per SM (cooperative launch, so every CTA is resident
// and the CTAs may wait for each other's flags), warp 0 the producer, the
// remaining warps the consumers.  CTA g owns row blocks g, g + G, ...; a row
// block is RB consecutive rows and fills one stage.
#pragma once

#include "gbn_common.cuh"
#include "gbnorm.h"

namespace gbn {

// Optional per-CTA timestamps for studying the ring kernels' phases: a
// build that defines GBN_RING_TRACE(point) records them; the library's own
// build compiles the hook away.
#ifndef GBN_RING_TRACE
#define GBN_RING_TRACE(point) ((void)0)
#endif

constexpr int kRowMaxStages = 8;
constexpr int kRowStaticSmem = 4096;  // bound on a ring kernel's static shared memory

// Static shared state of a ring kernel.
struct RowShared {
  uint64_t full[kRowMaxStages];   // stage landed (transaction count)
  uint64_t empty[kRowMaxStages];  // stage released by every consumer warp
  unsigned long long target;      // flag value of this launch
  unsigned long long epoch[2];    // the workspace's epoch pair as the kernel found it
  int issued[kRowMaxStages];      // stages the producer has issued into each slot
  volatile int abort;             // a wait expired: stop issuing and computing
};

// Workspace of the ring kernels, 64-bit words: [0, 1] the epoch pair, [2]
// the arrival counter (tag in the high 32 bits, arrivals in the low 32),
// [3] unused, [4 + 2k, 5 + 2k] the flag pair of CTA k; then, from the next
// 256-byte boundary, the column partials.
constexpr int kRingCounterWord = 2;
constexpr int kRingFlagWord = 4;
__host__ __device__ constexpr size_t row_sync_bytes(int G) {
  return ((size_t)8 * kRingFlagWord + (size_t)16 * (size_t)G + 255) & ~(size_t)255;
}

// Named barrier `id` (1 by default: all consumer warps; the producer never
// joins it) over nthreads threads.
__device__ __forceinline__ void consumers_bar(int nthreads, int id = 1) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// The same barrier, returning whether any participant passed p = true.
__device__ __forceinline__ bool consumers_bar_or(bool p, int nthreads, int id = 1) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// mbarrier wait that gives up after about a second, or as soon as another
// thread of the CTA has aborted.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

__device__ __forceinline__ void ring_abort(RowShared& sh, int* status) {
  if (!sh.abort) {
    sh.abort = 1;
    report_status(status, GBN_DEV_WAIT_TIMEOUT);
  }
}

// Next ring slot: s = i mod NS and lap = i / NS for i + 1.
__device__ __forceinline__ void ring_advance(int& s, uint32_t& lap, int NS) {
  if (++s == NS) {
    s = 0;
    ++lap;
  }
}

// The producer (one lane): stage i of this CTA goes to slot i % NS once the
// slot's previous stage has been released.  issue(i, slot) posts the stage's
// expect_tx and bulk copies on sh.full[slot].
template <typename IssueFn>
__device__ void ring_produce(RowShared& sh, int NS, int64_t nmine, int* status, IssueFn issue) {
  int s = 0;         // i mod NS
  uint32_t lap = 0;  // i / NS (no 64-bit division in the loop)
  for (int64_t i = 0; i < nmine; ++i, ring_advance(s, lap, NS)) {
    if (i >= NS) {
      if (!ring_wait(&sh.empty[s], (lap - 1u) & 1u, &sh.abort)) {
        ring_abort(sh, status);
        return;
      }
      fence_proxy_async_smem();  // the consumers' reads before the copy's writes
    } else if (sh.abort) {
      return;
    }
    issue(i, s);
    sh.issued[s] += 1;
  }
}

// Let every copy that was issued land before the CTA exits (only needed
// after a failure; bounded): the latest phase of each slot, whether or not
// a consumer waited for it.
__device__ __forceinline__ void ring_drain(RowShared& sh, int NS) {
  for (int s = 0; s < NS; ++s)
    if (sh.issued[s] > 0)
      mbar_wait_bounded(&sh.full[s], (uint32_t)((sh.issued[s] - 1) & 1), kWaitLimitNs / 8);
}

// Column outputs out[o][h] = sum over g < G of the partials
// part[o][plane][g][h] (plane 1, the low part of a double-fp32 sum, only
// when COMP), for this CTA's share of the nout * H/8 eight-column groups.
// Consumer warp cw takes groups u0 + cw, u0 + cw + ncw, ...; lane l reads
// the 16 bytes (l & 1) of the group's 32-byte sector in rows g = l/2,
// l/2 + 16, ... (all its loads in flight at once), then a fixed xor-shuffle
// tree adds the 16 row classes, so the order is fixed for a given G and
// every run gives the same bits.  outs[o] may be null (not written).  H is a
// multiple of 8.
template <typename T, bool COMP>
__device__ void colsum_warps(const float* __restrict__ part, int nout, int G, int64_t H,
                             T* const* outs, int cta, int ncta, int cw, int ncw, int lane) {
  const int64_t H8 = H / 8;
  const int64_t U = (int64_t)nout * H8;
  const int64_t u0 = (int64_t)cta * U / ncta, u1 = (int64_t)(cta + 1) * U / ncta;
  const int nplanes = COMP ? 2 : 1;
  const int half = lane & 1, r0 = lane >> 1;
  // u = o * H8 + jg, advanced without a division per group
  int o = (int)((u0 + cw) / H8);
  int64_t jg = (u0 + cw) - (int64_t)o * H8;
  for (int64_t u = u0 + cw; u < u1; u += ncw, jg += ncw) {
    while (jg >= H8) {
      jg -= H8;
      ++o;
    }
    const int64_t j = jg * 8 + 4 * half;
    const float* hi = part + (int64_t)o * nplanes * G * H + j;
    const float* lo = hi + (int64_t)G * H;
    DF acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    constexpr int NB = 10;  // loads per lane in flight: one round for G <= 160
    for (int g0 = r0; g0 < G; g0 += NB * 16) {
      float4 v[NB], w[NB];
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const int g = g0 + q * 16;
        v[q] = g < G ? __ldcg(reinterpret_cast<const float4*>(hi + (int64_t)g * H))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (COMP)
          w[q] = g < G ? __ldcg(reinterpret_cast<const float4*>(lo + (int64_t)g * H))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        if constexpr (COMP) {
          df_add(acc[0], v[q].x); acc[0].lo = __fadd_rn(acc[0].lo, w[q].x);
          df_add(acc[1], v[q].y); acc[1].lo = __fadd_rn(acc[1].lo, w[q].y);
          df_add(acc[2], v[q].z); acc[2].lo = __fadd_rn(acc[2].lo, w[q].z);
          df_add(acc[3], v[q].w); acc[3].lo = __fadd_rn(acc[3].lo, w[q].w);
        } else {
          acc[0].hi += v[q].x; acc[1].hi += v[q].y; acc[2].hi += v[q].z; acc[3].hi += v[q].w;
        }
      }
    }
    // add the 16 row classes (lane bits 1..4); lanes 0 and 1 hold the sums
#pragma unroll
    for (int m = 2; m < 32; m *= 2)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (COMP) acc[e] = df_sum(acc[e], shfl_xor_df(acc[e], m));
        else acc[e].hi += __shfl_xor_sync(0xffffffffu, acc[e].hi, m);
      }
    T* out = outs[o];
    if (lane < 2 && out != nullptr) {
#pragma unroll
      for (int e = 0; e < 4; ++e) out[j + e] = from_f32<T>(COMP ? df_round(acc[e]) : acc[e].hi);
    }
  }
}

// Consumer thread 0 reads the epoch pair into shared memory as the kernel
// starts: the value is needed only at the hand-off, and the first stage takes
// longer to land than the load, so the load stays off the ring's start.
__device__ __forceinline__ void epoch_read(RowShared& sh, const unsigned long long* sync, int t) {
  if (t == 0) {
    sh.epoch[0] = ld_relaxed_u64(sync);
    sh.epoch[1] = ld_relaxed_u64(sync + 1);
  }
}

// After this CTA's partials are written, the hand-off between CTAs: every
// CTA arrives on the workspace's counter (a fence, then one atomic add) and
// waits until all G have arrived; the last to arrive resets the counter for
// the next launch, tagged with the next launch's flag value (a waiter that
// sees the reset knows that every CTA has arrived).  A counter whose tag does not match this
// launch (a fresh workspace, or one a failed launch left behind) switches
// every CTA to per-CTA flags for this launch; CTA 0 then prepares the
// counter.  CTA 0 advances the epoch once it has seen every arrival.
// Consumer threads only; returns false (for every consumer) if a wait
// expired.
// sh.epoch holds the workspace's epoch pair (epoch_read at the kernel's
// start); `nonce` is the host's value for a workspace without a valid pair.
__device__ __forceinline__ bool ring_exchange(RowShared& sh, unsigned long long* sync, int G,
                                              int t, int nthreads, int* status,
                                              unsigned long long nonce) {
  __shared__ int use_flags;
  if (t == 0) sh.target = (sh.epoch[1] == ~sh.epoch[0] ? sh.epoch[0] : nonce) + 1ull;
  consumers_bar(nthreads);  // every consumer's partial stores precede the arrival
  unsigned long long* ctr = sync + kRingCounterWord;
  unsigned long long* flags = sync + kRingFlagWord;
  const unsigned int tag = (unsigned int)sh.target, next_tag = (unsigned int)(sh.target + 1ull);
  bool ok = true;
  if (t == 0) {
    // acq_rel: publishes this CTA's partials (every consumer's stores reach
    // this thread through the barrier above) and, for the last arrival,
    // acquires everyone else's
    unsigned long long old;
    asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
    const bool tagged = (unsigned int)(old >> 32) == tag;
    use_flags = !tagged;
    if (tagged) {
      if ((unsigned int)old == (unsigned int)(G - 1)) {
        // the last arrival: every partial is published; prepare the next launch
        atomicExch(ctr, (unsigned long long)next_tag << 32);
      } else {
        // done once all G have arrived, or the last has already reset the counter
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
          const unsigned long long v = ld_acquire_u64(ctr);
          if ((unsigned int)(v >> 32) != tag || (unsigned int)v >= (unsigned int)G) break;
          if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
      }
    } else {
      flag_publish(flags - 2, blockIdx.x, sh.target);  // flag pair k at word 4 + 2k
    }
  }
  consumers_bar(nthreads);
  if (use_flags)
    for (int k = t; k < G && ok; k += nthreads) ok = wait_flag(flags + 2 * (int64_t)k, sh.target);
  const bool failed = consumers_bar_or(!ok, nthreads);
  if (failed && t == 0) ring_abort(sh, status);
  if (blockIdx.x == 0 && t == 0) {
    if (use_flags && !failed) st_relaxed_u64(ctr, (unsigned long long)next_tag << 32);
    epoch_advance(sync, sh.target, !failed);
  }
  return !failed;
}

}  // namespace gbn
