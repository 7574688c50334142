// Persistent single-launch BatchNorm2d training forward and backward (NCHW).
//
// Method: Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
// statistics, finalize kernels" computes, per direction, a reduction pass
// (shifted sums d = x - x[0,c] and d^2; or sum dy and sum dy*(x - shift)),
// a finalize, and an elementwise pass (y = (x - mean)*scale + beta; or dx =
// dy*scale + (x - mean)*k1 + k2).  This file runs the three steps in ONE
// launch; the arithmetic is that of the two-launch kernels in bn_kernels.cu
// (same finalize helpers, same per-element formulas).
//
// GB300 design:
//   * One CTA per SM (cooperative launch, so every CTA is resident).  The
//     tensor is viewed channel-major -- channel c's M = B*HW elements in
//     (b, h, w) order -- and CTA k owns the contiguous range [k*W, (k+1)*W)
//     of that view: one to a few channel segments, each a run of whole or
//     partial planes.
//   * Warp 0 is the producer: it streams the range through a ring of
//     shared-memory stages with 1-D bulk copies (cp.async.bulk, one per plane
//     run, issued by the 32 lanes in parallel) completing on per-stage "full"
//     mbarriers.  Sixteen consumer warps reduce each stage and release it on
//     an "empty" mbarrier.
//   * Phase 1 (reduction) walks the range forward and writes one double-fp32
//     partial pair per (segment, channel) into partials[2][grid_y][C], slot j
//     = k - (first CTA of the channel), then publishes a per-CTA flag.
//   * Phase 2 waits only for the flags of the CTAs that share its channels,
//     finalizes each channel from those partials (fixed order, so all CTAs
//     of a channel hold identical values; the CTA holding the channel's first
//     element writes stats / grads and the running statistics), then walks
//     the range BACKWARD: the last ring-full of stages is still in shared
//     memory (no reload), and the stages before it were read last, so they
//     are the likeliest to be in L2.  Outputs are written with 16-byte stores.
//   * Tensor memory (TMEM, 256 KB per SM, otherwise idle in this kernel) is a
//     second on-chip tier: in phase 1 each consumer thread also copies its
//     vectors of the nt stages just before the resident tail into its own
//     TMEM columns (tcgen05.st), and phase 2 reads them back (tcgen05.ld)
//     instead of loading those stages again; the L2 window moves back by nt
//     stages.  The CTA holds all 512 columns for the whole launch (one CTA
//     per SM) and frees them before it exits, also after a failed wait.
//   * Work stealing at the end of phase 2: a CTA's first stages (the last
//     it would reload) form a small pool that other CTAs may take once they
//     run out of their own work, so that CTAs on slower SMs (the phase-2
//     time of a CTA depends on the SM it runs on) finish with the rest.  A
//     pool word per CTA holds the unclaimed stages [lo, hi): the owner
//     claims from the top with an atomic subtract, other CTAs from the
//     bottom with an atomic add, so every stage is processed exactly once,
//     with the owner's finalized channel parameters (published after its
//     finalize, behind a release flag) -- the same bits either way.  In
//     phase 2 the producer hands each loaded stage to the consumers with a
//     descriptor (channel, vectors, parameters) in shared memory.
//   * Flags carry an epoch: (e+1, ~(e+1)) per CTA, with e read at kernel
//     start from the workspace's epoch pair (or a host nonce if that pair is
//     not self-consistent); CTA 0 advances the epoch once every CTA has
//     published.  The flags need no memset and no atomics (the pool words
//     above are the kernel's only atomics); a relaunch on the same
//     workspace always waits for fresh flags.
//   * Both phases run close to the copy rate once the instruction count is
//     low: packed fp32x2 arithmetic in both passes, two accumulation chains
//     per thread in phase 1, ring slots and output offsets advanced by
//     counters, and the plane index by a precomputed multiplier -- no
//     division in any per-stage or per-vector path.
//   * Every wait is bounded (about one second).  On expiry the CTA records
//     GBN_DEV_WAIT_TIMEOUT in the status word, stops issuing and computing,
//     waits (bounded) for its own copies in flight and returns.
#include <atomic>

#include "bn_finalize.cuh"
#include "gbn_common.cuh"
#include "gbn_internal.h"

// Optional per-CTA timestamps for studying the kernel's phases: a build that
// defines GBN_RING_TRACE(point) records them; the library's own build
// compiles the hook away.
#ifndef GBN_RING_TRACE
#define GBN_RING_TRACE(point) ((void)0)
#endif

namespace gbn {

namespace {

constexpr int kFConsumerWarps = 16;
constexpr int kFConsumers = kFConsumerWarps * 32;  // 512
constexpr int kFThreads = kFConsumers + 32;        // + the producer warp
constexpr int kFMaxStages = 8;
constexpr int kFMaxSegs = 32;                      // channel segments per CTA
constexpr int kFStaticSmem = 4096;                 // bound on the static shared memory
constexpr int kPoolMax = 8;       // stages per CTA that other CTAs may take in phase 2, at most
constexpr int kPubFloats = 8;     // published parameters per segment (6 used)
constexpr int kStealScans = 64;   // claims (and victim scans) of a CTA's producer, at most
constexpr int kStealBatch = 2;    // pool stages taken per claim, at most
constexpr int kMaxCtas = 160;     // CTAs of a launch, at most (one per SM)
constexpr int kPoolMinStages = 16;  // reloaded stages per CTA from which the pool is used


struct FArgs {
  const void* x;
  const void* dy;        // backward
  void* out;             // y (forward) or dx (backward)
  const float* gamma;    // forward, may be null (1)
  const float* beta;     // may be null (0); the backward needs it only with an activation
  float* stats;          // forward: written; backward: read
  float* running_mean;   // forward, may be null
  float* running_var;    // forward, may be null
  float* grads;          // backward: written
  float momentum, eps;
  int32_t act;           // GBN_ACT_*: output act(pre) forward, gate on dy backward
  float slope;           // LeakyReLU negative slope
  unsigned long long* sync;  // [2] epoch pair, then [G][2] flag pairs
  uint32_t* steal;           // [G] pool words: unclaimed pool stages [lo, hi) as hi << 16 | lo
  unsigned long long* pubflag;  // [G] set (release) once the CTA's parameters are published
  float* pub;                // [G][kPoolMax][kPubFloats] parameters of a CTA's first segments
  float2* part;              // [2][grid_y][C]
  int* status;
  unsigned long long nonce;
  int64_t C;
  int64_t P;         // plane size in elements
  int64_t Wv;        // vectors per CTA
  int32_t Mv;        // vectors per channel
  int32_t Pv;        // vectors per plane
  int32_t stage_v;   // vectors per stage (per input)
  int32_t nstage;
  int32_t grid_y;
  int32_t G;
  int32_t dn, dp;    // kFConsumers / Pv, kFConsumers % Pv
  FastDiv pdiv;      // division by Pv
  int64_t ostep;     // output vector offset step of a thread: dn*C*Pv + dp
  int64_t owrap;     // added when the in-plane position wraps: C*Pv - Pv
  int32_t l2_window; // phase-1 stages before the TMEM stages kept at normal L2 priority
  int32_t nt;        // stages kept in TMEM between the phases (0: none)
  int32_t pool;      // a CTA's first stages (at most kPoolMax) open to other CTAs in phase 2
  int32_t stream_out; // outputs with the evict-first hint (tensors larger than L2 holds)
  float Mh, Ml;      // per-channel count M = Mh + Ml exactly
};

// A phase-2 stage as the producer hands it to the consumers: channel c,
// first vector rv0 inside the channel, len vectors, the channel's parameters
// (as seg_par), or the end of the CTA's work.
struct FDesc {
  int c, rv0, len, end;
  float par[6];
};

// Parameters per segment: [0] shift, [1] mean - shift (rounded),
// forward [2] scale, [3] beta; backward [2] scale, [3] k1, [4] k2, [5] beta.
struct FShared {
  uint64_t full[kFMaxStages];
  uint64_t empty[kFMaxStages];
  int issued[kFMaxStages];
  unsigned long long target;  // flag value of this launch (epoch + 1)
  int nseg;
  int nst;                    // stages in the range
  int t_lo, t_hi;             // stages [t_lo, t_hi) are kept in TMEM; stages < t_lo reload
  uint32_t tmem;              // TMEM base address (written by tcgen05.alloc)
  int pool;                   // this CTA's pool stages [0, pool)
  volatile int p2ready;       // set once this CTA has finalized (and published)
  FDesc desc[kFMaxStages];    // phase 2: what the producer loaded into each slot
  volatile int abort;
  int seg_c[kFMaxSegs];
  int seg_rv0[kFMaxSegs];     // first vector of the segment inside its channel
  int seg_len[kFMaxSegs];     // vectors
  int seg_klo[kFMaxSegs];     // first CTA of the channel
  int seg_khi[kFMaxSegs];     // last CTA of the channel
  float seg_par[kFMaxSegs][6];
  float2 red[2][kFConsumerWarps];
};
static_assert(sizeof(FShared) <= kFStaticSmem, "static shared memory bound");

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFConsumers) : "memory");
}

// mbarrier wait that also gives up once another warp has aborted.
__device__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
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

__device__ __forceinline__ void set_abort(FShared& sh, int* status) {
  if (!sh.abort) {
    sh.abort = 1;
    report_status(status, GBN_DEV_WAIT_TIMEOUT);
  }
}

// Warp-uniform stage wait: false (for every lane) if the CTA has aborted or
// any lane's wait expired.  Every lane waits, so each observes the phase.
__device__ __forceinline__ bool warp_wait_full(FShared& sh, int slot, uint32_t& fpar,
                                               int* status) {
  if (__any_sync(0xffffffffu, sh.abort != 0)) return false;
  bool ok = wait_or_abort(&sh.full[slot], (fpar >> slot) & 1u, &sh.abort);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) {
    if ((threadIdx.x & 31) == 0) set_abort(sh, status);
    return false;
  }
  fpar ^= 1u << slot;
  return true;
}

// 16-byte output store with the streaming (evict-first) cache hint, so the
// outputs do not push the inputs that phase 2 still re-reads out of L2.
__device__ __forceinline__ void store16_cs(float* p, const float (&e)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(e[0], e[1], e[2], e[3]));
}
__device__ __forceinline__ void store16_cs(bf16* p, const float (&e)[8]) {
  __stcs(reinterpret_cast<uint4*>(p), make_uint4(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                                                pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7])));
}

// ------------------------------------------------------------- TMEM tier --
// Thread t of warp w reaches TMEM lanes 32*(w % 4) .. 32*(w % 4) + 31 (its
// own lane is 32*(w % 4) + t); the 16 consumer warps share each lane quarter
// four ways, 128 of the 512 columns each.  Address: lane << 16 | column.

// Vectors per consumer thread and input of a stage at the usual stage size
// (227 KB of shared memory: 48 KB stages of x forward, 24 KB of x and dy
// backward): the phase-1 early release keeps that many in registers.
constexpr int kKVFwd = 6;
constexpr int kKVBwd = 3;
constexpr uint32_t kTmemCols = 512;
constexpr int kTmemColsPerThread = kTmemCols / (kFConsumerWarps / 4);  // 128

__device__ __forceinline__ void tmem_alloc_all(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "n"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free_all(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "n"(kTmemCols)
               : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 bytes of this thread into columns [col, col + 4) of its lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Loads and the wait for them in one statement, so that no use of the
// results can be scheduled before the wait.
__device__ __forceinline__ uint4 tmem_ld16(uint32_t taddr) {
  uint4 v;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(taddr)
      : "memory");
  return v;
}
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint4& a, uint4& b) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%8];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4, %5, %6, %7}, [%9];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "r"(ta), "r"(tb)
      : "memory");
}
// 24 consecutive columns of this thread's lane (three 8-column loads, each
// at a multiple of 8 columns like every other access here), then one wait:
// a whole TMEM stage of a thread on the device's stage size (6 vectors of x
// forward, 3 of x and dy backward).
__device__ __forceinline__ void tmem_ld24(uint32_t ta, uint32_t (&r)[24]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%24];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%25];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%26];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
      : "r"(ta), "r"(ta + 8u), "r"(ta + 16u)
      : "memory");
}

// This consumer thread's first TMEM column address (consumer warp cw).
__device__ __forceinline__ uint32_t tmem_thread_base(uint32_t tmem, int cw) {
  const uint32_t quarter = (uint32_t)((cw + 1) & 3);  // warp index cw + 1 in the CTA
  return tmem + ((quarter * 32u) << 16) + (uint32_t)(cw >> 2) * (uint32_t)kTmemColsPerThread;
}

// Stage q of segment s: its first vector inside the channel and its length.
__device__ __forceinline__ void stage_of(const FShared& sh, const FArgs& a, int s, int q,
                                         int& rv0, int& len) {
  const int off = q * a.stage_v;
  rv0 = sh.seg_rv0[s] + off;
  len = min(a.stage_v, sh.seg_len[s] - off);
}

__device__ __forceinline__ int stages_in(const FShared& sh, const FArgs& a, int s) {
  return (sh.seg_len[s] + a.stage_v - 1) / a.stage_v;
}

// Ring slots walked forward and backward without a division per stage.
__device__ __forceinline__ int slot_next(int s, int NS) { return s + 1 == NS ? 0 : s + 1; }
__device__ __forceinline__ int slot_prev(int s, int NS) { return s == 0 ? NS - 1 : s - 1; }


// Stage j (phase-1 numbering) of CTA v's range: its channel c, first vector
// rv0 inside the channel, length and segment index -- the segments computed
// the way the kernel's set-up computes its own.
__device__ bool range_stage(const FArgs& a, int v, int j, int& c, int& rv0, int& len, int& seg) {
  const int64_t e0 = (int64_t)v * a.Wv;
  const int64_t e1 = min(e0 + a.Wv, a.C * (int64_t)a.Mv);
  int sg = 0;
  for (int64_t e = e0; e < e1 && sg < kFMaxSegs; ++sg) {
    const int64_t cc = e / a.Mv;
    const int64_t cend = min((cc + 1) * (int64_t)a.Mv, e1);
    const int slen = (int)(cend - e);
    const int nq = (slen + a.stage_v - 1) / a.stage_v;
    if (j < nq) {
      c = (int)cc;
      rv0 = (int)(e - cc * a.Mv) + j * a.stage_v;
      len = min(a.stage_v, slen - j * a.stage_v);
      seg = sg;
      return true;
    }
    j -= nq;
    e = cend;
  }
  return false;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ld_relaxed_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// ------------------------------------------------------------- producer --

// Bulk copies of one stage (plane runs of channel c) into `slot`, issued by
// the whole producer warp: lane l copies runs l, l + 32, ... (one per plane
// the stage touches), so the per-copy address arithmetic runs in parallel.
template <typename T, bool BWD>
__device__ void issue_stage(const FArgs& a, FShared& sh, unsigned char* ring, int slot, int c,
                            int rv0, int len, uint64_t policy) {
  constexpr int VEC = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const uint32_t in_bytes = (uint32_t)a.stage_v * 16u;
  unsigned char* d0 = ring + (size_t)slot * (BWD ? 2u : 1u) * in_bytes;
  uint64_t* bar = &sh.full[slot];
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)len * 16u * (BWD ? 2u : 1u));
    sh.issued[slot] += 1;
  }
  __syncwarp();
  const int n0 = (int)fast_div((uint32_t)rv0, a.pdiv);
  const int nruns = (int)fast_div((uint32_t)(rv0 + len - 1), a.pdiv) - n0 + 1;
  for (int r = lane; r < nruns; r += 32) {
    const int n = n0 + r;
    const int b = max(rv0, n * a.Pv), e = min(rv0 + len, (n + 1) * a.Pv);
    const int64_t gvo = ((int64_t)n * a.C + c) * a.Pv + (b - n * a.Pv);
    const uint32_t bytes = (uint32_t)(e - b) * 16u;
    unsigned char* dst = d0 + (size_t)(b - rv0) * 16;
    bulk_g2s_hint(dst, static_cast<const T*>(a.x) + gvo * VEC, bytes, bar, policy);
    if (BWD)
      bulk_g2s_hint(dst + in_bytes, static_cast<const T*>(a.dy) + gvo * VEC, bytes, bar, policy);
  }
}

// Warp-uniform wait of the producer warp for a slot's release.
__device__ __forceinline__ bool producer_wait_empty(FShared& sh, int slot, uint32_t& epar,
                                                    int* status) {
  bool ok = wait_or_abort(&sh.empty[slot], (epar >> slot) & 1u, &sh.abort);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) {
    if ((threadIdx.x & 31) == 0) set_abort(sh, status);
    return false;
  }
  epar ^= 1u << slot;
  fence_proxy_async_smem();
  return true;
}

// The producer warp (all 32 lanes).  L2 policy of the loads: phase 2 reads
// the resident tail from shared memory, then the TMEM stages before it, and
// reloads the rest: the l2_window stages before those (which phase 1 loaded
// at normal priority, so they are likely still in L2) and the stages before
// the window from DRAM -- the window first in the forward, last in the
// backward; every other load is marked evict-first so that it does not
// displace that window.
template <typename T, bool BWD>
__device__ void producer(const FArgs& a, FShared& sh, unsigned char* ring) {
  const int NS = a.nstage, N1 = sh.nst;
  const uint64_t keep = l2_policy_evict_normal(), drop = l2_policy_evict_first();
  const int keep_lo = sh.t_lo - a.l2_window, keep_hi = sh.t_lo;  // phase-1 stages kept in L2
  uint32_t epar = 0;  // parity of the next "empty" completion per slot
  // Phase 1: forward.  A slot is refilled once its previous stage is released.
  int i = 0, slot = 0;  // slot = i mod NS
  for (int s = 0; s < sh.nseg; ++s) {
    const int nq = stages_in(sh, a, s);
    for (int q = 0; q < nq; ++q, ++i, slot = slot_next(slot, NS)) {
      if (i >= NS && !producer_wait_empty(sh, slot, epar, a.status)) return;
      if (__any_sync(0xffffffffu, sh.abort != 0)) return;
      int rv0, len;
      stage_of(sh, a, s, q, rv0, len);
      issue_stage<T, BWD>(a, sh, ring, slot, sh.seg_c[s], rv0, len,
                          (i >= keep_lo && i < keep_hi) ? keep : drop);
    }
  }
  // Phase 2.  The consumers first work through the resident tail and the
  // TMEM stages, which need no loads; everything else goes through the
  // slots they free, push j into slot (N1 - 1 - j) mod NS, each with a
  // descriptor: this CTA's stages from t_lo - 1 down to its pool, then the
  // pool stages it still claims (from the top), then stages it claims from
  // other CTAs' pools (from the bottom), then an end marker.  A pool word
  // holds the unclaimed pool stages [lo, hi) as hi << 16 | lo: the owner
  // takes hi - 1 by subtracting 1 << 16, another CTA takes lo by adding 1,
  // and the atomic order decides every stage exactly once.
  const int lane = threadIdx.x & 31;
  int j = 0, pslot = (N1 - 1) % NS;  // pslot = (N1 - 1 - j) mod NS
  auto push = [&](int c, int rv0, int len, const float* par, bool end) -> bool {
    const int slot = pslot;
    if (sh.issued[slot] > 0 && !producer_wait_empty(sh, slot, epar, a.status)) return false;
    if (__any_sync(0xffffffffu, sh.abort != 0)) return false;
    if (lane == 0) {
      FDesc& d = sh.desc[slot];
      d.c = c;
      d.rv0 = rv0;
      d.len = len;
      d.end = end ? 1 : 0;
      for (int f = 0; f < 6; ++f) d.par[f] = end ? 0.f : par[f];
    }
    __syncwarp();
    if (end) {
      if (lane == 0) {
        sh.issued[slot] += 1;
        mbar_arrive(&sh.full[slot]);
      }
      __syncwarp();
    } else {
      issue_stage<T, BWD>(a, sh, ring, slot, c, rv0, len, drop);
    }
    ++j;
    pslot = slot_prev(pslot, NS);
    return true;
  };
  // this CTA's stages below the on-chip ones, down to the pool: the stages
  // with phase-1 index in [lo, hi), from the top down
  auto push_range = [&](int lo, int hi) -> bool {
    int q2 = 0;
    for (int s = sh.nseg - 1; s >= 0; --s) {
      const int nq = stages_in(sh, a, s);
      for (int q = nq - 1; q >= 0; --q, ++q2) {
        const int i2 = N1 - 1 - q2;
        if (i2 >= hi || i2 < lo) continue;
        int rv0, len;
        stage_of(sh, a, s, q, rv0, len);
        if (!push(sh.seg_c[s], rv0, len, sh.seg_par[s], false)) return false;
      }
    }
    return true;
  };
  if constexpr (BWD) {
    // Backward: the stages that come from DRAM again first, so that their
    // loads overlap the consumers' on-chip stages, then the L2 window (its
    // lines have normal priority while every other load and store of the
    // kernel is evict-first, so they are still hits at the end); measured
    // 163.7 -> 162.2 us at bf16 [128,256,56,56], outputs bit-identical.  The
    // forward, with half the re-read, was no faster that way.
    const int wlo = max(sh.pool, keep_lo);
    if (!push_range(sh.pool, wlo)) return;
    if (!push_range(wlo, sh.t_lo)) return;
  } else {
    if (!push_range(sh.pool, sh.t_lo)) return;
  }
  // this CTA's pool stages that no other CTA has taken
  for (int left = sh.pool; left > 0; --left) {
    uint32_t old = 0;
    if (lane == 0) old = atomicSub(a.steal + blockIdx.x, 1u << 16);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int hi = (int)(old >> 16), lo = (int)(old & 0xffffu);
    if (hi <= lo) break;
    int rem = hi - 1, s = 0;
    while (s < sh.nseg - 1 && rem >= stages_in(sh, a, s)) rem -= stages_in(sh, a, s++);
    int rv0, len;
    stage_of(sh, a, s, rem, rv0, len);
    if (!push(sh.seg_c[s], rv0, len, sh.seg_par[s], false)) return;
  }
  // stages from the pools of other CTAs: the one with the most left first
  // (once this CTA's consumers have finalized: sh.target is set by then)
  bool ready = a.pool > 0;
  if (ready) {
    const uint64_t t0 = global_timer_ns();
    while (!sh.p2ready && !sh.abort) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        ready = false;
        break;
      }
    }
    ready = __all_sync(0xffffffffu, ready && !sh.abort);
  }
  // A claim takes up to kStealBatch stages at once; a CTA keeps claiming
  // from the same owner until that pool is empty, and keeps the owner's
  // parameters of the last segment it read.
  int victim = -1, pv_seg = -1;
  float par[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int scan = 0; scan < kStealScans && ready; ++scan) {
    if (victim < 0) {
      // Owners with at least half the largest number of unclaimed pool
      // stages qualify; each CTA takes the first of them after itself in
      // block order, so that the CTAs spread over the owners instead of all
      // contending for the one with the most left.
      constexpr int kWordsPerLane = (kMaxCtas + 31) / 32;
      int rem[kWordsPerLane];
      int rmax = 0;
#pragma unroll
      for (int u = 0; u < kWordsPerLane; ++u) {
        const int v = lane + 32 * u;
        rem[u] = 0;
        if (v < a.G && v != (int)blockIdx.x) {
          const uint32_t w = ld_relaxed_u32(a.steal + v);
          rem[u] = (int)(w >> 16) - (int)(w & 0xffffu);
        }
        rmax = max(rmax, rem[u]);
      }
      for (int o = 16; o > 0; o >>= 1) rmax = max(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
      if (rmax <= 0) break;
      const int thr = max(1, rmax / 2);
      int bd = a.G, best = -1;  // rotated distance from this CTA, and the owner
#pragma unroll
      for (int u = 0; u < kWordsPerLane; ++u) {
        const int v = lane + 32 * u;
        const int d = (v - (int)blockIdx.x + a.G) % a.G;
        if (rem[u] >= thr && d < bd) {
          bd = d;
          best = v;
        }
      }
      for (int o = 16; o > 0; o >>= 1) {
        const int d2 = __shfl_xor_sync(0xffffffffu, bd, o);
        const int b2 = __shfl_xor_sync(0xffffffffu, best, o);
        if (d2 < bd) {
          bd = d2;
          best = b2;
        }
      }
      if (best < 0) break;
      // the owner's parameters must be published before its pool is used
      int ok = 0;
      if (lane == 0) ok = ld_acquire_u64(a.pubflag + best) == sh.target;
      if (!__shfl_sync(0xffffffffu, ok, 0)) continue;
      victim = best;
      pv_seg = -1;
    }
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(a.steal + victim, (uint32_t)kStealBatch);
    old = __shfl_sync(0xffffffffu, old, 0);
    const int lo = (int)(old & 0xffffu), hi = (int)(old >> 16);
    if (lo >= hi) {
      victim = -1;
      continue;
    }
    for (int g = lo; g < min(lo + kStealBatch, hi); ++g) {
      int c = 0, rv0 = 0, len = 0, sg = 0;
      if (!range_stage(a, victim, g, c, rv0, len, sg) || sg >= kPoolMax) {
        // cannot happen for a consistent pool word
        if (lane == 0) set_abort(sh, a.status);
        return;
      }
      if (sg != pv_seg) {
        if (lane == 0) {
          const float* src = a.pub + ((int64_t)victim * kPoolMax + sg) * kPubFloats;
          for (int f = 0; f < 6; ++f) par[f] = ld_relaxed_f32(src + f);
        }
        pv_seg = sg;
      }
      if (!push(c, rv0, len, par, false)) return;
    }
  }
  push(0, 0, 0, nullptr, true);
}

// ------------------------------------------------------------ consumers --

// Phase-1 accumulation of one 16-byte vector.  Forward: sum d (d = x - shift)
// in double-fp32 so that the channel's sum d is exact to double-fp32
// precision (the backward's sum dy*(x - mean) relies on it: a constant dy
// must give 0): per element, with the rounding error of x - shift for fp32
// input; for bf16 input, per thread and stage when that is exact (below),
// else per element.  Sum d^2 in fp32 over the vector's lanes (fp32 input)
// or over the thread's vectors of the stage (bf16 input), then one
// double-fp32 add (its rounding enters the variance only relatively).
// Backward: sum dy*d per element in double-fp32 with each product's exact
// residual and, for fp32 input, the rounding error of x - shift; sum dy
// likewise for fp32, while ungated bf16 dy is first summed over the
// vector's four elements per lane in fp32 -- exact for 8-bit significands
// within 14 binades of each other -- and then added in double-fp32 once per
// vector.
//
// The bf16 sum per thread and stage: when the exponents of the thread's x
// in the stage and of shift lie in E_min .. E_max, every value is a
// multiple of Q = 2^(E_min - 7) below 2^(E_max + 1) in magnitude, so each
// d = x - shift is a multiple of Q below 2^(E_max + 2), and a partial sum
// of at most n of them is a multiple of Q below n 2^(E_max + 2).  With
// E_max - E_min <= 15 - ceil(log2 n) that is at most 2^24 Q: every fp32
// partial sum is exact, in any order.  n counts the terms of one lane (four
// per vector).  The magnitudes' largest and smallest come from the bf16x2
// max / min instructions over the stage, and only then is the sum added in
// double-fp32; a stage that fails the test (zeros, subnormals, a wide
// range) re-reads its vectors from the ring slot and sums per element.
// smag holds shift's bf16 magnitude bits in both halves.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// fp32 forward, one vector (bf16 input sums per stage: FwdStage below).
__device__ __forceinline__ void fwd_acc(uint4 r, f2 sh2, f2 nsh2, DF2 (&a1)[2], DF2& a2) {
  constexpr int NP = Pairs16<float>::NP;
  f2 p[NP], d[NP];
  Pairs16<float>::get(r, p);
  f2 l2 = 0ull;
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    d[k] = f2_sub(p[k], sh2);
    l2 = f2_fma(d[k], d[k], l2);
  }
  df2_add(a2, l2);
  // alternate pairs feed two accumulators (two dependency chains), each
  // with the rounding error of x - shift
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    DF2& acc = a1[k & 1];
    df2_add(acc, d[k]);
    const f2 bb = f2_sub(d[k], p[k]);
    acc.lo = f2_add(acc.lo, f2_add(f2_sub(p[k], f2_sub(d[k], bb)), f2_sub(nsh2, bb)));
  }
}

// bf16 forward: one thread's sums over its vectors of one stage.
struct FwdStage {
  f2 s0, s1;         // sum d, two chains
  f2 q0, q1;         // sum d^2, two chains
  uint32_t hi, lo;   // largest / smallest bf16 magnitude seen, per half
};

__device__ __forceinline__ void fwd_stage_begin(FwdStage& f, uint32_t smag) {
  f.s0 = f.s1 = f.q0 = f.q1 = 0ull;
  f.hi = f.lo = smag;
}

__device__ __forceinline__ void fwd_stage_vec(FwdStage& f, uint4 r, f2 sh2) {
  f2 p[4];
  Pairs16<bf16>::get(r, p);
  const f2 d0 = f2_sub(p[0], sh2), d1 = f2_sub(p[1], sh2);
  const f2 d2 = f2_sub(p[2], sh2), d3 = f2_sub(p[3], sh2);
  f.s0 = f2_add(f.s0, f2_add(d0, d1));
  f.s1 = f2_add(f.s1, f2_add(d2, d3));
  f.q0 = f2_fma(d0, d0, f.q0);
  f.q1 = f2_fma(d1, d1, f.q1);
  f.q0 = f2_fma(d2, d2, f.q0);
  f.q1 = f2_fma(d3, d3, f.q1);
  const uint32_t k7 = 0x7fff7fffu;
  const uint32_t m0 = r.x & k7, m1 = r.y & k7, m2 = r.z & k7, m3 = r.w & k7;
  f.hi = bf16x2_max(f.hi, bf16x2_max(bf16x2_max(m0, m1), bf16x2_max(m2, m3)));
  f.lo = bf16x2_min(f.lo, bf16x2_min(bf16x2_min(m0, m1), bf16x2_min(m2, m3)));
}

// Whether the stage's fp32 sums of d are exact: the exponent span of the
// magnitudes (both halves folded) at most span7 >> 7, no zero or subnormal.
__device__ __forceinline__ bool fwd_stage_exact(const FwdStage& f, uint32_t span7) {
  const uint32_t hi = bf16x2_max(f.hi, __byte_perm(f.hi, 0u, 0x1032));
  const uint32_t lo = bf16x2_min(f.lo, __byte_perm(f.lo, 0u, 0x1032));
  const uint32_t emax = hi & 0x7f80u, emin = lo & 0x7f80u;
  return emin != 0u && emax - emin <= span7;
}

// Per-element double-fp32 sum of one bf16 vector's d (the stage fallback).
__device__ __forceinline__ void fwd_sum_elems(uint4 r, f2 sh2, DF2 (&a1)[2]) {
  f2 p[4];
  Pairs16<bf16>::get(r, p);
#pragma unroll
  for (int k = 0; k < 4; ++k) df2_add(a1[k & 1], f2_sub(p[k], sh2));
}

// With an activation (ACT), dy is first gated by d act / d pre with
// pre = ((x - shift) - mean_d)*scale + beta, the forward's expression.
struct ActPar {
  f2 md2, sc2, be2;
  int act;
  float slope;
};

// ACT: GBN_ACT_* at compile time.  A ReLU gate (0 or 1) keeps bf16 dy
// exact, so its per-vector sum stays exact too; a LeakyReLU gate rounds.
template <typename T, int ACT>
__device__ __forceinline__ void bwd_acc(uint4 rx, uint4 rd, f2 sh2, f2 nsh2, const ActPar& ap,
                                        DF2& a0, DF2 (&a1)[2]) {
  constexpr int NP = Pairs16<T>::NP;
  f2 px[NP], pd[NP];
  Pairs16<T>::get(rx, px);
  Pairs16<T>::get(rd, pd);
  constexpr bool kLocalDy = sizeof(T) == 2 && ACT != GBN_ACT_LEAKY_RELU;
  f2 l0 = 0ull;
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const f2 d = f2_sub(px[k], sh2);
    if constexpr (ACT != GBN_ACT_NONE) {
      const float2 pre = f2_unpack(f2_fma(f2_sub(d, ap.md2), ap.sc2, ap.be2));
      pd[k] = f2_mul_rounded(pd[k], f2_pack(act_gate(pre.x, ACT, ap.slope),
                                            act_gate(pre.y, ACT, ap.slope)));
    }
    if constexpr (kLocalDy)
      l0 = f2_add(l0, pd[k]);
    else
      df2_add(a0, pd[k]);
    // alternate pairs feed two accumulators: two independent dependency
    // chains per thread
    DF2& acc = a1[k & 1];
    const f2 prod = f2_mul_rounded(pd[k], d);
    df2_add(acc, prod);
    // exact residual dy*d - prod (the negation flips the sign of both lanes)
    acc.lo = f2_add(acc.lo, f2_fma(pd[k], d, prod ^ 0x8000000080000000ull));
    if constexpr (sizeof(T) == 4) {
      const f2 bb = f2_sub(d, px[k]);
      const f2 d_lo = f2_add(f2_sub(px[k], f2_sub(d, bb)), f2_sub(nsh2, bb));
      acc.lo = f2_fma(pd[k], d_lo, acc.lo);
    }
  }
  if constexpr (kLocalDy) df2_add(a0, l0);
}

// Sum two (hi, lo) pairs over the consumer warps in a fixed tree; the result
// is valid in consumer warp 0.  Contains two consumer barriers.
__device__ __forceinline__ void consumers_sum2(FShared& sh, DF& a, DF& b) {
  const int ct = threadIdx.x - 32, lane = ct & 31, cw = ct >> 5;
  a = warp_sum_df(a);
  b = warp_sum_df(b);
  if (lane == 0) {
    sh.red[0][cw] = make_float2(a.hi, a.lo);
    sh.red[1][cw] = make_float2(b.hi, b.lo);
  }
  __syncwarp();
  consumers_sync();
  if (cw == 0) {
    const float2 u = lane < kFConsumerWarps ? sh.red[0][lane] : make_float2(0.f, 0.f);
    const float2 w = lane < kFConsumerWarps ? sh.red[1][lane] : make_float2(0.f, 0.f);
    a = warp_sum_df(DF{u.x, u.y});
    b = warp_sum_df(DF{w.x, w.y});
  }
  __syncwarp();
  consumers_sync();
}

template <typename T, bool BWD>
__device__ void consumer_phase1(const FArgs& a, FShared& sh, const unsigned char* ring,
                                uint32_t& fpar) {
  const int ct = threadIdx.x - 32, lane = ct & 31;
  const int NS = a.nstage, N1 = sh.nst;
  const uint32_t in_bytes = (uint32_t)a.stage_v * 16u;
  // TMEM stages: KV vector slots per thread and input, cps columns a stage.
  const int KV = a.stage_v / kFConsumers, cps = KV * (BWD ? 8 : 4);
  const uint32_t tbase = tmem_thread_base(sh.tmem, ct >> 5);
  // bf16 forward: exponent span (times 128) for which a lane's fp32 sum of
  // its n = 4 KV terms of a stage is exact, 15 - ceil(log2 n); none if < 0.
  constexpr bool kStageSum = !BWD && sizeof(T) == 2;
  const int span = 15 - (32 - __clz(4 * KV - 1));
  const uint32_t span7 = span >= 0 ? (uint32_t)span << 7 : 0u;
  const bool span_ok = span >= 0;
  int i = 0, slot = 0;  // slot = i mod NS
  for (int s = 0; s < sh.nseg; ++s) {
    const float shift = sh.seg_par[s][0];
    const f2 sh2 = f2_splat(shift), nsh2 = f2_splat(-shift);
    // shift's bf16 magnitude bits (shift is a bf16 value for bf16 input)
    const uint32_t sm16 = (__float_as_uint(shift) >> 16) & 0x7fffu;
    const uint32_t smag = sm16 | (sm16 << 16);
    ActPar ap;
    ap.md2 = f2_splat(sh.seg_par[s][1]);
    ap.sc2 = f2_splat(sh.seg_par[s][2]);
    ap.be2 = f2_splat(sh.seg_par[s][5]);
    ap.act = a.act;
    ap.slope = a.slope;
    DF2 a0{0ull, 0ull}, a1[2] = {{0ull, 0ull}, {0ull, 0ull}};  // see the fold below
    const int nq = stages_in(sh, a, s);
    for (int q = 0; q < nq; ++q, ++i, slot = slot_next(slot, NS)) {
      if (!warp_wait_full(sh, slot, fpar, a.status)) continue;
      if (i == 0 && ct == 0) GBN_RING_TRACE(1);
      int rv0, len;
      stage_of(sh, a, s, q, rv0, len);
      const unsigned char* st = ring + (size_t)slot * (BWD ? 2u : 1u) * in_bytes;
      if constexpr (kStageSum) {
        FwdStage f;
        fwd_stage_begin(f, smag);
        if (KV == kKVFwd && i + NS < N1) {
          // A stage that phase 1 refills: this thread's vectors into
          // registers and the slot released before the copies to TMEM (for
          // a TMEM stage) and the sums, so that the refill starts sooner.
          uint4 rx[kKVFwd];
#pragma unroll
          for (int k = 0; k < kKVFwd; ++k)
            rx[k] = *reinterpret_cast<const uint4*>(st + (size_t)(ct + k * kFConsumers) * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.empty[slot]);
          if (i >= sh.t_lo && i < sh.t_hi) {
            uint32_t ta = tbase + (uint32_t)((i - sh.t_lo) * cps);
#pragma unroll
            for (int k = 0; k < kKVFwd; ++k, ta += 4u) tmem_st16(ta, rx[k]);
          }
#pragma unroll
          for (int k = 0; k < kKVFwd; ++k)
            if (ct + k * kFConsumers < len) fwd_stage_vec(f, rx[k], sh2);
          df2_add(a0, f2_add(f.q0, f.q1));
          if (span_ok && fwd_stage_exact(f, span7)) {
            df2_add(a1[0], f2_add(f.s0, f.s1));
          } else {
#pragma unroll
            for (int k = 0; k < kKVFwd; ++k)
              if (ct + k * kFConsumers < len) fwd_sum_elems(rx[k], sh2, a1);
          }
          continue;
        }
        if (i >= sh.t_lo && i < sh.t_hi) {
          // a TMEM stage (see below): every slot copied, the valid ones summed
          uint32_t ta = tbase + (uint32_t)((i - sh.t_lo) * cps);
          for (int k = 0; k < KV; ++k, ta += 4u) {
            const int v = ct + k * kFConsumers;
            const uint4 rx = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
            tmem_st16(ta, rx);
            if (v < len) fwd_stage_vec(f, rx, sh2);
          }
        } else {
          for (int v = ct; v < len; v += kFConsumers)
            fwd_stage_vec(f, *reinterpret_cast<const uint4*>(st + (size_t)v * 16), sh2);
        }
        df2_add(a0, f2_add(f.q0, f.q1));
        if (span_ok && fwd_stage_exact(f, span7)) {
          df2_add(a1[0], f2_add(f.s0, f.s1));
        } else {
          for (int v = ct; v < len; v += kFConsumers)
            fwd_sum_elems(*reinterpret_cast<const uint4*>(st + (size_t)v * 16), sh2, a1);
        }
      } else if (BWD && KV == kKVBwd && i + NS < N1) {
        // Backward, a stage that phase 1 refills: as above, every vector
        // pair of this thread into registers and the slot released first.
        uint4 rx[kKVBwd], rd[kKVBwd];
#pragma unroll
        for (int k = 0; k < kKVBwd; ++k) {
          const int v = ct + k * kFConsumers;
          rx[k] = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
          rd[k] = *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
        if (i >= sh.t_lo && i < sh.t_hi) {
          uint32_t ta = tbase + (uint32_t)((i - sh.t_lo) * cps);
#pragma unroll
          for (int k = 0; k < kKVBwd; ++k, ta += 8u) {
            tmem_st16(ta, rx[k]);
            tmem_st16(ta + 4u, rd[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < kKVBwd; ++k) {
          if (ct + k * kFConsumers >= len) continue;
          if (a.act == GBN_ACT_NONE)
            bwd_acc<T, GBN_ACT_NONE>(rx[k], rd[k], sh2, nsh2, ap, a0, a1);
          else if (a.act == GBN_ACT_RELU)
            bwd_acc<T, GBN_ACT_RELU>(rx[k], rd[k], sh2, nsh2, ap, a0, a1);
          else
            bwd_acc<T, GBN_ACT_LEAKY_RELU>(rx[k], rd[k], sh2, nsh2, ap, a0, a1);
        }
        continue;
      } else if (i >= sh.t_lo && i < sh.t_hi) {
        // A TMEM stage: every lane copies all its vector slots of the stage
        // (the tcgen05 copies are warp-wide; a slot past len holds stale
        // ring bytes that phase 2 never uses) and sums the valid ones.
        uint32_t ta = tbase + (uint32_t)((i - sh.t_lo) * cps);
        for (int k = 0; k < KV; ++k, ta += (BWD ? 8u : 4u)) {
          const int v = ct + k * kFConsumers;
          const uint4 rx = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
          tmem_st16(ta, rx);
          if constexpr (!BWD) {
            if (v < len) fwd_acc(rx, sh2, nsh2, a1, a0);
          } else {
            const uint4 rd = *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16);
            tmem_st16(ta + 4u, rd);
            if (v < len) {
              if (a.act == GBN_ACT_NONE)
                bwd_acc<T, GBN_ACT_NONE>(rx, rd, sh2, nsh2, ap, a0, a1);
              else if (a.act == GBN_ACT_RELU)
                bwd_acc<T, GBN_ACT_RELU>(rx, rd, sh2, nsh2, ap, a0, a1);
              else
                bwd_acc<T, GBN_ACT_LEAKY_RELU>(rx, rd, sh2, nsh2, ap, a0, a1);
            }
          }
        }
      } else if constexpr (!BWD) {
        for (int v = ct; v < len; v += kFConsumers)
          fwd_acc(*reinterpret_cast<const uint4*>(st + (size_t)v * 16), sh2, nsh2, a1, a0);
      } else if (a.act == GBN_ACT_NONE) {
        for (int v = ct; v < len; v += kFConsumers)
          bwd_acc<T, GBN_ACT_NONE>(*reinterpret_cast<const uint4*>(st + (size_t)v * 16),
                                   *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16),
                                   sh2, nsh2, ap, a0, a1);
      } else if (a.act == GBN_ACT_RELU) {
        for (int v = ct; v < len; v += kFConsumers)
          bwd_acc<T, GBN_ACT_RELU>(*reinterpret_cast<const uint4*>(st + (size_t)v * 16),
                                   *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16),
                                   sh2, nsh2, ap, a0, a1);
      } else {
        for (int v = ct; v < len; v += kFConsumers)
          bwd_acc<T, GBN_ACT_LEAKY_RELU>(
              *reinterpret_cast<const uint4*>(st + (size_t)v * 16),
              *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16), sh2, nsh2, ap,
              a0, a1);
      }
      // Release the slot only if phase 1 refills it; the last NS stages stay
      // resident for phase 2.
      if (i + NS < N1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
      }
    }
    // forward: a1 holds sum d, a0 sum d^2; backward: a0 sum dy, a1 sum dy*d
    const DF sa = df_sum(df2_fold(a1[0]), df2_fold(a1[1]));
    DF s0 = BWD ? df2_fold(a0) : sa, s1 = BWD ? sa : df2_fold(a0);
    consumers_sum2(sh, s0, s1);
    if (ct == 0 && !sh.abort) {
      const int j = (int)blockIdx.x - sh.seg_klo[s];
      const int c = sh.seg_c[s];
      a.part[(int64_t)j * a.C + c] = make_float2(s0.hi, s0.lo);
      a.part[((int64_t)a.grid_y + j) * a.C + c] = make_float2(s1.hi, s1.lo);
    }
    __syncwarp();
  }
  // The TMEM copies complete before phase 2 reads them back.
  if (sh.t_hi > sh.t_lo) tmem_wait_st();
  // Publish: every partial of this CTA was written by this thread above.
  if (ct == 0 && !sh.abort) {
    unsigned long long* f = a.sync + 2 + 2 * (int64_t)blockIdx.x;
    __threadfence();
    st_relaxed_u64(f + 1, ~sh.target);
    st_release_u64(f, sh.target);
    GBN_RING_TRACE(2);
  }
  __syncwarp();
}

// Channel finalize for segment s by one consumer warp.
template <bool BWD>
__device__ void finalize_segment(const FArgs& a, FShared& sh, int s) {
  const int lane = (threadIdx.x - 32) & 31;
  const int c = sh.seg_c[s], klo = sh.seg_klo[s], n = sh.seg_khi[s] - klo + 1;
  DF p0{0.f, 0.f}, p1{0.f, 0.f};
  bool ok = true;
  for (int jj = lane; jj < n; jj += 32) {
    // Slot jj was written by CTA klo + jj; this lane acquires that CTA's flag
    // and then reads the slot itself.
    ok = ok && wait_flag(a.sync + 2 + 2 * (int64_t)(klo + jj), sh.target);
    if (ok) {
      const float2 u = ld_relaxed_f2(a.part + (int64_t)jj * a.C + c);
      const float2 w = ld_relaxed_f2(a.part + ((int64_t)a.grid_y + jj) * a.C + c);
      p0 = df_sum(p0, DF{u.x, u.y});
      p1 = df_sum(p1, DF{w.x, w.y});
    }
  }
  if (!__all_sync(0xffffffffu, ok)) {
    if (lane == 0) set_abort(sh, a.status);
    return;
  }
  p0 = warp_sum_df(p0);
  p1 = warp_sum_df(p1);
  const bool owner = (klo == (int)blockIdx.x);  // holds the channel's first element
  const float M = a.Mh + a.Ml;
  if constexpr (!BWD) {
    const BnFwdFinal f = bn_fwd_final(p0, p1, a.Mh, a.Ml, a.gamma ? a.gamma[c] : 1.f, a.eps);
    if (lane == 0) {
      sh.seg_par[s][1] = f.md.hi;
      sh.seg_par[s][2] = f.scale;
      sh.seg_par[s][3] = a.beta ? a.beta[c] : 0.f;
      if (owner)
        bn_fwd_write(f, sh.seg_par[s][0], a.C, c, M, a.stats, a.running_mean, a.running_var,
                     a.momentum);
    }
  } else {
    const int64_t C = a.C;
    const DF md{a.stats[6 * C + c], a.stats[7 * C + c]};
    const BnBwdFinal f = bn_bwd_final(p0, p1, md, a.stats[2 * C + c], sh.seg_par[s][2], M);
    if (lane == 0) {
      sh.seg_par[s][3] = f.k1;
      sh.seg_par[s][4] = f.k2;
      if (owner) {
        a.grads[c] = f.dgamma;
        a.grads[C + c] = f.dbeta;
        a.grads[2 * C + c] = f.k1;
        a.grads[3 * C + c] = f.k2;
      }
    }
  }
  __syncwarp();
}

// Outputs of one phase-2 stage (channel c, vectors [rv0, rv0 + len) of the
// channel, parameters par as seg_par) from ring slot st, or from TMEM at ta0
// when in_tmem.  A TMEM stage runs all KV slots on every lane (the TMEM
// loads are warp-wide); only slots v < len are computed and stored.  ACT is
// the activation (GBN_ACT_*) as a compile-time switch, so that the plain
// pass carries no per-element test.
template <typename T, bool BWD, int ACT>
__device__ __forceinline__ void stage_out(const FArgs& a, int c, int rv0, int len,
                                          const float* par, const unsigned char* st,
                                          uint32_t in_bytes, bool in_tmem, uint32_t ta0, int KV) {
  constexpr int VEC = 16 / sizeof(T);
  using V = Vec<T, VEC>;
  const int ct = threadIdx.x - 32;
  const float shift = par[0], mean_d = par[1], scale = par[2];
  const float p3 = par[3], p4 = par[4], beta = par[5];
  const float slope = a.slope;
  const f2 sh2 = f2_splat(shift), md2 = f2_splat(mean_d), sc2 = f2_splat(scale);
  const f2 p32 = f2_splat(p3), p42 = f2_splat(p4);
  T* out = static_cast<T*>(a.out);
  // Output position of vector v = ct, ct + 512, ...: plane n, in-plane pv,
  // and the vector offset gvo = (n*C + c)*Pv + pv, advanced per step.
  const int rv = rv0 + ct;
  const int n0 = (int)fast_div((uint32_t)rv, a.pdiv);
  int pv = rv - n0 * a.Pv;
  int64_t gvo = ((int64_t)n0 * a.C + c) * a.Pv + pv;
  // One output vector from its raw 16 bytes of x (and dy).
  auto emit = [&](uint4 rx, uint4 rd) {
    if constexpr (ACT == GBN_ACT_NONE) {
      // two elements per instruction (fp32x2), the same roundings as the
      // scalar form below
      using PK = Pairs16<T>;
      f2 px[PK::NP];
      PK::get(rx, px);
      if constexpr (!BWD) {
#pragma unroll
        for (int k = 0; k < PK::NP; ++k)
          px[k] = f2_fma(f2_sub(f2_sub(px[k], sh2), md2), sc2, p32);
      } else {
        f2 pg[PK::NP];
        PK::get(rd, pg);
#pragma unroll
        for (int k = 0; k < PK::NP; ++k)
          px[k] = f2_fma(pg[k], sc2, f2_fma(f2_sub(f2_sub(px[k], sh2), md2), p32, p42));
      }
      const uint4 w = PK::put(px);
      if (a.stream_out)
        __stcs(reinterpret_cast<uint4*>(out + gvo * VEC), w);
      else
        *reinterpret_cast<uint4*>(out + gvo * VEC) = w;
    } else {
      float e[VEC];
      V::cvt(rx, e);
      if constexpr (!BWD) {
#pragma unroll
        for (int k = 0; k < VEC; ++k)
          e[k] = act_out(fmaf((e[k] - shift) - mean_d, scale, p3), ACT, slope);
      } else {
        float g[VEC];
        V::cvt(rd, g);
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const float xc = (e[k] - shift) - mean_d;
          const float gk = ACT == GBN_ACT_NONE
                               ? g[k]
                               : __fmul_rn(g[k], act_gate(fmaf(xc, scale, beta), ACT, slope));
          e[k] = fmaf(gk, scale, fmaf(xc, p3, p4));
        }
      }
      if (a.stream_out)
        store16_cs(out + gvo * VEC, e);
      else
        V::store(out + gvo * VEC, e);
    }
  };
  auto step = [&]() {
    pv += a.dp;
    gvo += a.ostep;
    if (pv >= a.Pv) {
      pv -= a.Pv;
      gvo += a.owrap;
    }
  };
  // A TMEM stage of the device's usual size: all 24 of the thread's columns
  // in two loads and one wait (instead of a wait per vector).
  constexpr int KVT = BWD ? 3 : 6;  // vectors per thread, 24 columns
  if (in_tmem && KV == KVT) {
    uint32_t r[24];
    tmem_ld24(ta0, r);
#pragma unroll
    for (int u = 0; u < KVT; ++u) {
      const int v = ct + u * kFConsumers;
      const int o = BWD ? 8 * u : 4 * u;
      const uint4 rx = make_uint4(r[o], r[o + 1], r[o + 2], r[o + 3]);
      const uint4 rd = BWD ? make_uint4(r[o + 4], r[o + 5], r[o + 6], r[o + 7])
                           : make_uint4(0u, 0u, 0u, 0u);
      if (v < len) emit(rx, rd);
      step();
    }
    return;
  }
  for (int u = 0; u < KV; ++u) {
    const int v = ct + u * kFConsumers;
    if (!in_tmem && v >= len) break;
    uint4 rx, rd = make_uint4(0u, 0u, 0u, 0u);
    if (in_tmem) {
      if constexpr (BWD)
        tmem_ld16x2(ta0 + (uint32_t)u * 8u, ta0 + (uint32_t)u * 8u + 4u, rx, rd);
      else
        rx = tmem_ld16(ta0 + (uint32_t)u * 4u);
    } else {
      rx = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
      if constexpr (BWD) rd = *reinterpret_cast<const uint4*>(st + in_bytes + (size_t)v * 16);
    }
    if (v < len) emit(rx, rd);
    step();
  }
}

template <typename T, bool BWD, int ACT>
__device__ void consumer_phase2(const FArgs& a, FShared& sh, const unsigned char* ring,
                                uint32_t& fpar) {
  const int ct = threadIdx.x - 32, lane = ct & 31, cw = ct >> 5;
  const int NS = a.nstage, N1 = sh.nst;
  const uint32_t in_bytes = (uint32_t)a.stage_v * 16u;
  const size_t slot_bytes = (size_t)(BWD ? 2u : 1u) * in_bytes;
  const int KV = a.stage_v / kFConsumers, cps = KV * (BWD ? 8 : 4);
  const uint32_t tbase = tmem_thread_base(sh.tmem, cw);
  for (int s = cw; s < sh.nseg; s += kFConsumerWarps)
    if (!__any_sync(0xffffffffu, sh.abort != 0)) finalize_segment<BWD>(a, sh, s);
  __syncwarp();
  consumers_sync();
  if (ct == 0) GBN_RING_TRACE(3);
  // Publish the parameters of the first segments (those holding the pool
  // stages) for CTAs that take pool stages of this one.
  if (cw == 0 && a.pool > 0 && !__any_sync(0xffffffffu, sh.abort != 0)) {
    const int np = min(sh.nseg, kPoolMax);
    for (int x = lane; x < np * 6; x += 32)
      a.pub[((int64_t)blockIdx.x * kPoolMax + x / 6) * kPubFloats + x % 6] =
          sh.seg_par[x / 6][x % 6];
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      st_release_u64(a.pubflag + blockIdx.x, sh.target);
    }
    __syncwarp();
  }
  if (ct == 0) sh.p2ready = 1;
  if (ct == 0) GBN_RING_TRACE(10);
  // The on-chip stages: the resident tail (released afterwards, the
  // producer refills those slots) and the TMEM stages.
  int q2 = 0, slot = (N1 - 1) % NS;  // slot = i mod NS of stage i = N1 - 1 - q2
  for (int s = sh.nseg - 1; s >= 0; --s) {
    const int nq = stages_in(sh, a, s);
    for (int q = nq - 1; q >= 0; --q, ++q2, slot = slot_prev(slot, NS)) {
      const int i = N1 - 1 - q2;  // the stage's index in phase 1
      if (i < sh.t_lo) continue;
      if (__any_sync(0xffffffffu, sh.abort != 0)) continue;
      const bool in_tmem = i < sh.t_hi;
      if (ct == 0 && i == sh.t_hi - 1) GBN_RING_TRACE(8);
      int rv0, len;
      stage_of(sh, a, s, q, rv0, len);
      stage_out<T, BWD, ACT>(a, sh.seg_c[s], rv0, len, sh.seg_par[s],
                             ring + (size_t)slot * slot_bytes, in_bytes, in_tmem,
                             tbase + (uint32_t)((i - sh.t_lo) * cps), KV);
      if (!in_tmem) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
      }
    }
  }
  if (ct == 0) GBN_RING_TRACE(9);
  // Then what the producer loads, in its push order, until its end marker
  // (push j in slot (N1 - 1 - j) mod NS).
  slot = (N1 - 1) % NS;
  for (int j = 0;; ++j, slot = slot_prev(slot, NS)) {
    if (!warp_wait_full(sh, slot, fpar, a.status)) break;
    const FDesc& d = sh.desc[slot];
    if (d.end) break;
    if (ct == 0 && j == 0) GBN_RING_TRACE(5);
    float par[6];
#pragma unroll
    for (int f = 0; f < 6; ++f) par[f] = d.par[f];
    stage_out<T, BWD, ACT>(a, d.c, d.rv0, d.len, par, ring + (size_t)slot * slot_bytes,
                           in_bytes, false, 0u, KV);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[slot]);
  }
  if (ct == 0) GBN_RING_TRACE(6);
}

template <typename T, bool BWD>
__global__ void __launch_bounds__(kFThreads, 1) bn_fused_kernel(const FArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ FShared sh;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int s = 0; s < a.nstage; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kFConsumerWarps);
      sh.issued[s] = 0;
    }
    sh.abort = 0;
    // Segments of this CTA's range [k*Wv, (k+1)*Wv) of the channel-major view.
    const int64_t e0 = (int64_t)blockIdx.x * a.Wv;
    const int64_t e1 = min(e0 + a.Wv, a.C * (int64_t)a.Mv);
    int ns = 0, nst = 0;
    for (int64_t e = e0; e < e1 && ns < kFMaxSegs;) {
      const int64_t c = e / a.Mv;
      const int64_t cend = min((c + 1) * (int64_t)a.Mv, e1);
      sh.seg_c[ns] = (int)c;
      sh.seg_rv0[ns] = (int)(e - c * a.Mv);
      sh.seg_len[ns] = (int)(cend - e);
      sh.seg_klo[ns] = (int)((c * a.Mv) / a.Wv);
      sh.seg_khi[ns] = (int)(((c + 1) * a.Mv - 1) / a.Wv);
      nst += (sh.seg_len[ns] + a.stage_v - 1) / a.stage_v;
      ++ns;
      e = cend;
    }
    sh.nseg = ns;
    sh.nst = nst;
    sh.t_hi = max(nst - a.nstage, 0);
    sh.t_lo = max(sh.t_hi - a.nt, 0);
    sh.tmem = 0;
    sh.pool = min(a.pool, sh.t_lo);
    sh.p2ready = 0;
    // this CTA's pool word: stages [0, pool) unclaimed (published to the
    // other CTAs by the release of pubflag after the finalize)
    if (a.pool > 0) a.steal[blockIdx.x] = (uint32_t)sh.pool << 16;
    fence_mbarrier_init();
    GBN_RING_TRACE(0);
  }
  __syncthreads();

  if (tid < 32) {
    producer<T, BWD>(a, sh, ring);
    __syncwarp();
  } else {
    // The launch's flag value and the per-segment parameters: global loads,
    // off the producer's start path (the first stage takes longer to land).
    if (tid == 32) {
      const unsigned long long ea = ld_relaxed_u64(a.sync), eb = ld_relaxed_u64(a.sync + 1);
      sh.target = (eb == ~ea ? ea : a.nonce) + 1ull;
    }
    // Consumer warp 0 takes the SM's TMEM (all columns; the only CTA here).
    const bool use_tmem = sh.t_hi > sh.t_lo;
    if (use_tmem && tid < 64) tmem_alloc_all(&sh.tmem);
    if (tid - 32 < sh.nseg) {
      const int s = tid - 32;
      const int64_t c = sh.seg_c[s];
      if constexpr (!BWD) {
        sh.seg_par[s][0] = to_f32(static_cast<const T*>(a.x)[c * a.P]);  // x[0, c, 0, 0]
        sh.seg_par[s][4] = 0.f;
      } else {
        sh.seg_par[s][0] = a.stats[4 * a.C + c];
        sh.seg_par[s][1] = a.stats[5 * a.C + c];
        sh.seg_par[s][2] = a.stats[3 * a.C + c];
        sh.seg_par[s][5] = a.beta ? a.beta[c] : 0.f;
      }
    }
    if (use_tmem) tmem_fence_before_sync();
    consumers_sync();
    if (use_tmem) tmem_fence_after_sync();
    uint32_t fpar = 0;
    consumer_phase1<T, BWD>(a, sh, ring, fpar);
    if (a.act == GBN_ACT_RELU)
      consumer_phase2<T, BWD, GBN_ACT_RELU>(a, sh, ring, fpar);
    else if (a.act == GBN_ACT_LEAKY_RELU)
      consumer_phase2<T, BWD, GBN_ACT_LEAKY_RELU>(a, sh, ring, fpar);
    else
      consumer_phase2<T, BWD, GBN_ACT_NONE>(a, sh, ring, fpar);
    if (tid == 32) GBN_RING_TRACE(4);
    // Every consumer's TMEM loads have completed (each waited for its own);
    // warp 0 frees the columns.  Reached on every path, aborted or not.
    if (use_tmem) {
      tmem_fence_before_sync();
      consumers_sync();
      if (tid < 64) {
        tmem_fence_after_sync();
        tmem_free_all(sh.tmem);
      }
    }
  }
  __syncthreads();

  if (tid == 0) {
    // Let every copy this CTA issued land before the CTA exits.
    for (int s = 0; s < a.nstage; ++s)
      if (sh.issued[s] > 0 &&
          !mbar_wait_bounded(&sh.full[s], (uint32_t)(sh.issued[s] - 1) & 1u))
        report_status(a.status, GBN_DEV_WAIT_TIMEOUT);
  }
  // CTA 0 advances the epoch once every CTA has published (so every CTA has
  // read the old one); its threads check the G flags in parallel.  After a
  // failure it skips one epoch so that no flag of this launch can match the
  // next launch's target.
  if (blockIdx.x == 0) {
    bool ok = !sh.abort;
    for (int k = tid; k < a.G && ok; k += kFThreads)
      ok = wait_flag(a.sync + 2 + 2 * (int64_t)k, sh.target);
    const bool all = __syncthreads_and(ok) != 0;
    if (tid == 0) {
      if (!all) report_status(a.status, GBN_DEV_WAIT_TIMEOUT);
      const unsigned long long next = all ? sh.target : sh.target + 1ull;
      st_relaxed_u64(a.sync + 1, ~next);
      st_relaxed_u64(a.sync, next);
    }
  }
}

template <typename T, bool BWD>
cudaError_t launch_fused(const FArgs& a, const BnFusedPlan& p, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.G, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bn_fused_kernel<T, BWD>, a);
}


// Workspace of the persistent kernel: the epoch pair and a flag pair per CTA
// (16 bytes each), the pool words (4 bytes per CTA), the publish flags (8
// bytes per CTA), the published parameters (kPoolMax x kPubFloats floats per
// CTA), then, from the next 256-byte boundary, the partials.
size_t ws_steal_off(int G) { return ((size_t)16 + (size_t)16 * G + 15) & ~(size_t)15; }
size_t ws_pubflag_off(int G) { return (ws_steal_off(G) + (size_t)4 * G + 15) & ~(size_t)15; }
size_t ws_pub_off(int G) { return (ws_pubflag_off(G) + (size_t)8 * G + 15) & ~(size_t)15; }
size_t ws_part_off(int G) {
  return (ws_pub_off(G) + (size_t)G * kPoolMax * kPubFloats * sizeof(float) + 255) & ~(size_t)255;
}

FArgs make_args(const BnFusedPlan& p, void* ws) {
  FArgs a = {};
  unsigned char* w = static_cast<unsigned char*>(ws);
  a.sync = static_cast<unsigned long long*>(ws);
  a.steal = reinterpret_cast<uint32_t*>(w + ws_steal_off(p.G));
  a.pubflag = reinterpret_cast<unsigned long long*>(w + ws_pubflag_off(p.G));
  a.pub = reinterpret_cast<float*>(w + ws_pub_off(p.G));
  a.pool = p.pool;
  a.part = reinterpret_cast<float2*>(w + p.part_offset);
  a.nonce = next_nonce();
  a.C = p.C;
  a.P = p.P;
  a.Wv = p.Wv;
  a.Mv = (int32_t)p.Mv;
  a.Pv = (int32_t)p.Pv;
  a.stage_v = p.stage_v;
  a.nstage = p.nstage;
  a.grid_y = p.grid_y;
  a.G = p.G;
  a.dn = (int32_t)(kFConsumers / p.Pv);
  a.dp = (int32_t)(kFConsumers % p.Pv);
  a.ostep = (int64_t)a.dn * p.C * p.Pv + a.dp;
  a.pdiv = make_fast_div((uint32_t)p.Pv);
  a.owrap = p.C * p.Pv - p.Pv;
  a.l2_window = p.l2_window;
  a.nt = p.tmem_stages;
  a.stream_out = p.stream_out ? 1 : 0;
  a.Mh = (float)p.M;
  a.Ml = (float)(p.M - (int64_t)a.Mh);
  return a;
}

}  // namespace

namespace {
std::atomic<unsigned long long> g_nonce{0};
std::atomic<int> g_tmem{1};
std::atomic<int> g_steal{1};
}  // namespace

int bn_fused_set_tmem(int enable) { return g_tmem.exchange(enable != 0 ? 1 : 0); }
int bn_fused_set_steal(int enable) { return g_steal.exchange(enable != 0 ? 1 : 0); }

// A fresh 64-bit value per call (splitmix64 of a process counter): the flag
// epoch used when a workspace holds no valid epoch pair.
unsigned long long next_nonce() {
  unsigned long long z = g_nonce.fetch_add(0x9e3779b97f4a7c15ull) + 0x9e3779b97f4a7c15ull;
  z ^= reinterpret_cast<uintptr_t>(&g_nonce);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

bool bn_fused_plan(int dtype, bool backward, int64_t B, int64_t C, int64_t HW,
                   const DevInfo& dev, BnFusedPlan* p) {
  *p = BnFusedPlan();
  const int esize = dtype == GBN_F32 ? 4 : 2;
  const int64_t vec = 16 / esize;
  if (!dev.fused_ok || B <= 0 || C <= 0 || HW <= 0 || HW % vec != 0) return false;
  p->B = B;
  p->C = C;
  p->P = HW;
  p->M = B * HW;
  p->Pv = HW / vec;
  p->Mv = p->M / vec;
  const int64_t Ev = C * p->Mv;
  // One CTA per SM, each with at least kBnFusedMinVectors vectors.
  int64_t G = (Ev + kBnFusedMinVectors - 1) / kBnFusedMinVectors;
  if (G > dev.sms) G = dev.sms;
  if (G < 1) G = 1;
  p->Wv = (Ev + G - 1) / G;
  p->G = (int)((Ev + p->Wv - 1) / p->Wv);
  // Segments per CTA: at most ceil(Wv / Mv) + 1.
  if ((p->Wv + p->Mv - 1) / p->Mv + 1 > kFMaxSegs) return false;
  // CTAs per channel (partial slots): the largest over channels.
  int64_t gy = 1;
  for (int64_t c = 0; c < C; ++c) {
    const int64_t klo = (c * p->Mv) / p->Wv, khi = ((c + 1) * p->Mv - 1) / p->Wv;
    if (khi - klo + 1 > gy) gy = khi - klo + 1;
    if (c >= 4096) {  // a safe bound for the remaining channels
      gy = (p->Mv + p->Wv - 1) / p->Wv + 1;
      break;
    }
  }
  p->grid_y = (int)gy;
  // Ring: kBnFusedStages stages of whole 16-byte vectors (x and, backward, dy),
  // each a multiple of the consumer count.
  const int ninputs = backward ? 2 : 1;
  const int64_t budget = (int64_t)dev.smem_optin - kFStaticSmem;
  int64_t stage_v = budget / ((int64_t)kBnFusedStages * ninputs * 16);
  stage_v = stage_v / kFConsumers * kFConsumers;
  if (stage_v < kFConsumers) return false;
  p->stage_v = (int)stage_v;
  p->nstage = kBnFusedStages;
  p->smem = (size_t)kBnFusedStages * ninputs * (size_t)stage_v * 16;
  // Stages kept in TMEM between the phases: a consumer thread holds
  // stage_v / 512 vectors per input and stage in 4 columns each, within its
  // 128 columns.
  const int64_t cps = stage_v / kFConsumers * ninputs * 4;
  p->tmem_stages =
      (g_tmem.load() != 0 && cps <= kTmemColsPerThread) ? (int)(kTmemColsPerThread / cps) : 0;
  // Stages per CTA whose phase-1 loads stay at normal L2 priority: about
  // three quarters of L2, shared by the G CTAs.
  const int64_t stage_bytes = (int64_t)ninputs * stage_v * 16;
  p->l2_window = (int)((int64_t)dev.l2_bytes * 3 / 4 / ((int64_t)p->G * stage_bytes));
  // Outputs stream past L2 (evict-first) only when the call's tensors do not
  // fit in half of it: then they would push out the inputs that phase 2
  // re-reads; smaller outputs are left to L2, which absorbs the writes.
  const int64_t call_bytes = (int64_t)(ninputs + 1) * C * p->M * esize;
  p->stream_out = call_bytes > (int64_t)dev.l2_bytes / 2;
  // A CTA's first stages that other CTAs may take over in phase 2, so that
  // CTAs on slower SMs finish with the rest: only where a CTA reloads enough
  // stages in phase 2 for the claims to pay (measured: about 1-4 us slower
  // on short ranges, faster on [128,256,56,56] bf16).
  const int64_t reload = (p->Wv + stage_v - 1) / stage_v - kBnFusedStages - p->tmem_stages;
  p->pool =
      (g_steal.load() != 0 && reload >= kPoolMinStages && p->G <= kMaxCtas) ? kPoolMax : 0;
  p->part_offset = ws_part_off(p->G);
  p->ws_bytes = p->part_offset + (size_t)2 * p->grid_y * C * sizeof(float2);
  p->ws_bytes = (p->ws_bytes + 255) & ~(size_t)255;
  p->ok = true;
  return true;
}

cudaError_t bn_fused_forward(const BnFusedPlan& p, int dtype, const void* x, void* y,
                             const float* gamma, const float* beta, float* stats,
                             float* running_mean, float* running_var, float momentum, float eps,
                             int act, float slope, void* ws, int* status, cudaStream_t st) {
  FArgs a = make_args(p, ws);
  a.act = act;
  a.slope = slope;
  a.x = x;
  a.out = y;
  a.gamma = gamma;
  a.beta = beta;
  a.stats = stats;
  a.running_mean = running_mean;
  a.running_var = running_var;
  a.momentum = momentum;
  a.eps = eps;
  a.status = status;
  return dtype == GBN_F32 ? launch_fused<float, false>(a, p, st)
                          : launch_fused<bf16, false>(a, p, st);
}

cudaError_t bn_fused_backward(const BnFusedPlan& p, int dtype, const void* x, const void* dy,
                              void* dx, const float* stats, const float* beta, int act,
                              float slope, float* grads, void* ws, int* status,
                              cudaStream_t st) {
  FArgs a = make_args(p, ws);
  a.beta = beta;
  a.act = act;
  a.slope = slope;
  a.x = x;
  a.dy = dy;
  a.out = dx;
  a.stats = const_cast<float*>(stats);
  a.grads = grads;
  a.status = status;
  return dtype == GBN_F32 ? launch_fused<float, true>(a, p, st)
                          : launch_fused<bf16, true>(a, p, st);
}

cudaError_t bn_fused_configure(int smem_optin, bool* ok) {
  *ok = false;
  const int dyn = smem_optin - kFStaticSmem;
  if (dyn <= 0) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(bn_fused_kernel<float, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bn_fused_kernel<float, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bn_fused_kernel<bf16, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bn_fused_kernel<bf16, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) != cudaSuccess)
    return e;
  // The launch needs one resident CTA per SM with the full ring.
  int blocks = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, bn_fused_kernel<bf16, true>,
                                                    kFThreads, (size_t)dyn);
  if (e != cudaSuccess) return e;
  *ok = blocks >= 1;
  return cudaSuccess;
}

}  // namespace gbn
