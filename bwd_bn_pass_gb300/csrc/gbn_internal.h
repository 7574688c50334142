// Host-side declarations shared by the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gbnorm.h"

namespace gbn {

// Cached per-device facts.  Filled once per device by device_info().
struct DevInfo {
  int sms = 0;               // multiprocessor count (152 on GB300)
  int max_threads_sm = 0;    // resident threads per SM (2048)
  int smem_optin = 0;        // max dynamic shared memory per block (bytes)
  int smem_per_sm = 0;       // shared memory per SM (bytes)
  int smem_reserved = 0;     // shared memory the runtime reserves per block
  int l2_bytes = 0;          // L2 cache size
  int* status = nullptr;     // device address of the library status word
  bool fused_ok = false;     // the persistent BatchNorm kernel fits one CTA per SM
  bool ok = false;
};

// Returns nullptr (and leaves a CUDA error pending) if the device cannot be
// queried.  device < 0 means the current device.
const DevInfo* device_info(int device);

// Launch `kern` with the given configuration; `pdl` adds the programmatic
// stream serialization attribute so the kernel may start while the
// preceding kernel on the stream drains (it then calls griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------- BatchNorm --

constexpr int kBnThreads = 256;
constexpr int kBnBlocksPerSm = 4;   // resident 256-thread blocks per SM the grid fills
constexpr int64_t kBnMinElemsPerBlock = 4096;

// Shape facts derived once per call on the host.
struct BnPlan {
  int64_t B = 0, C = 0, P = 0;  // batch, channels, plane size (HW)
  int64_t M = 0;                // per-channel count B*P
  int grid_y = 0;               // blocks per channel
  int vec = 1;                  // elements per vector access
  size_t ws_partials = 0;       // two-launch partials bytes (2 * grid_y * C fp32 pairs, rounded)
  size_t ws_bytes = 0;          // workspace of the public calls: also fits the persistent path
};

// Fills grid_y / ws_bytes (device-dependent) for a shape; false on error.
int bn_set_wide_offsets(int force);  // 64-bit offsets in the two-launch kernels
bool bn_plan(int64_t B, int64_t C, int64_t HW, const DevInfo& dev, BnPlan* plan);

// Largest power-of-two vector width (<= 16 bytes) valid for all pointers.
int bn_vec_width(int dtype, int64_t P, const void* const* ptrs, int nptrs);

enum BnApplyMode { kApplyTrain = 0, kApplyStats = 1, kApplyInfer = 2 };

cudaError_t bn_launch_stats(const void* x, int dtype, const BnPlan& p, float2* part,
                            cudaStream_t st);
cudaError_t bn_launch_apply(const void* x, void* y, int dtype, const BnPlan& p, int mode,
                            const float2* part, const float* gamma, const float* beta,
                            float* stats, float* running_mean, float* running_var,
                            float momentum, float eps, const float* mean, const float* scale,
                            int act, float slope, cudaStream_t st, bool pdl);
// With act != GBN_ACT_NONE the backward kernels gate dy by d act / d pre,
// pre recomputed from x, the stats rows and beta (may be null: 0).
cudaError_t bn_launch_grad_sums(const void* x, const void* dy, int dtype, const BnPlan& p,
                                const float* stats, float2* part, const float* beta, int act,
                                float slope, cudaStream_t st);
cudaError_t bn_launch_dx(const void* x, const void* dy, void* dx, int dtype, const BnPlan& p,
                         const float* stats, const float2* part, float* grads, const float* beta,
                         int act, float slope, cudaStream_t st, bool pdl);

// Single-launch BatchNorm for small channels (bn_small.cu): one block per
// channel stages the channel's M <= lim elements in shared memory; up to
// kBnClusterMax * lim elements, a cluster of up to kBnClusterMax blocks per
// channel, each staging a share of at most lim (lim <= kBnSmallMaxM).
constexpr int64_t kBnSmallMaxM = 2048;
constexpr int kBnClusterMax = 8;
// Resident 256-thread blocks per SM the small-channel kernels are sized for
// (at most 64 registers a thread).
constexpr int kBnSmallBlocksPerSm = 4;
// Blocks per channel K (1, 2, 4 or 8) with which the small-channel kernels
// take a shape: the smallest K whose shares hold at most lim elements, and
// only while the grid is one latency chain per block (load, reduce,
// finalize, store) with no second wave: one block per channel while the C
// blocks fit kBnSmallBlocksPerSm per SM; a cluster while the C*K blocks fit
// one per SM (measured: 148 blocks beat the two-launch kernels by ~0.5 us,
// 256 tie, 608 lose by ~3 us).  0: not eligible.
int bn_small_blocks(int64_t M, int64_t C, int64_t lim, const DevInfo& dev);
cudaError_t bn_small_forward(int dtype, const void* x, void* y, int64_t B, int64_t C,
                             int64_t HW, const float* gamma, const float* beta, float* stats,
                             float* running_mean, float* running_var, float momentum, float eps,
                             int act, float slope, int K, cudaStream_t st);
cudaError_t bn_small_backward(int dtype, const void* x, const void* dy, void* dx, int64_t B,
                              int64_t C, int64_t HW, const float* stats, const float* beta,
                              int act, float slope, float* grads, int K, cudaStream_t st);

// Persistent single-launch BatchNorm (bn_fused.cu): one CTA per SM owns a
// contiguous range of the channel-major view; see that file.
constexpr int64_t kBnFusedMinVectors = 2048;  // 16-byte vectors per CTA, at least
constexpr int kBnFusedStages = 4;             // shared-memory ring depth

struct BnFusedPlan {
  bool ok = false;
  int64_t B = 0, C = 0, P = 0, M = 0;
  int64_t Pv = 0, Mv = 0;  // 16-byte vectors per plane / per channel
  int64_t Wv = 0;          // vectors per CTA
  int G = 0;               // CTAs
  int grid_y = 0;          // partial slots per channel
  int stage_v = 0;         // vectors per stage and input
  int nstage = 0;
  int l2_window = 0;       // phase-1 stages per CTA kept at normal L2 priority
  int tmem_stages = 0;     // stages per CTA kept in tensor memory between the phases
  int pool = 0;            // a CTA's first stages open to other CTAs in phase 2
  bool stream_out = true;  // outputs stored with the evict-first hint
  size_t smem = 0;         // dynamic shared memory (the ring)
  size_t part_offset = 0;  // partials offset in the workspace (sync words first)
  size_t ws_bytes = 0;
};

// False when the shape or device does not take the persistent path (plane
// not a whole number of 16-byte vectors, too many channels per CTA, ...).
bool bn_fused_plan(int dtype, bool backward, int64_t B, int64_t C, int64_t HW,
                   const DevInfo& dev, BnFusedPlan* plan);
// Whether later plans keep stages in TMEM (process-wide); returns the previous setting.
int bn_fused_set_tmem(int enable);
// Whether later plans let CTAs take other CTAs' last stages; returns the previous setting.
int bn_fused_set_steal(int enable);
cudaError_t bn_fused_forward(const BnFusedPlan& p, int dtype, const void* x, void* y,
                             const float* gamma, const float* beta, float* stats,
                             float* running_mean, float* running_var, float momentum, float eps,
                             int act, float slope, void* ws, int* status, cudaStream_t st);
cudaError_t bn_fused_backward(const BnFusedPlan& p, int dtype, const void* x, const void* dy,
                              void* dx, const float* stats, const float* beta, int act,
                              float slope, float* grads, void* ws, int* status,
                              cudaStream_t st);
// A fresh 64-bit value per call: the epoch of a launch whose workspace holds
// no valid epoch pair (kernels that hand results between resident CTAs).
unsigned long long next_nonce();
// Shared-memory limits and the one-CTA-per-SM check (called from device_info).
cudaError_t bn_fused_configure(int smem_optin, bool* ok);

// Training forward with a caller-fixed scratch buffer (the allocation-free
// entry point): `ws` must hold at least bn_partials_bytes(B, C, HW) bytes;
// the persistent kernel is used when `ws_bytes` also fits its workspace,
// else the two-launch kernels.  Same status codes as gbn_bn_forward_train.
size_t bn_partials_bytes(int64_t B, int64_t C, int64_t HW);
// The argument checks of the training forward that need no CUDA call (dtype,
// sizes, null pointers, stats alignment, eps / momentum): GBN_OK or the
// status the forward would return for them.
int bn_forward_check_args(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                          const void* y, const float* stats, float momentum, float eps);
int bn_forward_train_scratch(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                             const float* gamma, const float* beta, float* running_mean,
                             float* running_var, float momentum, float eps, void* y,
                             float* stats, void* ws, size_t ws_bytes, void* stream);

// ------------------------------------------------------------ row-wise --

// Column partials: [nout][nplanes][G][H] fp32; nplanes = 2 (hi, lo) when the
// outputs are fp32 (double-fp32 accumulation), 1 otherwise.
struct RowPlan {
  int64_t R = 0, H = 0;
  int kind = GBN_ROW_RMS;
  int dtype = GBN_F32;
  bool fast = false;   // bulk-copy persistent kernel (else the generic kernel)
  int threads = 0;     // block size
  int kv = 0;          // 16-byte vectors per thread per row (fast path)
  int rb = 1;          // rows per pipeline stage (fast path)
  int cps = 1;         // blocks per SM the launch is sized for (fast path)
  int nstage = 0;      // pipeline depth (fast path)
  int G = 0;           // blocks (= rows of column partials)
  int nout = 1;        // column outputs
  int nplanes = 1;     // 2 when fp32 outputs use hi/lo partials
  size_t smem = 0;     // dynamic shared memory per block
  uint32_t stage_bytes = 0;
  uint32_t off[5] = {0, 0, 0, 0, 0};  // per-stage offsets: dy, x, residual, mask, dz_extra
  int tprw = 0;        // LayerNorm ring: consumer warps per row slot
  int rs = 0;          // LayerNorm ring: row slots
  size_t part_offset = 0;  // column partials' offset in the workspace (flags first)
  size_t ws_bytes = 0;
};

// Consumer warps of the LayerNorm ring kernel: at most 14 when a thread owns
// one 16-byte vector of a row, 8 when it owns two (register budget).
constexpr int kLnRingWarpsKV1 = 14;
constexpr int kLnRingWarpsKVn = 8;

struct LnPtrs {
  const void* dy = nullptr;
  const void* x = nullptr;
  const void* residual = nullptr;
  const void* bias = nullptr;
  const uint8_t* mask = nullptr;
  const float* dz_extra = nullptr;
  const float* mean = nullptr;
  const float* rstd = nullptr;
  const void* gamma = nullptr;
  float scale = 1.f;
  void* dx = nullptr;
  void* dres = nullptr;
  void* dgamma = nullptr;
  void* dbeta = nullptr;
  void* dbias = nullptr;
  bool saved_z = false;   // x is the saved LayerNorm input z (fused outputs, no residual)
  bool dres_f32 = false;  // dres is fp32
};

// Plans the launch.  `fast_ok` says whether pointers/shape allow the
// bulk-copy path; the workspace query plans with fast_ok=false and true and
// takes the larger size.
bool row_plan(int64_t R, int64_t H, int kind, int dtype, bool fast_ok, bool has_mask,
              bool has_dzx, const DevInfo& dev, RowPlan* plan);

cudaError_t rms_launch(const RowPlan& p, const void* dy, const void* x, const void* w,
                       const float* rstd, void* dx, void* dw, void* ws, int* status,
                       cudaStream_t st);
cudaError_t ln_launch(const RowPlan& p, const LnPtrs& a, void* ws, int* status,
                      cudaStream_t st);

// Row-wise training forwards (fwd_kernels.cu).
struct RowFwdPtrs {
  const void* x = nullptr;         // RMSNorm x / LayerNorm input
  const void* residual = nullptr;  // fused LayerNorm
  const void* bias = nullptr;
  const uint8_t* mask = nullptr;
  const void* w = nullptr;         // RMSNorm weight / LayerNorm gamma
  const void* beta = nullptr;
  void* y = nullptr;
  void* z = nullptr;
  float* mean = nullptr;
  float* rstd = nullptr;
};

// kind: GBN_ROW_RMS, GBN_ROW_LN or GBN_ROW_LN_FUSED.  vec_ok: every tensor
// is 16-byte aligned and a row is a whole number of 16-byte vectors (and of
// 8-byte mask words), so the register-resident vector kernels may run.
cudaError_t row_fwd_launch(int kind, int dtype, const RowFwdPtrs& p, int64_t R, int64_t H,
                           float eps, float scale, bool vec_ok, const DevInfo& dev,
                           cudaStream_t st);
cudaError_t row_fwd_configure();  // shared-memory limits (called from device_info)

// Column-partials reduction: out[o][h] = sum_g part[o][*][g][h] in a fixed
// order; outs[o] may be nullptr (skipped).  Launched with PDL after the row
// kernel when `pdl` is set.
cudaError_t colsum_launch(const float* part, int nout, int nplanes, int G, int64_t H, int dtype,
                          void* const* outs, cudaStream_t st, bool pdl);

// Set the kernels' dynamic shared memory limits (called from device_info).
cudaError_t row_kernels_configure(int smem_optin);

// Launches one block that waits on an mbarrier nothing completes, through
// the library's bounded wait, for at most limit_ns; the expired wait sets
// GBN_DEV_WAIT_TIMEOUT in *status.
cudaError_t selftest_bounded_wait(int* status, uint64_t limit_ns, cudaStream_t st);

// -------------------------------------------- BatchNorm, channels last --

struct NhwcPlan {
  int64_t M = 0, C = 0;  // rows (N*H*W) and channels
  int vec = 1;           // channels per vector (divides C)
  int TX = 1;            // vectors per block row
  int grid_y = 1;        // row slices
  size_t ws_bytes = 0;   // partials [2][grid_y][C] float2
};
bool nhwc_plan(int64_t M, int64_t C, int vec, const DevInfo& dev, NhwcPlan* p);
size_t nhwc_ws_bound(int64_t M, int64_t C, const DevInfo& dev);
cudaError_t nhwc_forward(const NhwcPlan& p, int dtype, const void* x, void* y,
                         const float* gamma, const float* beta, float* stats,
                         float* running_mean, float* running_var, float momentum, float eps,
                         int act, float slope, void* ws, cudaStream_t st);
// y = act(((x - shift) - (mean - shift))*scale + beta) from a training
// stats buffer, or (stats NULL) act((x - mean)*scale + beta) from
// per-channel mean and scale.
cudaError_t nhwc_apply(const NhwcPlan& p, int dtype, const void* x, void* y, const float* stats,
                       const float* mean, const float* scale, const float* beta, int act,
                       float slope, cudaStream_t st);
cudaError_t nhwc_backward(const NhwcPlan& p, int dtype, const void* x, const void* dy, void* dx,
                          const float* stats, const float* beta, int act, float slope,
                          float* grads, void* ws, cudaStream_t st);

}  // namespace gbn
