/*
 * gbnorm.h -- C ABI of libgbnorm.so: training-mode normalization forward and
 * backward on one GB300 (sm_103a) GPU.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers of the current CUDA device (for example
 *   torch's tensor.data_ptr()), except where a comment says otherwise.  The
 *   caller owns all memory; the library allocates nothing and keeps no
 *   per-call state.  It caches only device attributes and the address of its
 *   device status word (see gbn_get_device_status).
 * - `stream` is a cudaStream_t passed as void*.  Every call is asynchronous
 *   on that stream; no call synchronises the host.
 * - Tensors are dense and contiguous in the layout stated per call.  Sizes
 *   are int64_t element counts.
 * - `dtype` selects the storage type of the large tensors: GBN_F32 or
 *   GBN_BF16.  All accumulation is fp32 on the GPU, with error-free (double
 *   fp32) summation where a fp32 output needs it; per-channel and per-row
 *   reductions across blocks are combined in fp64 or double-fp32 in a fixed
 *   order, so two runs on the same device give bit-identical results.  No
 *   float atomics are used anywhere.
 * - Return value: GBN_OK (0) or a negative GBN_E* code.  On an argument
 *   error nothing is launched and no output is touched.  GBN_ECUDA reports
 *   the error returned by a CUDA query or launch.  Errors that can
 *   only be seen on the device (a bounded wait that ran out) are recorded in
 *   the device status word, read with gbn_get_device_status.
 * - Alignment: any element-aligned pointer is accepted for the large
 *   tensors; 16-byte aligned pointers (and rows/planes whose byte length is
 *   a multiple of 16) take the vectorised / bulk-copy fast paths.  `stats`
 *   must be 8-byte aligned and workspaces 16-byte aligned (else GBN_EALIGN).
 *
 * Source pages (titles; the numbers in brackets are the sections used):
 *   [P4] Aether-ML PR #18 "perf(batchnorm): device-sized grid, one-pass
 *        statistics, finalize kernels" -- sections "Reduction grid",
 *        "One-pass statistics", "Backward finalize", "Behavior changes".
 *   [P2] nvFuser issue #1473 "Why is LayerNorm Backward Segmenting?" --
 *        the bias+dropout+add+layer_norm backward repro (fusion_id9) and the
 *        layer_norm backward repro (fusion_id14), "Perf on A100".
 *   [P3] nvFuser issue #3629 "Performance gap between manual nvfuser
 *        definition and thunder.jit for rmsnorm" -- "nvfuser pre-generated
 *        definition" (rmsnorm_bwd_fusion) and the Thunder definition.
 *   [P1] Lightning-Thunder PR #182 "Improve batch_norm backward performance
 *        for automatically generated backward" (BN backward as one pass).
 */
#ifndef GBNORM_H
#define GBNORM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GBN_API __attribute__((visibility("default")))
#else
#define GBN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GBN_OK 0
#define GBN_EINVAL -1     /* null pointer, negative/overflowing size, M < 2 in training, bad combination */
#define GBN_EDTYPE -2     /* dtype is not GBN_F32 / GBN_BF16 */
#define GBN_EALIGN -3     /* stats not 8-byte aligned or workspace not 16-byte aligned */
#define GBN_EWORKSPACE -4 /* ws_bytes smaller than the matching *_workspace_bytes() */
#define GBN_ECUDA -5      /* CUDA runtime error while querying the device or launching */
#define GBN_EDEVICE -6    /* a kernel reported an error in the device status word */

/* ---- storage types ----------------------------------------------------- */
#define GBN_F32 0
#define GBN_BF16 1

/* ---- device status bits (gbn_get_device_status) ------------------------ */
#define GBN_DEV_WAIT_TIMEOUT 1 /* a bulk-copy wait in a row kernel ran out (about 1 s) */

/* ---- BatchNorm buffer sizes -------------------------------------------- */
/* stats: 8*C floats (32*C bytes, 8-byte aligned).  Rows 0..3 are public,
 * fp32 [4, C] = (mean, var, inv_std, scale = gamma*inv_std) as in [P4]
 * "One-pass statistics".  Rows 4..7 are private to this library: row 4 the
 * channel's shift x[0,c,0,0], row 5 mean - shift rounded to fp32, rows 6 and
 * 7 the same mean - shift as an unevaluated fp32 pair (hi, lo) that the
 * backward uses.                                                            */
#define GBN_BN_STATS_FLOATS(C) (8 * (int64_t)(C))
/* grads: fp32 [4, C] = (dgamma, dbeta, k1, k2), [P4] "Backward finalize".  */
#define GBN_BN_GRADS_FLOATS(C) (4 * (int64_t)(C))

/* ---- activations fused into BatchNorm (gbn_bn_*_act) ------------------- */
/* [P4] "Part 2": the BatchNorm output pre = (x - mean)*scale + beta goes
 * through act in the same pass.  RELU: max(pre, 0).  LEAKY_RELU: pre where
 * pre > 0, else slope*pre.  The backward gates dy by d act / d pre (1 where
 * pre > 0, else 0 or slope), recomputing pre from x, stats and beta, so no
 * mask or pre-activation tensor is stored.                                  */
#define GBN_ACT_NONE 0
#define GBN_ACT_RELU 1
#define GBN_ACT_LEAKY_RELU 2

/* ---- row-wise workspace kinds ------------------------------------------ */
#define GBN_ROW_RMS 0      /* rmsnorm_backward: dweight partials           */
#define GBN_ROW_LN 1       /* layernorm_backward, plain: dgamma, dbeta     */
#define GBN_ROW_LN_FUSED 2 /* layernorm_backward, fused: + dbias           */

/* Version of this ABI (increments on any signature change). */
GBN_API int gbn_abi_version(void);

/* Static, human-readable text for a status code. */
GBN_API const char* gbn_status_string(int status);

/* Prepare `device` (-1: current): cache its attributes, resolve the device
 * status word and raise the kernels' shared-memory limits.  Every entry
 * point does this on its first call on a device; call it explicitly before
 * capturing a CUDA graph.  Returns GBN_OK or GBN_ECUDA.  The cached facts
 * include device addresses (the status word, the allocation-free call's
 * scratch array) that a cudaDeviceReset invalidates: do not use the library
 * on a device after resetting it in the same process.                      */
GBN_API int gbn_init(int device);

/* The pages have no counterpart: a self-test of the failure detection.  It
 * launches one block on `stream` that waits, through the bounded wait every
 * ring and flag wait of the library uses, on a barrier nothing completes;
 * after about limit_ns nanoseconds (0 < limit_ns <= 2e9) the wait gives up
 * and sets GBN_DEV_WAIT_TIMEOUT in the current device's status word, and
 * the kernel returns.  Read and clear the word with gbn_get_device_status.
 * Nothing faults, traps or hangs; the context stays usable.               */
GBN_API int gbn_selftest_bounded_wait(int64_t limit_ns, void* stream);

/* Read the device status word of `device` (-1: current) into *status, a
 * HOST pointer (bit set of GBN_DEV_*; 0 = no device-side error), and clear it
 * when `clear` is nonzero.  Synchronises with the device (it is a copy).     */
GBN_API int gbn_get_device_status(int device, int* status, int clear);

/* =========================================================================
 * BatchNorm2d, training mode, NCHW  ([P4]; [P1] for the one-pass backward)
 *
 * x, y, dy, dx: [B, C, HW] contiguous (HW = H*W), storage `dtype`.
 * gamma, beta, running_mean, running_var: fp32 [C].  gamma/beta may be NULL
 * (treated as 1 and 0); running_mean/running_var may be NULL (not updated).
 * Per channel, M = B*HW elements are reduced.
 *
 * The forward is two launches: a device-sized grid of one-pass shifted-sum
 * blocks writes per-block partials (sum d, sum d^2 with d = x - x[0,c], each
 * an fp32 (hi, lo) pair) into `ws` without atomics; a second kernel, launched with programmatic
 * dependent launch, reduces the partials of its channel in a fixed order
 * (the "finalize"), writes stats and the running-stat update from the
 * channel's first block, and applies y = (x - mean)*scale + beta in the
 * centred form.  The backward mirrors it: grad_sums partials (sum dy,
 * sum dy*(x - shift)), then finalize + dx = dy*scale + (x-mean)*k1 + k2.
 * ======================================================================= */

/* Workspace bytes for the BN partials of this shape on `device` (-1:
 * current): 16 * grid_y * C rounded up to 256, where grid_y is the number of
 * blocks per channel ([P4] "Reduction grid": fill every resident 256-thread
 * block slot once).  Returns 0 on a bad shape or a CUDA error.              */
GBN_API size_t gbn_bn_workspace_bytes(int64_t B, int64_t C, int64_t HW, int device);

/* The composite calls below (gbn_bn_forward_train[_act], gbn_bn_backward[_act],
 * gbn_bn_forward_train_noalloc) run the single-launch persistent kernel
 * only when the input bytes of the call (x forward; x and dy backward) are
 * at least this threshold, and the two-launch kernels otherwise; both give
 * results within the parity tolerance.  Default 128 MiB: on GB300 the
 * cooperative launch and its flag handshake cost more than the re-read the
 * persistent kernel saves on smaller tensors.  Sets the process-wide value
 * (negative: 0, i.e. always when eligible) and returns the previous one.
 * The pages have no counterpart: it is a tuning knob of this library.     */
GBN_API int64_t gbn_bn_set_persistent_min_bytes(int64_t bytes);
/* The current threshold (bytes).                                           */
GBN_API int64_t gbn_bn_persistent_min_bytes(void);

/* Below the persistent kernel's threshold, the composite calls run channels
 * of at most 8 * m elements (M = B*HW per channel), m this limit, in ONE
 * launch while the grid is a single wave (gbn_bn_small_blocks_per_channel) ([P4]'s stats / finalize / apply, or grad_sums / finalize / dx,
 * fused for latency-bound shapes): a channel of at most m elements takes a
 * block that stages it in shared memory as it reads it once, reduces,
 * finalizes and writes the outputs; a larger one a thread-block cluster of
 * K = 2, 4 or 8 blocks (the smallest K whose shares hold at most m
 * elements), whose partial sums meet in distributed shared memory behind
 * the cluster barrier.  Default and maximum 2048; 0 sends every shape to
 * the two-launch kernels.  Results are within the parity tolerance of the
 * other paths.  Process-wide; returns the previous value.  The pages have
 * no counterpart: a tuning knob.                                           */
GBN_API int64_t gbn_bn_set_small_max_elems(int64_t m);
/* The current limit (elements per channel).                               */
GBN_API int64_t gbn_bn_small_max_elems(void);
/* Blocks per channel (1, 2, 4 or 8) with which the composite calls, below
 * the persistent kernel's threshold, run an NCHW [B, C, HW] shape in the
 * single-launch small-channel kernels on the current device, or 0 when they
 * run the two-launch kernels: eligible are channels of at most 8 * m
 * elements (m the limit above) whose blocks run as one latency chain each
 * with no second wave -- one block per channel (K = 1) while C is at most 4
 * blocks per SM, a cluster (K > 1) while C * K is at most the SM count;
 * beyond that the two-launch kernels are faster.  Host arithmetic and a
 * cached device query only; 0 also for invalid dimensions.                */
GBN_API int gbn_bn_small_blocks_per_channel(int64_t B, int64_t C, int64_t HW);

/* The persistent BatchNorm kernel keeps a few stages per SM in tensor
 * memory (TMEM) between its reduction and output passes, instead of loading
 * them again.  enable = 0 turns that off for later calls, nonzero turns it
 * back on (the default).  Results are bit-identical either way; only where
 * phase 2 reads those stages from changes.  Process-wide; returns the
 * previous setting.  The pages have no counterpart: a tuning knob.         */
GBN_API int gbn_bn_set_persistent_tmem(int enable);

/* The persistent BatchNorm kernel lets CTAs that run out of work take the
 * last stages of others at the end of its output pass (on tensors large
 * enough for it to pay).  enable = 0 turns that off for later calls,
 * nonzero back on (the default).  Results are bit-identical either way.
 * Process-wide; returns the previous setting.  A tuning knob; the pages
 * have no counterpart.                                                     */
GBN_API int gbn_bn_set_persistent_steal(int enable);

/* The two-launch BatchNorm kernels (NCHW) address vectors with 32-bit
 * offsets while the tensor holds fewer than 2^32 16-byte-or-smaller vectors,
 * and with 64-bit offsets beyond.  A nonzero `force` makes every later call
 * take the 64-bit form (results are identical; it exists so that the wide
 * form can be tested on small tensors).  Process-wide; returns the previous
 * setting.  The pages have no counterpart.                                 */
GBN_API int gbn_bn_set_wide_offsets(int force);

/* Full training forward: stats pass + finalize/apply.  Writes y, stats
 * (8*C floats, see GBN_BN_STATS_FLOATS), and updates the running stats in
 * place: running_mean = (1-momentum)*running_mean + momentum*mean,
 * running_var = (1-momentum)*running_var + momentum*var*M/(M-1); var in
 * stats is biased (divides by M).  Requires M >= 2 (GBN_EINVAL otherwise).
 * y may alias x.  ws: >= gbn_bn_workspace_bytes(B, C, HW, -1) bytes.       */
GBN_API int gbn_bn_forward_train(const void* x, int dtype, int64_t B, int64_t C,
                         int64_t HW, const float* gamma, const float* beta,
                         float* running_mean, float* running_var,
                         float momentum, float eps, void* y, float* stats,
                         void* ws, size_t ws_bytes, void* stream);

/* The paper has no counterpart to this call: it exists for callers that
 * cannot allocate device memory (code inside a CUDA-graph capture or a
 * real-time loop where cudaMalloc is forbidden, plugins whose host framework
 * owns every allocation, C callers without an allocator).  Same as
 * gbn_bn_forward_train without `ws`/`ws_bytes`: the scratch (stats partials
 * and, for the single-launch kernel, its per-block flags) goes to a fixed
 * 64 KiB file-scope device array inside the library, which every GPU that
 * loads the library holds until the process exits.  Shapes whose two-launch
 * partials need more (16 * grid_y * C bytes; all C <= 4096 fit on GB300) are
 * rejected with GBN_EWORKSPACE; shapes whose single-launch scratch does not
 * fit run the two-launch kernels.  Allocates nothing and nothing needs
 * zeroing: every call rewrites the partials it reads and the flags carry a
 * launch epoch checked on the device.  All calls share the one array,
 * so calls that overlap on the GPU (other streams, other threads) race; order
 * them on one stream.  The first call on a device resolves the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Argument errors (dtype, sizes, null x / y
 * / stats, stats alignment, eps, momentum) return GBN_EINVAL / GBN_EDTYPE /
 * GBN_EALIGN before any CUDA call, as for the other entry points.          */
GBN_API int gbn_bn_forward_train_noalloc(const void* x, int dtype, int64_t B, int64_t C,
                                         int64_t HW, const float* gamma, const float* beta,
                                         float* running_mean, float* running_var,
                                         float momentum, float eps, void* y, float* stats,
                                         void* stream);

/* gbn_bn_forward_train followed by the activation `act` (GBN_ACT_*) in the
 * same kernels: y = act((x - mean)*scale + beta).  slope is LeakyReLU's
 * negative slope (finite; ignored for the others).  stats and the running
 * update are those of gbn_bn_forward_train.  GBN_EINVAL for an unknown act
 * or a non-finite LeakyReLU slope.                                          */
GBN_API int gbn_bn_forward_train_act(const void* x, int dtype, int64_t B, int64_t C,
                                     int64_t HW, const float* gamma, const float* beta,
                                     float* running_mean, float* running_var, float momentum,
                                     float eps, int act, float slope, void* y, float* stats,
                                     void* ws, size_t ws_bytes, void* stream);

/* Phase 1 of the forward alone: writes the stats partials into ws.        */
GBN_API int gbn_bn_stats(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                 void* ws, size_t ws_bytes, void* stream);

/* Phases 2+3 of the forward: finalize the partials left in ws by
 * gbn_bn_stats (same x, same shape, same device), write stats and the
 * running update, and apply.  Arguments as gbn_bn_forward_train.           */
GBN_API int gbn_bn_finalize_apply(const void* x, int dtype, int64_t B, int64_t C,
                          int64_t HW, const float* gamma, const float* beta,
                          float* running_mean, float* running_var,
                          float momentum, float eps, void* y, float* stats,
                          const void* ws, size_t ws_bytes, void* stream);

/* Centred apply y = (x - mean)*scale + beta, shared by training and
 * inference ([P4] "One-pass statistics", _bn_apply_ew).  If `stats` is
 * non-NULL it is a buffer written by a training forward and mean/scale are
 * ignored; otherwise `mean` and `scale` (fp32 [C], e.g. running_mean and
 * gamma/sqrt(running_var + eps)) are used.  beta may be NULL (0).           */
GBN_API int gbn_bn_apply(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                 const float* stats, const float* mean, const float* scale,
                 const float* beta, void* y, void* stream);

/* gbn_bn_apply followed by the activation `act` (arguments as
 * gbn_bn_forward_train_act).                                                */
GBN_API int gbn_bn_apply_act(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                             const float* stats, const float* mean, const float* scale,
                             const float* beta, int act, float slope, void* y, void* stream);

/* Full training backward: grad_sums pass + finalize/dx.  `stats` is the
 * buffer written by the matching training forward of the same x.  Writes
 * dx and grads (fp32 [4, C] = dgamma, dbeta, k1, k2; [P4] "Backward
 * finalize") with k1 = -scale*inv_std^2*sum(dy*(x-mean))/M and
 * k2 = -scale*dbeta/M.  dx may alias dy.  ws as for the forward.            */
GBN_API int gbn_bn_backward(const void* x, const void* dy, int dtype, int64_t B,
                    int64_t C, int64_t HW, const float* stats, void* dx,
                    float* grads, void* ws, size_t ws_bytes, void* stream);

/* Backward of gbn_bn_forward_train_act: dy is first multiplied by
 * d act / d pre, with pre = (x - mean)*scale + beta recomputed from x, the
 * forward's stats and the forward's beta (fp32 [C], NULL if the forward had
 * none), evaluated exactly as the forward did; then as gbn_bn_backward,
 * grads' dbeta and dgamma being those of the gated gradient.  act and slope
 * must be the forward's.                                                    */
GBN_API int gbn_bn_backward_act(const void* x, const void* dy, int dtype, int64_t B,
                                int64_t C, int64_t HW, const float* stats, const float* beta,
                                int act, float slope, void* dx, float* grads, void* ws,
                                size_t ws_bytes, void* stream);

/* Phase 1 of the backward alone: grad_sums partials into ws.              */
GBN_API int gbn_bn_grad_sums(const void* x, const void* dy, int dtype, int64_t B,
                     int64_t C, int64_t HW, const float* stats, void* ws,
                     size_t ws_bytes, void* stream);

/* Phases 2+3 of the backward: finalize the grad_sums partials in ws and
 * write grads and dx.                                                       */
GBN_API int gbn_bn_finalize_dx(const void* x, const void* dy, int dtype, int64_t B,
                       int64_t C, int64_t HW, const float* stats, void* dx,
                       float* grads, const void* ws, size_t ws_bytes,
                       void* stream);

/* =========================================================================
 * BatchNorm2d, training mode, channels last (NHWC)  ([P4]; "Part 2" act)
 *
 * x, y, dy, dx: [M, C] row-major in `dtype` with M = N*H*W and the channel
 * innermost (a channels-last [N, H, W, C] tensor).  The statistics, the
 * finalize, the centred apply, the backward finalize and the activation are
 * those of the NCHW entry points, and stats / grads have the same layout
 * (GBN_BN_STATS_FLOATS, GBN_BN_GRADS_FLOATS) with shift = x[0, c].  Three
 * launches per direction: a row-streaming sum kernel writing per-block
 * (hi, lo) partials for every channel, a finalize kernel (one warp per
 * channel, fixed order), and the apply / dx kernel.  act / slope as for
 * gbn_bn_forward_train_act (GBN_ACT_NONE for plain BatchNorm).  Requires
 * M >= 2 and M < 2^31.  ws must be 16-byte aligned.                       */

/* Workspace bytes for an NHWC forward or backward of this shape on `device`
 * (-1: current): the partials, 16 * grid_y * C rounded up to 256.  Returns
 * 0 on a bad shape or a CUDA error.                                        */
GBN_API size_t gbn_bn_nhwc_workspace_bytes(int64_t M, int64_t C, int device);

/* Training forward: writes y, stats (8*C floats) and the running update as
 * gbn_bn_forward_train does.  y may alias x.                               */
GBN_API int gbn_bn_nhwc_forward_train(const void* x, int dtype, int64_t M, int64_t C,
                                      const float* gamma, const float* beta,
                                      float* running_mean, float* running_var, float momentum,
                                      float eps, int act, float slope, void* y, float* stats,
                                      void* ws, size_t ws_bytes, void* stream);

/* Centred apply (optionally through act) for channels-last x, as
 * gbn_bn_apply_act: from a training stats buffer when `stats` is non-NULL,
 * else from per-channel mean and scale (fp32 [C], e.g. the running mean and
 * gamma/sqrt(running_var + eps)).  No workspace.  y may alias x.          */
GBN_API int gbn_bn_nhwc_apply(const void* x, int dtype, int64_t M, int64_t C,
                              const float* stats, const float* mean, const float* scale,
                              const float* beta, int act, float slope, void* y, void* stream);

/* Training backward from the matching forward's stats (and its beta when an
 * activation is fused): writes dx and grads (fp32 [4, C]).  dx may alias dy. */
GBN_API int gbn_bn_nhwc_backward(const void* x, const void* dy, int dtype, int64_t M,
                                 int64_t C, const float* stats, const float* beta, int act,
                                 float slope, void* dx, float* grads, void* ws,
                                 size_t ws_bytes, void* stream);

/* =========================================================================
 * Row-wise backward passes: RMSNorm ([P3]) and LayerNorm ([P2]).
 *
 * Tensors are [R, H] row-major in `dtype` unless stated.  One persistent
 * launch streams rows through shared memory with bulk copies, reduces each
 * row with warp shuffles while the row is on chip (x and dy are read once),
 * and accumulates the per-column sums of its rows in registers; a second
 * small launch (programmatic dependent launch) adds the per-block column
 * partials in a fixed order.  The column reductions therefore never re-read
 * the [R, H] inputs.
 * ======================================================================= */

/* Workspace bytes for a row-wise backward of kind GBN_ROW_* and `dtype` on
 * `device` (-1: current).  Returns 0 on a bad shape or a CUDA error.        */
GBN_API size_t gbn_rowwise_workspace_bytes(int64_t R, int64_t H, int kind, int dtype,
                                   int device);

/* RMSNorm backward ([P3] rmsnorm_bwd_fusion, with the saved statistic taken
 * as rstd = 1/rms, fp32 [R]):
 *   S_r   = sum_j w_j*dy_rj*x_rj
 *   dx_rj = rstd_r*w_j*dy_rj - x_rj*rstd_r^3*S_r/H
 *   dw_j  = sum_r dy_rj*x_rj*rstd_r        (written in `dtype`)
 * dy, x, dx: [R, H]; w, dw: [H].                                            */
GBN_API int gbn_rmsnorm_backward(const void* dy, const void* x, const void* w,
                         int dtype, const float* rstd, int64_t R, int64_t H,
                         void* dx, void* dw, void* ws, size_t ws_bytes,
                         void* stream);

/* LayerNorm backward, plain or fused with bias+dropout+add ([P2]).
 * mean, rstd: fp32 [R] saved by the forward; gamma: [H].
 *
 * Plain (residual == NULL; bias, mask, dresidual, dbias must be NULL):
 *   z = x_or_input (the LayerNorm input), dx = dz (+ dz_extra).
 * Fused (residual != NULL): the LayerNorm input is recomputed in fp32 as
 *   z = residual + mask*dropout_scale*(x_or_input + bias)
 *   dresidual = dz (+ dz_extra), dx = dresidual*dropout_scale*mask,
 *   dbias = sum_rows dx.
 * with xhat = (z-mean)*rstd, g = dy*gamma and
 *   dz = rstd*(g - mean_j(g) - xhat*mean_j(g*xhat)).
 * Column sums: dgamma = sum_rows dy*xhat, dbeta = sum_rows dy.
 * mask: uint8 [R, H] (nonzero = kept) or NULL (all kept).  bias: [H] or NULL.
 * dz_extra: fp32 [R, H] or NULL (an extra gradient arriving at z).
 * dresidual, dgamma, dbeta, dbias may be NULL (not written).  Outputs are in
 * `dtype`.                                                                 */
GBN_API int gbn_layernorm_backward(const void* dy, const void* x_or_input, int dtype,
                           const float* mean, const float* rstd,
                           const void* gamma, int64_t R, int64_t H,
                           const void* residual, const void* bias,
                           const uint8_t* mask, float dropout_scale,
                           const float* dz_extra, void* dx, void* dresidual,
                           void* dgamma, void* dbeta, void* dbias, void* ws,
                           size_t ws_bytes, void* stream);

/* Flags of gbn_layernorm_backward_ex.                                       */
#define GBN_LN_SAVED_Z  1  /* x_or_input is the saved LayerNorm input z        */
#define GBN_LN_DRES_F32 2  /* dresidual is written as fp32 (as [P2] emits it)  */

/* gbn_layernorm_backward with variants ([P2] nvfuser_fusion_id9, where the
 * LayerNorm input and the residual gradient are fp32 tensors):
 *   GBN_LN_SAVED_Z: x_or_input is z itself (e.g. the z written by
 *     gbn_layernorm_forward) instead of the dropout input; residual and bias
 *     must be NULL.  The fused outputs are still produced from mask and
 *     dropout_scale: dresidual = dz (+ dz_extra), dx = dresidual*scale*mask,
 *     dbias = sum_rows dx (each may be NULL).
 *   GBN_LN_DRES_F32: dresidual is an fp32 [R, H] tensor (no effect when
 *     dtype is already GBN_F32).
 * Unknown flag bits return GBN_EINVAL.  flags = 0 is gbn_layernorm_backward. */
GBN_API int gbn_layernorm_backward_ex(const void* dy, const void* x_or_input, int dtype,
                                      const float* mean, const float* rstd,
                                      const void* gamma, int64_t R, int64_t H,
                                      const void* residual, const void* bias,
                                      const uint8_t* mask, float dropout_scale,
                                      const float* dz_extra, void* dx, void* dresidual,
                                      void* dgamma, void* dbeta, void* dbias, void* ws,
                                      size_t ws_bytes, int flags, void* stream);

/* =========================================================================
 * Row-wise training forwards: RMSNorm ([P3]) and LayerNorm ([P2]), writing
 * the statistics the backward passes above take.  Tensors are [R, H]
 * row-major in `dtype`; statistics are fp32 [R].  Each row is loaded once
 * into registers (one warp per row up to 256 16-byte vectors, one block per
 * row up to 2048), reduced with warp shuffles and written back; longer or
 * unaligned rows take a block-per-row kernel that re-reads the row from L2.
 * No workspace.  H must be positive when R > 0.
 * ======================================================================= */

/* RMSNorm forward ([P3] the rmsnorm_prims / F.rms_norm section):
 *   rstd_r = 1/sqrt(mean_j x_rj^2 + eps),   y_rj = x_rj*rstd_r*w_j.
 * x, y: [R, H]; w: [H] or NULL (ones); rstd: fp32 [R] (written); eps >= 0.
 * Returns GBN_EINVAL for a null x / y / rstd or H == 0 with R > 0.        */
GBN_API int gbn_rmsnorm_forward(const void* x, const void* w, int dtype, int64_t R,
                                int64_t H, float eps, void* y, float* rstd, void* stream);

/* LayerNorm forward, plain or fused with bias+dropout+add ([P2]: the
 * forward whose saved fp32 mean and rstd the backward repros take).
 * Plain (residual == NULL; bias, mask, z must be NULL): z = x_or_input.
 * Fused (residual != NULL): z = residual + mask*dropout_scale*(x_or_input +
 *   bias) in fp32, written to `z` (the residual-stream output) unless NULL.
 * Then mean_r = mean_j z_rj, rstd_r = 1/sqrt(mean_j (z_rj - mean_r)^2 + eps)
 * (biased variance, as a second pass) and
 *   y_rj = (z_rj - mean_r)*rstd_r*gamma_j + beta_j.
 * gamma, beta, bias: [H] or NULL (ones / zeros / none); mask: uint8 [R, H]
 * (nonzero = kept) or NULL; mean, rstd: fp32 [R] (written).               */
GBN_API int gbn_layernorm_forward(const void* x_or_input, int dtype, int64_t R, int64_t H,
                                  const void* residual, const void* bias,
                                  const uint8_t* mask, float dropout_scale,
                                  const void* gamma, const void* beta, float eps, void* y,
                                  void* z, float* mean, float* rstd, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBNORM_H */
