// extern "C" entry points of libgbnorm.so (declared in include/gbnorm.h).
//
// Every entry point validates its arguments before touching CUDA, so an
// argument error launches nothing and writes nothing; then it plans the
// launch from cached device attributes and launches on the caller's stream.
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>

#include "gbn_internal.h"

namespace gbn {

namespace {

// Device status word (bit set of GBN_DEV_*).  Kernels receive its device
// address; the host reads it with gbn_get_device_status.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  explicit DeviceGuard(int device) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != device) {
      switched = cudaSetDevice(device) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// a*b without int64 overflow; false on overflow or negative operands.
inline bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > LLONG_MAX / a) return false;
  *out = a * b;
  return true;
}

int bn_check(int dtype, int64_t B, int64_t C, int64_t HW, bool training, int64_t* M) {
  if (dtype != GBN_F32 && dtype != GBN_BF16) return GBN_EDTYPE;
  if (B < 0 || C < 0 || HW < 0) return GBN_EINVAL;
  if (C > INT32_MAX || HW > INT32_MAX) return GBN_EINVAL;
  int64_t bc, n;
  if (!mul_ok(B, C, &bc) || !mul_ok(bc, HW, &n) || n > (LLONG_MAX >> 3)) return GBN_EINVAL;
  if (!mul_ok(B, HW, M) || *M > INT32_MAX) return GBN_EINVAL;  // per-channel count < 2^31
  if (training && C > 0 && *M < 2) return GBN_EINVAL;
  return GBN_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? GBN_OK : GBN_ECUDA; }

}  // namespace

const DevInfo* device_info(int device) {
  if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return nullptr;
  if (device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[device];
  if (d.ok) return &d;
  DeviceGuard guard(device);
  DevInfo n;
  if (cudaDeviceGetAttribute(&n.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&n.max_threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&n.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&n.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                             device) != cudaSuccess ||
      cudaDeviceGetAttribute(&n.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&n.l2_bytes, cudaDevAttrL2CacheSize, device) != cudaSuccess)
    return nullptr;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
  n.status = static_cast<int*>(addr);
  if (row_kernels_configure(n.smem_optin) != cudaSuccess) return nullptr;
  if (bn_fused_configure(n.smem_optin, &n.fused_ok) != cudaSuccess) return nullptr;
  if (row_fwd_configure() != cudaSuccess) return nullptr;
  n.ok = true;
  d = n;
  return &d;
}

}  // namespace gbn

using namespace gbn;

extern "C" {

int gbn_abi_version(void) { return 1; }

const char* gbn_status_string(int status) {
  switch (status) {
    case GBN_OK: return "ok";
    case GBN_EINVAL: return "invalid argument (null pointer, bad size or combination)";
    case GBN_EDTYPE: return "unsupported dtype (expected GBN_F32 or GBN_BF16)";
    case GBN_EALIGN: return "misaligned buffer (stats needs 8 bytes, workspace 16 bytes)";
    case GBN_EWORKSPACE: return "workspace too small";
    case GBN_ECUDA: return "CUDA runtime error";
    case GBN_EDEVICE: return "a kernel reported an error in the device status word";
    default: return "unknown status";
  }
}

int gbn_init(int device) { return device_info(device) ? GBN_OK : GBN_ECUDA; }

int gbn_get_device_status(int device, int* status, int clear) {
  if (status == nullptr) return GBN_EINVAL;
  if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return GBN_ECUDA;
  if (!device_info(device)) return GBN_ECUDA;
  DeviceGuard guard(device);
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return GBN_ECUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return GBN_ECUDA;
  }
  *status = v;
  return GBN_OK;
}

int gbn_selftest_bounded_wait(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000ll) return GBN_EINVAL;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  return to_status(selftest_bounded_wait(dev->status, (uint64_t)limit_ns,
                                         static_cast<cudaStream_t>(stream)));
}

// ----------------------------------------------------------- BatchNorm --

size_t gbn_bn_workspace_bytes(int64_t B, int64_t C, int64_t HW, int device) {
  int64_t M;
  if (bn_check(GBN_F32, B, C, HW, false, &M) != GBN_OK) return 0;
  const DevInfo* dev = device_info(device);
  if (!dev) return 0;
  BnPlan p;
  if (!bn_plan(B, C, HW, *dev, &p)) return 0;
  return p.ws_bytes;
}

static int bn_prepare(int dtype, int64_t B, int64_t C, int64_t HW, bool training,
                      const void* const* ptrs, int nptrs, const void* ws, size_t ws_bytes,
                      bool need_ws, BnPlan* plan, const DevInfo** dev_out,
                      bool partials_only = false) {
  int64_t M;
  const int rc = bn_check(dtype, B, C, HW, training, &M);
  if (rc != GBN_OK) return rc;
  if (need_ws && ws != nullptr && !aligned(ws, 16)) return GBN_EALIGN;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  if (!bn_plan(B, C, HW, *dev, plan)) return GBN_EINVAL;
  if (need_ws && (ws == nullptr)) return GBN_EINVAL;
  if (need_ws && ws_bytes < (partials_only ? plan->ws_partials : plan->ws_bytes))
    return GBN_EWORKSPACE;
  plan->vec = bn_vec_width(dtype, HW, ptrs, nptrs);
  *dev_out = dev;
  return GBN_OK;
}

static bool bn_empty(int64_t B, int64_t C, int64_t HW) { return C == 0 || B == 0 || HW == 0; }

// Inputs (x, and dy backward) below this many bytes per call run the
// two-launch kernels even when the persistent kernel could take them: the
// cooperative launch and its flag handshake cost more than the re-read they
// save on small tensors (GB300: two-launch ahead up to ~100 MB, behind from
// ~200 MB).
static std::atomic<int64_t> g_fused_min_bytes{128ll << 20};

// Channels of at most this many elements (M = B*HW) run the single-launch
// small-channel kernels in the composite calls (below the persistent
// kernel's threshold); 0 disables them.
static std::atomic<int64_t> g_small_max_m{kBnSmallMaxM};

// act one of GBN_ACT_*; LeakyReLU's slope finite.
static bool act_ok(int act, float slope) {
  if (act == GBN_ACT_NONE || act == GBN_ACT_RELU) return true;
  return act == GBN_ACT_LEAKY_RELU && slope - slope == 0.f;
}

int gbn_bn_stats(const void* x, int dtype, int64_t B, int64_t C, int64_t HW, void* ws,
                 size_t ws_bytes, void* stream) {
  int64_t M;
  int rc = bn_check(dtype, B, C, HW, true, &M);
  if (rc != GBN_OK) return rc;
  if (C == 0) return GBN_OK;
  if (x == nullptr || ws == nullptr) return GBN_EINVAL;
  const void* ptrs[1] = {x};
  BnPlan p;
  const DevInfo* dev;
  rc = bn_prepare(dtype, B, C, HW, true, ptrs, 1, ws, ws_bytes, true, &p, &dev);
  if (rc != GBN_OK) return rc;
  return to_status(bn_launch_stats(x, dtype, p, static_cast<float2*>(ws),
                                   static_cast<cudaStream_t>(stream)));
}

static int bn_finalize_apply_impl(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                                  const float* gamma, const float* beta, float* running_mean,
                                  float* running_var, float momentum, float eps, void* y,
                                  float* stats, const void* ws, size_t ws_bytes, void* stream,
                                  bool with_stats_pass, bool partials_only = false,
                                  int act = GBN_ACT_NONE, float slope = 0.f) {
  int64_t M;
  int rc = bn_check(dtype, B, C, HW, true, &M);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (C == 0) return GBN_OK;
  if (x == nullptr || y == nullptr || stats == nullptr || ws == nullptr) return GBN_EINVAL;
  if (!aligned(stats, 8)) return GBN_EALIGN;
  if (!(eps >= 0.f) || momentum != momentum) return GBN_EINVAL;
  const void* ptrs[2] = {x, y};
  BnPlan p;
  const DevInfo* dev;
  rc = bn_prepare(dtype, B, C, HW, true, ptrs, 2, ws, ws_bytes, true, &p, &dev, partials_only);
  if (rc != GBN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float2* part = static_cast<float2*>(const_cast<void*>(ws));
  BnFusedPlan fp;
  const int64_t in_bytes = B * C * HW * (dtype == GBN_F32 ? 4 : 2);
  if (with_stats_pass && in_bytes >= g_fused_min_bytes.load() && aligned(x, 16) &&
      aligned(y, 16) && bn_fused_plan(dtype, false, B, C, HW, *dev, &fp) &&
      ws_bytes >= fp.ws_bytes)
    return to_status(bn_fused_forward(fp, dtype, x, y, gamma, beta, stats, running_mean,
                                      running_var, momentum, eps, act, slope,
                                      const_cast<void*>(ws), dev->status, st));
  const int K = with_stats_pass ? bn_small_blocks(M, C, g_small_max_m.load(), *dev) : 0;
  if (K > 0)
    return to_status(bn_small_forward(dtype, x, y, B, C, HW, gamma, beta, stats, running_mean,
                                      running_var, momentum, eps, act, slope, K, st));
  if (with_stats_pass) {
    cudaError_t e = bn_launch_stats(x, dtype, p, part, st);
    if (e != cudaSuccess) return GBN_ECUDA;
  }
  return to_status(bn_launch_apply(x, y, dtype, p, kApplyTrain, part, gamma, beta, stats,
                                   running_mean, running_var, momentum, eps, nullptr, nullptr, act,
                                   slope, st, /*pdl=*/true));
}

}  // extern "C"

namespace gbn {

size_t bn_partials_bytes(int64_t B, int64_t C, int64_t HW) {
  int64_t M;
  if (bn_check(GBN_F32, B, C, HW, false, &M) != GBN_OK) return 0;
  const DevInfo* dev = device_info(-1);
  BnPlan p;
  if (!dev || !bn_plan(B, C, HW, *dev, &p)) return 0;
  return p.ws_partials;
}

int bn_forward_check_args(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                          const void* y, const float* stats, float momentum, float eps) {
  int64_t M;
  const int rc = bn_check(dtype, B, C, HW, true, &M);
  if (rc != GBN_OK || C == 0) return rc;
  if (x == nullptr || y == nullptr || stats == nullptr) return GBN_EINVAL;
  if (!aligned(stats, 8)) return GBN_EALIGN;
  if (!(eps >= 0.f) || momentum != momentum) return GBN_EINVAL;
  return GBN_OK;
}

int bn_forward_train_scratch(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                             const float* gamma, const float* beta, float* running_mean,
                             float* running_var, float momentum, float eps, void* y,
                             float* stats, void* ws, size_t ws_bytes, void* stream) {
  return bn_finalize_apply_impl(x, dtype, B, C, HW, gamma, beta, running_mean, running_var,
                                momentum, eps, y, stats, ws, ws_bytes, stream, true, true);
}

}  // namespace gbn

extern "C" {

int64_t gbn_bn_set_persistent_min_bytes(int64_t bytes) {
  return g_fused_min_bytes.exchange(bytes < 0 ? 0 : bytes);
}

int64_t gbn_bn_persistent_min_bytes(void) { return g_fused_min_bytes.load(); }

int64_t gbn_bn_small_max_elems(void) { return g_small_max_m.load(); }

int gbn_bn_small_blocks_per_channel(int64_t B, int64_t C, int64_t HW) {
  int64_t M;
  if (bn_check(GBN_F32, B, C, HW, false, &M) != GBN_OK) return 0;
  const DevInfo* dev = device_info(-1);
  if (dev == nullptr) {
    cudaGetLastError();
    return 0;
  }
  return bn_small_blocks(M, C, g_small_max_m.load(), *dev);
}

int64_t gbn_bn_set_small_max_elems(int64_t m) {
  if (m < 0) m = 0;
  if (m > kBnSmallMaxM) m = kBnSmallMaxM;
  return g_small_max_m.exchange(m);
}

int gbn_bn_set_wide_offsets(int force) { return bn_set_wide_offsets(force); }

int gbn_bn_set_persistent_tmem(int enable) { return bn_fused_set_tmem(enable); }

int gbn_bn_set_persistent_steal(int enable) { return bn_fused_set_steal(enable); }

int gbn_bn_forward_train(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                         const float* gamma, const float* beta, float* running_mean,
                         float* running_var, float momentum, float eps, void* y, float* stats,
                         void* ws, size_t ws_bytes, void* stream) {
  return bn_finalize_apply_impl(x, dtype, B, C, HW, gamma, beta, running_mean, running_var,
                                momentum, eps, y, stats, ws, ws_bytes, stream, true);
}

int gbn_bn_finalize_apply(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                          const float* gamma, const float* beta, float* running_mean,
                          float* running_var, float momentum, float eps, void* y, float* stats,
                          const void* ws, size_t ws_bytes, void* stream) {
  return bn_finalize_apply_impl(x, dtype, B, C, HW, gamma, beta, running_mean, running_var,
                                momentum, eps, y, stats, ws, ws_bytes, stream, false);
}

int gbn_bn_forward_train_act(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                             const float* gamma, const float* beta, float* running_mean,
                             float* running_var, float momentum, float eps, int act, float slope,
                             void* y, float* stats, void* ws, size_t ws_bytes, void* stream) {
  return bn_finalize_apply_impl(x, dtype, B, C, HW, gamma, beta, running_mean, running_var,
                                momentum, eps, y, stats, ws, ws_bytes, stream, true, false, act,
                                slope);
}

static int bn_apply_impl(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                         const float* stats, const float* mean, const float* scale,
                         const float* beta, int act, float slope, void* y, void* stream) {
  int64_t M;
  int rc = bn_check(dtype, B, C, HW, false, &M);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (bn_empty(B, C, HW)) return GBN_OK;
  if (x == nullptr || y == nullptr) return GBN_EINVAL;
  if (stats == nullptr && (mean == nullptr || scale == nullptr)) return GBN_EINVAL;
  if (stats != nullptr && !aligned(stats, 8)) return GBN_EALIGN;
  const void* ptrs[2] = {x, y};
  BnPlan p;
  const DevInfo* dev;
  rc = bn_prepare(dtype, B, C, HW, false, ptrs, 2, nullptr, 0, false, &p, &dev);
  if (rc != GBN_OK) return rc;
  return to_status(bn_launch_apply(x, y, dtype, p, stats ? kApplyStats : kApplyInfer, nullptr,
                                   nullptr, beta, const_cast<float*>(stats), nullptr, nullptr,
                                   0.f, 0.f, mean, scale, act, slope,
                                   static_cast<cudaStream_t>(stream), /*pdl=*/false));
}

int gbn_bn_apply(const void* x, int dtype, int64_t B, int64_t C, int64_t HW, const float* stats,
                 const float* mean, const float* scale, const float* beta, void* y,
                 void* stream) {
  return bn_apply_impl(x, dtype, B, C, HW, stats, mean, scale, beta, GBN_ACT_NONE, 0.f, y,
                       stream);
}

int gbn_bn_apply_act(const void* x, int dtype, int64_t B, int64_t C, int64_t HW,
                     const float* stats, const float* mean, const float* scale, const float* beta,
                     int act, float slope, void* y, void* stream) {
  return bn_apply_impl(x, dtype, B, C, HW, stats, mean, scale, beta, act, slope, y, stream);
}

static int bn_backward_impl(const void* x, const void* dy, int dtype, int64_t B, int64_t C,
                            int64_t HW, const float* stats, void* dx, float* grads,
                            const void* ws, size_t ws_bytes, void* stream, bool sums,
                            bool finalize, const float* beta = nullptr, int act = GBN_ACT_NONE,
                            float slope = 0.f) {
  int64_t M;
  int rc = bn_check(dtype, B, C, HW, true, &M);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (C == 0) return GBN_OK;
  if (x == nullptr || dy == nullptr || stats == nullptr || ws == nullptr) return GBN_EINVAL;
  if (finalize && (dx == nullptr || grads == nullptr)) return GBN_EINVAL;
  if (!aligned(stats, 8)) return GBN_EALIGN;
  const void* ptrs[3] = {x, dy, finalize ? dx : nullptr};
  BnPlan p;
  const DevInfo* dev;
  rc = bn_prepare(dtype, B, C, HW, true, ptrs, 3, ws, ws_bytes, true, &p, &dev);
  if (rc != GBN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float2* part = static_cast<float2*>(const_cast<void*>(ws));
  BnFusedPlan fp;
  const int64_t in_bytes = 2 * B * C * HW * (dtype == GBN_F32 ? 4 : 2);
  if (sums && finalize && in_bytes >= g_fused_min_bytes.load() && aligned(x, 16) &&
      aligned(dy, 16) && aligned(dx, 16) && bn_fused_plan(dtype, true, B, C, HW, *dev, &fp) &&
      ws_bytes >= fp.ws_bytes)
    return to_status(bn_fused_backward(fp, dtype, x, dy, dx, stats, beta, act, slope, grads,
                                       const_cast<void*>(ws), dev->status, st));
  const int K = sums && finalize ? bn_small_blocks(M, C, g_small_max_m.load(), *dev) : 0;
  if (K > 0)
    return to_status(bn_small_backward(dtype, x, dy, dx, B, C, HW, stats, beta, act, slope,
                                       grads, K, st));
  if (sums) {
    cudaError_t e = bn_launch_grad_sums(x, dy, dtype, p, stats, part, beta, act, slope, st);
    if (e != cudaSuccess) return GBN_ECUDA;
  }
  if (finalize)
    return to_status(bn_launch_dx(x, dy, dx, dtype, p, stats, part, grads, beta, act, slope, st,
                                  /*pdl=*/true));
  return GBN_OK;
}

int gbn_bn_backward(const void* x, const void* dy, int dtype, int64_t B, int64_t C, int64_t HW,
                    const float* stats, void* dx, float* grads, void* ws, size_t ws_bytes,
                    void* stream) {
  return bn_backward_impl(x, dy, dtype, B, C, HW, stats, dx, grads, ws, ws_bytes, stream, true,
                          true);
}

int gbn_bn_backward_act(const void* x, const void* dy, int dtype, int64_t B, int64_t C,
                        int64_t HW, const float* stats, const float* beta, int act, float slope,
                        void* dx, float* grads, void* ws, size_t ws_bytes, void* stream) {
  return bn_backward_impl(x, dy, dtype, B, C, HW, stats, dx, grads, ws, ws_bytes, stream, true,
                          true, beta, act, slope);
}

int gbn_bn_grad_sums(const void* x, const void* dy, int dtype, int64_t B, int64_t C, int64_t HW,
                     const float* stats, void* ws, size_t ws_bytes, void* stream) {
  return bn_backward_impl(x, dy, dtype, B, C, HW, stats, nullptr, nullptr, ws, ws_bytes, stream,
                          true, false);
}

int gbn_bn_finalize_dx(const void* x, const void* dy, int dtype, int64_t B, int64_t C,
                       int64_t HW, const float* stats, void* dx, float* grads, const void* ws,
                       size_t ws_bytes, void* stream) {
  return bn_backward_impl(x, dy, dtype, B, C, HW, stats, dx, grads, ws, ws_bytes, stream, false,
                          true);
}

// ------------------------------------------------- BatchNorm, NHWC --

static int nhwc_check(int dtype, int64_t M, int64_t C, bool training) {
  if (dtype != GBN_F32 && dtype != GBN_BF16) return GBN_EDTYPE;
  if (M < 0 || C < 0 || C > INT32_MAX || M > INT32_MAX) return GBN_EINVAL;
  int64_t n;
  if (!mul_ok(M, C, &n) || n > (LLONG_MAX >> 3)) return GBN_EINVAL;
  if (training && C > 0 && M < 2) return GBN_EINVAL;
  return GBN_OK;
}

size_t gbn_bn_nhwc_workspace_bytes(int64_t M, int64_t C, int device) {
  if (nhwc_check(GBN_F32, M, C, false) != GBN_OK) return 0;
  if (C == 0) return 256;
  const DevInfo* dev = device_info(device);
  if (!dev) return 0;
  return nhwc_ws_bound(M, C, *dev);
}

int gbn_bn_nhwc_forward_train(const void* x, int dtype, int64_t M, int64_t C, const float* gamma,
                              const float* beta, float* running_mean, float* running_var,
                              float momentum, float eps, int act, float slope, void* y,
                              float* stats, void* ws, size_t ws_bytes, void* stream) {
  int rc = nhwc_check(dtype, M, C, true);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (C == 0) return GBN_OK;
  if (x == nullptr || y == nullptr || stats == nullptr || ws == nullptr) return GBN_EINVAL;
  if (!aligned(ws, 16) || !aligned(stats, 4)) return GBN_EALIGN;
  if (!(eps >= 0.f) || momentum != momentum) return GBN_EINVAL;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const void* ptrs[2] = {x, y};
  NhwcPlan p;
  if (!nhwc_plan(M, C, bn_vec_width(dtype, C, ptrs, 2), *dev, &p)) return GBN_EINVAL;
  if (ws_bytes < p.ws_bytes) return GBN_EWORKSPACE;
  return to_status(nhwc_forward(p, dtype, x, y, gamma, beta, stats, running_mean, running_var,
                                momentum, eps, act, slope, ws, static_cast<cudaStream_t>(stream)));
}

int gbn_bn_nhwc_apply(const void* x, int dtype, int64_t M, int64_t C, const float* stats,
                      const float* mean, const float* scale, const float* beta, int act,
                      float slope, void* y, void* stream) {
  int rc = nhwc_check(dtype, M, C, false);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (C == 0 || M == 0) return GBN_OK;
  if (x == nullptr || y == nullptr) return GBN_EINVAL;
  if (stats == nullptr && (mean == nullptr || scale == nullptr)) return GBN_EINVAL;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const void* ptrs[2] = {x, y};
  NhwcPlan p;
  if (!nhwc_plan(M, C, bn_vec_width(dtype, C, ptrs, 2), *dev, &p)) return GBN_EINVAL;
  return to_status(nhwc_apply(p, dtype, x, y, stats, mean, scale, beta, act, slope,
                              static_cast<cudaStream_t>(stream)));
}

int gbn_bn_nhwc_backward(const void* x, const void* dy, int dtype, int64_t M, int64_t C,
                         const float* stats, const float* beta, int act, float slope, void* dx,
                         float* grads, void* ws, size_t ws_bytes, void* stream) {
  int rc = nhwc_check(dtype, M, C, true);
  if (rc != GBN_OK) return rc;
  if (!act_ok(act, slope)) return GBN_EINVAL;
  if (C == 0) return GBN_OK;
  if (x == nullptr || dy == nullptr || dx == nullptr || stats == nullptr || grads == nullptr ||
      ws == nullptr)
    return GBN_EINVAL;
  if (!aligned(ws, 16) || !aligned(stats, 4)) return GBN_EALIGN;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const void* ptrs[3] = {x, dy, dx};
  NhwcPlan p;
  if (!nhwc_plan(M, C, bn_vec_width(dtype, C, ptrs, 3), *dev, &p)) return GBN_EINVAL;
  if (ws_bytes < p.ws_bytes) return GBN_EWORKSPACE;
  return to_status(nhwc_backward(p, dtype, x, dy, dx, stats, beta, act, slope, grads, ws,
                                 static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------ row-wise --

static int row_check(int dtype, int64_t R, int64_t H) {
  if (dtype != GBN_F32 && dtype != GBN_BF16) return GBN_EDTYPE;
  if (R < 0 || H < 0 || H > INT32_MAX / 16) return GBN_EINVAL;
  int64_t n;
  if (!mul_ok(R, H, &n) || n > (LLONG_MAX >> 3)) return GBN_EINVAL;
  return GBN_OK;
}

size_t gbn_rowwise_workspace_bytes(int64_t R, int64_t H, int kind, int dtype, int device) {
  if (row_check(dtype, R, H) != GBN_OK) return 0;
  const DevInfo* dev = device_info(device);
  if (!dev) return 0;
  RowPlan a, b;
  if (!row_plan(R, H, kind, dtype, true, false, false, *dev, &a)) return 0;
  if (!row_plan(R, H, kind, dtype, false, false, false, *dev, &b)) return 0;
  return a.ws_bytes > b.ws_bytes ? a.ws_bytes : b.ws_bytes;
}

int gbn_rmsnorm_backward(const void* dy, const void* x, const void* w, int dtype,
                         const float* rstd, int64_t R, int64_t H, void* dx, void* dw, void* ws,
                         size_t ws_bytes, void* stream) {
  int rc = row_check(dtype, R, H);
  if (rc != GBN_OK) return rc;
  if (H == 0) return GBN_OK;
  if (w == nullptr || dw == nullptr || ws == nullptr) return GBN_EINVAL;
  if (R > 0 && (dy == nullptr || x == nullptr || rstd == nullptr || dx == nullptr))
    return GBN_EINVAL;
  if (!aligned(ws, 16)) return GBN_EALIGN;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const bool fast_ok = aligned(dy, 16) && aligned(x, 16) && aligned(w, 16) && aligned(dx, 16);
  RowPlan p;
  if (!row_plan(R, H, GBN_ROW_RMS, dtype, fast_ok, false, false, *dev, &p)) return GBN_EINVAL;
  if (ws_bytes < p.ws_bytes) return GBN_EWORKSPACE;
  return to_status(rms_launch(p, dy, x, w, rstd, dx, dw, ws, dev->status,
                              static_cast<cudaStream_t>(stream)));
}

int gbn_layernorm_backward_ex(const void* dy, const void* x_or_input, int dtype,
                              const float* mean, const float* rstd, const void* gamma, int64_t R,
                              int64_t H, const void* residual, const void* bias,
                              const uint8_t* mask, float dropout_scale, const float* dz_extra,
                              void* dx, void* dresidual, void* dgamma, void* dbeta, void* dbias,
                              void* ws, size_t ws_bytes, int flags, void* stream) {
  int rc = row_check(dtype, R, H);
  if (rc != GBN_OK) return rc;
  if (flags & ~(GBN_LN_SAVED_Z | GBN_LN_DRES_F32)) return GBN_EINVAL;
  const bool saved_z = (flags & GBN_LN_SAVED_Z) != 0;
  if (saved_z && (residual || bias)) return GBN_EINVAL;  // z already holds them
  const bool fused = residual != nullptr || saved_z;
  if (!fused && (bias || mask || dresidual || dbias)) return GBN_EINVAL;
  if (H == 0) return GBN_OK;
  if (gamma == nullptr || ws == nullptr) return GBN_EINVAL;
  if (R > 0 && (dy == nullptr || x_or_input == nullptr || mean == nullptr || rstd == nullptr ||
                dx == nullptr))
    return GBN_EINVAL;
  if (dropout_scale != dropout_scale) return GBN_EINVAL;
  if (!aligned(ws, 16)) return GBN_EALIGN;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const bool fast_ok = aligned(dy, 16) && aligned(x_or_input, 16) && aligned(gamma, 16) &&
                       aligned(dx, 16) && aligned(residual, 16) && aligned(bias, 16) &&
                       aligned(mask, 16) && aligned(dz_extra, 16) && aligned(dresidual, 16);
  const int kind = fused ? GBN_ROW_LN_FUSED : GBN_ROW_LN;
  RowPlan p;
  if (!row_plan(R, H, kind, dtype, fast_ok, mask != nullptr, dz_extra != nullptr, *dev, &p))
    return GBN_EINVAL;
  if (ws_bytes < p.ws_bytes) return GBN_EWORKSPACE;
  LnPtrs q;
  q.dy = dy;
  q.x = x_or_input;
  q.residual = residual;
  q.bias = bias;
  q.mask = mask;
  q.dz_extra = dz_extra;
  q.mean = mean;
  q.rstd = rstd;
  q.gamma = gamma;
  q.scale = fused ? dropout_scale : 1.f;
  q.dx = dx;
  q.dres = dresidual;
  q.dgamma = dgamma;
  q.dbeta = dbeta;
  q.dbias = dbias;
  q.saved_z = saved_z;
  q.dres_f32 = (flags & GBN_LN_DRES_F32) != 0 && dtype != GBN_F32;
  return to_status(ln_launch(p, q, ws, dev->status,
                             static_cast<cudaStream_t>(stream)));
}

int gbn_layernorm_backward(const void* dy, const void* x_or_input, int dtype, const float* mean,
                           const float* rstd, const void* gamma, int64_t R, int64_t H,
                           const void* residual, const void* bias, const uint8_t* mask,
                           float dropout_scale, const float* dz_extra, void* dx,
                           void* dresidual, void* dgamma, void* dbeta, void* dbias, void* ws,
                           size_t ws_bytes, void* stream) {
  return gbn_layernorm_backward_ex(dy, x_or_input, dtype, mean, rstd, gamma, R, H, residual,
                                   bias, mask, dropout_scale, dz_extra, dx, dresidual, dgamma,
                                   dbeta, dbias, ws, ws_bytes, 0, stream);
}

// ------------------------------------------------------ row-wise forward --

int gbn_rmsnorm_forward(const void* x, const void* w, int dtype, int64_t R, int64_t H, float eps,
                        void* y, float* rstd, void* stream) {
  int rc = row_check(dtype, R, H);
  if (rc != GBN_OK) return rc;
  if (!(eps >= 0.f)) return GBN_EINVAL;
  if (R == 0) return GBN_OK;
  if (rstd == nullptr) return GBN_EINVAL;
  if (H > 0 && (x == nullptr || y == nullptr)) return GBN_EINVAL;
  if (H == 0) return GBN_EINVAL;  // the mean over an empty row is undefined
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const int64_t esize = dtype == GBN_F32 ? 4 : 2;
  const bool vec_ok = (H * esize) % 16 == 0 && aligned(x, 16) && aligned(w, 16) && aligned(y, 16);
  RowFwdPtrs q;
  q.x = x;
  q.w = w;
  q.y = y;
  q.rstd = rstd;
  return to_status(row_fwd_launch(GBN_ROW_RMS, dtype, q, R, H, eps, 1.f, vec_ok, *dev,
                                  static_cast<cudaStream_t>(stream)));
}

int gbn_layernorm_forward(const void* x_or_input, int dtype, int64_t R, int64_t H,
                          const void* residual, const void* bias, const uint8_t* mask,
                          float dropout_scale, const void* gamma, const void* beta, float eps,
                          void* y, void* z, float* mean, float* rstd, void* stream) {
  int rc = row_check(dtype, R, H);
  if (rc != GBN_OK) return rc;
  const bool fused = residual != nullptr;
  if (!fused && (bias || mask || z)) return GBN_EINVAL;
  if (!(eps >= 0.f) || dropout_scale != dropout_scale) return GBN_EINVAL;
  if (R == 0) return GBN_OK;
  if (mean == nullptr || rstd == nullptr) return GBN_EINVAL;
  if (H == 0) return GBN_EINVAL;  // the mean over an empty row is undefined
  if (x_or_input == nullptr || y == nullptr) return GBN_EINVAL;
  const DevInfo* dev = device_info(-1);
  if (!dev) return GBN_ECUDA;
  const int64_t esize = dtype == GBN_F32 ? 4 : 2;
  const bool vec_ok = (H * esize) % 16 == 0 && (mask == nullptr || H % 16 == 0) &&
                      aligned(x_or_input, 16) && aligned(residual, 16) && aligned(bias, 16) &&
                      aligned(mask, 16) && aligned(gamma, 16) && aligned(beta, 16) &&
                      aligned(y, 16) && aligned(z, 16);
  RowFwdPtrs q;
  q.x = x_or_input;
  q.residual = residual;
  q.bias = bias;
  q.mask = mask;
  q.w = gamma;
  q.beta = beta;
  q.y = y;
  q.z = z;
  q.mean = mean;
  q.rstd = rstd;
  return to_status(row_fwd_launch(fused ? GBN_ROW_LN_FUSED : GBN_ROW_LN, dtype, q, R, H, eps,
                                  fused ? dropout_scale : 1.f, vec_ok, *dev,
                                  static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
