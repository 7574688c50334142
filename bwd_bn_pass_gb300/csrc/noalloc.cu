// BatchNorm2d training forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to provide the workspace that gbn_bn_forward_train
// needs: code running inside a CUDA-graph capture or a real-time loop where a
// cudaMalloc would synchronise or is forbidden, plugins whose host framework
// owns every device allocation, or C callers without an allocator at all.
// This file gives them one entry point whose scratch (the per-block
// statistics partials) lives in a fixed, file-scope device array that every
// GPU loading the library holds until the process exits.
//
// The entry point allocates nothing: it resolves the array's device address
// once per device (the host-side symbol is only a stand-in, never a device
// address) and then runs the ordinary forward with that address as the
// workspace.  Nothing needs zeroing: the partials are rewritten by every
// call, and the persistent kernel's flags carry a launch epoch that the
// kernel validates and advances itself.
#include <mutex>

#include "gbn_internal.h"

namespace {

// 64 KiB.  The two-launch kernels need 16 * grid_y * C bytes of partials,
// where grid_y (blocks per channel) fills the device's resident 256-thread
// block slots (608 on GB300, 4 per SM) at least once:
//   * C <= slots: grid_y * C stays within about one slot per channel-block,
//     at most ~608 * 16 bytes = 9.5 KiB, far below the limit;
//   * C > slots: grid_y = 1 and the partials are 16 * C bytes, so every
//     C <= 4096 fits and larger C is rejected with GBN_EWORKSPACE.
// The single-launch persistent kernel also needs its per-CTA flags (16 bytes
// per SM) and its own partials; it runs whenever those fit the array too
// (and the call's size threshold selects it), otherwise the two-launch
// kernels do.  Channels of at most 8 x 2048 elements run the single-launch
// small-channel kernels (a block or a cluster of blocks per channel), which
// use no scratch (the size check above still applies to them).
constexpr size_t kNoAllocScratchBytes = 64 * 1024;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; nullptr if the
// CUDA runtime refuses.  Done once per device, with that device current.
void* scratch_on_current_device() {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[device] = p;
  }
  return g_noalloc_ptr[device];
}

}  // namespace

extern "C" int gbn_bn_forward_train_noalloc(const void* x, int dtype, int64_t B, int64_t C,
                                            int64_t HW, const float* gamma, const float* beta,
                                            float* running_mean, float* running_var,
                                            float momentum, float eps, void* y, float* stats,
                                            void* stream) {
  // Argument errors come back before any CUDA call, as for every entry point.
  const int rc = gbn::bn_forward_check_args(x, dtype, B, C, HW, y, stats, momentum, eps);
  if (rc != GBN_OK) return rc;
  if (C == 0 || B == 0 || HW == 0) return GBN_OK;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return GBN_ECUDA;
  const size_t need = gbn::bn_partials_bytes(B, C, HW);
  if (need == 0) return GBN_ECUDA;
  if (need > kNoAllocScratchBytes) return GBN_EWORKSPACE;
  return gbn::bn_forward_train_scratch(x, dtype, B, C, HW, gamma, beta, running_mean,
                                       running_var, momentum, eps, y, stats, scratch,
                                       kNoAllocScratchBytes, stream);
}
