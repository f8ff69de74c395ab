// moe_tail_latent_up_noalloc: the latent tail for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin that an
// inference runtime gives only its input and output buffers, or a host
// process whose device memory is entirely reserved by its own pool allocator.
// Others must not call cudaMalloc on their hot path because it can
// synchronise the device.  This entry point enqueues the same two steps as
// moe_tail_latent_up (through the same internal calls), but keeps the
// intermediate y rows in a fixed array in device memory that is part of the
// library itself, so the caller passes only inputs and outputs and nothing is
// allocated per call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe_tail.h"
#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace {

// The y rows (BF16 [b][L]) of a no-alloc latent tail call.  Every GPU that
// loads the library holds this array until the process exits; all calls share
// it.  Host code must not use this name as a device address: the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_y[MOE_TAIL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddress {
  CUcontext ctx;  // the context the address belongs to
  void* ptr;
};
ScratchAddress g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mutex;

using CtxGetCurrent = CUresult (*)(CUcontext*);

// The calling thread's current context, or null when it has none yet.
CUcontext current_context() {
  static const CtxGetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrent>(p);
    return static_cast<CtxGetCurrent>(nullptr);
  }();
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// The device address of g_noalloc_y on the current device.  It is looked up
// with cudaGetSymbolAddress once per device (the first call on a device does
// this), and again only if the device's context has changed since -- after a
// cudaDeviceReset the library's module is loaded anew and the array may move.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const CUcontext ctx = current_context();
  if (!g_scratch[dev].ptr || !ctx || g_scratch[dev].ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_y);  // with the device current; creates its context if needed
    if (e != cudaSuccess) return e;
    g_scratch[dev] = ScratchAddress{current_context(), p};
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return an && bn && a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

MOE_API int moe_tail_latent_up_noalloc(const void* latent, const void* gamma, float eps, const void* w_up,
                                       const void* shared, int tp_s, int b, int tp, int L, int H, void* out,
                                       void* stream) {
  // the limits of moe_tail_latent_up (one definition for both)
  if (!moetail::latent_sizes_ok(b, tp, L) || !moetail::up_sizes_ok(b, tp_s, L, H)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  // y must fit the library's fixed scratch array
  if ((size_t)b * (size_t)L * 2 > (size_t)MOE_TAIL_NOALLOC_SCRATCH_BYTES) return MOE_TAIL_EINVAL;
  if (!latent || !gamma || !w_up || !out) return MOE_TAIL_EINVAL;
  if ((tp_s > 0) != (shared != nullptr)) return MOE_TAIL_EINVAL;
  if (!aligned16(latent) || !aligned16(gamma) || !aligned16(w_up) || !aligned16(out) ||
      (shared && !aligned16(shared)))
    return MOE_TAIL_EINVAL;
  const size_t out_n = (size_t)b * H * 2;
  if (overlaps(out, out_n, latent, (size_t)tp * b * L * 2) || overlaps(out, out_n, gamma, (size_t)L * 2) ||
      overlaps(out, out_n, w_up, (size_t)H * L * 2) || overlaps(out, out_n, shared, (size_t)tp_s * b * H * 2))
    return MOE_TAIL_EINVAL;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The one-kernel form, where pinned, keeps y in shared memory (no scratch array).
  moetail::GemmPlan plan;
  if (moetail::latent_tail_fused(b, tp, L, H, &plan))
    return moetail::enqueue_latent_fused(plan, latent, gamma, eps, w_up, shared, tp_s, b, tp, L, H, out, nullptr, 0,
                                         st);
  void* y = nullptr;
  cudaError_t e = scratch_on_current_device(&y);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_TAIL_ECUDA;
  }
  // The array belongs to the library, so no caller buffer can legitimately
  // overlap it; check anyway, with the same rule as a caller's workspace.
  const size_t y_n = (size_t)b * L * 2;
  if (overlaps(y, y_n, out, out_n) || overlaps(y, y_n, latent, (size_t)tp * b * L * 2) ||
      overlaps(y, y_n, gamma, (size_t)L * 2) || overlaps(y, y_n, w_up, (size_t)H * L * 2) ||
      overlaps(y, y_n, shared, (size_t)tp_s * b * H * 2))
    return MOE_TAIL_EINVAL;
  // 1. y (every element written, so nothing has to start at zero), 2. the
  // up-projection, which follows this call's own norm kernel
  e = moetail::enqueue_latent_norm(latent, gamma, eps, b, tp, L, y, false, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_TAIL_ECUDA;
  }
  return moetail::enqueue_up_project(y, w_up, shared, tp_s, b, L, H, out, true, st);
}
