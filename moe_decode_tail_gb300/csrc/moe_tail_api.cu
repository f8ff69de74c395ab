// C ABI of the MoE decode tail: argument checks, TMA descriptors, launches.
// Every check runs before the first CUDA call, so a refused call touches no
// device state ([MS] _check_tail_args: refuse before anything launches).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/moe_tail.h"
#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

// ============================================================================ host-side configuration

namespace moetail {

namespace {
std::atomic<int> g_forms[kFormCalls];  // zero-initialised: the library's choice
std::atomic<unsigned long long> g_stage_wait_ns{0};  // 0: the kernels' default limit

int env_int(const char* name) {
  const char* v = getenv(name);
  return v ? atoi(v) : 0;
}

int env_split(const char* name) {
  const int s = env_int(name);
  return (s == 1 || s == 2 || s == 4 || s == 8) ? s : 0;
}

void env_plan(const char* name, int (&plan)[3]) {
  plan[0] = plan[1] = plan[2] = 0;
  const char* v = getenv(name);
  int tm = 0, ks = 0, st = 0;
  if (!v || sscanf(v, "%d,%d,%d", &tm, &ks, &st) != 3) return;
  if ((tm != 64 && tm != 128 && tm != 256) || ks < 1 || ks > 8 || st < 2 || st > 12) return;
  plan[0] = tm;
  plan[1] = ks;
  plan[2] = st;
}
}  // namespace

int kernel_form(int call) { return call >= 0 && call < kFormCalls ? g_forms[call].load(std::memory_order_relaxed) : 0; }

unsigned long long stage_wait_limit_ns() { return g_stage_wait_ns.load(std::memory_order_relaxed); }

const Tuning& tuning() {
  static const Tuning t = [] {
    Tuning r{};
    r.fin_split = env_split("MOE_TAIL_FIN_SPLIT");
    r.fin_ep_split = env_split("MOE_TAIL_FIN_EP_SPLIT");
    r.fin_latent_split = env_split("MOE_TAIL_FIN_LATENT_SPLIT");
    r.fin_ring_kb = env_int("MOE_TAIL_FIN_RING_KB");
    r.fin_groups = env_int("MOE_TAIL_FIN_GROUPS");
    r.fin_routes = env_int("MOE_TAIL_FIN_ROUTES");
    env_plan("MOE_TAIL_GEMM_PLAN_UP", r.gemm_plan[0]);
    env_plan("MOE_TAIL_GEMM_PLAN_GATEUP", r.gemm_plan[1]);
    env_plan("MOE_TAIL_GEMM_PLAN_DOWN", r.gemm_plan[2]);
    env_plan("MOE_TAIL_GEMM_PLAN_DOWNUP", r.gemm_plan[3]);
    return r;
  }();
  return t;
}

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex m;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(m);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
  if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

}  // namespace moetail

MOE_API int moe_tail_set_stage_wait_limit(unsigned long long limit_ns) {
  if (limit_ns > 1000000000ull) return MOE_TAIL_EINVAL;
  moetail::g_stage_wait_ns.store(limit_ns, std::memory_order_relaxed);
  return MOE_TAIL_OK;
}

MOE_API int moe_tail_set_kernel_form(int call, int form) {
  static const int kForms[moetail::kFormCalls] = {3, 3, 3};  // forms 0..2 of each call
  if (call < 0 || call >= moetail::kFormCalls || form < 0 || form >= kForms[call]) return MOE_TAIL_EINVAL;
  moetail::g_forms[call].store(form, std::memory_order_relaxed);
  return MOE_TAIL_OK;
}

namespace {

using moetail::device_sms;
using moetail::FinalizeArgs;
using moetail::GemmArgs;
using moetail::GemmPlan;

using moetail::kMaxK;
using moetail::kMaxP;
using moetail::kMaxTokens;
using moetail::kMaxTp;
using moetail::kMaxWidth;

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

struct Range {
  uintptr_t lo, hi;
};
Range span(const void* p, size_t bytes) { return Range{(uintptr_t)p, (uintptr_t)p + bytes}; }
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

int finish(cudaError_t e) {
  if (e == cudaSuccess) return MOE_TAIL_OK;
  (void)cudaGetLastError();
  return MOE_TAIL_ECUDA;
}

// ---- TMA descriptors --------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// Row-major BF16 matrix [rows][cols] read in boxes of box_rows x 64 columns
// (128 bytes: the swizzle span), 128-byte swizzle; out-of-range boxes read zeros.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
                    CUtensorMapL2promotion promo) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

int check_finalize_common(const void* w, int weight_dtype, const void* gamma, int b, int tp, int K, int P,
                          void* out) {
  if (b < 0 || tp < 1 || tp > kMaxTp || K < 1 || K > kMaxK || P < 8 || P > kMaxP || P % 8) return MOE_TAIL_EINVAL;
  if (b > kMaxTokens) return MOE_TAIL_EINVAL;
  if (weight_dtype != MOE_TAIL_W_FP32 && weight_dtype != MOE_TAIL_W_BF16) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!w || !gamma || !out) return MOE_TAIL_EINVAL;
  if (!aligned(gamma, 16) || !aligned(out, 16)) return MOE_TAIL_EINVAL;
  if (!aligned(w, weight_dtype == MOE_TAIL_W_FP32 ? 4 : 2)) return MOE_TAIL_EINVAL;
  return MOE_TAIL_OK;
}

}  // namespace

// ============================================================================ EP finalize

namespace {

// EP or expert-TP finalize after the common checks; flags: 0 or MOE_TAIL_INPUTS_READY.
int finalize_call(int mode, const void* rows, int64_t num_rows, const int32_t* permuted_idx,
                  const void* route_weights, int weight_dtype, const void* gamma, float gain_center, float eps,
                  int weight_before_norm, int b, int tp, int K, int P, void* out, int flags, void* stream) {
  int rc = check_finalize_common(route_weights, weight_dtype, gamma, b, tp, K, P, out);
  if (rc == MOE_TAIL_OK && (flags & ~MOE_TAIL_INPUTS_READY)) rc = MOE_TAIL_EINVAL;
  if (rc != MOE_TAIL_OK || b == 0) return rc;
  if (num_rows < 0 || num_rows > ((int64_t)1 << 31) - 1) return MOE_TAIL_EINVAL;
  if (!permuted_idx || !aligned(permuted_idx, 4)) return MOE_TAIL_EINVAL;
  if (num_rows > 0 && (!rows || !aligned(rows, 16))) return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * P * 2);
  const size_t wsz = weight_dtype == MOE_TAIL_W_FP32 ? 4 : 2;
  const size_t idx_count = (mode == moetail::kFinalizeEP ? (size_t)tp : 1) * b * K;  // EP: [tp][b][K]
  if (overlaps(o, span(rows, (size_t)tp * num_rows * P * 2)) || overlaps(o, span(permuted_idx, idx_count * 4)) ||
      overlaps(o, span(route_weights, (size_t)b * K * wsz)) || overlaps(o, span(gamma, (size_t)P * 2)))
    return MOE_TAIL_EINVAL;
  FinalizeArgs a;
  a.inputs_before_wait = (flags & MOE_TAIL_INPUTS_READY) ? 1 : 0;
  a.rows = static_cast<const uint16_t*>(rows);
  a.num_rows = num_rows;
  a.slot_stride = num_rows * P;
  a.idx = permuted_idx;
  a.w = route_weights;
  a.gamma = static_cast<const uint16_t*>(gamma);
  a.gain_center = gain_center;
  a.eps = eps;
  a.rcpP = (float)(1.0 / (double)P);
  a.b = b;
  a.tp = tp;
  a.K = K;
  a.P = P;
  a.out = static_cast<uint16_t*>(out);
  return finish(moetail::launch_finalize(mode, a, weight_before_norm != 0, weight_dtype, device_sms(),
                                         static_cast<cudaStream_t>(stream)));
}

}  // namespace

MOE_API int moe_tail_ep_finalize(const void* rows, int64_t rows_per_slot, const int32_t* permuted_idx,
                                 const void* route_weights, int weight_dtype, const void* gamma,
                                 float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                                 int P, void* out, void* stream) {
  return finalize_call(moetail::kFinalizeEP, rows, rows_per_slot, permuted_idx, route_weights, weight_dtype, gamma,
                       gain_center, eps, weight_before_norm, b, tp, K, P, out, 0, stream);
}

MOE_API int moe_tail_ep_finalize_flags(const void* rows, int64_t rows_per_slot, const int32_t* permuted_idx,
                                       const void* route_weights, int weight_dtype, const void* gamma,
                                       float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                                       int P, void* out, int flags, void* stream) {
  return finalize_call(moetail::kFinalizeEP, rows, rows_per_slot, permuted_idx, route_weights, weight_dtype, gamma,
                       gain_center, eps, weight_before_norm, b, tp, K, P, out, flags, stream);
}

// ============================================================================ expert-TP finalize

MOE_API int moe_tail_tp_finalize(const void* partials, int64_t num_rows, const int32_t* permuted_idx,
                                 const void* route_weights, int weight_dtype, const void* gamma,
                                 float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                                 int P, void* out, void* stream) {
  return finalize_call(moetail::kFinalizeTP, partials, num_rows, permuted_idx, route_weights, weight_dtype, gamma,
                       gain_center, eps, weight_before_norm, b, tp, K, P, out, 0, stream);
}

MOE_API int moe_tail_tp_finalize_flags(const void* partials, int64_t num_rows, const int32_t* permuted_idx,
                                       const void* route_weights, int weight_dtype, const void* gamma,
                                       float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                                       int P, void* out, int flags, void* stream) {
  return finalize_call(moetail::kFinalizeTP, partials, num_rows, permuted_idx, route_weights, weight_dtype, gamma,
                       gain_center, eps, weight_before_norm, b, tp, K, P, out, flags, stream);
}

// ============================================================================ latent tail

MOE_API size_t moe_tail_workspace_bytes(int which, int b, int dim) {
  if (b < 0 || dim < 1 || (which != 0 && which != 1)) return 0;
  return round256((size_t)b * dim * 2);
}

namespace moetail {

// Step 1 of the latent tail: y = RMS norm of the slot-summed latent (an
// expert-TP finalize with one "route" per token: row = token, unit weight,
// gain center 0).  Arguments already checked.
cudaError_t enqueue_latent_norm(const void* latent, const void* gamma, float eps, int b, int tp, int L, void* y,
                                bool inputs_ready, cudaStream_t st) {
  FinalizeArgs n;
  n.inputs_before_wait = inputs_ready ? 1 : 0;
  n.rows = static_cast<const uint16_t*>(latent);
  n.num_rows = b;
  n.slot_stride = (int64_t)b * L;
  n.idx = nullptr;
  n.w = nullptr;
  n.gamma = static_cast<const uint16_t*>(gamma);
  n.gain_center = 0.0f;
  n.eps = eps;
  n.rcpP = (float)(1.0 / (double)L);
  n.b = b;
  n.tp = tp;
  n.K = 1;
  n.P = L;
  n.out = static_cast<uint16_t*>(y);
  return moetail::launch_finalize(moetail::kFinalizeLatent, n, false, moetail::kWeightUnit, device_sms(), st);
}

// Step 2: out = y . w_up^T + sum_s shared[s].  Arguments already checked.
int enqueue_up_project(const void* y, const void* w_up, const void* shared, int tp_s, int b, int L, int H, void* out,
                       bool weights_before_wait, cudaStream_t st) {
  const GemmPlan plan = moetail::plan_gemm(moetail::kGemmUpShared, H, L, b, device_sms());
  CUtensorMap mw, mx;
  if (!encode_bf16_2d(&mw, w_up, H, L, plan.tm, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mx, y, b, L, plan.n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return MOE_TAIL_ECUDA;
  GemmArgs g;
  g.M = H;
  g.K = L;
  g.n_tok = b;
  g.kblocks = (L + 63) / 64;
  g.shared = static_cast<const uint16_t*>(shared);
  g.tp_s = tp_s;
  g.out = static_cast<uint16_t*>(out);
  g.accumulate = 0;
  g.weights_before_wait = weights_before_wait ? 1 : 0;
  return finish(moetail::launch_decode_gemm(moetail::kGemmUpShared, plan, mw, mw, mx, g, true, st));
}

// The one-kernel form is taken only on request (moe_tail_set_kernel_form):
// measured on GB300 it is slower than the norm kernel followed by the
// up-projection at every batch size (b = 1: 14.5 vs 13.9 us in one call,
// 12.3 vs 10.5 us with both promises).  Its CTAs form y on the MMA's critical
// path -- a trip for the latent rows under the weight stream's load, the
// cluster exchange, then y -- and every M tile's cluster re-reads the latent
// partials, while the separate norm runs ahead of the weight stream under
// programmatic dependent launch.
bool latent_tail_fused(int b, int tp, int L, int H, GemmPlan* plan) {
  if (kernel_form(kFormCallLatent) != MOE_TAIL_FORM_LATENT_ONE_KERNEL) return false;
  return moetail::plan_latent_fused(H, L, b, tp, device_sms(), plan);
}

int enqueue_latent_fused(const GemmPlan& plan, const void* latent, const void* gamma, float eps, const void* w_up,
                         const void* shared, int tp_s, int b, int tp, int L, int H, void* out, void* y, int flags,
                         cudaStream_t st) {
  CUtensorMap mw;
  if (!encode_bf16_2d(&mw, w_up, H, L, plan.tm, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)) return MOE_TAIL_ECUDA;
  GemmArgs g;
  g.M = H;
  g.K = L;
  g.n_tok = b;
  g.kblocks = (L + 63) / 64;
  g.shared = static_cast<const uint16_t*>(shared);
  g.tp_s = tp_s;
  g.out = static_cast<uint16_t*>(out);
  g.accumulate = 0;
  g.weights_before_wait = (flags & MOE_TAIL_WEIGHTS_STATIC) ? 1 : 0;
  g.latent = static_cast<const uint16_t*>(latent);
  g.gamma = static_cast<const uint16_t*>(gamma);
  g.y = static_cast<uint16_t*>(y);
  g.tp = tp;
  g.eps = eps;
  g.rcpK = (float)(1.0 / (double)L);
  g.chunks = (L + 255) / 256;
  g.inputs_before_wait = (flags & MOE_TAIL_INPUTS_READY) ? 1 : 0;
  // the token-tile map is not used by this mode
  return finish(moetail::launch_decode_gemm(moetail::kGemmLatentUp, plan, mw, mw, mw, g, true, st));
}

int enqueue_latent_tail(const void* latent, const void* gamma, float eps, const void* w_up, const void* shared,
                        int tp_s, int b, int tp, int L, int H, void* out, void* y, int flags, cudaStream_t st) {
  GemmPlan plan;
  if (latent_tail_fused(b, tp, L, H, &plan))
    return enqueue_latent_fused(plan, latent, gamma, eps, w_up, shared, tp_s, b, tp, L, H, out, y, flags, st);
  // 1. y, 2. the up-projection; the GEMM follows this call's own norm kernel,
  // which never writes w_up, so it requests its weights before waiting.
  const cudaError_t e =
      enqueue_latent_norm(latent, gamma, eps, b, tp, L, y, (flags & MOE_TAIL_INPUTS_READY) != 0, st);
  if (e != cudaSuccess) return finish(e);
  return enqueue_up_project(y, w_up, shared, tp_s, b, L, H, out, true, st);
}

}  // namespace moetail

namespace {

using moetail::enqueue_latent_norm;
using moetail::enqueue_up_project;

using moetail::latent_sizes_ok;
using moetail::up_sizes_ok;

}  // namespace

MOE_API int moe_tail_latent_up(const void* latent, const void* gamma, float eps, const void* w_up,
                               const void* shared, int tp_s, int b, int tp, int L, int H, void* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!latent_sizes_ok(b, tp, L) || !up_sizes_ok(b, tp_s, L, H)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!latent || !gamma || !w_up || !out || !workspace) return MOE_TAIL_EINVAL;
  if ((tp_s > 0) != (shared != nullptr)) return MOE_TAIL_EINVAL;
  if (!aligned(latent, 16) || !aligned(gamma, 16) || !aligned(w_up, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16) || (shared && !aligned(shared, 16)))
    return MOE_TAIL_EINVAL;
  if (workspace_bytes < moe_tail_workspace_bytes(0, b, L)) return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  const Range ws = span(workspace, (size_t)b * L * 2);
  if (overlaps(o, span(latent, (size_t)tp * b * L * 2)) || overlaps(o, span(gamma, (size_t)L * 2)) ||
      overlaps(o, span(w_up, (size_t)H * L * 2)) || overlaps(o, span(shared, (size_t)tp_s * b * H * 2)) ||
      overlaps(o, ws) || overlaps(ws, span(latent, (size_t)tp * b * L * 2)) || overlaps(ws, span(w_up, (size_t)H * L * 2)) ||
      overlaps(ws, span(shared, (size_t)tp_s * b * H * 2)) || overlaps(ws, span(gamma, (size_t)L * 2)))
    return MOE_TAIL_EINVAL;
  return moetail::enqueue_latent_tail(latent, gamma, eps, w_up, shared, tp_s, b, tp, L, H, out, workspace, 0,
                                      static_cast<cudaStream_t>(stream));
}

MOE_API int moe_tail_latent_up_flags(const void* latent, const void* gamma, float eps, const void* w_up,
                                     const void* shared, int tp_s, int b, int tp, int L, int H, void* out, void* y,
                                     int flags, void* stream) {
  if (!latent_sizes_ok(b, tp, L) || !up_sizes_ok(b, tp_s, L, H)) return MOE_TAIL_EINVAL;
  if (flags & ~(MOE_TAIL_INPUTS_READY | MOE_TAIL_WEIGHTS_STATIC)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!latent || !gamma || !w_up || !out || !y) return MOE_TAIL_EINVAL;
  if ((tp_s > 0) != (shared != nullptr)) return MOE_TAIL_EINVAL;
  if (!aligned(latent, 16) || !aligned(gamma, 16) || !aligned(w_up, 16) || !aligned(out, 16) || !aligned(y, 16) ||
      (shared && !aligned(shared, 16)))
    return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  const Range yr = span(y, (size_t)b * L * 2);
  if (overlaps(o, span(latent, (size_t)tp * b * L * 2)) || overlaps(o, span(gamma, (size_t)L * 2)) ||
      overlaps(o, span(w_up, (size_t)H * L * 2)) || overlaps(o, span(shared, (size_t)tp_s * b * H * 2)) ||
      overlaps(o, yr) || overlaps(yr, span(latent, (size_t)tp * b * L * 2)) || overlaps(yr, span(w_up, (size_t)H * L * 2)) ||
      overlaps(yr, span(shared, (size_t)tp_s * b * H * 2)) || overlaps(yr, span(gamma, (size_t)L * 2)))
    return MOE_TAIL_EINVAL;
  return moetail::enqueue_latent_tail(latent, gamma, eps, w_up, shared, tp_s, b, tp, L, H, out, y, flags,
                                      static_cast<cudaStream_t>(stream));
}

MOE_API int moe_tail_latent_norm(const void* latent, const void* gamma, float eps, int b, int tp, int L, void* y,
                                 int flags, void* stream) {
  if (!latent_sizes_ok(b, tp, L) || (flags & ~MOE_TAIL_INPUTS_READY)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!latent || !gamma || !y) return MOE_TAIL_EINVAL;
  if (!aligned(latent, 16) || !aligned(gamma, 16) || !aligned(y, 16)) return MOE_TAIL_EINVAL;
  const Range yr = span(y, (size_t)b * L * 2);
  if (overlaps(yr, span(latent, (size_t)tp * b * L * 2)) || overlaps(yr, span(gamma, (size_t)L * 2)))
    return MOE_TAIL_EINVAL;
  return finish(enqueue_latent_norm(latent, gamma, eps, b, tp, L, y, (flags & MOE_TAIL_INPUTS_READY) != 0,
                                    static_cast<cudaStream_t>(stream)));
}

MOE_API int moe_tail_up_project(const void* y, const void* w_up, const void* shared, int tp_s, int b, int L, int H,
                                void* out, int flags, void* stream) {
  if (!up_sizes_ok(b, tp_s, L, H) || (flags & ~MOE_TAIL_WEIGHTS_STATIC)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!y || !w_up || !out) return MOE_TAIL_EINVAL;
  if ((tp_s > 0) != (shared != nullptr)) return MOE_TAIL_EINVAL;
  if (!aligned(y, 16) || !aligned(w_up, 16) || !aligned(out, 16) || (shared && !aligned(shared, 16)))
    return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  if (overlaps(o, span(y, (size_t)b * L * 2)) || overlaps(o, span(w_up, (size_t)H * L * 2)) ||
      overlaps(o, span(shared, (size_t)tp_s * b * H * 2)))
    return MOE_TAIL_EINVAL;
  return enqueue_up_project(y, w_up, shared, tp_s, b, L, H, out, (flags & MOE_TAIL_WEIGHTS_STATIC) != 0,
                            static_cast<cudaStream_t>(stream));
}

MOE_API int moe_tail_up_project_shared_down(const void* y, const void* w_up, const void* shared, int tp_s,
                                            const void* h, const void* w_down, int b, int L, int I, int H,
                                            void* out, void* d_out, int flags, void* stream) {
  if (!up_sizes_ok(b, tp_s, L, H) || I < 8 || I % 8 || I > kMaxWidth || (flags & ~MOE_TAIL_WEIGHTS_STATIC))
    return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!y || !w_up || !h || !w_down || !out) return MOE_TAIL_EINVAL;
  if ((tp_s > 0) != (shared != nullptr)) return MOE_TAIL_EINVAL;
  if (!aligned(y, 16) || !aligned(w_up, 16) || !aligned(h, 16) || !aligned(w_down, 16) || !aligned(out, 16) ||
      (shared && !aligned(shared, 16)) || (d_out && !aligned(d_out, 16)))
    return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2), dr = span(d_out, (size_t)b * H * 2);
  const Range ins[5] = {span(y, (size_t)b * L * 2), span(w_up, (size_t)H * L * 2),
                        span(shared, (size_t)tp_s * b * H * 2), span(h, (size_t)b * I * 2),
                        span(w_down, (size_t)H * I * 2)};
  if (overlaps(o, dr)) return MOE_TAIL_EINVAL;
  for (const Range& r : ins)
    if (overlaps(o, r) || overlaps(dr, r)) return MOE_TAIL_EINVAL;
  const GemmPlan plan = moetail::plan_gemm(moetail::kGemmDownUp, H, I, b, device_sms(), L);
  CUtensorMap md, mh, mu, my;
  if (!encode_bf16_2d(&md, w_down, H, I, plan.tm, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mh, h, b, I, plan.n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !encode_bf16_2d(&mu, w_up, H, L, plan.tm, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&my, y, b, L, plan.n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return MOE_TAIL_ECUDA;
  GemmArgs g;
  g.M = H;
  g.K = I;
  g.n_tok = b;
  g.kblocks = (I + 63) / 64;
  g.K2 = L;
  g.kblocks2 = (L + 63) / 64;
  g.shared = static_cast<const uint16_t*>(shared);
  g.tp_s = tp_s;
  g.out = static_cast<uint16_t*>(out);
  g.d_out = static_cast<uint16_t*>(d_out);
  g.accumulate = 0;
  g.weights_before_wait = (flags & MOE_TAIL_WEIGHTS_STATIC) ? 1 : 0;
  return finish(moetail::launch_decode_gemm(moetail::kGemmDownUp, plan, md, mu, mh, g, true,
                                            static_cast<cudaStream_t>(stream), &my));
}

// ============================================================================ shared expert

namespace {

bool shared_sizes_ok(int b, int H, int I) {
  return b >= 0 && b <= kMaxTokens && H >= 8 && H % 8 == 0 && I >= 8 && I % 8 == 0 && H <= kMaxWidth &&
         I <= kMaxWidth;
}

// h = bf16(silu(bf16(x . w_gate^T)) * bf16(x . w_up^T)).  Arguments already checked.
int launch_gate_up(const void* x, const void* w_gate, const void* w_up, int b, int H, int I, void* h,
                   bool weights_before_wait, cudaStream_t st, bool inputs_before_wait = false) {
  const GemmPlan p1 = moetail::plan_gemm(moetail::kGemmGateUpSilu, I, H, b, device_sms());
  CUtensorMap mg, mu, mx;
  if (!encode_bf16_2d(&mg, w_gate, I, H, p1.tm / 2, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mu, w_up, I, H, p1.tm / 2, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mx, x, b, H, p1.n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return MOE_TAIL_ECUDA;
  GemmArgs g;
  g.M = I;
  g.K = H;
  g.n_tok = b;
  g.kblocks = (H + 63) / 64;
  g.shared = nullptr;
  g.tp_s = 0;
  g.out = static_cast<uint16_t*>(h);
  g.accumulate = 0;
  g.weights_before_wait = weights_before_wait ? 1 : 0;
  g.inputs_before_wait = inputs_before_wait ? 1 : 0;
  return finish(moetail::launch_decode_gemm(moetail::kGemmGateUpSilu, p1, mg, mu, mx, g, true, st));
}

// out = accumulate ? bf16(out + bf16(h . w_down^T)) : bf16(h . w_down^T).  Arguments already checked.
int launch_down(const void* h, const void* w_down, int b, int H, int I, void* out, bool accumulate,
                bool weights_before_wait, cudaStream_t st) {
  const GemmPlan p2 = moetail::plan_gemm(moetail::kGemmDown, H, I, b, device_sms());
  CUtensorMap md, mh;
  if (!encode_bf16_2d(&md, w_down, H, I, p2.tm, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mh, h, b, I, p2.n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return MOE_TAIL_ECUDA;
  GemmArgs d;
  d.M = H;
  d.K = I;
  d.n_tok = b;
  d.kblocks = (I + 63) / 64;
  d.shared = nullptr;
  d.tp_s = 0;
  d.out = static_cast<uint16_t*>(out);
  d.accumulate = accumulate ? 1 : 0;
  d.weights_before_wait = weights_before_wait ? 1 : 0;
  return finish(moetail::launch_decode_gemm(moetail::kGemmDown, p2, md, md, mh, d, true, st));
}

}  // namespace

MOE_API int moe_shared_expert(const void* x, const void* w_gate, const void* w_up, const void* w_down, int b,
                              int H, int I, void* out, int accumulate, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!shared_sizes_ok(b, H, I)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!x || !w_gate || !w_up || !w_down || !out || !workspace) return MOE_TAIL_EINVAL;
  if (!aligned(x, 16) || !aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16))
    return MOE_TAIL_EINVAL;
  if (workspace_bytes < moe_tail_workspace_bytes(1, b, I)) return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  const Range ws = span(workspace, (size_t)b * I * 2);
  const Range rx = span(x, (size_t)b * H * 2), rg = span(w_gate, (size_t)I * H * 2),
              ru = span(w_up, (size_t)I * H * 2), rd = span(w_down, (size_t)H * I * 2);
  if (overlaps(o, rx) || overlaps(o, rg) || overlaps(o, ru) || overlaps(o, rd) || overlaps(o, ws) ||
      overlaps(ws, rx) || overlaps(ws, rg) || overlaps(ws, ru) || overlaps(ws, rd))
    return MOE_TAIL_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // gate/up is the first kernel of the call: the caller may just have written the weights
  const int rc = launch_gate_up(x, w_gate, w_up, b, H, I, workspace, false, st);
  if (rc != MOE_TAIL_OK) return rc;
  // the down projection follows this call's own gate/up kernel, which never writes w_down
  return launch_down(workspace, w_down, b, H, I, out, accumulate != 0, true, st);
}

MOE_API int moe_shared_gate_up(const void* x, const void* w_gate, const void* w_up, int b, int H, int I, void* h,
                               int flags, void* stream) {
  if (!shared_sizes_ok(b, H, I) || (flags & ~(MOE_TAIL_WEIGHTS_STATIC | MOE_TAIL_INPUTS_READY))) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!x || !w_gate || !w_up || !h) return MOE_TAIL_EINVAL;
  if (!aligned(x, 16) || !aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(h, 16)) return MOE_TAIL_EINVAL;
  const Range rh = span(h, (size_t)b * I * 2);
  if (overlaps(rh, span(x, (size_t)b * H * 2)) || overlaps(rh, span(w_gate, (size_t)I * H * 2)) ||
      overlaps(rh, span(w_up, (size_t)I * H * 2)))
    return MOE_TAIL_EINVAL;
  return launch_gate_up(x, w_gate, w_up, b, H, I, h, (flags & MOE_TAIL_WEIGHTS_STATIC) != 0,
                        static_cast<cudaStream_t>(stream), (flags & MOE_TAIL_INPUTS_READY) != 0);
}

MOE_API int moe_shared_down(const void* h, const void* w_down, int b, int H, int I, void* out, int accumulate,
                            int flags, void* stream) {
  if (!shared_sizes_ok(b, H, I) || (flags & ~MOE_TAIL_WEIGHTS_STATIC)) return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!h || !w_down || !out) return MOE_TAIL_EINVAL;
  if (!aligned(h, 16) || !aligned(w_down, 16) || !aligned(out, 16)) return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  if (overlaps(o, span(h, (size_t)b * I * 2)) || overlaps(o, span(w_down, (size_t)H * I * 2)))
    return MOE_TAIL_EINVAL;
  return launch_down(h, w_down, b, H, I, out, accumulate != 0, (flags & MOE_TAIL_WEIGHTS_STATIC) != 0,
                     static_cast<cudaStream_t>(stream));
}

MOE_API int moe_shared_down_persistent(const void* h, const void* w_down, int b, int H, int I, void* out,
                                       int accumulate, int ctas, int flags, void* stream) {
  if (!shared_sizes_ok(b, H, I) || ctas < 0 || ctas > 65535 || (flags & ~MOE_TAIL_WEIGHTS_STATIC))
    return MOE_TAIL_EINVAL;
  if (b == 0) return MOE_TAIL_OK;
  if (!h || !w_down || !out) return MOE_TAIL_EINVAL;
  if (!aligned(h, 16) || !aligned(w_down, 16) || !aligned(out, 16)) return MOE_TAIL_EINVAL;
  const Range o = span(out, (size_t)b * H * 2);
  if (overlaps(o, span(h, (size_t)b * I * 2)) || overlaps(o, span(w_down, (size_t)H * I * 2)))
    return MOE_TAIL_EINVAL;
  const int n_tile = b <= 16 ? 16 : b <= 32 ? 32 : b <= 64 ? 64 : 128;
  const int64_t tiles = (int64_t)((H + 127) / 128) * ((b + n_tile - 1) / n_tile);
  const int grid = (int)std::min<int64_t>(tiles, ctas > 0 ? ctas : device_sms());
  CUtensorMap md, mh;
  if (!encode_bf16_2d(&md, w_down, H, I, 128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_bf16_2d(&mh, h, b, I, n_tile, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return MOE_TAIL_ECUDA;
  GemmArgs d;
  d.M = H;
  d.K = I;
  d.n_tok = b;
  d.kblocks = (I + 63) / 64;
  d.shared = nullptr;
  d.tp_s = 0;
  d.out = static_cast<uint16_t*>(out);
  d.accumulate = accumulate != 0 ? 1 : 0;
  d.weights_before_wait = (flags & MOE_TAIL_WEIGHTS_STATIC) ? 1 : 0;
  return finish(moetail::launch_persistent_down(md, mh, d, n_tile, grid, true, static_cast<cudaStream_t>(stream)));
}

// ============================================================================ misc

MOE_API const char* moe_tail_status_str(int status) {
  switch (status) {
    case MOE_TAIL_OK: return "ok";
    case MOE_TAIL_EINVAL: return "invalid argument";
    case MOE_TAIL_ECUDA: return "CUDA error";
    case MOE_TAIL_ENOTSUP: return "not supported";
    default: return "unknown status";
  }
}

MOE_API int moe_tail_take_device_error(unsigned int* bits) {
  if (!bits) return MOE_TAIL_EINVAL;
  unsigned g = 0, f = 0;
  cudaError_t e = moetail::take_device_error(&g);
  if (e == cudaSuccess) e = moetail::take_finalize_error(&f);
  *bits = g | f;
  return finish(e);
}

MOE_API int moe_tail_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return MOE_TAIL_EINVAL;
  return finish(moetail::launch_selftest_wait((unsigned long long)limit_us * 1000ull, static_cast<cudaStream_t>(stream)));
}

#ifdef MOE_TAIL_TRACE
#include "../../include/moe_tail_trace.h"

MOE_API int moe_tail_trace_attach(void* buf, unsigned int capacity) {
  if (buf && (!aligned(buf, 16) || capacity < 2)) return MOE_TAIL_EINVAL;
  // GEMM records fill the buffer's first half, finalize records its second
  const unsigned half = buf ? capacity / 2 : 0;
  void* second = buf ? static_cast<uint8_t*>(buf) + (size_t)half * MOE_TAIL_TRACE_RECORD_BYTES : nullptr;
  cudaError_t e = moetail::trace_attach_gemm(buf, half);
  if (e == cudaSuccess) e = moetail::trace_attach_finalize(second, buf ? capacity - half : 0);
  return finish(e);
}

MOE_API int moe_tail_trace_counts(unsigned int* gemm_records, unsigned int* finalize_records) {
  if (!gemm_records || !finalize_records) return MOE_TAIL_EINVAL;
  *gemm_records = moetail::trace_count_gemm();
  *finalize_records = moetail::trace_count_finalize();
  return finish(cudaGetLastError());
}
#endif
