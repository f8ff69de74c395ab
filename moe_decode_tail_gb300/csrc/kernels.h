// Internal interface between the C-ABI layer and the kernels (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moetail {

enum { kWeightF32 = 0, kWeightBF16 = 1, kWeightUnit = 2 };

// Limits of the C ABI's sizes (every entry point checks against these).
constexpr int kMaxTp = 32, kMaxK = 32, kMaxP = 32768, kMaxTokens = 65535, kMaxWidth = 1 << 24;

// The latent tail's sizes: tp latent slots of b tokens, width L.
inline bool latent_sizes_ok(int b, int tp, int L) {
  return b >= 0 && b <= kMaxTokens && tp >= 1 && tp <= kMaxTp && L >= 8 && L <= kMaxP && L % 8 == 0;
}
// The up-projection's sizes: tp_s shared slots, y of width L, output width H.
inline bool up_sizes_ok(int b, int tp_s, int L, int H) {
  return b >= 0 && b <= kMaxTokens && tp_s >= 0 && tp_s <= kMaxTp && L >= 8 && L <= kMaxP && L % 8 == 0 &&
         H >= 8 && H % 8 == 0 && H <= kMaxWidth;
}

// Rows of one finalize call: slot s's row j starts at rows + s * slot_stride + j * P.
struct FinalizeArgs {
  const uint16_t* rows;   // EP: GEMM2 rows [tp][num_rows][P]; TP: K-partials; latent: [tp][b][L]
  int64_t num_rows;       // rows per slot (EP rows_per_slot, TP num_rows, latent b)
  int64_t slot_stride;    // elements between slots
  const int32_t* idx;     // EP [tp][b][K]; TP [b][K]; latent unused
  const void* w;          // [b][K] FP32 or BF16; latent unused (unit weight)
  const uint16_t* gamma;  // BF16 [P]
  float gain_center, eps, rcpP;
  int b, tp, K, P;
  int chunks, band_vectors, routes_per_pass, stages;  // set by the launcher
  uint16_t* out;          // BF16 [b][P]
  // 1: the inputs are complete before the preceding kernel of the stream ends,
  // so they are read before the grid dependency wait (out is written after it)
  int inputs_before_wait = 0;
  unsigned long long stage_wait_ns = 0;  // the staged kernel's consumer wait limit (0: the default)
};

enum { kFinalizeEP = 0, kFinalizeTP = 1, kFinalizeLatent = 2 };

cudaError_t launch_finalize(int mode, const FinalizeArgs& a, bool wbn, int wmode, int sms, cudaStream_t stream);
// Read and clear the finalize kernels' device error word (synchronises).
cudaError_t take_finalize_error(unsigned* bits);

// ---- decode GEMM (tcgen05) ---------------------------------------------------

enum GemmMode { kGemmUpShared = 0, kGemmGateUpSilu = 1, kGemmDown = 2, kGemmLatentUp = 3, kGemmDownUp = 4 };

struct GemmArgs {
  int M;             // output features of one weight (rows of W; gate/up: I)
  int K;             // reduction length
  int n_tok;         // tokens b (<= N tile)
  int kblocks;       // ceil(K / 64)
  const uint16_t* shared;  // mode 0: BF16 [tp_s][b][M] partials added in slot order, or null
  int tp_s;
  uint16_t* out;     // mode 0, 2: BF16 [b][M]; mode 1: h BF16 [b][M]
  int accumulate;    // mode 2: out = bf16(out + bf16(d))
  int weights_before_wait;  // 1 only when the preceding kernel is this library's own
  // mode 3 (latent tail in one kernel: y formed in shared memory, then mode 0's product)
  const uint16_t* latent = nullptr;  // BF16 [tp][n_tok][K]
  const uint16_t* gamma = nullptr;   // BF16 [K]
  uint16_t* y = nullptr;             // BF16 [n_tok][K], written by the first M tile's CTAs, or null
  int tp = 0;
  float eps = 0.f, rcpK = 0.f;
  int chunks = 0;                    // 256-column chunks of K (at most 32)
  int inputs_before_wait = 0;        // mode 3: latent and gamma, mode 1: x, complete before the
                                     // preceding kernel ends (read before its grid dependency wait)
  unsigned long long stage_wait_ns = 0;  // the MMA issuer's operand-stage wait limit (0: the default)
  // mode 4 (the shared expert's down projection and the up-projection in one
  // kernel): M, K, kblocks, map_w0 and map_x describe the down projection
  // (W_down [M][K], h [n_tok][K]); K2, kblocks2, map_w1 and map_x1 the
  // up-projection (W_up [M][K2], y [n_tok][K2]); out = bf16(u + (sum_s shared[s]
  // + bf16(d))), and d_out (BF16 [n_tok][M], or null) receives bf16(d)
  int K2 = 0, kblocks2 = 0;
  uint16_t* d_out = nullptr;
};

// Mode 4's cluster of ksplit >= 2 CTAs: ranks 0 .. n-1 stream the down
// projection's K range, ranks n .. ksplit-1 the up-projection's, each range
// split evenly over its ranks.  n minimises the longest per-CTA range (the
// smallest such n).
__host__ __device__ inline int downup_down_ranks(int ksplit, int kblocks, int kblocks2) {
  int best = 1, best_len = 1 << 30;
  for (int n = 1; n < ksplit; ++n) {
    const int d = (kblocks + n - 1) / n, u = (kblocks2 + ksplit - n - 1) / (ksplit - n);
    const int len = d > u ? d : u;
    if (len < best_len) {
      best = n;
      best_len = len;
    }
  }
  return best;
}

struct GemmPlan {
  int tm;       // MMA M: weight rows per CTA (64 or 128)
  int n_tile;   // MMA N (tokens, padded)
  int ksplit;   // cluster size (K split)
  int stages;   // shared-memory ring depth
  int m_tiles;  // CTAs clusters along M
};

// K2: the up-projection's reduction length in mode kGemmDownUp (0 otherwise).
GemmPlan plan_gemm(int mode, int M, int K, int b, int sms, int K2 = 0);
// The persistent down projection (out = [accumulate ? out + ] bf16(h . w^T)):
// ctas CTAs walk the output tiles of 128 rows x n_tile tokens over the whole
// K range with two alternating TMEM accumulators.  Uses M, K, kblocks, n_tok,
// out, accumulate and weights_before_wait of a; w: [M][K] (box 128 rows),
// h: [n_tok][K] (box n_tile rows).
cudaError_t launch_persistent_down(const CUtensorMap& w, const CUtensorMap& h, const GemmArgs& a, int n_tile,
                                   int ctas, bool pdl, cudaStream_t stream);
// The one-kernel latent tail's plan at b tokens and tp slots: the
// up-projection's tiles and K split (so the product is bit for bit the
// two-kernel one) and a ring that fits beside the CTA's y operand and can
// stage a token's tp latent rows per epilogue warp; false where that is not
// possible (more than 32 tokens, more than 32 chunks of 256 columns, a plan
// override with other tiles, too little shared memory).
bool plan_latent_fused(int H, int L, int b, int tp, int sms, GemmPlan* plan);
cudaError_t launch_decode_gemm(int mode, const GemmPlan& plan, const CUtensorMap& w0, const CUtensorMap& w1,
                               const CUtensorMap& x, const GemmArgs& a, bool pdl, cudaStream_t stream,
                               const CUtensorMap* x1 = nullptr);

// The latent tail's two steps, shared by its entry points (arguments already
// checked; enqueue_up_project returns a moe_tail status).
cudaError_t enqueue_latent_norm(const void* latent, const void* gamma, float eps, int b, int tp, int L, void* y,
                                bool inputs_ready, cudaStream_t st);
int enqueue_up_project(const void* y, const void* w_up, const void* shared, int tp_s, int b, int L, int H, void* out,
                       bool weights_before_wait, cudaStream_t st);
// The whole latent tail in one kernel (kGemmLatentUp)?  Only when the
// latent-tail kernel form is pinned to it and plan_latent_fused finds a plan
// at these sizes (the two-kernel form is faster on GB300).
bool latent_tail_fused(int b, int tp, int L, int H, GemmPlan* plan);
// Enqueue it (y: BF16 [b][L] written, or null); flags as moe_tail_latent_up_flags.
int enqueue_latent_fused(const GemmPlan& plan, const void* latent, const void* gamma, float eps, const void* w_up,
                         const void* shared, int tp_s, int b, int tp, int L, int H, void* out, void* y, int flags,
                         cudaStream_t st);
// Either form, as moe_tail_latent_up_flags (y required).
int enqueue_latent_tail(const void* latent, const void* gamma, float eps, const void* w_up, const void* shared,
                        int tp_s, int b, int tp, int L, int H, void* out, void* y, int flags, cudaStream_t st);

// Read and clear the device error word (synchronises with the device).
cudaError_t take_device_error(unsigned* bits);

// ---- host-side configuration -------------------------------------------------

// Kernel forms a caller may pin with moe_tail_set_kernel_form (the values of
// the MOE_TAIL_FORM_* constants of the public header); 0: the library's choice.
enum { kFormCallEP = 0, kFormCallTP = 1, kFormCallLatent = 2, kFormCalls = 3 };
int kernel_form(int call);

// Tuning overrides for sweeps, read from the environment once (at the first
// call that needs them), never per call.  0 means "not set".
struct Tuning {
  int fin_split;         // MOE_TAIL_FIN_SPLIT: column bands per token (1, 2, 4 or 8), any finalize
  int fin_ep_split;      // MOE_TAIL_FIN_EP_SPLIT: the same for EP finalize alone
  int fin_latent_split;  // MOE_TAIL_FIN_LATENT_SPLIT: the same for the latent norm alone
  int fin_ring_kb;       // MOE_TAIL_FIN_RING_KB: staged finalize ring budget (KB)
  int fin_groups;        // MOE_TAIL_FIN_GROUPS: staged finalize CTAs along the tokens
  int fin_routes;        // MOE_TAIL_FIN_ROUTES: route-parallel finalize routes per pass
  int gemm_plan[4][3];   // MOE_TAIL_GEMM_PLAN_<UP|GATEUP|DOWN|DOWNUP> = "tm,ksplit,stages"
};
const Tuning& tuning();

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per (kernel, device) and safe to call from several host threads.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Multiprocessors of the current device (cached per device).
int device_sms();

// The operand-stage wait limit set by moe_tail_set_stage_wait_limit (0: the
// kernels' default), copied into each call's arguments.
unsigned long long stage_wait_limit_ns();
#ifdef MOE_TAIL_TRACE
cudaError_t trace_attach_gemm(void* buf, unsigned cap);
unsigned trace_count_gemm();
cudaError_t trace_attach_finalize(void* buf, unsigned cap);
unsigned trace_count_finalize();
#endif
// A one-thread kernel whose bounded wait expires after limit_ns.
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace moetail
