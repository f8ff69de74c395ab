// Internal interface between the C-ABI layer and the kernels (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moetail {

enum { kWeightF32 = 0, kWeightBF16 = 1, kWeightUnit = 2 };

struct EpArgs {
  const uint16_t* rows;  // BF16 [tp][rows_per_slot][P]
  int64_t rows_per_slot;
  const int32_t* idx;    // [tp][b][K]
  const void* w;         // [b][K] FP32 or BF16
  const uint16_t* gamma; // BF16 [P]
  float gain_center, eps, rcpP;
  int b, tp, K, P, chunks;
  uint16_t* out;         // BF16 [b][P]
};

struct TpArgs {
  const uint16_t* partials;  // BF16 [tp][num_rows][P]
  int64_t num_rows;
  int64_t slot_stride;       // elements between slots (num_rows * P)
  const int32_t* idx;        // [b][K], or null: row = token (K = 1)
  const void* w;             // [b][K] FP32 or BF16, or null with unit weights
  const uint16_t* gamma;     // BF16 [P]
  float gain_center, eps, rcpP;
  int b, tp, K, P, chunks;
  uint16_t* out;             // BF16 [b][P]
};

cudaError_t launch_ep_finalize(const EpArgs& a, bool wbn, int wmode, int sms, int force_split,
                               cudaStream_t stream);
cudaError_t launch_tp_finalize(const TpArgs& a, bool wbn, int wmode, int sms, int force_split,
                               cudaStream_t stream);

// ---- decode GEMM (tcgen05) ---------------------------------------------------

enum GemmMode { kGemmUpShared = 0, kGemmGateUpSilu = 1, kGemmDown = 2 };

struct GemmArgs {
  int M;             // output features of one weight (rows of W; gate/up: I)
  int K;             // reduction length
  int n_tok;         // tokens b (<= N tile)
  int kblocks;       // ceil(K / 64)
  const uint16_t* shared;  // mode 0: BF16 [tp_s][b][M] partials added in slot order, or null
  int tp_s;
  uint16_t* out;     // mode 0, 2: BF16 [b][M]; mode 1: h BF16 [b][M]
  int accumulate;    // mode 2: out = bf16(out + bf16(d))
};

struct GemmPlan {
  int n_tile;   // MMA N (tokens, padded)
  int ksplit;   // cluster size (K split)
  int stages;   // shared-memory ring depth
  int m_tiles;  // CTAs clusters along M
};

GemmPlan plan_gemm(int mode, int M, int K, int b, int sms);
cudaError_t launch_decode_gemm(int mode, const GemmPlan& plan, const CUtensorMap& w0, const CUtensorMap& w1,
                               const CUtensorMap& x, const GemmArgs& a, bool pdl, cudaStream_t stream);

// Read and clear the device error word (synchronises with the device).
cudaError_t take_device_error(unsigned* bits);

}  // namespace moetail
