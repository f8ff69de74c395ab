// Finalize kernels of the MoE decode tail (sm_103a).
//
// EP finalize and expert-TP finalize follow the Muse Spark MoE tail page
// ("vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.moe.tail"):
// module docstring (both formulas) and _TpTailKernel (gains, per-lane sum of
// squares of 8 columns, xor butterfly, normalisation order, each product
// rounded alone before the route sum, BF16 round-to-nearest with -0 made +0).
// The latent norm follows the Kimi-K3 tail runtime page
// ("...kimi_k3...moe.tail_runtime", module docstring): the latent partials are
// summed over slots, RMS-normalised per row, then up-projected.
//
// One kernel serves all three.  A CTA works on one column band of one token;
// the bands of a token form a thread-block cluster.  Its threads are R route
// groups of VB threads: thread (r, v) owns 16-byte vector v of the band
// (columns 8v..8v+7) of the r-th route of the current pass, so the routes of
// a token run side by side, as in the page's kernel (TOP_K x band threads).
// Each thread issues all of its loads at once -- EP: its route row; expert-TP
// and latent: the route's row in every slot, summed in slot order and rounded
// to BF16 -- so a pass costs one trip to memory.  Every warp covers one
// 256-column chunk of one route: it forms the chunk's sum of squares with the
// xor butterfly and stores it into every cluster CTA's shared memory (DSMEM).
// After one cluster barrier each thread folds its route's chunk sums in chunk
// order from +0 (the same bits whatever the split), normalises, weights, and
// leaves the product in shared memory; the first route group then adds the
// products in route order (EP: per slot, each slot's partial rounded to BF16,
// slots summed in order).  All arithmetic is single IEEE binary32 operations
// (__fmul_rn / __fadd_rn: never contracted into an FMA), the inverse RMS is
// 1 / sqrt(.) with IEEE square root and division, and subnormals are kept.
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moetail {

enum { kModeEP = kFinalizeEP, kModeTP = kFinalizeTP, kModeLatent = kFinalizeLatent };

constexpr int kMaxRoutesPerPass = 8;
constexpr int kMaxChunks = 128;  // P <= 32768
constexpr int kMaxList = 1024;   // tp * K <= 32 * 32
constexpr int kMaxThreads = 1024;

struct __align__(16) FinalizeSmem {
  float ss[2][kMaxRoutesPerPass][kMaxChunks];  // chunk sums of squares, per pass parity
  int32_t list_row[kMaxList];                  // the token's routes: row within the slot
  int16_t list_slot[kMaxList];                 // EP: the slot holding it
  int16_t list_route[kMaxList];                // route index k (for its weight)
  float w[32];                                 // the token's route weights
  int warp_count[32];
  int warp_base[32];
  int count;
};

template <int WMODE>
__device__ __forceinline__ float route_weight(const void* w, int64_t i) {
  if (WMODE == kWeightBF16) return __uint_as_float((uint32_t)((const uint16_t*)w)[i] << 16);
  if (WMODE == kWeightUnit) return 1.0f;
  return ((const float*)w)[i];
}

template <int MODE, bool WBN, int WMODE>
__global__ void __launch_bounds__(kMaxThreads) finalize_kernel(const FinalizeArgs a) {
  extern __shared__ __align__(16) float prod[];  // [R][VB][8] products of a pass
  __shared__ FinalizeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int VB = a.band_vectors, R = a.routes_per_pass;
  const int r_local = tid / VB, vb = tid - r_local * VB;
  const int t = blockIdx.y;
  const uint32_t split = cluster_size();
  const int band = (int)cluster_rank();
  const int vec = band * VB + vb;
  const int col = vec * 8;
  const int chunk = vec >> 5;  // VB is a multiple of 32: a warp is one chunk of one route
  const bool valid = col < a.P;
  const int nthreads = blockDim.x;

  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  grid_dependency_wait();
  launch_dependents();  // a kernel chained behind this one may start its own prologue

  // One trip for the gains, the route weights and the route indices.
  const uint4 gv = valid ? ld_v4(a.gamma + col) : make_uint4(0, 0, 0, 0);
  if (MODE != kModeLatent && tid < a.K) sm.w[tid] = route_weight<WMODE>(a.w, (int64_t)t * a.K + tid);
  int count = 1;
  if (MODE == kModeLatent) {
    if (tid == 0) {
      sm.list_row[0] = t;
      sm.list_slot[0] = 0;
      sm.list_route[0] = 0;
      sm.w[0] = 1.0f;
    }
    __syncthreads();
  } else {
    // The token's routes with a row, in the order their sums run: EP in
    // (slot, route) order over the slots' local routes, expert-TP in route order.
    const int n = MODE == kModeEP ? a.tp * a.K : a.K;
    int running = 0;
    for (int base = 0; base < n; base += nthreads) {
      const int i = base + tid;
      int j = -1, s = 0, k = i;
      if (i < n) {
        if (MODE == kModeEP) {
          s = i / a.K;
          k = i - s * a.K;
          j = a.idx[((int64_t)s * a.b + t) * a.K + k];
        } else {
          j = a.idx[(int64_t)t * a.K + i];
        }
      }
      const bool has_row = i < n && j >= 0 && (int64_t)j < a.num_rows;
      const unsigned ballot = __ballot_sync(0xffffffffu, has_row);
      if (lane == 0) sm.warp_count[warp] = __popc(ballot);
      __syncthreads();
      if (tid == 0) {
        int acc = 0;
        for (int w = 0; w < (nthreads >> 5); ++w) {
          sm.warp_base[w] = acc;
          acc += sm.warp_count[w];
        }
        sm.count = acc;
      }
      __syncthreads();
      if (has_row) {
        const int pos = running + sm.warp_base[warp] + __popc(ballot & ((1u << lane) - 1u));
        sm.list_row[pos] = j;
        sm.list_slot[pos] = (int16_t)s;
        sm.list_route[pos] = (int16_t)k;
      }
      running += sm.count;
      __syncthreads();
    }
    count = running;
  }

  float g[8];
  unpack8(gv, g);
#pragma unroll
  for (int i = 0; i < 8; ++i) g[i] = __fadd_rn(g[i], a.gain_center);
  float o[8], part[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = part[i] = 0.0f;
  int cur_slot = -1;

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers started: DSMEM is live

  for (int base = 0, pass = 0; base < count; base += R, ++pass) {
    const int e = base + r_local;  // this thread's route in the pass
    const bool active = e < count;
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    if (active && valid) {
      const int64_t row = sm.list_row[e];
      if (MODE == kModeEP) {
        const uint4 v = ld_stream_v4(a.rows + (int64_t)sm.list_slot[e] * a.slot_stride + row * a.P + col);
        unpack8(v, x);
      } else {
        const uint16_t* src = a.rows + row * a.P + col;
        for (int s0 = 0; s0 < a.tp; s0 += 8) {  // eight slots in flight at a time
          uint4 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            v[q] = s0 + q < a.tp ? ld_stream_v4(src + (int64_t)(s0 + q) * a.slot_stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (s0 + q < a.tp) {  // slot order, FP32 from +0
              float f[8];
              unpack8(v[q], f);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] = __fadd_rn(x[i], f[i]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = bf16_round(x[i]);
      }
    }
    // this warp's chunk sum of squares, published to every CTA of the cluster
    float* ssp = sm.ss[pass & 1][r_local];
    {
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float v = WBN ? __fmul_rn(x[i], g[i]) : x[i];
        acc = __fadd_rn(acc, __fmul_rn(v, v));
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      if (active && chunk < a.chunks && lane < (int)split)
        st_cluster_f32(map_to_rank(smem_addr(&ssp[chunk]), (uint32_t)lane), acc);
    }
    cluster_sync_all();
    if (active) {
      float ss = 0.0f;
      for (int c = 0; c < a.chunks; ++c) ss = __fadd_rn(ss, ssp[c]);
      const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, a.rcpP), a.eps)));
      const float w = MODE == kModeLatent ? 1.0f : sm.w[sm.list_route[e]];
      float4* dst = reinterpret_cast<float4*>(prod + ((size_t)r_local * VB + vb) * 8);
      float p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float nv = WBN ? __fmul_rn(__fmul_rn(x[i], g[i]), inv) : __fmul_rn(__fmul_rn(x[i], inv), g[i]);
        p[i] = __fmul_rn(nv, w);  // each product rounded alone
      }
      dst[0] = make_float4(p[0], p[1], p[2], p[3]);
      dst[1] = make_float4(p[4], p[5], p[6], p[7]);
    }
    __syncthreads();
    if (r_local == 0) {  // the route sum, in route order
      const int n_pass = min(R, count - base);
      for (int rr = 0; rr < n_pass; ++rr) {
        const float4* src = reinterpret_cast<const float4*>(prod + ((size_t)rr * VB + vb) * 8);
        const float4 p0 = src[0], p1 = src[1];
        const float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        if (MODE == kModeEP) {
          const int s = sm.list_slot[base + rr];
          if (s != cur_slot) {  // slot boundary: its BF16 partial joins the slot sum
            if (cur_slot >= 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                o[i] = __fadd_rn(o[i], bf16_round(part[i]));
                part[i] = 0.0f;
              }
            }
            cur_slot = s;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) part[i] = __fadd_rn(part[i], p[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = __fadd_rn(o[i], p[i]);
        }
      }
    }
    __syncthreads();  // the products of this pass are consumed
  }
  if (MODE == kModeEP && cur_slot >= 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __fadd_rn(o[i], bf16_round(part[i]));
  }
  if (r_local == 0 && valid) {
    uint4 r;
    r.x = pack_bf16x2_pz(o[0], o[1]);
    r.y = pack_bf16x2_pz(o[2], o[3]);
    r.z = pack_bf16x2_pz(o[4], o[5]);
    r.w = pack_bf16x2_pz(o[6], o[7]);
    st_v4(a.out + (int64_t)t * a.P + col, r);
  }
}

// ---------------------------------------------------------------- launcher

// Tuning override of the column split: MOE_TAIL_FIN_SPLIT=<1|2|4|8>.
static int split_override() {
  const char* v = getenv("MOE_TAIL_FIN_SPLIT");
  const int s = v ? atoi(v) : 0;
  return (s == 1 || s == 2 || s == 4 || s == 8) ? s : 0;
}

template <int MODE, bool WBN, int WMODE>
static cudaError_t launch_t(const FinalizeArgs& a, int split, cudaStream_t stream) {
  auto k = finalize_kernel<MODE, WBN, WMODE>;
  const size_t smem = (size_t)a.routes_per_pass * a.band_vectors * 32;
  static int configured[64] = {0};  // raise the limit once per device, not per call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, a.b, 1);
  cfg.blockDim = dim3(a.routes_per_pass * a.band_vectors, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: this kernel touches no global memory before
  // griddepcontrol.wait, so it may be scheduled while its predecessor drains.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_finalize(int mode, const FinalizeArgs& args, bool wbn, int wmode, int sms, cudaStream_t stream) {
  FinalizeArgs a = args;
  a.chunks = (a.P + 255) / 256;
  const int routes = mode == kModeLatent ? 1 : (mode == kModeEP ? a.tp * a.K : a.K);
  // Bands per token: enough CTAs to cover the SMs about twice, at most 8
  // (portable cluster size), one band per chunk at most.
  int split = split_override();
  if (split == 0) {
    split = 1;
    while (split < 8 && split < a.chunks && (int64_t)a.b * split < 2 * sms) split *= 2;
  }
  while (split < 8 && (a.chunks + split - 1) / split > 32) split *= 2;
  a.band_vectors = 32 * ((a.chunks + split - 1) / split);
  if (a.band_vectors > kMaxThreads) return cudaErrorInvalidValue;
  a.routes_per_pass = std::min(std::min(kMaxRoutesPerPass, std::max(1, routes)), kMaxThreads / a.band_vectors);
  if (mode == kModeEP) {  // a token has about K local rows in all: more groups would idle
    a.routes_per_pass = std::max(1, std::min(a.routes_per_pass, a.K));
  }
  if (mode == kModeEP) {
    if (wbn) return wmode == kWeightBF16 ? launch_t<kModeEP, true, kWeightBF16>(a, split, stream)
                                         : launch_t<kModeEP, true, kWeightF32>(a, split, stream);
    return wmode == kWeightBF16 ? launch_t<kModeEP, false, kWeightBF16>(a, split, stream)
                                : launch_t<kModeEP, false, kWeightF32>(a, split, stream);
  }
  if (mode == kModeTP) {
    if (wbn) return wmode == kWeightBF16 ? launch_t<kModeTP, true, kWeightBF16>(a, split, stream)
                                         : launch_t<kModeTP, true, kWeightF32>(a, split, stream);
    return wmode == kWeightBF16 ? launch_t<kModeTP, false, kWeightBF16>(a, split, stream)
                                : launch_t<kModeTP, false, kWeightF32>(a, split, stream);
  }
  return launch_t<kModeLatent, false, kWeightUnit>(a, split, stream);
}

}  // namespace moetail
