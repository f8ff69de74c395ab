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
// (__fmul_rn / __fadd_rn and the paired mul.rn.f32x2 / add.rn.f32x2, which
// round each component alike: never contracted into an FMA), the inverse RMS
// is 1 / sqrt(.) with IEEE square root and division, and subnormals are kept.
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moetail {

enum { kModeEP = kFinalizeEP, kModeTP = kFinalizeTP, kModeLatent = kFinalizeLatent };

constexpr int kMaxRoutesPerPass = 8;
constexpr int kMaxChunks = 128;  // P <= 32768
// A route's chunk sums sit kChunkStride floats apart: the lanes that form
// different routes' 1/rms at once then read different shared-memory banks.
constexpr int kChunkStride = kMaxChunks + 1;
constexpr int kMaxList = 1024;   // tp * K <= 32 * 32
// At most 512 threads of at most 64 registers (half an SM's register file), so
// that a finalize CTA fits on an SM beside the GEMM CTAs of a concurrent
// weight stream; a 1024-thread CTA at 64 registers would need a whole SM.
constexpr int kMaxThreads = 512;

struct __align__(16) FinalizeSmem {
  float ss[2][kMaxRoutesPerPass][kChunkStride];  // chunk sums of squares, per pass parity
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

// 1/rms of one route from its chunk sums of squares: the sums added in chunk
// order from +0, then 1 / sqrt(ss * (1/P) + eps) with IEEE square root and
// division.
__device__ __forceinline__ float inv_rms_of_route(const float* chunk_ss, const FinalizeArgs& a) {
  float ss = 0.0f;
  for (int c = 0; c < a.chunks; ++c) ss = __fadd_rn(ss, chunk_ss[c]);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, a.rcpP), a.eps)));
}

// The token's route weights into sm.w and its routes that have a row into
// sm.list_* (EP in (slot, route) order over the slots' local routes, expert-TP
// in route order; the latent norm has one "route", the token's own row);
// returns their count.  Called by every thread of the CTA.
template <int MODE, int WMODE>
__device__ int load_route_list(const FinalizeArgs& a, FinalizeSmem& sm, int t) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  if (MODE != kModeLatent && tid < a.K) sm.w[tid] = route_weight<WMODE>(a.w, (int64_t)t * a.K + tid);
  if (MODE == kModeLatent) {
    if (tid == 0) {
      sm.list_row[0] = t;
      sm.list_slot[0] = 0;
      sm.list_route[0] = 0;
      sm.w[0] = 1.0f;
    }
    __syncthreads();
    return 1;
  }
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
  return running;
}

template <int MODE, bool WBN, int WMODE>
__global__ void __launch_bounds__(kMaxThreads, 2) finalize_kernel(const FinalizeArgs a) {
  MOE_TRACE_SCOPE(10 + MODE);
  extern __shared__ __align__(16) float prod[];  // [R][VB][8] products of a pass
  __shared__ FinalizeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31;
  const int VB = a.band_vectors, R = a.routes_per_pass;
  const int r_local = tid / VB, vb = tid - r_local * VB;
  const int t = blockIdx.y;
  const uint32_t split = cluster_size();
  const int band = (int)cluster_rank();
  const int vec = band * VB + vb;
  const int col = vec * 8;
  const int chunk = vec >> 5;  // VB is a multiple of 32: a warp is one chunk of one route
  const bool valid = col < a.P;

  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (!a.inputs_before_wait) grid_dependency_wait();
  // A kernel chained behind this one may start its own prologue.  The latent
  // norm that waited first, from 8 tokens on, lets it start only once this
  // thread's latent row loads are issued (below): the up-projection behind it
  // requests its weights at once, and that flood would otherwise queue ahead
  // of the norm's own loads (one call at b = 16: 15.1 -> 14.4 us with the
  // start held back until the rows were summed, 13.9 -> 13.5 us once it
  // followed their issue; b = 8: 14.8 -> 14.1 -> 13.0).  At b = 1 the early
  // start is worth more (12.3 vs 13.2 us).
  const bool late_trigger = MODE == kModeLatent && !a.inputs_before_wait && a.b >= 8;
  if (!late_trigger) launch_dependents();

  // One trip for the gains, the route weights and the route indices.
  const uint4 gv = valid ? ld_v4(a.gamma + col) : make_uint4(0, 0, 0, 0);
  const int count = load_route_list<MODE, WMODE>(a, sm, t);

  float2 g[4];
  unpack8p(gv, g);
#pragma unroll
  for (int k = 0; k < 4; ++k) g[k] = add2(g[k], splat2(a.gain_center));
  float2 o[4], part[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = part[k] = splat2(0.0f);
  int cur_slot = -1;

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers started: DSMEM is live

  for (int base = 0, pass = 0; base < count; base += R, ++pass) {
    const int e = base + r_local;  // this thread's route in the pass
    const bool active = e < count;
    float2 x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = splat2(0.0f);
    if (active && valid) {
      const int64_t row = sm.list_row[e];
      if (MODE == kModeEP) {
        const uint4 v = ld_stream_v4(a.rows + (int64_t)sm.list_slot[e] * a.slot_stride + row * a.P + col);
        unpack8p(v, x);
      } else {
        const uint16_t* src = a.rows + row * a.P + col;
        for (int s0 = 0; s0 < a.tp; s0 += 8) {  // eight slots in flight at a time
          uint4 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            v[q] = s0 + q < a.tp ? ld_stream_v4(src + (int64_t)(s0 + q) * a.slot_stride) : make_uint4(0, 0, 0, 0);
          if (late_trigger && pass == 0 && s0 == 0) launch_dependents();  // the first slots' loads are out
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (s0 + q < a.tp) {  // slot order, FP32 from +0
              float2 f[4];
              unpack8p(v[q], f);
#pragma unroll
              for (int k = 0; k < 4; ++k) x[k] = add2(x[k], f[k]);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = bf16_round2(x[k]);
      }
    }
    if (late_trigger && pass == 0) launch_dependents();  // threads without a row (a repeat is harmless)
    // this warp's chunk sum of squares, published to every CTA of the cluster
    float* ssp = sm.ss[pass & 1][r_local];
    {
      float acc = 0.0f;  // the lane's eight squares, added in column order
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 v = WBN ? mul2(x[k], g[k]) : x[k];
        const float2 sq = mul2(v, v);
        acc = __fadd_rn(__fadd_rn(acc, sq.x), sq.y);
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      if (active && chunk < a.chunks && lane < (int)split)
        st_cluster_f32(map_to_rank(smem_addr(&ssp[chunk]), (uint32_t)lane), acc);
    }
    cluster_sync_all();
    if (active) {
      const float inv = inv_rms_of_route(ssp, a);
      const float w = MODE == kModeLatent ? 1.0f : sm.w[sm.list_route[e]];
      const float2 inv2 = splat2(inv);
      float4* dst = reinterpret_cast<float4*>(prod + ((size_t)r_local * VB + vb) * 8);
      float2 p[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 nv = WBN ? mul2(mul2(x[k], g[k]), inv2) : mul2(mul2(x[k], inv2), g[k]);
        p[k] = mul_each(nv, w);  // each product rounded alone (summed after the barrier)
      }
      dst[0] = make_float4(p[0].x, p[0].y, p[1].x, p[1].y);
      dst[1] = make_float4(p[2].x, p[2].y, p[3].x, p[3].y);
    }
    __syncthreads();
    if (r_local == 0) {  // the route sum, in route order
      const int n_pass = min(R, count - base);
      for (int rr = 0; rr < n_pass; ++rr) {
        const float4* src = reinterpret_cast<const float4*>(prod + ((size_t)rr * VB + vb) * 8);
        const float4 p0 = src[0], p1 = src[1];
        const float2 p[4] = {make_float2(p0.x, p0.y), make_float2(p0.z, p0.w), make_float2(p1.x, p1.y),
                             make_float2(p1.z, p1.w)};
        if (MODE == kModeEP) {
          const int s = sm.list_slot[base + rr];
          if (s != cur_slot) {  // slot boundary: its BF16 partial joins the slot sum
            if (cur_slot >= 0) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                o[k] = add2(o[k], bf16_round2(part[k]));
                part[k] = splat2(0.0f);
              }
            }
            cur_slot = s;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) part[k] = add2(part[k], p[k]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) o[k] = add2(o[k], p[k]);
        }
      }
    }
    __syncthreads();  // the products of this pass are consumed
  }
  if (MODE == kModeEP && cur_slot >= 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = add2(o[k], bf16_round2(part[k]));
  }
  if (r_local == 0 && valid) {
    const uint4 r = pack8p_pz(o);
    if (a.inputs_before_wait) grid_dependency_wait();  // the preceding kernel may still read out
    st_v4(a.out + (int64_t)t * a.P + col, r);
  }
}

// ------------------------------------------- EP: a token's routes in registers
//
// The same arithmetic as finalize_kernel in EP mode, with one thread per
// 16-byte vector of the band holding up to kEpRoutes of the token's routes at
// once: their rows are loaded together, their chunk sums of squares are
// published together, and one cluster barrier serves them all, so a token
// whose local routes number at most kEpRoutes (the usual top-K) costs one trip
// to memory and one barrier.  The products never leave registers: each thread
// adds its columns' products in (slot, route) order itself, rounding each
// slot's partial to BF16 at the slot boundary.
constexpr int kEpRoutes = 8;
constexpr int kEpMaxThreads = 512;

template <bool WBN, int WMODE>
__global__ void __launch_bounds__(kEpMaxThreads, 1) ep_finalize_kernel(const FinalizeArgs a) {
  MOE_TRACE_SCOPE(40);
  __shared__ FinalizeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31;
  const int t = blockIdx.y;
  const uint32_t split = cluster_size();
  const int vec = (int)cluster_rank() * a.band_vectors + tid;
  const int col = vec * 8;
  const int chunk = vec >> 5;  // a warp is one 256-column chunk
  const bool valid = col < a.P;

  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (!a.inputs_before_wait) grid_dependency_wait();
  launch_dependents();

  const uint4 gv = valid ? ld_v4(a.gamma + col) : make_uint4(0, 0, 0, 0);
  const int count = load_route_list<kModeEP, WMODE>(a, sm, t);
  MOE_TRACE_MARK(0);  // the token's route list resolved
  float2 g[4];
  unpack8p(gv, g);
#pragma unroll
  for (int k = 0; k < 4; ++k) g[k] = add2(g[k], splat2(a.gain_center));
  float2 o[4], part[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = part[k] = splat2(0.0f);
  int cur_slot = -1;

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers started: DSMEM is live

  for (int base = 0, pass = 0; base < count; base += kEpRoutes, ++pass) {
    const int n_pass = min(kEpRoutes, count - base);  // the same in every thread of the cluster
    uint4 raw[kEpRoutes];
#pragma unroll
    for (int q = 0; q < kEpRoutes; ++q) {
      raw[q] = make_uint4(0, 0, 0, 0);
      if (q < n_pass && valid) {
        const int e = base + q;
        raw[q] = ld_stream_v4(a.rows + (int64_t)sm.list_slot[e] * a.slot_stride + (int64_t)sm.list_row[e] * a.P + col);
      }
    }
    // the routes' weights and slots, read while the rows are in flight
    float wq[kEpRoutes];
    int sq[kEpRoutes];
#pragma unroll
    for (int q = 0; q < kEpRoutes; ++q) {
      const int e = min(base + q, count - 1);
      wq[q] = sm.w[sm.list_route[e]];
      sq[q] = sm.list_slot[e];
    }
    float* ssp = &sm.ss[pass & 1][0][0];  // [route of the pass][chunk]
#pragma unroll
    for (int q = 0; q < kEpRoutes; ++q) {
      if (q < n_pass) {
        float2 x[4];
        unpack8p(raw[q], x);
        float acc = 0.0f;  // the lane's eight squares, added in column order
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 v = WBN ? mul2(x[k], g[k]) : x[k];
          const float2 sq = mul2(v, v);
          acc = __fadd_rn(__fadd_rn(acc, sq.x), sq.y);
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        if (chunk < a.chunks && lane < (int)split)
          st_cluster_f32(map_to_rank(smem_addr(&ssp[q * kChunkStride + chunk]), (uint32_t)lane), acc);
      }
    }
    if (pass == 0) MOE_TRACE_MARK(1);  // rows landed, chunk sums published
    cluster_sync_all();
    if (pass == 0) MOE_TRACE_MARK(2);  // cluster barrier passed
    // lane q of every warp forms route q's 1/rms; the warp shares them
    const float my_inv = inv_rms_of_route(ssp + (lane & (kEpRoutes - 1)) * kChunkStride, a);
    float invq[kEpRoutes];
#pragma unroll
    for (int q = 0; q < kEpRoutes; ++q) invq[q] = __shfl_sync(0xffffffffu, my_inv, q);
#pragma unroll
    for (int q = 0; q < kEpRoutes; ++q) {
      if (q < n_pass) {
        const float inv = invq[q], w = wq[q];
        const int s = sq[q];
        if (s != cur_slot) {  // slot boundary: its BF16 partial joins the slot sum
          if (cur_slot >= 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              o[k] = add2(o[k], bf16_round2(part[k]));
              part[k] = splat2(0.0f);
            }
          }
          cur_slot = s;
        }
        float2 x[4];
        unpack8p(raw[q], x);
        const float2 inv2 = splat2(inv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 nv = WBN ? mul2(mul2(x[k], g[k]), inv2) : mul2(mul2(x[k], inv2), g[k]);
          part[k] = add2(part[k], mul_each(nv, w));  // each product rounded alone
        }
      }
    }
  }
  if (cur_slot >= 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = add2(o[k], bf16_round2(part[k]));
  }
  MOE_TRACE_MARK(3);  // products summed
  if (valid) {
    const uint4 r = pack8p_pz(o);
    if (a.inputs_before_wait) grid_dependency_wait();
    st_v4(a.out + (int64_t)t * a.P + col, r);
  }
}

// ------------------------------------------- expert-TP / latent: staged rows
//
// The same arithmetic as finalize_kernel for expert-TP and the latent norm,
// with the rows staged in shared memory: for each route of each token the
// CTA owns (in route order), the route's rows of this column band in every
// slot arrive by 1-D bulk asynchronous copies in a ring of stages (one route
// = one stage = tp band rows), tracked by mbarriers.  Thread v owns 16-byte
// vector v of the band.  There is no producer thread: the last warp to finish
// with a stage (a shared-memory counter) issues the copies of the route S
// places on, so no thread ever waits for a free stage and a refill goes out
// as soon as the stage is free (expert-TP at b = 128 alone: 16.9 -> 16.0 us,
// against a copy issuer that also consumed and waited for each release).
// A CTA finalizes tokens blockIdx.y, + gridDim.y, ... so the ring keeps
// streaming across tokens.  Every wait is bounded; once a wait gives up, all
// later waits return at once and nothing more is issued, so the kernel ends
// without skipping a barrier, and the copies still in flight are waited for
// (with the full limit) before the CTA's shared memory goes away.

constexpr int kStagedMaxStages = 16;

__device__ unsigned int g_finalize_error = 0;

struct __align__(16) StagedSmem {
  float ss[2][kMaxRoutesPerPass][kChunkStride];
  unsigned long long full[kStagedMaxStages];
  uint32_t released[kStagedMaxStages];  // warps done with the stage's current route
  uint32_t issued;                      // routes issued (a prefix of the CTA's route numbers)
  uint32_t abort_flag;
};

__device__ __forceinline__ void sb_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void sb_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void sb_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool sb_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity; false once the limit has passed --
// the first wait to give up raises the abort flag and the error bit -- or at
// once when the flag is already up.  A limit of 1 ns (the failure-detection
// tests' setting) gives up at once, whether or not the phase has completed.
__device__ __forceinline__ bool sb_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                        unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns > 1 && sb_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (limit_ns <= 1 || !sb_try(bar, parity)) {
    if (*abort_flag) return false;
    if (limit_ns <= 1 || global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(&g_finalize_error, 1u);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

template <bool WBN, int WMODE, bool LATENT>
__global__ void __launch_bounds__(512) staged_finalize_kernel(const FinalizeArgs a) {
  MOE_TRACE_SCOPE(20 + (LATENT ? 1 : 0));
  extern __shared__ __align__(128) uint8_t ring_raw[];
  __shared__ StagedSmem sm;
  const int tid = threadIdx.x, lane = tid & 31;
  const int VB = a.band_vectors;  // one 16-byte vector of the band per thread
  const int S = a.stages;
  const uint32_t n_warps = (uint32_t)(VB / 32);
  const uint32_t split = cluster_size();
  const int band = (int)cluster_rank();
  const int col0 = band * VB * 8;
  const uint32_t band_bytes = (uint32_t)VB * 16;
  const uint32_t copy_bytes = col0 < a.P ? (uint32_t)min(VB * 8, a.P - col0) * 2 : 0u;
  const uint32_t stage_bytes = band_bytes * (uint32_t)a.tp;
  const uint32_t ring = smem_addr(ring_raw);
  volatile uint32_t* abort_flag = &sm.abort_flag;
  // route number m of this CTA: token blockIdx.y + (m / K) * gridDim.y, route m % K
  const int n_tok = a.b > (int)blockIdx.y ? (a.b - (int)blockIdx.y + (int)gridDim.y - 1) / (int)gridDim.y : 0;
  const uint32_t total = (uint32_t)n_tok * (uint32_t)a.K;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      sb_init(smem_addr(&sm.full[i]), 1);
      sm.released[i] = 0;
    }
    sm.issued = 0;
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (!a.inputs_before_wait) grid_dependency_wait();
  launch_dependents();

  // Route m goes into stage m % S.  It is issued by the last warp to finish
  // with route m - S (or at the start), so no thread waits for a free stage;
  // a route without a row completes its stage's phase with a plain arrive.
  // Once any wait has given up nothing more is issued.
  auto issue = [&](uint32_t m) {
    if (*abort_flag) return;
    const int st = (int)(m % (uint32_t)S);
    const int t = (int)blockIdx.y + (int)(m / (uint32_t)a.K) * (int)gridDim.y;
    const int k = (int)(m % (uint32_t)a.K);
    const int64_t j = LATENT ? (int64_t)t : (int64_t)a.idx[(int64_t)t * a.K + k];
    const uint32_t bar = smem_addr(&sm.full[st]);
    if (j >= 0 && j < a.num_rows && copy_bytes) {
      sb_expect(bar, copy_bytes * (uint32_t)a.tp);
      const uint16_t* src = a.rows + j * a.P + col0;
      const uint32_t dst = ring + (uint32_t)st * stage_bytes;
      for (int s = 0; s < a.tp; ++s) bulk_copy(dst + (uint32_t)s * band_bytes, src + (int64_t)s * a.slot_stride, copy_bytes, bar);
    } else {
      sb_arrive(bar);
    }
    atomicAdd(&sm.issued, 1u);
  };
  if (tid == 0)
    for (uint32_t m = 0; m < (uint32_t)S && m < total; ++m) issue(m);

  const int vb = tid;
  const int vec = band * VB + vb;
  const bool valid = vec * 8 < a.P;
  const int chunk = vec >> 5;
  float2 g8[4];
  {
    const uint4 gv = valid ? ld_v4(a.gamma + vec * 8) : make_uint4(0, 0, 0, 0);
    unpack8p(gv, g8);
#pragma unroll
    for (int k = 0; k < 4; ++k) g8[k] = add2(g8[k], splat2(a.gain_center));
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers started: DSMEM is live

  uint32_t m = 0;  // routes consumed
  int pass = 0;
  // the consumers' stage wait (its limit can be shortened for failure-detection tests)
  const unsigned long long stage_limit = a.stage_wait_ns ? a.stage_wait_ns : kWaitLimitNs;
  for (int t = blockIdx.y; t < a.b; t += gridDim.y) {
    float2 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = splat2(0.0f);
    for (int base = 0; base < a.K; base += kMaxRoutesPerPass, ++pass) {
      float2 xr[kMaxRoutesPerPass][4];
      bool has[kMaxRoutesPerPass];
      float wr[kMaxRoutesPerPass];
      float* ss = &sm.ss[pass & 1][0][0];
#pragma unroll
      for (int rr = 0; rr < kMaxRoutesPerPass; ++rr) {
        const int k = base + rr;
        int64_t j = -1;
        if (k < a.K) j = LATENT ? (int64_t)t : (int64_t)a.idx[(int64_t)t * a.K + k];
        has[rr] = k < a.K && j >= 0 && j < a.num_rows;
        wr[rr] = has[rr] ? route_weight<WMODE>(a.w, (int64_t)t * a.K + k) : 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) xr[rr][k] = splat2(0.0f);
        if (k < a.K) {
          const int st = (int)(m % (uint32_t)S);
          sb_wait(smem_addr(&sm.full[st]), (m / S) & 1, abort_flag, stage_limit);
          if (m == 0) MOE_TRACE_MARK(0);  // first route's rows landed
          if (m == 3) MOE_TRACE_MARK(1);  // fourth route's rows landed
          if (has[rr] && valid) {
            const uint8_t* src = ring_raw + (size_t)st * stage_bytes + (size_t)vb * 16;
            for (int s = 0; s < a.tp; ++s, src += band_bytes) {  // slot order, FP32 from +0
              float2 f[4];
              unpack8p(*reinterpret_cast<const uint4*>(src), f);
#pragma unroll
              for (int k = 0; k < 4; ++k) xr[rr][k] = add2(xr[rr][k], f[k]);
            }
          }
          __syncwarp();
          if (lane == 0) {  // the last warp done with route m issues route m + S into its stage
            __threadfence_block();
            if (atomicAdd(&sm.released[st], 1u) == n_warps - 1) {
              sm.released[st] = 0;
              __threadfence_block();
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              if (m + (uint32_t)S < total) issue(m + (uint32_t)S);
            }
          }
          ++m;
        }
        if (has[rr]) {
#pragma unroll
          for (int k = 0; k < 4; ++k) xr[rr][k] = bf16_round2(xr[rr][k]);
          float sq = 0.0f;  // the lane's eight squares, added in column order
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 v = WBN ? mul2(xr[rr][k], g8[k]) : xr[rr][k];
            const float2 s2 = mul2(v, v);
            sq = __fadd_rn(__fadd_rn(sq, s2.x), s2.y);
          }
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, off));
          if (chunk < a.chunks && lane < (int)split)
            st_cluster_f32(map_to_rank(smem_addr(&ss[rr * kChunkStride + chunk]), (uint32_t)lane), sq);
        }
      }
      if (m <= (uint32_t)kMaxRoutesPerPass) MOE_TRACE_MARK(2);  // first pass: all its routes consumed
      cluster_sync_all();
      if (m <= (uint32_t)kMaxRoutesPerPass) MOE_TRACE_MARK(3);
      // lane r of every warp folds route r's chunk sums in chunk order and forms
      // its 1/rms (one square root and division per thread); the warp shares them
      const float my_inv = inv_rms_of_route(ss + (lane & (kMaxRoutesPerPass - 1)) * kChunkStride, a);
#pragma unroll
      for (int rr = 0; rr < kMaxRoutesPerPass; ++rr) {
        const float inv = __shfl_sync(0xffffffffu, my_inv, rr);
        if (has[rr]) {  // a route with no row contributes nothing
          const float2 inv2 = splat2(inv);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 x = xr[rr][k];
            const float2 nv = WBN ? mul2(mul2(x, g8[k]), inv2) : mul2(mul2(x, inv2), g8[k]);
            acc[k] = add2(acc[k], mul_each(nv, wr[rr]));  // each product rounded alone
          }
        }
      }
    }
    if (valid) {
      const uint4 r = pack8p_pz(acc);
      if (a.inputs_before_wait) grid_dependency_wait();  // the preceding kernel may still read out
      st_v4(a.out + (int64_t)t * a.P + vec * 8, r);
    }
  }
  // on abort, let copies in flight land before the CTA's memory goes away
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    const uint32_t issued = sm.issued;
    for (uint32_t i = issued > (uint32_t)S ? issued - S : 0; i < issued; ++i) {
      const unsigned long long t0 = global_ns();
      while (!sb_try(smem_addr(&sm.full[i % S]), (i / S) & 1))
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
  }
}

#ifdef MOE_TAIL_TRACE
cudaError_t trace_attach_finalize(void* buf, unsigned cap) { return trace_attach_tu(buf, cap); }
unsigned trace_count_finalize() { return trace_count_tu(); }
#endif

cudaError_t take_finalize_error(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_finalize_error, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_finalize_error, &zero, sizeof zero);
  *bits = v;
  return e;
}

// ---------------------------------------------------------------- launcher

template <int MODE, bool WBN, int WMODE>
static cudaError_t launch_t(const FinalizeArgs& a, int split, cudaStream_t stream) {
  auto k = finalize_kernel<MODE, WBN, WMODE>;
  const size_t smem = (size_t)a.routes_per_pass * a.band_vectors * 32;
  cudaError_t e = ensure_smem_limit((const void*)k, 64 * 1024);  // once per device, not per call
  if (e != cudaSuccess) return e;
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

template <bool WBN, int WMODE>
static cudaError_t launch_ep_t(const FinalizeArgs& a, int split, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, a.b, 1);
  cfg.blockDim = dim3(a.band_vectors, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ep_finalize_kernel<WBN, WMODE>, a);
}

template <bool WBN, int WMODE, bool LATENT>
static cudaError_t launch_staged_t(const FinalizeArgs& a, int split, int groups, size_t smem, cudaStream_t stream) {
  auto k = staged_finalize_kernel<WBN, WMODE, LATENT>;
  cudaError_t e = ensure_smem_limit((const void*)k, 192 * 1024);  // once per device, not per call
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, groups, 1);
  cfg.blockDim = dim3(a.band_vectors, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, a);
}

// Expert-TP and latent with the rows staged in shared memory; returns
// cudaErrorNotSupported when a stage (one route's rows of a band in every
// slot) does not fit, so the caller can fall back to finalize_kernel.
static cudaError_t launch_staged(int mode, const FinalizeArgs& args, bool wbn, int wmode, int sms, cudaStream_t stream) {
  FinalizeArgs a = args;
  a.stage_wait_ns = stage_wait_limit_ns();
  a.chunks = (a.P + 255) / 256;
  // Bands per token: the fewest that keep a stage (one route's band rows in
  // every slot) within 32 KB, then more while the batch leaves over half of
  // the SMs idle (measured on GB300: tp = 8, P = 4096 is best at 2 bands for
  // b = 64 and b = 128).
  int split = tuning().fin_split;
  if (split == 0) {
    split = 1;
    while (split < 8 && split < a.chunks && (size_t)a.tp * ((a.P + split - 1) / split) * 2 > 32 * 1024) split *= 2;
    while (split < 8 && split < a.chunks && (int64_t)a.b * split < sms / 2) split *= 2;
  }
  while (split < 8 && (a.chunks + split - 1) / split > 16) split *= 2;
  a.band_vectors = 32 * ((a.chunks + split - 1) / split);
  if (a.band_vectors > 512) return cudaErrorNotSupported;
  const size_t stage_bytes = (size_t)a.tp * a.band_vectors * 16;
  const size_t budget = (size_t)(tuning().fin_ring_kb > 0 ? tuning().fin_ring_kb : 64) * 1024;
  a.stages = (int)std::min<size_t>(16, budget / stage_bytes);
  if (a.stages < 2) return cudaErrorNotSupported;
  const int group_cap = tuning().fin_groups;  // tuning override: CTAs along the tokens
  const int groups = (int)std::min<int64_t>(
      a.b, group_cap > 0 ? group_cap : std::max<int64_t>(1, 2 * (int64_t)sms / split));
  const size_t smem = (size_t)a.stages * stage_bytes;
  if (mode == kModeLatent) return launch_staged_t<false, kWeightUnit, true>(a, split, groups, smem, stream);
  if (wbn) return wmode == kWeightBF16 ? launch_staged_t<true, kWeightBF16, false>(a, split, groups, smem, stream)
                                       : launch_staged_t<true, kWeightF32, false>(a, split, groups, smem, stream);
  return wmode == kWeightBF16 ? launch_staged_t<false, kWeightBF16, false>(a, split, groups, smem, stream)
                              : launch_staged_t<false, kWeightF32, false>(a, split, groups, smem, stream);
}

cudaError_t launch_finalize(int mode, const FinalizeArgs& args, bool wbn, int wmode, int sms, cudaStream_t stream) {
  // Staged rows pay off for expert-TP (tp rows per route) once a call has
  // enough routes to keep the ring streaming (measured: b * K >= 512, i.e.
  // b >= 64 at top-8); fewer routes finish sooner on the route-parallel
  // kernel's single trip (b = 1: 4.6 vs 13.5 us).  The latent norm (one route
  // per token) is faster on the route-parallel kernel.  A pinned kernel form
  // (1 staged, 2 route-parallel) takes precedence.
  const int staged = kernel_form(kFormCallTP);
  if (mode == kModeTP && (staged == 1 || (staged != 2 && (int64_t)args.b * args.K >= 512))) {
    const cudaError_t e = launch_staged(mode, args, wbn, wmode, sms, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  FinalizeArgs a = args;
  a.chunks = (a.P + 255) / 256;
  const int routes = mode == kModeLatent ? 1 : (mode == kModeEP ? a.tp * a.K : a.K);
  // Bands per token: EP and the latent norm move little data per token, so
  // about one wave of CTAs (b * split >= 3/4 of the SMs; fewer, smaller
  // clusters also find room beside a running weight stream: the latent norm
  // at b = 64 with 2 bands instead of 8 shortened the composed step by 1.3 us);
  // expert-TP about two waves.  At most 8 bands (portable cluster size), one
  // band per chunk at most.
  int split = tuning().fin_split;
  if (mode == kModeEP && tuning().fin_ep_split) split = tuning().fin_ep_split;  // tuning overrides for EP
  if (mode == kModeLatent && tuning().fin_latent_split) split = tuning().fin_latent_split;  // or the latent norm alone
  if (split == 0) {
    const int64_t target = mode == kModeTP ? 2 * (int64_t)sms : (3 * (int64_t)sms) / 4;
    split = 1;
    while (split < 8 && split < a.chunks && (int64_t)a.b * split < target) split *= 2;
    // The latent norm of up to 4 tokens in at most 2 bands: its 2-CTA clusters
    // hand over to the up-projection sooner (one call at b = 1: 12.4 vs 13.7
    // us; b = 4: 13.5 vs 14.6).  From b = 8 the wide bands are far slower
    // there (~20 us), and the composed step is the same either way.
    if (mode == kModeLatent && a.b <= 4) split = std::min(split, 2);
    // An EP CTA of 512 threads holds a whole SM's registers (about 114 each),
    // so none of a concurrent weight stream's CTAs fits beside it: at most 8
    // warps per band where the row allows (the decode step at b = 128: 87.8 ->
    // 82.0 us per step with 2 bands instead of 1; b = 32 and 96 unchanged).
    if (mode == kModeEP)
      while (split < 8 && split < a.chunks && (a.chunks + split - 1) / split > 8) split *= 2;
  }
  while (split < 8 && (a.chunks + split - 1) / split > kMaxThreads / 32) split *= 2;
  a.band_vectors = 32 * ((a.chunks + split - 1) / split);
  if (a.band_vectors > kMaxThreads) return cudaErrorInvalidValue;
  a.routes_per_pass = std::min(std::min(kMaxRoutesPerPass, std::max(1, routes)), kMaxThreads / a.band_vectors);
  if (mode == kModeEP) {  // a token has about K local rows in all: more groups would idle
    a.routes_per_pass = std::max(1, std::min(a.routes_per_pass, a.K));
  }
  const int routes_cap = tuning().fin_routes;  // tuning override
  if (routes_cap >= 1 && routes_cap <= kMaxRoutesPerPass) a.routes_per_pass = std::min(a.routes_per_pass, routes_cap);
  if (mode == kModeEP && a.band_vectors <= kEpMaxThreads && kernel_form(kFormCallEP) != 2) {
    if (wbn) return wmode == kWeightBF16 ? launch_ep_t<true, kWeightBF16>(a, split, stream)
                                         : launch_ep_t<true, kWeightF32>(a, split, stream);
    return wmode == kWeightBF16 ? launch_ep_t<false, kWeightBF16>(a, split, stream)
                                : launch_ep_t<false, kWeightF32>(a, split, stream);
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
