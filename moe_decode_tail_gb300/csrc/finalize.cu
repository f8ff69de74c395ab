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
// Layout of the work: one CTA per (column band, token); the bands of a token
// form a thread-block cluster.  Every warp owns one 256-column chunk of the
// row (lane l: columns 8l..8l+7 of it, one 16-byte vector), computes that
// chunk's sum of squares with the xor butterfly and stores it into every
// cluster CTA's shared memory (DSMEM).  After one cluster barrier each CTA
// folds all chunk sums of the row in chunk order from +0, so the result is
// the same bits whatever the split.  All arithmetic is single IEEE binary32
// operations (__fmul_rn / __fadd_rn: never contracted into an FMA), the
// inverse RMS is 1 / sqrt(.) with IEEE square root and division, and
// subnormals are kept.
#include "common.cuh"
#include "kernels.h"

namespace moetail {

constexpr int kBatch = 8;        // route rows normalised per pass
constexpr int kMaxChunks = 128;  // P <= 32768
constexpr int kMaxList = 1024;   // tp * K <= 32 * 32

struct __align__(16) FinalizeSmem {
  float ss[2][kBatch][kMaxChunks];  // chunk sums of squares, double-buffered
  int list_sk[kMaxList];            // EP: local routes as s * K + k, in (s, k) order
  int list_j[kMaxList];             // EP: their rows within the slot
  int warp_count[32];
  int warp_base[32];
  int count;
};

__device__ __forceinline__ float lane_sum_of_squares(const float (&v)[8]) {
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(v[i], v[i]));
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
  return acc;
}

__device__ __forceinline__ float inverse_rms(const float* chunk_ss, int chunks, float rcpP, float eps) {
  float ss = 0.0f;
  for (int c = 0; c < chunks; ++c) ss = __fadd_rn(ss, chunk_ss[c]);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, rcpP), eps)));
}

// Lane 0 of each warp publishes its chunk's sum to every CTA of the cluster.
__device__ __forceinline__ void publish_chunk_sum(float* slot, float value, int lane, uint32_t split) {
  if (lane == 0) {
    uint32_t addr = smem_addr(slot);
    for (uint32_t q = 0; q < split; ++q) st_cluster_f32(map_to_rank(addr, q), value);
  }
}

template <int WMODE>
__device__ __forceinline__ float route_weight(const void* w, int64_t i) {
  if (WMODE == kWeightBF16) return __uint_as_float((uint32_t)((const uint16_t*)w)[i] << 16);
  if (WMODE == kWeightUnit) return 1.0f;
  return ((const float*)w)[i];
}

// ---------------------------------------------------------------- EP finalize

template <bool WBN, int WMODE>
__global__ void __launch_bounds__(512) ep_finalize_kernel(const EpArgs a) {
  __shared__ FinalizeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
  const int t = blockIdx.y;
  const uint32_t split = cluster_size();
  const int band = (int)cluster_rank();
  const int chunk = band * (nthreads >> 5) + warp;  // this warp's 256-column chunk
  const int col = chunk * 256 + lane * 8;
  const bool valid = chunk < a.chunks && col < a.P;

  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  grid_dependency_wait();

  // Local routes of token t in (slot, route) order: the slot sums run in slot
  // order and each slot's routes in route order.
  const int n = a.tp * a.K;
  int running = 0;
  for (int base = 0; base < n; base += nthreads) {
    const int i = base + tid;
    int j = -1;
    if (i < n) {
      const int s = i / a.K, k = i - s * a.K;
      j = a.idx[((int64_t)s * a.b + t) * a.K + k];
    }
    const bool local = i < n && j >= 0 && (int64_t)j < a.rows_per_slot;
    const unsigned ballot = __ballot_sync(0xffffffffu, local);
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
    if (local) {
      const int pos = running + sm.warp_base[warp] + __popc(ballot & ((1u << lane) - 1u));
      sm.list_sk[pos] = i;
      sm.list_j[pos] = j;
    }
    running += sm.count;
    __syncthreads();
  }
  const int count = running;

  float g[8];
  {
    uint4 gv = valid ? ld_v4(a.gamma + col) : make_uint4(0, 0, 0, 0);
    unpack8(gv, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = __fadd_rn(g[i], a.gain_center);
  }
  float o[8], part[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = part[i] = 0.0f;
  int cur_slot = -1;

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // peers started: DSMEM is live

  for (int base = 0, pass = 0; base < count; base += kBatch, ++pass) {
    const int nb = min(kBatch, count - base);
    uint4 xv[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      xv[r] = make_uint4(0, 0, 0, 0);
      if (r < nb && valid) {
        const int s = sm.list_sk[base + r] / a.K;
        const int64_t row = (int64_t)s * a.rows_per_slot + sm.list_j[base + r];
        xv[r] = ld_stream_v4(a.rows + row * a.P + col);
      }
    }
    float(*ss)[kMaxChunks] = sm.ss[pass & 1];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      if (r < nb) {
        float x[8];
        unpack8(xv[r], x);
        if (WBN) {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], g[i]);
        }
        const float s = lane_sum_of_squares(x);
        if (chunk < a.chunks) publish_chunk_sum(&ss[r][chunk], s, lane, split);
      }
    }
    cluster_sync_all();
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      if (r < nb) {
        const float inv = inverse_rms(ss[r], a.chunks, a.rcpP, a.eps);
        const int sk = sm.list_sk[base + r];
        const int s = sk / a.K, k = sk - s * a.K;
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
        const float w = route_weight<WMODE>(a.w, (int64_t)t * a.K + k);
        float x[8];
        unpack8(xv[r], x);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float nv = WBN ? __fmul_rn(__fmul_rn(x[i], g[i]), inv) : __fmul_rn(__fmul_rn(x[i], inv), g[i]);
          part[i] = __fadd_rn(part[i], __fmul_rn(nv, w));
        }
      }
    }
  }
  if (cur_slot >= 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __fadd_rn(o[i], bf16_round(part[i]));
  }
  launch_dependents();
  if (valid) {
    uint4 r;
    r.x = pack_bf16x2_pz(o[0], o[1]);
    r.y = pack_bf16x2_pz(o[2], o[3]);
    r.z = pack_bf16x2_pz(o[4], o[5]);
    r.w = pack_bf16x2_pz(o[6], o[7]);
    st_v4(a.out + (int64_t)t * a.P + col, r);
  }
}

// ------------------------------------------------ expert-TP finalize / latent norm
//
// Route (t, k)'s row j = idx[t, k] (or j = t for the latent norm) has a
// K-partial in every slot; x = bf16(sum over slots in order), then the same
// normalisation as EP, routes summed in order from +0.

template <bool WBN, int WMODE>
__global__ void __launch_bounds__(512) tp_finalize_kernel(const TpArgs a) {
  __shared__ FinalizeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
  const int t = blockIdx.y;
  const uint32_t split = cluster_size();
  const int band = (int)cluster_rank();
  const int chunk = band * (nthreads >> 5) + warp;
  const int col = chunk * 256 + lane * 8;
  const bool valid = chunk < a.chunks && col < a.P;
  (void)tid;

  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  grid_dependency_wait();

  float g[8];
  {
    uint4 gv = valid ? ld_v4(a.gamma + col) : make_uint4(0, 0, 0, 0);
    unpack8(gv, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = __fadd_rn(g[i], a.gain_center);
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

  for (int base = 0, pass = 0; base < a.K; base += kBatch, ++pass) {
    const int nb = min(kBatch, a.K - base);
    int64_t rowoff[kBatch];
    bool local[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      int64_t j = -1;
      if (r < nb) j = a.idx ? (int64_t)a.idx[(int64_t)t * a.K + base + r] : (int64_t)t;
      local[r] = r < nb && j >= 0 && j < a.num_rows;
      rowoff[r] = local[r] ? j * a.P + col : 0;
    }
    float xs[kBatch][8];
#pragma unroll
    for (int r = 0; r < kBatch; ++r)
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[r][i] = 0.0f;
    const uint16_t* slot_base = a.partials;
#pragma unroll 1
    for (int s = 0; s < a.tp; ++s, slot_base += a.slot_stride) {
      uint4 v[kBatch];
#pragma unroll
      for (int r = 0; r < kBatch; ++r)
        v[r] = (local[r] && valid) ? ld_stream_v4(slot_base + rowoff[r]) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        float f[8];
        unpack8(v[r], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) xs[r][i] = __fadd_rn(xs[r][i], f[i]);
      }
    }
    float(*ss)[kMaxChunks] = sm.ss[pass & 1];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[r][i] = bf16_round(xs[r][i]);
      if (local[r]) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = WBN ? __fmul_rn(xs[r][i], g[i]) : xs[r][i];
        const float s = lane_sum_of_squares(v);
        if (chunk < a.chunks) publish_chunk_sum(&ss[r][chunk], s, lane, split);
      }
    }
    cluster_sync_all();
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      if (local[r]) {  // a route with no row contributes nothing
        const float inv = inverse_rms(ss[r], a.chunks, a.rcpP, a.eps);
        const float w = route_weight<WMODE>(a.w, (int64_t)t * a.K + base + r);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x = xs[r][i];
          const float nv = WBN ? __fmul_rn(__fmul_rn(x, g[i]), inv) : __fmul_rn(__fmul_rn(x, inv), g[i]);
          acc[i] = __fadd_rn(acc[i], __fmul_rn(nv, w));
        }
      }
    }
  }
  launch_dependents();
  if (valid) {
    uint4 r;
    r.x = pack_bf16x2_pz(acc[0], acc[1]);
    r.y = pack_bf16x2_pz(acc[2], acc[3]);
    r.z = pack_bf16x2_pz(acc[4], acc[5]);
    r.w = pack_bf16x2_pz(acc[6], acc[7]);
    st_v4(a.out + (int64_t)t * a.P + col, r);
  }
}

// ---------------------------------------------------------------- launchers

// Column bands per token: enough CTAs to cover the SMs about twice, at most
// 8 (portable cluster size) and at most one band per chunk.
static int choose_split(int b, int chunks, int sms, int force) {
  if (force > 0) return force;
  int split = 1;
  while (split < 8 && split < chunks && (int64_t)b * split < 2 * sms) split *= 2;
  while (split < chunks && (chunks + split - 1) / split > 16) split *= 2;  // <= 512 threads
  return split;
}

template <typename Kernel, typename Args>
static cudaError_t launch_cluster(Kernel kernel, const Args& a, int b, int chunks, int split, bool pdl,
                                  cudaStream_t stream) {
  const int warps = (chunks + split - 1) / split;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, b, 1);
  cfg.blockDim = dim3(32 * warps, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch_ep_finalize(const EpArgs& a, bool wbn, int wmode, int sms, int force_split,
                               cudaStream_t stream) {
  const int split = choose_split(a.b, a.chunks, sms, force_split);
  EpArgs args = a;
  if (wbn) {
    if (wmode == kWeightBF16) return launch_cluster(ep_finalize_kernel<true, kWeightBF16>, args, a.b, a.chunks, split, false, stream);
    return launch_cluster(ep_finalize_kernel<true, kWeightF32>, args, a.b, a.chunks, split, false, stream);
  }
  if (wmode == kWeightBF16) return launch_cluster(ep_finalize_kernel<false, kWeightBF16>, args, a.b, a.chunks, split, false, stream);
  return launch_cluster(ep_finalize_kernel<false, kWeightF32>, args, a.b, a.chunks, split, false, stream);
}

cudaError_t launch_tp_finalize(const TpArgs& a, bool wbn, int wmode, int sms, int force_split,
                               cudaStream_t stream) {
  const int split = choose_split(a.b, a.chunks, sms, force_split);
  TpArgs args = a;
  if (wmode == kWeightUnit)  // latent norm: gain after the norm, unit weight
    return launch_cluster(tp_finalize_kernel<false, kWeightUnit>, args, a.b, a.chunks, split, false, stream);
  if (wbn) {
    if (wmode == kWeightBF16) return launch_cluster(tp_finalize_kernel<true, kWeightBF16>, args, a.b, a.chunks, split, false, stream);
    return launch_cluster(tp_finalize_kernel<true, kWeightF32>, args, a.b, a.chunks, split, false, stream);
  }
  if (wmode == kWeightBF16) return launch_cluster(tp_finalize_kernel<false, kWeightBF16>, args, a.b, a.chunks, split, false, stream);
  return launch_cluster(tp_finalize_kernel<false, kWeightF32>, args, a.b, a.chunks, split, false, stream);
}

}  // namespace moetail
