// Latency floors of a finalize-shaped call: kernels that do only a finalize
// call's memory traffic, launched as the finalize kernels are.  Measurement
// only (libmoetail_floor.so); see include/moe_tail_floor.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_tail_floor.h"
#include "common.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace {

using moetail::grid_dependency_wait;
using moetail::launch_dependents;
using moetail::ld_stream_v4;

constexpr int kMaxVec = 16;  // 16-byte loads in flight per thread, at most

__global__ void floor_empty_kernel() {
  grid_dependency_wait();
  launch_dependents();
}

__device__ __forceinline__ void cta_sink(uint32_t v, uint32_t* sink) {
  __shared__ uint32_t warp_x[32];
  for (int o = 16; o > 0; o >>= 1) v ^= __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) warp_x[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t x = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) x ^= warp_x[w];
    sink[blockIdx.y * gridDim.x + blockIdx.x] = x;
  }
}

// Thread i of the grid loads vectors i, i + n_threads, ... (at most kMaxVec),
// all before using any.
__global__ void floor_read_kernel(const uint4* src, int64_t n_vec, uint32_t* sink) {
  grid_dependency_wait();
  launch_dependents();
  const int64_t n_threads = (int64_t)gridDim.x * gridDim.y * blockDim.x;
  const int64_t i = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  uint4 v[kMaxVec];
#pragma unroll
  for (int q = 0; q < kMaxVec; ++q) {
    const int64_t e = i + q * n_threads;
    v[q] = e < n_vec ? ld_stream_v4(src + e) : make_uint4(0, 0, 0, 0);
  }
  uint32_t x = 0;
#pragma unroll
  for (int q = 0; q < kMaxVec; ++q) x ^= v[q].x ^ v[q].y ^ v[q].z ^ v[q].w;
  cta_sink(x, sink);
}

// CTA (x, y): the nk indices of row y of idx, then 16 bytes per thread of
// band x of every indexed row (at most kMaxVec rows in flight).
__global__ void floor_gather_kernel(const int32_t* idx, int nk, const uint8_t* rows, int64_t n_rows,
                                    int64_t row_bytes, uint32_t* sink) {
  grid_dependency_wait();
  launch_dependents();
  const int64_t col = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 16;
  uint32_t x = 0;
  for (int k0 = 0; k0 < nk; k0 += kMaxVec) {
    int32_t j[kMaxVec];
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q) j[q] = k0 + q < nk ? idx[(int64_t)blockIdx.y * nk + k0 + q] : -1;
    uint4 v[kMaxVec];
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q)
      v[q] = (j[q] >= 0 && j[q] < n_rows) ? ld_stream_v4(rows + (int64_t)j[q] * row_bytes + col)
                                          : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q) x ^= v[q].x ^ v[q].y ^ v[q].z ^ v[q].w;
  }
  cta_sink(x, sink);
}

bool shape_ok(int grid_x, int grid_y, int threads, int cluster) {
  return grid_x > 0 && grid_y > 0 && grid_y <= 65535 && threads >= 32 && threads <= 1024 && threads % 32 == 0 &&
         cluster >= 1 && cluster <= 8 && grid_x % cluster == 0;
}

template <class K, class... Args>
int launch(K kernel, int grid_x, int grid_y, int threads, int cluster, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, grid_y, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
    (void)cudaGetLastError();
    return 2;
  }
  return 0;
}

}  // namespace

MOE_API int moe_tail_floor_empty(int grid_x, int grid_y, int threads, int cluster, void* stream) {
  if (!shape_ok(grid_x, grid_y, threads, cluster)) return 1;
  return launch(floor_empty_kernel, grid_x, grid_y, threads, cluster, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_tail_floor_read(const void* src, size_t bytes, int grid_x, int grid_y, int threads, int cluster,
                                uint32_t* sink, void* stream) {
  if (!shape_ok(grid_x, grid_y, threads, cluster) || !src || !sink || bytes == 0 || bytes % 16 ||
      ((uintptr_t)src & 15) || ((uintptr_t)sink & 3))
    return 1;
  if ((int64_t)(bytes / 16) > (int64_t)grid_x * grid_y * threads * kMaxVec) return 1;  // one trip per thread
  return launch(floor_read_kernel, grid_x, grid_y, threads, cluster, static_cast<cudaStream_t>(stream),
                static_cast<const uint4*>(src), (int64_t)(bytes / 16), sink);
}

MOE_API int moe_tail_floor_gather(const int32_t* idx, int nk, const void* rows, int64_t n_rows, int grid_x,
                                  int grid_y, int threads, int cluster, uint32_t* sink, void* stream) {
  if (!shape_ok(grid_x, grid_y, threads, cluster) || !idx || !rows || !sink || nk < 1 || n_rows < 1 ||
      ((uintptr_t)idx & 3) || ((uintptr_t)rows & 15) || ((uintptr_t)sink & 3))
    return 1;
  return launch(floor_gather_kernel, grid_x, grid_y, threads, cluster, static_cast<cudaStream_t>(stream), idx, nk,
                static_cast<const uint8_t*>(rows), n_rows, (int64_t)grid_x * threads * 16, sink);
}
