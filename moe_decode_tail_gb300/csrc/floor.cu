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

constexpr int kMaxVec = 16;  // 16-byte loads in flight per thread, at most
constexpr int kMaxThreads = 768;  // kMaxVec slots of 16 bytes per thread in shared memory: 192 KB

// The loads are asynchronous copies into shared memory (one 16-byte slot per
// load and thread), so that every one of them is in flight before any is
// waited for: loads into registers leave that to the compiler's schedule.
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

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

// Thread i of the grid copies vectors i, i + n_threads, ... (at most kMaxVec)
// into its slots, all before waiting for any.
__global__ void floor_read_kernel(const uint4* src, int64_t n_vec, uint32_t* sink) {
  extern __shared__ uint4 slots[];  // [kMaxVec][blockDim.x]
  grid_dependency_wait();
  launch_dependents();
  const int64_t n_threads = (int64_t)gridDim.x * gridDim.y * blockDim.x;
  const int64_t i = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
  for (int q = 0; q < kMaxVec; ++q) {
    const int64_t e = i + q * n_threads;
    uint4* slot = &slots[q * blockDim.x + threadIdx.x];
    if (e < n_vec) cp16(smem_u32(slot), src + e);
    else *slot = make_uint4(0, 0, 0, 0);
  }
  cp_wait_all();
  uint32_t x = 0;
#pragma unroll
  for (int q = 0; q < kMaxVec; ++q) {
    const uint4 v = slots[q * blockDim.x + threadIdx.x];
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  cta_sink(x, sink);
}

// CTA (x, y): the nk indices of row y of idx, then 16 bytes per thread of
// band x of every indexed row (at most kMaxVec rows in flight).
__global__ void floor_gather_kernel(const int32_t* idx, int nk, const uint8_t* rows, int64_t n_rows,
                                    int64_t row_bytes, uint32_t* sink) {
  extern __shared__ uint4 slots[];  // [kMaxVec][blockDim.x]
  grid_dependency_wait();
  launch_dependents();
  const int64_t col = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 16;
  uint32_t x = 0;
  for (int k0 = 0; k0 < nk; k0 += kMaxVec) {
    int32_t j[kMaxVec];
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q) j[q] = k0 + q < nk ? idx[(int64_t)blockIdx.y * nk + k0 + q] : -1;
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q) {
      uint4* slot = &slots[q * blockDim.x + threadIdx.x];
      if (j[q] >= 0 && j[q] < n_rows) cp16(smem_u32(slot), rows + (int64_t)j[q] * row_bytes + col);
      else *slot = make_uint4(0, 0, 0, 0);
    }
    cp_wait_all();
#pragma unroll
    for (int q = 0; q < kMaxVec; ++q) {
      const uint4 v = slots[q * blockDim.x + threadIdx.x];
      x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  cta_sink(x, sink);
}

bool shape_ok(int grid_x, int grid_y, int threads, int cluster) {
  return grid_x > 0 && grid_y > 0 && grid_y <= 65535 && threads >= 32 && threads <= kMaxThreads &&
         threads % 32 == 0 && cluster >= 1 && cluster <= 8 && grid_x % cluster == 0;
}

template <class K, class... Args>
int launch(K kernel, int grid_x, int grid_y, int threads, int cluster, size_t smem, cudaStream_t st, Args... args) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, grid_y, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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
  return launch(floor_empty_kernel, grid_x, grid_y, threads, cluster, 0, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_tail_floor_read(const void* src, size_t bytes, int grid_x, int grid_y, int threads, int cluster,
                                uint32_t* sink, void* stream) {
  if (!shape_ok(grid_x, grid_y, threads, cluster) || !src || !sink || bytes == 0 || bytes % 16 ||
      ((uintptr_t)src & 15) || ((uintptr_t)sink & 3))
    return 1;
  if ((int64_t)(bytes / 16) > (int64_t)grid_x * grid_y * threads * kMaxVec) return 1;  // one trip per thread
  return launch(floor_read_kernel, grid_x, grid_y, threads, cluster, (size_t)threads * kMaxVec * 16,
                static_cast<cudaStream_t>(stream),
                static_cast<const uint4*>(src), (int64_t)(bytes / 16), sink);
}

MOE_API int moe_tail_floor_gather(const int32_t* idx, int nk, const void* rows, int64_t n_rows, int grid_x,
                                  int grid_y, int threads, int cluster, uint32_t* sink, void* stream) {
  if (!shape_ok(grid_x, grid_y, threads, cluster) || !idx || !rows || !sink || nk < 1 || n_rows < 1 ||
      ((uintptr_t)idx & 3) || ((uintptr_t)rows & 15) || ((uintptr_t)sink & 3))
    return 1;
  return launch(floor_gather_kernel, grid_x, grid_y, threads, cluster, (size_t)threads * kMaxVec * 16,
                static_cast<cudaStream_t>(stream), idx, nk,
                static_cast<const uint8_t*>(rows), n_rows, (int64_t)grid_x * threads * 16, sink);
}
