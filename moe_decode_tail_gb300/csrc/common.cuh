// Device helpers shared by the MoE decode tail kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moetail {

// Error word the kernels raise instead of trapping: a bounded wait that runs
// out sets a bit here, skips its remaining work and returns.  The host reads
// and clears it with moe_tail_take_device_error().
enum : unsigned {
  kErrWaitFull = 1u << 0,    // an operand stage never arrived
  kErrWaitEmpty = 1u << 1,   // a stage was never released by the MMA
  kErrWaitAccum = 1u << 2,   // the accumulator never completed
  kErrWaitDrain = 1u << 3,   // an in-flight copy did not land while aborting
  kErrTmemAlloc = 1u << 4,   // tensor memory allocation returned a bad address
};

// Wall-clock bound on every spin in these kernels.
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}


// ---- BF16 vectors --------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round to BF16 (nearest, ties to even); -0 becomes +0.
__device__ __forceinline__ uint32_t bf16_bits_pz(float f) {
  uint32_t h = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
  return h == 0x8000u ? 0u : h;
}
__device__ __forceinline__ float bf16_round(float f) {
  return __bfloat162float(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf16x2_pz(float lo, float hi) {
  return bf16_bits_pz(lo) | (bf16_bits_pz(hi) << 16);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// ---- paired FP32 arithmetic ----------------------------------------------------
//
// Eight consecutive values as four pairs (2k, 2k + 1).  add.rn.f32x2 and
// mul.rn.f32x2 do two binary32 operations in one instruction, each component
// rounded to nearest even as add.rn.f32 / mul.rn.f32 round it, so the paired
// loops give the bits of the scalar ones -- with one rule: a paired product
// never feeds a paired add.  Measured on GB300, such a pair gave sums as if
// the product had not been rounded (one ulp off in rare elements), despite
// the explicit rounding modes and with contraction switched off; a product
// that goes into a sum is formed by mul_each (two __fmul_rn, which are never
// merged) instead.
__device__ __forceinline__ void unpack8p(const uint4& v, float2 (&f)[4]) {
  f[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
  f[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
  f[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
  f[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
}
__device__ __forceinline__ uint64_t pair_bits(float2 v) {
  return ((uint64_t)__float_as_uint(v.y) << 32) | __float_as_uint(v.x);
}
__device__ __forceinline__ float2 pair_of(uint64_t b) {
  return make_float2(__uint_as_float((uint32_t)b), __uint_as_float((uint32_t)(b >> 32)));
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pair_bits(a)), "l"(pair_bits(b)));
  return pair_of(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pair_bits(a)), "l"(pair_bits(b)));
  return pair_of(d);
}
// Each component times s, as two scalar products that are never merged into a
// following add (the form to use for a product that is summed).
__device__ __forceinline__ float2 mul_each(float2 v, float s) { return make_float2(__fmul_rn(v.x, s), __fmul_rn(v.y, s)); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
// Both components rounded to BF16 as bf16_round rounds each, by one paired
// conversion (cvt.rn.bf16x2.f32 puts its first source in the upper half).
__device__ __forceinline__ float2 bf16_round2(float2 v) {
  uint32_t b;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(v.y), "f"(v.x));
  return make_float2(bf16_lo(b), bf16_hi(b));
}
__device__ __forceinline__ uint4 pack8p_pz(const float2 (&o)[4]) {
  return make_uint4(pack_bf16x2_pz(o[0].x, o[0].y), pack_bf16x2_pz(o[1].x, o[1].y), pack_bf16x2_pz(o[2].x, o[2].y),
                    pack_bf16x2_pz(o[3].x, o[3].y));
}

// 16-byte streaming load of data read once (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---- clusters and distributed shared memory -------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// Every thread of every CTA of the cluster: release our writes, acquire peers'.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---- programmatic dependent launch -------------------------------------------

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


// ---- per-CTA timeline trace (only in builds with MOE_TAIL_TRACE) -----------
//
// Thread 0 of every CTA records %globaltimer at kernel entry, at up to four
// marks inside the kernel and at exit, with the kernel's id, the CTA index and
// the SM, into a device buffer the host attaches.  Each translation unit has
// its own copy of the buffer pointer; moe_tail_trace_attach sets them all.
#ifdef MOE_TAIL_TRACE
struct TraceRec {
  unsigned long long t0, mark[4], t1, ids, pad;  // ids: kernel id << 48 | SM << 32 | CTA
};
static_assert(sizeof(TraceRec) == 64, "trace record layout");
static __device__ TraceRec* g_trace_buf = nullptr;
static __device__ unsigned g_trace_n = 0;
static __device__ unsigned g_trace_cap = 0;
struct TraceScope {
  unsigned long long t0, mark[4];
  unsigned kid;
  __device__ explicit TraceScope(unsigned k) : t0(global_ns()), mark{0, 0, 0, 0}, kid(k) {}
  __device__ ~TraceScope() {
    if (threadIdx.x != 0 || g_trace_buf == nullptr) return;
    const unsigned i = atomicAdd(&g_trace_n, 1u);
    if (i >= g_trace_cap) return;
    unsigned sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    g_trace_buf[i] = TraceRec{t0, {mark[0], mark[1], mark[2], mark[3]}, global_ns(),
                              ((unsigned long long)kid << 48) | ((unsigned long long)sm << 32) | cta, 0};
  }
};
// attach (or detach, buf = null) this translation unit's copy and reset its count
static inline cudaError_t trace_attach_tu(void* buf, unsigned cap) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyToSymbol(g_trace_buf, &buf, sizeof buf);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_trace_cap, &cap, sizeof cap);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_trace_n, &zero, sizeof zero);
  return e;
}
static inline unsigned trace_count_tu() {
  unsigned n = 0;
  cudaMemcpyFromSymbol(&n, g_trace_n, sizeof n);
  return n;
}
#define MOE_TRACE_SCOPE(kid) ::moetail::TraceScope moe_trace_scope_(kid)
#define MOE_TRACE_MARK(k) \
  do {                    \
    if (threadIdx.x == 0) moe_trace_scope_.mark[k] = ::moetail::global_ns(); \
  } while (0)
#else
#define MOE_TRACE_SCOPE(kid) \
  do {                       \
  } while (0)
#define MOE_TRACE_MARK(k) \
  do {                    \
  } while (0)
#endif

}  // namespace moetail
