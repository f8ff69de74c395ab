// Small-batch decode GEMM on the 5th-generation tensor cores (sm_103a).
//
//   D[m, t] = sum_k W[m, k] * X[t, k]       (W: weights [M, K], X: tokens [b, K])
//
// The weights are the MMA's M operand (64 or 128 rows per CTA) and the tokens
// its N operand ("swap AB"), so a decode batch of b <= 128 tokens is one N
// tile and the kernel is a stream of weight tiles: its roofline is the weight
// bytes over HBM bandwidth.  Per CTA: warp 4 (one thread) streams Mx64 BF16
// weight tiles and Nx64 token tiles with TMA (128-byte swizzle) into a ring of
// shared-memory stages guarded by mbarriers; warp 5 (one thread) issues four
// K=16 tcgen05.mma per stage into an FP32 accumulator in tensor memory and
// releases the stage with tcgen05.commit; warps 0-3 read the accumulator
// (tcgen05.ld, one TMEM lane = one weight row per thread).  The K range may
// be split over the CTAs of a thread-block cluster; their FP32 partial tiles
// are then added in cluster-rank order over distributed shared memory, so the
// result is deterministic, and the fused epilogue writes BF16:
//
//   kGemmUpShared   out = bf16(acc + sum_s shared[s])   (latent tail up-projection
//                   plus the shared-expert partials, Kimi-K3 tail runtime page,
//                   module docstring)
//   kGemmGateUpSilu the first half of the tile's rows are gate rows, the second
//                   half the matching up rows; h = bf16(silu(bf16(gate)) * bf16(up))  (Kimi-K3
//                   shared expert page: SharedUmma.load_tile pairs gate and up
//                   rows in one M tile; owned_h rounds gate and up to BF16)
//   kGemmDown       out = bf16(out + bf16(d)) or bf16(d)  (the down projection
//                   pushed as BF16, -0 made +0, added into the tail's output)
//   kGemmLatentUp   kGemmUpShared with y formed on chip from the latent partials
//                   (the latent tail in one kernel; taken only on request)
//   kGemmDownUp     the shared expert's down projection d and the up-projection
//                   u in one kernel: out = bf16(u + (sum_s shared[s] + bf16(d)))
//                   (Kimi-K3 tail runtime page, module docstring: the shared
//                   expert's output is one more shared partial).  The cluster's
//                   first ranks split W_down's K range, the others W_up's; one
//                   epilogue adds each projection's partials in rank order.
//
// Every wait is bounded in time; on expiry the kernel raises a bit in the
// device error word, drains what it started, frees its tensor memory and
// returns.
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moetail {

constexpr int kBlockK = 64;                        // BF16 per K block: one 128-byte swizzle row
constexpr int kThreads = 192;                      // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kMaxStages = 12;

// The device error word of this library (see the enum in common.cuh).
__device__ unsigned int g_device_error = 0;
__device__ __forceinline__ void raise_error(unsigned bit) { atomicOr(&g_device_error, bit); }

cudaError_t take_device_error(unsigned* bits) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  *bits = v;
  return e;
}

// ---- PTX wrappers --------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
// Wait for the phase of the given parity to complete; false if the time limit
// ran out, or (given abort_flag) once another thread of the CTA has aborted.
// A limit of 1 ns (the failure-detection tests' setting) gives up at once,
// whether or not the phase has completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs,
                                          volatile uint32_t* abort_flag = nullptr) {
  if (limit_ns <= 1) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (abort_flag && *abort_flag) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled TMA load of box (x = inner coordinate, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 16 consecutive FP32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes, written by TMA with 128-byte swizzle: 8-row groups 1024 bytes
// apart (stride byte offset), the leading byte offset unused by this layout,
// descriptor version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: FP32 accumulate (bits 4-5 = 1), BF16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

struct GemmSmem {  // offsets from the 1024-aligned base of dynamic shared memory
  uint32_t ring, full, empty, accum, tmem_slot, abort_flag;
  // latent tail in one kernel: y operand, chunk sums, 1/rms, gamma of the K
  // range; y ready for the MMA; latent loads issued (the weights may follow)
  uint32_t yop, ss, inv, gam, ybar, latbar;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Barrier 1 over the four epilogue warps only.
__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Byte offset, in a K-major operand tile of 128-byte rows written with the
// 128-byte swizzle, of the 16-byte unit u (columns 8u..8u+7) of row r: the
// unit index is XORed with the row's position in its 8-row group, as a TMA
// box lands with CU_TENSOR_MAP_SWIZZLE_128B (tile bases 1024-aligned).
__device__ __forceinline__ uint32_t sw128_offset(int r, int u) {
  return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
}

// Cluster rank whose K range holds K block kb under the even split of
// kblocks over ksplit ranks (the first kb_rem ranks take one more).
__device__ __forceinline__ uint32_t kblock_owner(int kb, int kb_per, int kb_rem) {
  const int big = kb_rem * (kb_per + 1);
  return (uint32_t)(kb < big ? kb / (kb_per + 1) : kb_rem + (kb - big) / kb_per);
}

// TM = weight rows per CTA: 64 (one M=64 MMA), 128 (one M=128 MMA) or 256
// (two M=128 MMAs per K step sharing the token tile, into two accumulators
// at TMEM columns [0, N) and [N, 2N)).  With M = 128 accumulator row r sits
// in TMEM lane r; with M = 64 it sits in lane 32 * (r / 16) + r % 16 (lanes
// 16..31 of each warp's quarter stay unused).  Gate/up tiles hold TM/2 gate
// rows then the TM/2 matching up rows.
//
// kGemmLatentUp is the whole latent tail in one kernel (Kimi-K3 tail runtime
// page, module docstring: latent sum over the slots, RMS norm, up-projection,
// shared partials): instead of loading token tiles, the epilogue warps form y
// for the CTA's K range in shared memory, in the swizzled operand layout, while
// the weight ring fills.  Each CTA forms x (the slot sum, rounded to BF16) for
// every 256-column chunk its K range touches, with the chunk's sum of squares
// in the finalize kernels' canonical tree (lane l: columns 8l..8l+7 in order,
// xor butterfly); after one cluster barrier each token's chunk sums are read
// from the CTA that holds the chunk's first K block and added in chunk order
// from +0, so y is bit for bit the norm kernel's y.  The K split and the MMA
// sequence are the up-projection's, so out is bit for bit the two-kernel
// result as well.
template <int MODE, int N, int TM>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                       const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_x1,
                       const GemmArgs a, const int stages) {
  MOE_TRACE_SCOPE(30 + MODE);
  extern __shared__ uint8_t smem_raw[];
  constexpr bool kFused = MODE == kGemmLatentUp;
  constexpr bool kDU = MODE == kGemmDownUp;  // d on some ranks of the cluster, u on the rest, one epilogue
  constexpr bool kUp = MODE == kGemmUpShared || kFused || kDU;  // out = bf16(acc + slot sum of shared)
  constexpr int kATile = TM * kBlockK * 2;
  constexpr int kBTileBytes = N * kBlockK * 2;
  constexpr int kStageBytes = kFused ? kATile : kATile + kBTileBytes;
  constexpr int kMmaM = TM == 64 ? 64 : 128;
  constexpr int kNumAcc = TM / kMmaM;
  constexpr int kAccCols = N * kNumAcc;  // the accumulator's TMEM columns
  constexpr uint32_t kTmemCols = kAccCols < 32 ? 32 : kAccCols;
  constexpr uint32_t kIdesc = idesc_bf16(kMmaM, N);
  constexpr int kOutRows = (MODE == kGemmGateUpSilu) ? TM / 2 : TM;  // output features per tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank(), ksplit = cluster_size();
  const int m_tile = blockIdx.y;
  const int tok0 = blockIdx.z * N;

  // K blocks of this CTA: an even split of the tile's K range over the cluster
  // (down + up: the first n_down ranks split the down projection's K range,
  // the others the up-projection's; a rank streams one weight into one
  // accumulator).
  const int n_down = kDU ? downup_down_ranks((int)ksplit, a.kblocks, a.kblocks2) : 0;
  const bool up_rank = kDU && (int)rank >= n_down;  // down + up: this CTA streams W_up against y
  const int g_rank = up_rank ? (int)rank - n_down : (int)rank;
  const int g_size = kDU ? (up_rank ? (int)ksplit - n_down : n_down) : (int)ksplit;
  const int g_blocks = up_rank ? a.kblocks2 : a.kblocks;
  const int kb_per = g_blocks / g_size, kb_rem = g_blocks % g_size;
  const int kb0 = g_rank * kb_per + min(g_rank, kb_rem);
  const int nk = kb_per + (g_rank < kb_rem ? 1 : 0);
  const int nk_all = nk;

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  GemmSmem L;
  L.ring = base;
  uint32_t tail = base + stages * kStageBytes;
  if (kFused) {  // y operand of the CTA's K range, chunk sums [N][chunks], 1/rms [N]
    L.yop = tail;  // 1024-aligned: kATile is a multiple of 1024
    tail += (uint32_t)((kb_per + (kb_rem > 0 ? 1 : 0)) * kBTileBytes);
    L.ss = tail;
    tail += (uint32_t)(4 * N * a.chunks);
    L.inv = tail;
    tail += 4u * N;
    L.gam = tail;  // 16-aligned: the offsets before it are multiples of 64
    tail = (tail + (uint32_t)((kb_per + (kb_rem > 0 ? 1 : 0)) * kBlockK * 2) + 7u) & ~7u;
  }
  L.full = tail;
  L.empty = L.full + 8 * stages;
  L.accum = L.empty + 8 * stages;
  L.ybar = L.accum + 8;
  L.latbar = L.accum + 16;
  L.tmem_slot = L.accum + (kFused ? 24 : 8);
  L.abort_flag = L.tmem_slot + 4;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (L.tmem_slot - base));
  volatile uint32_t* abort_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (L.abort_flag - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(L.full + 8 * s, 1);
      mbar_init(L.empty + 8 * s, 1);
    }
    mbar_init(L.accum, 1);
    if (kFused) {
      mbar_init(L.ybar, 128);
      mbar_init(L.latbar, 128);
    }
    *abort_ptr = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w0);
    if (MODE == kGemmGateUpSilu || kDU) prefetch_map(&map_w1);
    if (!kFused) prefetch_map(&map_x);
    if (kDU) prefetch_map(&map_x1);
  }
  if (warp == 5) tmem_alloc(L.tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  launch_dependents();  // the next kernel may be scheduled as this one's CTAs retire
  // The epilogue warps exchange chunk sums over one cluster barrier; the
  // producer and MMA warps take part in it without waiting here.
  if (kFused && ksplit > 1 && warp >= 4) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // Tokens whose outputs this CTA finishes (the tile's tokens split over the cluster).
  const int n_valid = min(N, a.n_tok - tok0);
  const int t_per = n_valid / (int)ksplit, t_rem = n_valid % (int)ksplit;
  const int t_begin = (int)rank * t_per + min((int)rank, t_rem);
  const int t_count = t_per + ((int)rank < t_rem ? 1 : 0);
  constexpr int kQuads = kOutRows / 4;  // an epilogue item: 4 output features of one token
  const int n_items = t_count * kQuads;
  // The epilogue's addend of an item -- the slot sum of the shared partials
  // (up-projection) or the old out (accumulating down projection) -- does not
  // depend on the accumulator, so the four epilogue warps gather it while the
  // K loop runs when each holds at most kPre items.
  constexpr int kPre = 4;
  const bool has_addend = kDU || (kUp ? a.shared != nullptr : (MODE == kGemmDown && a.accumulate != 0));
  const bool pre = has_addend && n_items <= 128 * kPre;
  float4 pre_add[kPre];
  auto addend = [&](int item) -> float4 {
    const int tg = tok0 + t_begin + item / kQuads;
    const int n = m_tile * kOutRows + 4 * (item % kQuads);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (n >= a.M) return v;
    if (kUp) {  // slot order, from +0
      for (int s = 0; s < a.tp_s; ++s) {
        const uint2 sv = *reinterpret_cast<const uint2*>(a.shared + ((int64_t)s * a.n_tok + tg) * a.M + n);
        v.x = __fadd_rn(v.x, bf16_lo(sv.x)); v.y = __fadd_rn(v.y, bf16_hi(sv.x));
        v.z = __fadd_rn(v.z, bf16_lo(sv.y)); v.w = __fadd_rn(v.w, bf16_hi(sv.y));
      }
    } else {
      const uint2 ov = *reinterpret_cast<const uint2*>(a.out + (int64_t)tg * a.M + n);
      v = make_float4(bf16_lo(ov.x), bf16_hi(ov.x), bf16_lo(ov.y), bf16_hi(ov.y));
    }
    return v;
  };

  // Weight box of the CTA's i-th K block into stage st (two half-height boxes
  // for gate/up; down + up: W_down, or W_up on the up-projection's ranks).
  auto load_weights = [&](uint32_t st, uint32_t bar, int i, uint64_t policy) {
    if (MODE == kGemmGateUpSilu) {
      const int kx = (kb0 + i) * kBlockK;
      tma_load_2d(st, &map_w0, bar, kx, m_tile * (TM / 2), policy);
      tma_load_2d(st + kATile / 2, &map_w1, bar, kx, m_tile * (TM / 2), policy);
    } else {
      tma_load_2d(st, up_rank ? &map_w1 : &map_w0, bar, (kb0 + i) * kBlockK, m_tile * TM, policy);
    }
  };
  // Token box of the CTA's i-th K block (down + up: h, or y on the up-projection's ranks).
  auto load_tokens = [&](uint32_t st, uint32_t bar, int i, uint64_t policy) {
    tma_load_2d(st + kATile, up_rank ? &map_x1 : &map_x, bar, (kb0 + i) * kBlockK, tok0, policy);
  };

  // Fused mode, the four epilogue warps: y of the tile's tokens over this
  // CTA's K range into the operand tile, then release it to the MMA warp.
  auto form_y = [&]() {
    constexpr int kChunk = 256, kKbPerChunk = kChunk / kBlockK;
    const int c_first = kb0 / kKbPerChunk;
    const int ncc = nk > 0 ? (kb0 + nk - 1) / kKbPerChunk - c_first + 1 : 0;  // chunks the range touches
    const int n_work = n_valid * ncc;                                          // (token, chunk) items
    float* ss_sm = reinterpret_cast<float*>(base_ptr + (L.ss - base));
    float* inv_sm = reinterpret_cast<float*>(base_ptr + (L.inv - base));
    const int64_t slot_stride = (int64_t)a.n_tok * a.K;
    if (!a.inputs_before_wait) grid_dependency_wait();
    // gamma of the K range into shared memory, asynchronously (read in step 3)
    const int gvecs = nk * (kBlockK / 8);
    for (int v = threadIdx.x; v < gvecs; v += 128)
      if (kb0 * kBlockK + 8 * v < a.K) cp_async_16(L.gam + 16u * v, a.gamma + kb0 * kBlockK + 8 * v);
    asm volatile("cp.async.commit_group;" ::: "memory");
    // 1. x = bf16(slot sum) of whole chunks (a warp per token and chunk; lane
    //    l holds columns 8l..8l+7), the chunk's sum of squares, and x of the
    //    CTA's own K blocks into the operand tile.  The latent rows are staged
    //    with cp.async in the weight ring, which is still empty: each warp
    //    takes a quarter of it, so a batch of items is one trip to memory made
    //    before the CTA's weight stream starts.  Rows of padding tokens are left
    //    as they are: they only feed accumulator columns that are never read.
    const uint32_t quarter = (uint32_t)(stages * kStageBytes / 4) & ~511u;
    const int per_batch = max(1, (int)(quarter / (uint32_t)(a.tp * 512)));  // the host keeps this >= 1
    const uint32_t wstage = L.ring + (uint32_t)warp * quarter;
    const int my_items = warp < n_work ? (n_work - warp + 3) / 4 : 0;  // items warp + 4j
    for (int j0 = 0; j0 < my_items; j0 += per_batch) {
      const int nb = min(per_batch, my_items - j0);
      for (int j = 0; j < nb; ++j) {
        const int it = warp + 4 * (j0 + j);
        const int t = it / ncc, c = c_first + (it - t * ncc);
        const int col = c * kChunk + 8 * lane;
        if (col < a.K) {
          const uint16_t* src = a.latent + (int64_t)(tok0 + t) * a.K + col;
          for (int sl = 0; sl < a.tp; ++sl)
            cp_async_16(wstage + (uint32_t)(((j * a.tp + sl) * 32 + lane) * 16), src + (int64_t)sl * slot_stride);
        }
      }
      cp_async_wait_all();  // this lane's own copies (and gamma's)
      for (int j = 0; j < nb; ++j) {
        const int it = warp + 4 * (j0 + j);
        const int t = it / ncc, c = c_first + (it - t * ncc);
        const int col = c * kChunk + 8 * lane;
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.0f;
        if (col < a.K) {
          for (int sl = 0; sl < a.tp; ++sl) {  // slot order, FP32 from +0
            float f[8];
            unpack8(ld_shared_v4(wstage + (uint32_t)(((j * a.tp + sl) * 32 + lane) * 16)), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __fadd_rn(x[i], f[i]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = bf16_round(x[i]);
        }
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(x[i], x[i]));
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        if (lane == 0) ss_sm[t * a.chunks + c] = acc;
        const int kb = c * kKbPerChunk + (lane >> 3);
        if (kb >= kb0 && kb < kb0 + nk) {  // x is BF16-exact: the high half of each float is its BF16
          uint4 pk;
          pk.x = (__float_as_uint(x[0]) >> 16) | (__float_as_uint(x[1]) & 0xffff0000u);
          pk.y = (__float_as_uint(x[2]) >> 16) | (__float_as_uint(x[3]) & 0xffff0000u);
          pk.z = (__float_as_uint(x[4]) >> 16) | (__float_as_uint(x[5]) & 0xffff0000u);
          pk.w = (__float_as_uint(x[6]) >> 16) | (__float_as_uint(x[7]) & 0xffff0000u);
          st_shared_v4(L.yop + (uint32_t)((kb - kb0) * kBTileBytes) + sw128_offset(t, lane & 7), pk);
        }
      }
      __syncwarp();  // the batch's staging is read before the next batch overwrites it
    }
    cp_async_wait_all();  // gamma, where this thread had no latent batch
    // the ring is free for the weights (ordered before the async proxy's writes)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(L.latbar);
    MOE_TRACE_MARK(1);  // fused: latent rows read, x and chunk sums formed
    if (ksplit > 1) cluster_sync_all();  // chunk sums published (producer and MMA warps arrived at entry)
    else epilogue_bar();
    // 2. per token: the chunk sums in chunk order from +0, then 1/rms; chunk c
    //    is read from the CTA whose K range holds its first K block.
    for (int t = warp; t < n_valid; t += 4) {
      float v = 0.0f;
      if (lane < a.chunks) {
        const uint32_t owner = ksplit > 1 ? kblock_owner(kKbPerChunk * lane, kb_per, kb_rem) : 0u;
        const int idx = t * a.chunks + lane;
        v = owner == rank ? ss_sm[idx] : ld_cluster_f32(map_to_rank(L.ss + (uint32_t)(4 * idx), owner));
      }
      float ss = 0.0f;
      for (int c = 0; c < a.chunks; ++c) ss = __fadd_rn(ss, __shfl_sync(0xffffffffu, v, c));
      if (lane == 0) inv_sm[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, a.rcpK), a.eps)));
    }
    epilogue_bar();  // 1/rms and gamma (each thread waited for its copies) for every warp
    // 3. y = bf16((x * inv) * gamma), -0 made +0, in place.
    for (int it = warp; it < n_work; it += 4) {
      const int t = it / ncc, c = c_first + (it - t * ncc);
      const int kb = c * kKbPerChunk + (lane >> 3);
      const int col = c * kChunk + 8 * lane;
      if (kb < kb0 || kb >= kb0 + nk || col >= a.K) continue;  // outside the range, or zeros past K
      const uint32_t addr = L.yop + (uint32_t)((kb - kb0) * kBTileBytes) + sw128_offset(t, lane & 7);
      float x[8], g[8], yv[8];
      unpack8(ld_shared_v4(addr), x);
      unpack8(ld_shared_v4(L.gam + (uint32_t)(2 * (col - kb0 * kBlockK))), g);
      const float inv = inv_sm[t];
#pragma unroll
      for (int i = 0; i < 8; ++i) yv[i] = __fmul_rn(__fmul_rn(x[i], inv), __fadd_rn(g[i], 0.0f));
      st_shared_v4(addr, make_uint4(pack_bf16x2_pz(yv[0], yv[1]), pack_bf16x2_pz(yv[2], yv[3]),
                                    pack_bf16x2_pz(yv[4], yv[5]), pack_bf16x2_pz(yv[6], yv[7])));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
    mbar_arrive(L.ybar);
    MOE_TRACE_MARK(2);  // fused: y in the operand tile
  };

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();     // token tiles: re-read by every M tile
      const uint64_t stream = policy_evict_first();  // weights: read once
      int issued = 0;
      bool ok = true;
      // Inside the library's own kernel chains the weights never depend on the
      // preceding kernel, so the first ring's worth is requested before waiting
      // for it; the first kernel of a call waits first.  With the inputs-ready
      // promise (gate/up: x complete before the preceding kernel ends) the
      // token tiles are read without waiting as well, and only the epilogue
      // waits, before it writes.
      const int pre = min(nk_all, stages);
      const bool tokens_ready = !kFused && a.inputs_before_wait;
      if (!a.weights_before_wait) grid_dependency_wait();
      if (kFused && !mbar_wait(L.latbar, 0)) {  // the ring holds the latent rows until y's inputs are read
        raise_error(kErrWaitFull);
        *abort_ptr = 1;
      }
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(L.full + 8 * i, kStageBytes);
        load_weights(L.ring + i * kStageBytes, L.full + 8 * i, i, stream);
      }
      if (!kFused) {  // the token tiles are the preceding kernel's output, unless promised ready
        if (a.weights_before_wait && !tokens_ready) grid_dependency_wait();
        for (int i = 0; i < pre; ++i) load_tokens(L.ring + i * kStageBytes, L.full + 8 * i, i, keep);
      }
      issued = pre;
      for (int i = pre; i < nk_all; ++i) {
        const int s = i % stages;
        const uint32_t round = (uint32_t)(i / stages);
        if (!mbar_wait(L.empty + 8 * s, (round - 1u) & 1u, kWaitLimitNs, abort_ptr)) {
          if (!*abort_ptr) raise_error(kErrWaitEmpty);  // (else the MMA issuer aborted: stop issuing)
          *abort_ptr = 1;
          ok = false;
          break;
        }
        const uint32_t st = L.ring + s * kStageBytes;
        const uint32_t bar = L.full + 8 * s;
        mbar_expect_tx(bar, kStageBytes);
        load_weights(st, bar, i, stream);
        if (!kFused) load_tokens(st, bar, i, keep);
        ++issued;
      }
      if (!ok) {  // let the copies already in flight land before the CTA's memory goes away
        for (int i = max(0, issued - stages); i < issued; ++i)
          if (!mbar_wait(L.full + 8 * (i % stages), (uint32_t)(i / stages) & 1u)) raise_error(kErrWaitDrain);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (!kFused && !a.inputs_before_wait) grid_dependency_wait();  // fused: reads shared memory only
    if (lane == 0) {
      bool ok = true;
      if (kFused) {  // y is in shared memory (and visible to the tensor cores)
        ok = mbar_wait(L.ybar, 0);
        if (!ok) {
          raise_error(kErrWaitFull);
          *abort_ptr = 1;
        }
        tc_fence_after();
      }
      // the operand-stage wait (its limit can be shortened for failure-detection tests)
      const unsigned long long stage_limit = a.stage_wait_ns ? a.stage_wait_ns : kWaitLimitNs;
      for (int i = 0; ok && i < nk_all; ++i) {
        const int s = i % stages;
        if (!mbar_wait(L.full + 8 * s, (uint32_t)(i / stages) & 1u, stage_limit)) {
          raise_error(kErrWaitFull);
          *abort_ptr = 1;
          break;
        }
        tc_fence_after();
        const uint32_t st = L.ring + s * kStageBytes;
        const uint64_t adesc = smem_desc_sw128(st);
        const uint64_t bdesc = smem_desc_sw128(kFused ? L.yop + (uint32_t)(i * kBTileBytes) : st + kATile);
#pragma unroll
        for (int kk = 0; kk < kBlockK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled row
#pragma unroll
          for (int acc = 0; acc < kNumAcc; ++acc)  // accumulator acc: weight rows acc*128 .. +127
            mma_bf16(tmem + (uint32_t)(acc * N), adesc + (uint64_t)(acc * (kMmaM * 128 >> 4)) + 2 * kk,
                     bdesc + 2 * kk, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(L.empty + 8 * s);
      }
      if (nk_all > 0) mma_commit(L.accum);  // also on abort: completes once the issued MMAs are done
      else mbar_arrive(L.accum);             // an empty K range (the epilogue stages zeros)
    }
    __syncwarp();
  } else {
    // ---------------- (fused: y) accumulator -> FP32 staging tile [N tokens][TM rows] ----------------
    if (kFused) {
      form_y();
      if (a.inputs_before_wait) grid_dependency_wait();  // before the shared partials and any store
    } else {
      grid_dependency_wait();
    }
    if (pre) {
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const int item = threadIdx.x + 128 * j;
        if (item < n_items) pre_add[j] = addend(item);
      }
    }
    if (kFused && a.y != nullptr && m_tile == 0) {  // y of the CTA's K range, from the operand tile
      const int vecs = nk * (kBlockK / 8);
      for (int e = threadIdx.x; e < n_valid * vecs; e += 128) {
        const int t = e / vecs, v = e - t * vecs;
        const int col = kb0 * kBlockK + 8 * v;
        if (col < a.K)
          st_v4(a.y + (int64_t)(tok0 + t) * a.K + col,
                ld_shared_v4(L.yop + (uint32_t)((v >> 3) * kBTileBytes) + sw128_offset(t, v & 7)));
      }
    }
    const bool got = mbar_wait(L.accum, 0);
    MOE_TRACE_MARK(0);  // accumulator complete
    if (!got) {
      if (lane == 0) raise_error(kErrWaitAccum);
      *abort_ptr = 1;
    }
    tc_fence_after();
    const bool holds_row = kMmaM == 128 || lane < 16;
    const int row = kMmaM == 128 ? warp * 32 + lane : warp * 16 + lane;
    float* stage = reinterpret_cast<float*>(base_ptr);
    for (int acc = 0; acc < kNumAcc; ++acc) {
      const int r = acc * kMmaM + row;
      if (got && nk > 0) {
#pragma unroll 1
        for (int c = 0; c < N; c += 16) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * N + c), v);
          if (holds_row) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stage[(c + i) * TM + r] = v[i];
          }
        }
      } else if (got && holds_row) {  // an empty K range contributes zeros
        for (int c = 0; c < N; ++c) stage[c * TM + r] = 0.0f;
      }
    }
    tc_fence_before();
  }
  if (kFused && ksplit > 1 && warp >= 4) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  __syncthreads();
  const bool aborted = *abort_ptr != 0;
  if (!kFused) MOE_TRACE_MARK(1);      // partial tile staged
  if (ksplit > 1) cluster_sync_all();  // every CTA's partial tile is staged
  if (!kFused) MOE_TRACE_MARK(2);

  // ---------------- rank-order reduction over the cluster + fused epilogue ----------------
  auto finish_item = [&](int item, float4 add) {
    const int t = t_begin + item / kQuads;
    const int q = item % kQuads;
    const int tg = tok0 + t;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc2 = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t off = base + (uint32_t)((t * TM + 4 * q) * 4);
    // down + up: d is the sum over the down projection's ranks, u over the
    // up-projection's, each in rank order
    for (uint32_t p = 0; p < ksplit; ++p) {
      const float4 v = ld_cluster_v4(map_to_rank(off, p));
      if (kDU && (int)p >= n_down) {
        acc2.x = __fadd_rn(acc2.x, v.x); acc2.y = __fadd_rn(acc2.y, v.y);
        acc2.z = __fadd_rn(acc2.z, v.z); acc2.w = __fadd_rn(acc2.w, v.w);
      } else {
        acc.x = __fadd_rn(acc.x, v.x); acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z); acc.w = __fadd_rn(acc.w, v.w);
      }
      if (MODE == kGemmGateUpSilu) {  // the up rows of the tile
        const float4 u = ld_cluster_v4(map_to_rank(off + (TM / 2) * 4, p));
        acc2.x = __fadd_rn(acc2.x, u.x); acc2.y = __fadd_rn(acc2.y, u.y);
        acc2.z = __fadd_rn(acc2.z, u.z); acc2.w = __fadd_rn(acc2.w, u.w);
      }
    }
    float r[4] = {acc.x, acc.y, acc.z, acc.w};
    if (MODE == kGemmGateUpSilu) {
      const int j = m_tile * kOutRows + 4 * q;
      if (j >= a.M) return;
      const float u[4] = {acc2.x, acc2.y, acc2.z, acc2.w};
      uint32_t hb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) hb[e] = bf16_bits_pz(silu(bf16_round(r[e])) * bf16_round(u[e]));
      uint2 pk = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
      *reinterpret_cast<uint2*>(a.out + (int64_t)tg * a.M + j) = pk;
    } else {
      const int n = m_tile * kOutRows + 4 * q;
      if (n >= a.M) return;
      const float ad[4] = {add.x, add.y, add.z, add.w};
      if (kDU) {  // d = acc rounded to BF16 joins the shared partials as their last slot; u = acc2
        uint32_t db[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) db[e] = bf16_bits_pz(r[e]);
        if (a.d_out != nullptr)
          *reinterpret_cast<uint2*>(a.d_out + (int64_t)tg * a.M + n) =
              make_uint2(db[0] | (db[1] << 16), db[2] | (db[3] << 16));
        const float u[4] = {acc2.x, acc2.y, acc2.z, acc2.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = __fadd_rn(u[e], __fadd_rn(ad[e], __uint_as_float(db[e] << 16)));
      } else if (kUp) {  // out = bf16(acc + slot sum of the shared partials)
        if (has_addend) {
#pragma unroll
          for (int e = 0; e < 4; ++e) r[e] = __fadd_rn(r[e], ad[e]);
        }
      } else if (has_addend) {  // down projection added into out: bf16(out + bf16(d))
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = __fadd_rn(ad[e], __uint_as_float(bf16_bits_pz(r[e]) << 16));
      }
      uint2 pk = make_uint2(pack_bf16x2_pz(r[0], r[1]), pack_bf16x2_pz(r[2], r[3]));
      *reinterpret_cast<uint2*>(a.out + (int64_t)tg * a.M + n) = pk;
    }
  };
  if (!aborted) {
    if (pre) {  // the items whose addends the epilogue warps gathered
      if (threadIdx.x < 128) {
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
          const int item = threadIdx.x + 128 * j;
          if (item < n_items) finish_item(item, pre_add[j]);
        }
      }
    } else {
      for (int item = threadIdx.x; item < n_items; item += kThreads)
        finish_item(item, has_addend ? addend(item) : make_float4(0.f, 0.f, 0.f, 0.f));
    }
  }
  MOE_TRACE_MARK(3);                   // reduction and epilogue stores done
  if (ksplit > 1) cluster_sync_all();  // peers are done reading this CTA's staging tile
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- persistent down projection ----------------------------------------------------
//
//   out[t, n] = accumulate ? bf16(out[t, n] + bf16(d)) : bf16(d),   d = sum_k W[n, k] * h[t, k]
//
// The Kimi-K3 shared expert page's down projection (SharedDown): a persistent
// grid whose CTAs walk output tiles of 128 weight rows x N tokens, tile
// blockIdx.x, + gridDim.x, ..., each over the whole K range (no K split, no
// cluster), with two tensor-memory accumulators that alternate between a
// CTA's consecutive tiles: the MMA issuer fills one while the epilogue warps
// drain the other, so a tile's epilogue overlaps the next tile's weight
// stream.  Warp 4 streams the weight and token tiles of all the CTA's tiles
// through one ring, warp 5 issues the MMAs, warps 0-3 read an accumulator (one
// TMEM lane = one weight row per thread) and write out directly: per token a
// warp's 32 rows are 64 contiguous bytes.  Waits are bounded as in
// decode_gemm_kernel; after an abort no copy or MMA is issued, the epilogue
// skips its stores, and the CTA waits for what it started before freeing its
// tensor memory.
template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    persistent_down_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                           const GemmArgs a, const int stages) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kATile = 128 * kBlockK * 2;
  constexpr int kStageBytes = kATile + N * kBlockK * 2;
  constexpr uint32_t kTmemCols = 2 * N < 32 ? 32 : 2 * N;  // two accumulators of N columns
  constexpr uint32_t kIdesc = idesc_bf16(128, N);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (a.M + 127) / 128;
  const int n_items = m_tiles * ((a.n_tok + N - 1) / N);
  const int my_items =
      (int)blockIdx.x < n_items ? (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int total = my_items * a.kblocks;  // ring stages this CTA streams

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t ring = base;
  const uint32_t full = ring + (uint32_t)(stages * kStageBytes);  // [stages]
  const uint32_t empty = full + 8u * stages;                       // [stages]
  const uint32_t acc_full = empty + 8u * stages;                   // [2]: accumulator holds a finished tile
  const uint32_t acc_empty = acc_full + 16;                        // [2]: the epilogue has read it
  const uint32_t mma_done = acc_empty + 16;                        // the issuer's MMAs have all completed
  const uint32_t tmem_slot = mma_done + 8;
  const uint32_t abort_off = tmem_slot + 4;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  volatile uint32_t* abort_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (abort_off - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(acc_full + 8 * k, 1);
      mbar_init(acc_empty + 8 * k, 4);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    *abort_ptr = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w);
    prefetch_map(&map_h);
  }
  if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  launch_dependents();

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();     // token tiles: re-read by every weight tile
      const uint64_t stream = policy_evict_first();  // weights: read once
      // stage g of the CTA: its tile g / kblocks, K block g % kblocks
      auto load = [&](int g, bool weights, bool tokens) {
        const int j = g / a.kblocks, kb = g - j * a.kblocks;
        const int item = (int)blockIdx.x + j * (int)gridDim.x;
        const uint32_t st = ring + (uint32_t)((g % stages) * kStageBytes), bar = full + 8u * (g % stages);
        if (weights) tma_load_2d(st, &map_w, bar, kb * kBlockK, (item % m_tiles) * 128, stream);
        if (tokens) tma_load_2d(st + kATile, &map_h, bar, kb * kBlockK, (item / m_tiles) * N, keep);
      };
      const int pre = min(total, stages);
      if (!a.weights_before_wait) grid_dependency_wait();
      for (int g = 0; g < pre; ++g) {
        mbar_expect_tx(full + 8u * g, kStageBytes);
        load(g, true, false);
      }
      if (a.weights_before_wait) grid_dependency_wait();  // h is the preceding kernel's output
      for (int g = 0; g < pre; ++g) load(g, false, true);
      int issued = pre;
      bool ok = true;
      for (int g = pre; g < total; ++g) {
        const int s = g % stages;
        if (!mbar_wait(empty + 8u * s, (uint32_t)(g / stages - 1) & 1u, kWaitLimitNs, abort_ptr)) {
          if (!*abort_ptr) raise_error(kErrWaitEmpty);  // (else the MMA issuer aborted: stop issuing)
          *abort_ptr = 1;
          ok = false;
          break;
        }
        mbar_expect_tx(full + 8u * s, kStageBytes);
        load(g, true, true);
        ++issued;
      }
      if (!ok) {  // let the copies already in flight land before the CTA's memory goes away
        for (int g = max(0, issued - stages); g < issued; ++g)
          if (!mbar_wait(full + 8u * (g % stages), (uint32_t)(g / stages) & 1u)) raise_error(kErrWaitDrain);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer: accumulator j % 2 for the CTA's tile j ----------------
    if (lane == 0) {
      const unsigned long long stage_limit = a.stage_wait_ns ? a.stage_wait_ns : kWaitLimitNs;
      bool ok = true;
      int g = 0;
      for (int j = 0; ok && j < my_items; ++j) {
        const uint32_t acc = (uint32_t)(j & 1);
        // the epilogue has read this accumulator's previous tile (j - 2)
        if (j >= 2 && !mbar_wait(acc_empty + 8u * acc, (uint32_t)(j / 2 - 1) & 1u, kWaitLimitNs, abort_ptr)) {
          if (!*abort_ptr) raise_error(kErrWaitAccum);
          *abort_ptr = 1;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < a.kblocks; ++kb, ++g) {
          const int s = g % stages;
          if (!mbar_wait(full + 8u * s, (uint32_t)(g / stages) & 1u, stage_limit)) {
            raise_error(kErrWaitFull);
            *abort_ptr = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = ring + (uint32_t)(s * kStageBytes);
          const uint64_t adesc = smem_desc_sw128(st), bdesc = smem_desc_sw128(st + kATile);
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled row
            mma_bf16(tmem + acc * (uint32_t)N, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(empty + 8u * s);
        }
        mma_commit(acc_full + 8u * acc);  // also on abort: the epilogue then skips the tile
      }
      mma_commit(mma_done);  // completes once every MMA issued above has
      if (!mbar_wait(mma_done, 0)) raise_error(kErrWaitAccum);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps ----------------
    grid_dependency_wait();  // out may still be read (or, accumulating, written) by the preceding kernel
    const int row = warp * 32 + lane;
    for (int j = 0; j < my_items; ++j) {
      const uint32_t acc = (uint32_t)(j & 1);
      const int item = (int)blockIdx.x + j * (int)gridDim.x;
      const int n = (item % m_tiles) * 128 + row;
      const int tok0 = (item / m_tiles) * N;
      // lane 0 waits and the warp follows its outcome, so the warp stays converged
      // for the tcgen05.ld below (an abort seen by some lanes only would split it)
      bool got = true;
      if (lane == 0) {
        got = mbar_wait(acc_full + 8u * acc, (uint32_t)(j / 2) & 1u, kWaitLimitNs, abort_ptr);
        if (!got) {
          if (!*abort_ptr) raise_error(kErrWaitAccum);
          *abort_ptr = 1;
        }
      }
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) break;
      __syncwarp();
      tc_fence_after();
      const bool skip = __shfl_sync(0xffffffffu, *abort_ptr != 0 ? 1 : 0, 0) != 0;
      if (!skip) {
#pragma unroll 1
        for (int c = 0; c < N; c += 16) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + acc * (uint32_t)N + (uint32_t)c, v);
          if (n < a.M) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = tok0 + c + i;
              if (t < a.n_tok) {
                uint16_t* o = a.out + (int64_t)t * a.M + n;
                const uint32_t db = bf16_bits_pz(v[i]);  // d pushed as BF16, -0 made +0
                *o = (uint16_t)(a.accumulate ? bf16_bits_pz(__fadd_rn(__uint_as_float((uint32_t)*o << 16),
                                                                      __uint_as_float(db << 16)))
                                             : db);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + 8u * acc);
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Failure-detection self-test: one thread waits, with the kernels' bounded
// wait, on an mbarrier that nothing arrives at; after limit_ns it gives up,
// raises kErrWaitFull and returns, so the host sees the error and the context
// stays usable.
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait(b, 0, limit_ns)) raise_error(kErrWaitFull);
}

#ifdef MOE_TAIL_TRACE
cudaError_t trace_attach_gemm(void* buf, unsigned cap) { return trace_attach_tu(buf, cap); }
unsigned trace_count_gemm() { return trace_count_tu(); }
#endif

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

// ---- host side ---------------------------------------------------------------------

static int stage_bytes(int tm, int n_tile) { return tm * kBlockK * 2 + n_tile * kBlockK * 2; }

// Plan override for tuning (tm, ksplit, stages; read once from the environment).
static bool plan_override(int mode, GemmPlan& p) {
  const int slot = mode == kGemmDownUp ? 3 : mode;
  if (slot < 0 || slot > 3) return false;
  const int* v = tuning().gemm_plan[slot];
  if (v[0] == 0) return false;
  p.tm = v[0];
  p.ksplit = v[1];
  p.stages = v[2];
  return true;
}

GemmPlan plan_gemm(int mode, int M, int K, int b, int sms, int K2) {
  GemmPlan p;
  p.n_tile = b <= 16 ? 16 : b <= 32 ? 32 : b <= 64 ? 64 : 128;
  const int tok_tiles = (b + p.n_tile - 1) / p.n_tile;
  const int kblocks = (K + kBlockK - 1) / kBlockK;
  const int kblocks2 = (K2 + kBlockK - 1) / kBlockK;  // down + up: the up-projection's K blocks
  p.tm = 128;
  p.stages = 0;
  const bool forced = plan_override(mode, p);
  if (mode == kGemmDownUp) p.tm = 128;  // the only tile height this mode is built for
  const int rows_per_tile = mode == kGemmGateUpSilu ? p.tm / 2 : p.tm;
  p.m_tiles = (M + rows_per_tile - 1) / rows_per_tile;
  // The up-projection of at most 16 tokens (18 KB stages) runs three CTAs per
  // SM with 3-stage rings: the latent tail alone at b = 16 with both promises
  // 11.9 -> 11.3 us, at b = 1 10.7 -> 10.2, b = 8 11.5 -> 10.9; without them
  // the same at b = 16, faster at b = 1 and 8.
  const bool small_up = mode == kGemmUpShared && p.n_tile <= 16;
  // The gate/up projection takes a 4-way K split (384 CTAs at I = 6144, about
  // 2.5 per SM) with rings of up to 3 stages and 72 KB.  Alone it is 4-6 %
  // faster than the 3-way split at b = 40 ... 128 (b = 64: 32.5 -> 31.2 us,
  // b = 128: 38.5 -> 36.1); in the decode step b = 64 59.8 -> 56.7 us, b = 40
  // 63.6 -> 60.5, b = 96 71.6 -> 69.2, b = 128 80.2 -> 79.2, b = 32 59.0 ->
  // 55.1, b = 8 52.3 -> 51.5, b = 1 50.9 -> 50.5 (b = 48 and 56 +1.7 and +1.4;
  // at b = 128 a 3-stage, 96 KB ring leaves too few CTAs per SM: 84.7 us).
  const bool small_gateup = mode == kGemmGateUpSilu;
  if (!forced) {  // K split over a cluster: about two CTAs per SM
    // Above 32 tokens the down projection takes about 1.5 per SM (K split 4
    // at H = 7168; with its 96 KB rings the shared expert alone at b = 64
    // measured 49.4 us against 51.0 / 52.6 with a 5- / 3-way split, at b = 128
    // 59.3 against 63.8 / 63.4).  Small batches keep two (b = 1 alone: 45.9
    // vs 48.5 us for the shared expert).
    // The down + up kernel above 64 tokens (128-token tiles, 2-stage rings) takes
    // a 6-way split (about 2.2 CTAs per SM): the decode step at b = 128 84.4 ->
    // 81.7 us (5-way; 7-way 83.1, 8-way 88.8, 3-stage rings 91-93).
    const int slots = (mode == kGemmDown && b > 32) ? 3 * sms / 2 : small_up ? 3 * sms
                      : small_gateup ? 8 * sms / 3 : (mode == kGemmDownUp && b > 64) ? 9 * sms / 4 : 2 * sms;
    int ks = slots / std::max(1, p.m_tiles * tok_tiles);
    p.ksplit = std::max(1, std::min(ks, 8));
  }
  if (mode == kGemmDownUp) {  // at least one rank for each projection, and a K block for every rank
    p.ksplit = std::max(2, std::min(p.ksplit, 8));
    for (int n; p.ksplit > 2 && ((n = downup_down_ranks(p.ksplit, kblocks, kblocks2)) > kblocks ||
                                 p.ksplit - n > kblocks2);)
      --p.ksplit;
  } else {
    p.ksplit = std::min(p.ksplit, kblocks);
  }
  const int sb = stage_bytes(p.tm, p.n_tile);
  // Ring budget 72 KB at TM <= 128 (3 stages at b = 64): two GEMM CTAs then
  // leave room on their SM for one finalize CTA of a concurrent stream (up to
  // ~80 KB of shared memory), which measured faster in the composed decode
  // step than deeper rings that keep the finalize kernels waiting for an SM.
  // The up-projection ends the step, after the finalize kernels, and takes a
  // 96 KB ring (4 stages at b = 64: 71.4 -> 70.3 us per step with the down
  // projection's split above).
  // The down + up kernel takes 72 KB as well: in a decode step it runs while
  // the expert-TP finalize still holds SMs, and two of its CTAs beside one
  // finalize CTA fit an SM only at this size (b = 64: 63.3 vs 66.9 us per
  // step with 96 KB, whose second CTA waits for the finalize to end).  The
  // down projection on its own (moe_shared_down, moe_shared_expert; the
  // decode step streams it in the down + up kernel) takes 96 KB: the shared
  // expert alone at b = 64 52.9 -> 49.4 us, b = 128 65.8 -> 59.3, b = 1..32
  // 2-3 % faster.
  const int budget = p.tm == 256 ? 200 * 1024 : small_up ? 3 * sb : small_gateup ? std::min(3 * sb, 72 * 1024)
                     : ((mode == kGemmUpShared || mode == kGemmDown) ? 96 * 1024 : 72 * 1024);
  if (p.stages == 0) p.stages = std::max(2, std::min(kMaxStages, budget / sb));
  int per_cta = (kblocks + p.ksplit - 1) / p.ksplit;  // the longest K range of a CTA
  if (mode == kGemmDownUp) {
    const int n = downup_down_ranks(p.ksplit, kblocks, kblocks2);
    per_cta = std::max((kblocks + n - 1) / n, (kblocks2 + p.ksplit - n - 1) / (p.ksplit - n));
  }
  p.stages = std::min(p.stages, std::max(2, per_cta));
  // the FP32 staging tile reuses the ring
  while (p.stages * sb < p.n_tile * p.tm * 4) ++p.stages;
  return p;
}

// Fused latent tail: everything but the weight ring (alignment slack, the y
// operand of the longest K range, chunk sums, 1/rms, barriers and slots).
static size_t fused_fixed_bytes(int n_tile, int kblocks, int ksplit, int chunks) {
  const size_t per_cta = (size_t)((kblocks + ksplit - 1) / ksplit);
  return 1024 + per_cta * n_tile * kBlockK * 2 + 4 * (size_t)n_tile * chunks + 4 * (size_t)n_tile +
         per_cta * kBlockK * 2 + 8 + 8 + 8 + 8 + 8 + 64;
}

static size_t smem_bytes(const GemmPlan& p, int mode, const GemmArgs& a) {
  if (mode == kGemmLatentUp)
    return fused_fixed_bytes(p.n_tile, a.kblocks, p.ksplit, a.chunks) +
           (size_t)p.stages * (p.tm * kBlockK * 2 + 16);
  return 1024 + (size_t)p.stages * stage_bytes(p.tm, p.n_tile) + 16 * (size_t)p.stages + 8 + 8 + 64;
}

// Two fused CTAs per SM: 2 x (this + the 1 KB the hardware keeps per CTA)
// within an SM's 228 KB of shared memory.
constexpr size_t kFusedSmemCap = 112 * 1024;

bool plan_latent_fused(int H, int L, int b, int tp, int sms, GemmPlan* plan) {
  const int chunks = (L + 255) / 256;
  if (b < 1 || b > 32 || chunks > 32 || tp < 1) return false;
  GemmPlan p = plan_gemm(kGemmUpShared, H, L, b, sms, 0);  // the two-kernel tiles and K split
  if (p.tm != 128 || p.n_tile > 32) return false;
  const int kblocks = (L + kBlockK - 1) / kBlockK;
  const size_t fixed = fused_fixed_bytes(p.n_tile, kblocks, p.ksplit, chunks);
  const size_t a_tile = (size_t)p.tm * kBlockK * 2, per_stage = a_tile + 16;
  if (fixed + 2 * per_stage > kFusedSmemCap) return false;
  // as many stages as fit: the ring also stages the latent rows (a quarter per
  // epilogue warp, which must hold one item's tp rows of 512 bytes)
  p.stages = (int)std::min<size_t>((kFusedSmemCap - fixed) / per_stage, (size_t)kMaxStages);
  if ((size_t)tp * 512 > (p.stages * a_tile / 4 & ~(size_t)511)) return false;
  // the FP32 staging tile [n_tile][tm] reuses the ring
  if ((size_t)p.stages * a_tile < (size_t)p.n_tile * p.tm * 4) return false;
  *plan = p;
  return true;
}

template <int MODE, int N, int TM>
static cudaError_t launch_t(const GemmPlan& p, const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& x,
                            const CUtensorMap& x1, const GemmArgs& a, bool pdl, cudaStream_t stream) {
  auto kernel = decode_gemm_kernel<MODE, N, TM>;
  const size_t smem = smem_bytes(p, MODE, a);
  // Raise the kernel's shared-memory limit once per device (not per call, so
  // that a captured stream sees only launches).
  const cudaError_t e = ensure_smem_limit((const void*)kernel, 220 * 1024);
  if (e != cudaSuccess) return e;
  if (smem > 220 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ksplit, p.m_tiles, (a.n_tok + N - 1) / N);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  ++n;
  if (p.ksplit > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = p.ksplit;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, w0, w1, x, x1, a, p.stages);
}

template <int MODE, int TM>
static cudaError_t launch_n(const GemmPlan& p, const CUtensorMap& w0, const CUtensorMap& w1,
                            const CUtensorMap& x, const CUtensorMap& x1, const GemmArgs& a, bool pdl,
                            cudaStream_t stream) {
  switch (p.n_tile) {
    case 16: return launch_t<MODE, 16, TM>(p, w0, w1, x, x1, a, pdl, stream);
    case 32: return launch_t<MODE, 32, TM>(p, w0, w1, x, x1, a, pdl, stream);
    case 64: return launch_t<MODE, 64, TM>(p, w0, w1, x, x1, a, pdl, stream);
    case 128: return launch_t<MODE, 128, TM>(p, w0, w1, x, x1, a, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
static cudaError_t launch_mode(const GemmPlan& p, const CUtensorMap& w0, const CUtensorMap& w1,
                               const CUtensorMap& x, const GemmArgs& a, bool pdl, cudaStream_t stream) {
  if (p.tm == 256) return launch_n<MODE, 256>(p, w0, w1, x, x, a, pdl, stream);
  return p.tm == 128 ? launch_n<MODE, 128>(p, w0, w1, x, x, a, pdl, stream)
                     : launch_n<MODE, 64>(p, w0, w1, x, x, a, pdl, stream);
}

cudaError_t launch_decode_gemm(int mode, const GemmPlan& p, const CUtensorMap& w0, const CUtensorMap& w1,
                               const CUtensorMap& x, const GemmArgs& args, bool pdl, cudaStream_t stream,
                               const CUtensorMap* x1) {
  GemmArgs a = args;
  a.stage_wait_ns = stage_wait_limit_ns();
  switch (mode) {
    case kGemmUpShared: return launch_mode<kGemmUpShared>(p, w0, w1, x, a, pdl, stream);
    case kGemmGateUpSilu: return launch_mode<kGemmGateUpSilu>(p, w0, w1, x, a, pdl, stream);
    case kGemmDown: return launch_mode<kGemmDown>(p, w0, w1, x, a, pdl, stream);
    case kGemmLatentUp:  // built for the small batches plan_latent_fused admits
      if (p.tm != 128 || a.chunks < 1 || a.chunks > 32) return cudaErrorInvalidValue;
      if (p.n_tile == 16) return launch_t<kGemmLatentUp, 16, 128>(p, w0, w1, x, x, a, pdl, stream);
      if (p.n_tile == 32) return launch_t<kGemmLatentUp, 32, 128>(p, w0, w1, x, x, a, pdl, stream);
      return cudaErrorInvalidValue;
    case kGemmDownUp:  // tm = 128 only, a rank for each projection; x1 is the up-projection's token map (y)
      if (p.tm != 128 || p.ksplit < 2 || p.ksplit > 8 || x1 == nullptr || a.kblocks < 1 || a.kblocks2 < 1)
        return cudaErrorInvalidValue;
      return launch_n<kGemmDownUp, 128>(p, w0, w1, x, *x1, a, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Ring of the persistent down projection: one CTA per SM with a deep ring
// (about 192 KB, as the page's SharedDown budget), at most kMaxStages stages.
static int persistent_stages(int n_tile) {
  return std::max(2, std::min(kMaxStages, (192 * 1024) / stage_bytes(128, n_tile)));
}

template <int N>
static cudaError_t launch_persistent_t(const CUtensorMap& w, const CUtensorMap& h, const GemmArgs& a, int ctas,
                                       bool pdl, cudaStream_t stream) {
  auto kernel = persistent_down_kernel<N>;
  const int stages = persistent_stages(N);
  const size_t smem = 1024 + (size_t)stages * stage_bytes(128, N) + 16 * (size_t)stages + 16 + 16 + 8 + 8 + 64;
  const cudaError_t e = ensure_smem_limit((const void*)kernel, 220 * 1024);
  if (e != cudaSuccess) return e;
  if (smem > 220 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, w, h, a, stages);
}

cudaError_t launch_persistent_down(const CUtensorMap& w, const CUtensorMap& h, const GemmArgs& args, int n_tile,
                                   int ctas, bool pdl, cudaStream_t stream) {
  GemmArgs a = args;
  a.stage_wait_ns = stage_wait_limit_ns();
  if (ctas < 1 || a.kblocks < 1) return cudaErrorInvalidValue;
  switch (n_tile) {
    case 16: return launch_persistent_t<16>(w, h, a, ctas, pdl, stream);
    case 32: return launch_persistent_t<32>(w, h, a, ctas, pdl, stream);
    case 64: return launch_persistent_t<64>(w, h, a, ctas, pdl, stream);
    case 128: return launch_persistent_t<128>(w, h, a, ctas, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moetail
