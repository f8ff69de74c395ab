/*
 * moe_tail_floor.h -- latency floors of a finalize-shaped call (measurement
 * only; no counterpart on the pages).
 *
 * libmoetail_floor.so (moe_decode_tail_gb300.build, floor=True) holds three
 * kernels that do only the memory traffic of a finalize call, launched the
 * way the finalize kernels are (programmatic dependent launch: each waits for
 * the stream's preceding kernel, then lets its own dependents be scheduled;
 * thread-block clusters of `cluster` CTAs along x).  Timed back to back in a
 * CUDA graph, they give the time below which a finalize call of the same grid
 * cannot go:
 *   - moe_tail_floor_empty: the launch and the dependency wait alone;
 *   - moe_tail_floor_read:  one trip to memory for `bytes` bytes, every thread
 *     loading its share (16-byte asynchronous copies into shared memory, up
 *     to 16 per thread, all issued before any is waited for);
 *   - moe_tail_floor_gather: two dependent trips -- a token's nk route indices,
 *     then the indexed rows of the CTA's column band, 16 rows in flight per
 *     thread (asynchronous copies as above) -- the access pattern of EP and
 *     expert-TP finalize without their arithmetic or cluster exchange.
 * Each writes one 32-bit word per CTA into sink (grid_x * grid_y words), so
 * that no load is dead.  Pointers are device pointers, 16-byte aligned (idx:
 * 4-byte); stream is a cudaStream_t.  Returns 0, 1 for refused arguments
 * (non-positive sizes, threads not a multiple of 32 or above 768, cluster
 * not dividing grid_x or above 8, a null or misaligned pointer), 2 for a CUDA
 * launch error.
 */
#ifndef MOE_TAIL_FLOOR_H
#define MOE_TAIL_FLOOR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int moe_tail_floor_empty(int grid_x, int grid_y, int threads, int cluster, void* stream);

/* src: `bytes` bytes (a multiple of 16), read once over the grid. */
int moe_tail_floor_read(const void* src, size_t bytes, int grid_x, int grid_y, int threads, int cluster,
                        uint32_t* sink, void* stream);

/* idx: int32 [grid_y][nk], each in [0, n_rows); rows: [n_rows][row_bytes]
 * (row_bytes = grid_x * threads * 16: CTA x reads 16 bytes per thread of its
 * band of every indexed row). */
int moe_tail_floor_gather(const int32_t* idx, int nk, const void* rows, int64_t n_rows, int grid_x, int grid_y,
                          int threads, int cluster, uint32_t* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TAIL_FLOOR_H */
