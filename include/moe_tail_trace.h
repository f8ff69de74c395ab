/*
 * moe_tail_trace.h -- per-CTA timeline trace of the MoE decode tail kernels.
 *
 * Only libraries built with MOE_TAIL_TRACE (moe_decode_tail_gb300.build
 * with trace=True: _build/libmoetail_trace.so) export these calls; the normal
 * library has no trace code at all.  Thread 0 of every CTA of every kernel
 * writes one record when the CTA exits:
 *
 *   struct { uint64 t0, mark[4], t1, ids, pad; }      (64 bytes, %globaltimer ns)
 *   ids = kernel id << 48 | SM id << 32 | linear CTA index
 *   kernel ids: 10 + mode route-parallel finalize (0 EP, 1 expert-TP, 2 latent norm),
 *               20 staged expert-TP finalize, 40 EP finalize (routes in registers),
 *               30 + mode decode GEMM (0 up-projection, 1 gate/up, 2 down,
 *               3 latent tail in one kernel, 4 down projection with the up-projection)
 *   GEMM marks: 0 accumulator complete, 1 partial tile staged, 2 first cluster
 *               barrier passed, 3 reduction and epilogue stores done (0 when the
 *               K range is not split); finalize kernels leave the marks at 0.
 */
#ifndef MOE_TAIL_TRACE_H
#define MOE_TAIL_TRACE_H

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_TAIL_TRACE_RECORD_BYTES 64

/* Attach a device buffer of `capacity` records (16-byte aligned; GEMM records
 * fill its first half, finalize records its second) and reset the counts;
 * buf = NULL detaches.  Records beyond a half's capacity are dropped.
 * Returns MOE_TAIL_EINVAL for a misaligned buffer or a capacity below 2. */
int moe_tail_trace_attach(void* buf, unsigned int capacity);

/* Records written since the last attach (may exceed the capacity: the excess
 * was dropped).  Synchronises with the device. */
int moe_tail_trace_counts(unsigned int* gemm_records, unsigned int* finalize_records);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TAIL_TRACE_H */
