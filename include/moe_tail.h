/*
 * moe_tail.h -- C ABI of the GB300 MoE decode tail.
 *
 * The MoE decode tail is the per-token finalize that turns the routed
 * experts' output rows into the layer's BF16 output row, plus the dense
 * latent up-projection and the fused shared expert that add into it.  One
 * process drives one GPU: the "ranks" (partitions) of the multi-GPU method
 * are the leading [tp, ...] dimension of a partial-slot tensor in device
 * memory, so there are no mailboxes, peer stores or collectives.
 *
 * Sources (vLLM API pages, cited by page and section):
 *   [MS] vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.moe.tail --
 *        module docstring, BoundTail.run, _check_tail_args, _TpTailKernel.
 *   [KT] vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.tail_runtime --
 *        module docstring, MoeTailBox, MoeTailWeights.
 *   [KS] vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.shared --
 *        module docstring, SharedUmma (load_tile, owned_h), SharedBase.push.
 *
 * Conventions of every call
 *   - Pointers are DEVICE pointers owned by the caller; nothing is allocated,
 *     freed or retained.  `stream` is a cudaStream_t (NULL: legacy default
 *     stream); the call only enqueues work and returns.
 *   - BF16 is IEEE bfloat16 in uint16 storage; FP32 is IEEE binary32.
 *     Tensors are dense, row-major, with the shapes given below.
 *   - Arguments are checked on the host before anything is launched ([MS]
 *     _check_tail_args: a refused call launches nothing).  b = 0 succeeds and
 *     launches nothing ([MS] BoundTail.run).  Refusal reasons: a negative or
 *     out-of-range size, a null pointer with b > 0, a vector pointer not
 *     16-byte aligned (BF16 rows, gamma, out, workspace; the index 4-byte,
 *     route weights 4- or 2-byte), a width not a multiple of 8, an unknown
 *     dtype, a workspace smaller than moe_tail_workspace_bytes(), or `out`
 *     overlapping any input or the workspace.
 *   - Every BF16 result is rounded to nearest-even with -0 written as +0.
 *   - Errors are returned synchronously; a launch failure returns
 *     MOE_TAIL_ECUDA (the CUDA error is cleared).  Faults inside a kernel
 *     surface through the stream like any CUDA error; a bounded internal wait
 *     that expires sets a bit read by moe_tail_take_device_error().
 */
#ifndef MOE_TAIL_H
#define MOE_TAIL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_TAIL_OK = 0,
  MOE_TAIL_EINVAL = 1,  /* arguments refused before any launch */
  MOE_TAIL_ECUDA = 2,   /* a CUDA call failed */
  MOE_TAIL_ENOTSUP = 3  /* valid arguments the library does not support */
} moe_tail_status;

enum { MOE_TAIL_W_FP32 = 0, MOE_TAIL_W_BF16 = 1 };

/*
 * EP finalize ([MS] module docstring, expert parallelism).  Per token t:
 *   g[c]       = fp32(gamma[c]) + gain_center
 *   for slot s in 0..tp-1 (rank order), over the routes k (in order) with
 *   j = permuted_idx[s][t][k] in [0, rows_per_slot)  ("local to s"):
 *     x = rows[s][j][:];  v = weight_before_norm ? x*g : x
 *     inv = 1 / sqrt(sum_squares(v) * (1/P) + eps)
 *     n = weight_before_norm ? v*inv : (x*inv)*g
 *     part_s += n * w[t][k]                     (FP32 from +0, each product rounded)
 *   out[t] = bf16( sum over s of fp32(bf16(part_s)) )   (FP32 from +0)
 * sum_squares: per 256-column chunk, lane l squares and adds columns
 * 8l..8l+7 in order, 32 lanes combine by xor butterfly (1,2,4,8,16), chunk
 * sums are added in chunk order.  Routes with no local row contribute nothing.
 *
 *   rows          BF16 [tp][rows_per_slot][P]  slot s's GEMM2 output rows
 *   rows_per_slot rows per slot (>= 0)
 *   permuted_idx  int32 [tp][b][K]
 *   route_weights [b][K], FP32 or BF16 per weight_dtype (MOE_TAIL_W_*)
 *   gamma         BF16 [P] norm weight (ones when the norm has none)
 *   out           BF16 [b][P]
 * Limits: 1 <= tp <= 32, 1 <= K <= 32, 8 <= P <= 32768, P % 8 == 0, b <= 65535.
 */
int moe_tail_ep_finalize(const void* rows, int64_t rows_per_slot, const int32_t* permuted_idx,
                         const void* route_weights, int weight_dtype, const void* gamma,
                         float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                         int P, void* out, void* stream);

/*
 * Expert-TP finalize ([MS] module docstring, expert TP; _TpTailKernel).
 * Every slot holds a K-partial of every route row.  Per token t, routes k in
 * order with j = permuted_idx[t][k] in [0, num_rows):
 *   x_k = bf16( sum over s in slot order of fp32(partials[s][j][:]) )
 *   out[t] = bf16( sum over k from +0 of fp32(w[t][k] * norm(x_k)) )
 * with norm() the EP finalize's normalisation.  A route whose index is out
 * of range contributes nothing.
 *
 *   partials      BF16 [tp][num_rows][P]
 *   permuted_idx  int32 [b][K] (shared by all slots)
 *   route_weights, gamma, out, limits: as moe_tail_ep_finalize.
 */
int moe_tail_tp_finalize(const void* partials, int64_t num_rows, const int32_t* permuted_idx,
                         const void* route_weights, int weight_dtype, const void* gamma,
                         float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                         int P, void* out, void* stream);

/*
 * The two finalize calls with a scheduling promise (no counterpart on the
 * pages as calls): the same arguments, results and refusals as
 * moe_tail_ep_finalize / moe_tail_tp_finalize, plus
 *   flags: 0, or MOE_TAIL_INPUTS_READY (defined below) -- a promise that the
 *   rows or partials, the indices, the route weights and gamma are not being
 *   written by work still in flight on the stream when the call is enqueued.
 *   The kernel then reads them while the stream's preceding kernel still runs
 *   (with programmatic dependent launch) and waits for that kernel only
 *   before it writes out, which in-flight work may still be reading.
 * Back to back on static inputs this hides most of a call's first trip to
 * memory behind the previous call.
 */
int moe_tail_ep_finalize_flags(const void* rows, int64_t rows_per_slot, const int32_t* permuted_idx,
                               const void* route_weights, int weight_dtype, const void* gamma,
                               float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                               int P, void* out, int flags, void* stream);
int moe_tail_tp_finalize_flags(const void* partials, int64_t num_rows, const int32_t* permuted_idx,
                               const void* route_weights, int weight_dtype, const void* gamma,
                               float gain_center, float eps, int weight_before_norm, int b, int tp, int K,
                               int P, void* out, int flags, void* stream);

/*
 * Latent tail ([KT] module docstring): the latent partials of the tp slots
 * are summed, RMS-normalised per row, up-projected and the shared expert's
 * partials are added:
 *   x    = bf16( sum over s in slot order of fp32(latent[s][t][:]) )
 *   y    = bf16( (x * inv) * fp32(gamma) ),  inv as above with 1/L, eps
 *   out  = bf16( y . w_up^T  (FP32 accumulate)  + sum over s of fp32(shared[s][t][:]) )
 *
 *   latent     BF16 [tp][b][L]
 *   gamma      BF16 [L]
 *   w_up       BF16 [H][L] row-major (output feature n is row n)
 *   shared     BF16 [tp_s][b][H] or NULL when tp_s == 0
 *   out        BF16 [b][H]
 *   workspace  >= moe_tail_workspace_bytes(0, b, L) bytes, 16-byte aligned;
 *              holds y (BF16 [b][L]) after the call
 * Limits: 1 <= tp <= 32, 0 <= tp_s <= 32, 8 <= L <= 32768, 8 <= H <= 16777216,
 * L % 8 == 0, H % 8 == 0, b <= 65535.
 */
int moe_tail_latent_up(const void* latent, const void* gamma, float eps, const void* w_up,
                       const void* shared, int tp_s, int b, int tp, int L, int H, void* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * The latent tail's two steps as separate calls ([KT] module docstring), for
 * callers that schedule them apart: the norm needs only the latent partials,
 * the up-projection only y, the weights and the shared partials, so the norm
 * can run early (beside other work) and the up-projection right after the
 * last shared partial is written.  moe_tail_latent_up is these two calls in
 * a row, and each gives bit for bit the same result as that step there.
 *
 * moe_tail_latent_norm:  y = the x and y lines of moe_tail_latent_up.
 *   latent BF16 [tp][b][L];  gamma BF16 [L];  y BF16 [b][L] (written)
 *   flags: 0, or MOE_TAIL_INPUTS_READY -- a promise that latent and gamma are
 *   not being written by work still in flight on the stream when the call is
 *   enqueued.  The kernel then reads and normalises them while the stream's
 *   preceding kernel still runs and waits for that kernel only before it
 *   writes y (which in-flight work may still be reading).
 *   Limits: 1 <= tp <= 32, 8 <= L <= 32768, L % 8 == 0, b <= 65535; y must
 *   not overlap latent or gamma.
 *
 * moe_tail_up_project:  out = the out line of moe_tail_latent_up, from y.
 *   y BF16 [b][L];  w_up BF16 [H][L];  shared BF16 [tp_s][b][H] or NULL when
 *   tp_s == 0;  out BF16 [b][H] (written; must not overlap an input).
 *   flags: 0, or MOE_TAIL_WEIGHTS_STATIC -- a promise that w_up is not being
 *   written by work still in flight on the stream when the call is enqueued
 *   (model weights loaded before serving).  The kernel then requests its
 *   first weight tiles before it waits for the stream's preceding kernel, so
 *   with programmatic dependent launch the weight stream starts while that
 *   kernel drains; y and shared are always read after the wait.
 *   Limits: 0 <= tp_s <= 32, 8 <= L <= 32768, 8 <= H <= 16777216,
 *   L % 8 == 0, H % 8 == 0, b <= 65535.
 */
#define MOE_TAIL_WEIGHTS_STATIC 1
#define MOE_TAIL_INPUTS_READY 2
int moe_tail_latent_norm(const void* latent, const void* gamma, float eps, int b, int tp, int L, void* y,
                         int flags, void* stream);
int moe_tail_up_project(const void* y, const void* w_up, const void* shared, int tp_s, int b, int L, int H,
                        void* out, int flags, void* stream);

/*
 * The latent tail in one call with the scheduling promises of the split calls
 * ([KT] module docstring, as moe_tail_latent_up).  Same arguments as
 * moe_tail_latent_up, with y (BF16 [b][L], written, 16-byte aligned,
 * overlapping no other argument) in place of the workspace, plus
 *   flags: any of MOE_TAIL_INPUTS_READY (latent and gamma, as for
 *   moe_tail_latent_norm) and MOE_TAIL_WEIGHTS_STATIC (w_up, as for
 *   moe_tail_up_project); shared is always read, and y and out written, after
 *   the wait for the stream's preceding kernel.
 * It runs moe_tail_latent_norm then moe_tail_up_project.  With the latent
 * tail's kernel form pinned to MOE_TAIL_FORM_LATENT_ONE_KERNEL
 * (moe_tail_set_kernel_form) it runs instead, wherever the sizes allow
 * (b <= 32, L <= 8192, tp <= 8 x the ring's stages), one kernel
 * in the pages' fused-tail shape ([KT] WaveMoeTail keeps the normalised
 * latent on chip): the up-projection's CTAs form y for their own K range in
 * shared memory -- each CTA sums and squares the 256-column chunks its range
 * touches and the cluster exchanges the chunk sums -- and then stream the
 * weights.  It is slower on GB300 at every batch size and so not the default.
 * Both forms give bit for bit the same y and out as the two split calls;
 * moe_tail_latent_up and moe_tail_latent_up_noalloc take the same path with
 * flags 0 (the one-kernel form of the latter does not touch its scratch
 * array).  Limits: those of moe_tail_latent_up.
 */
int moe_tail_latent_up_flags(const void* latent, const void* gamma, float eps, const void* w_up,
                             const void* shared, int tp_s, int b, int tp, int L, int H, void* out, void* y,
                             int flags, void* stream);

/*
 * Fused shared expert ([KS] module docstring, SharedUmma.owned_h,
 * SharedBase.push): gate/up projection, gated activation, down projection,
 * added into the tail's output:
 *   gate = bf16(x . w_gate^T), up = bf16(x . w_up^T)     (FP32 accumulate)
 *   h    = bf16( silu(gate) * up ),  silu(g) = g / (1 + exp(-g))
 *   d    = h . w_down^T                                   (FP32 accumulate)
 *   out  = accumulate ? bf16( fp32(out) + fp32(bf16(d)) ) : bf16(d)
 *
 *   x          BF16 [b][H]
 *   w_gate     BF16 [I][H];  w_up BF16 [I][H];  w_down BF16 [H][I]
 *   out        BF16 [b][H] (read as well when accumulate != 0)
 *   workspace  >= moe_tail_workspace_bytes(1, b, I) bytes, 16-byte aligned;
 *              holds h (BF16 [b][I]) after the call
 * Limits: 8 <= H <= 16777216, 8 <= I <= 16777216, H % 8 == 0, I % 8 == 0,
 * b <= 65535.
 */
int moe_shared_expert(const void* x, const void* w_gate, const void* w_up, const void* w_down,
                      int b, int H, int I, void* out, int accumulate, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * The shared expert's two GEMMs as separate calls ([KS] module docstring), for
 * callers that schedule other work between them -- e.g. the latent tail's
 * up-projection between gate/up and down, with down then adding d into the
 * tail's output.  moe_shared_expert is these two calls in a row, and each
 * gives bit for bit the same result as that step there.
 *
 * moe_shared_gate_up:  h = the gate, up and h lines of moe_shared_expert.
 *   x BF16 [b][H];  w_gate, w_up BF16 [I][H];  h BF16 [b][I] (written; must
 *   not overlap an input).
 * moe_shared_down:  out = the d and out lines of moe_shared_expert, from h.
 *   h BF16 [b][I];  w_down BF16 [H][I];  out BF16 [b][H] (read as well when
 *   accumulate != 0; must not overlap an input).
 *   flags (both calls): 0, or MOE_TAIL_WEIGHTS_STATIC (as for
 *   moe_tail_up_project: the first weight tiles are requested before the
 *   kernel waits for the stream's preceding kernel).  moe_shared_gate_up
 *   also takes MOE_TAIL_INPUTS_READY: a promise that x is not being written
 *   by work still in flight on the stream.  The kernel then reads x and runs
 *   its whole K loop while the preceding kernel drains, and waits for that
 *   kernel only before it writes h (which the preceding kernel may still be
 *   reading).  The flags change only when memory is read, never the result.
 *   Limits: 8 <= H <= 16777216, 8 <= I <= 16777216, H % 8 == 0, I % 8 == 0,
 *   b <= 65535.
 */
int moe_shared_gate_up(const void* x, const void* w_gate, const void* w_up, int b, int H, int I, void* h,
                       int flags, void* stream);
int moe_shared_down(const void* h, const void* w_down, int b, int H, int I, void* out, int accumulate,
                    int flags, void* stream);

/*
 * The down projection as the Kimi-K3 shared expert page's persistent kernel
 * ([KS] SharedDown): the same out as moe_shared_down, up to the order of d's
 * FP32 sum (here no K split: a few elements may round differently).  ctas
 * CTAs (one per SM; 0: one per output tile, at most the GPU's SM count) walk
 * the output tiles of 128 rows x the token tile (16, 32, 64 or 128 tokens),
 * tile c, c + ctas, ..., each over the whole K range, with two tensor-memory
 * accumulators that alternate between a CTA's consecutive tiles, so each
 * tile's epilogue overlaps the next tile's weight stream.  A caller that runs
 * other work beside it gives it the SMs that work leaves free.
 *   h, w_down, out, accumulate, flags: as moe_shared_down.
 *   ctas: 0 .. 65535.
 * Limits and refusals: those of moe_shared_down, plus ctas out of range.
 */
int moe_shared_down_persistent(const void* h, const void* w_down, int b, int H, int I, void* out, int accumulate,
                               int ctas, int flags, void* stream);

/*
 * The latent tail's up-projection with the shared expert's down projection
 * in one kernel ([KT] module docstring: the shared expert's output joins the
 * tail's shared partials before the up-projection's epilogue; [KS]
 * SharedBase.push: the down projection is pushed as BF16, -0 made +0):
 *   d   = h . w_down^T                     (FP32 accumulate)
 *   u   = y . w_up^T                       (FP32 accumulate)
 *   out = bf16( u + ( sum_s fp32(shared[s]) + fp32(bf16(d)) ) )
 * with the shared partials added in slot order from +0 and bf16(d) last --
 * the result of moe_shared_down (accumulate = 0) writing bf16(d) into one
 * more shared slot, then moe_tail_up_project over tp_s + 1 slots, up to the
 * order of the FP32 sums of d and u (each K range is split differently, so
 * a few elements may round differently).  One kernel streams both weights:
 * some CTAs of each cluster take slices of W_down's K range, the others of
 * W_up's, and one epilogue adds each projection's partials, so the pair
 * costs one kernel's ramp and tail instead of two.
 *   y       BF16 [b][L] (moe_tail_latent_norm's output)
 *   w_up    BF16 [H][L];  shared BF16 [tp_s][b][H] or NULL (tp_s = 0)
 *   h       BF16 [b][I] (moe_shared_gate_up's output);  w_down BF16 [H][I]
 *   out     BF16 [b][H] (written)
 *   d_out   BF16 [b][H] receiving bf16(d), or NULL
 *   flags   0, or MOE_TAIL_WEIGHTS_STATIC (w_up and w_down, as for
 *           moe_tail_up_project: weight tiles requested before the kernel
 *           waits for the stream's preceding kernel)
 * Neither out nor d_out may overlap an input or each other.  Limits: those of
 * moe_tail_up_project, plus 8 <= I <= 16777216, I % 8 == 0.
 */
int moe_tail_up_project_shared_down(const void* y, const void* w_up, const void* shared, int tp_s,
                                    const void* h, const void* w_down, int b, int L, int I, int H,
                                    void* out, void* d_out, int flags, void* stream);

/*
 * Latent tail without a workspace (no counterpart on the pages: an addition
 * of this library).  Same computation and arguments as moe_tail_latent_up,
 * minus the workspace: for callers that cannot allocate device memory -- a
 * plugin that its host runtime hands only input and output buffers, a
 * process whose device memory is all reserved by its own pool, or a hot path
 * that must not call cudaMalloc because it can synchronise the device.
 *
 * The intermediate y rows live in a fixed array of
 * MOE_TAIL_NOALLOC_SCRATCH_BYTES bytes inside the library's device code,
 * which every GPU that loads the library keeps until the process exits.  The
 * call allocates and frees nothing.  Limits and refusals are those of
 * moe_tail_latent_up, plus: b * L * 2 > MOE_TAIL_NOALLOC_SCRATCH_BYTES
 * returns MOE_TAIL_EINVAL before anything runs.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  If the device's context has been replaced since (a
 *     cudaDeviceReset), the next call looks the address up again.
 *   - The array is private to the library, so no caller buffer can overlap
 *     it; the call still refuses one that does, as it would a workspace.
 *   - All calls share the one array and each overwrites all of the y rows it
 *     uses, so nothing has to start at zero; calls that may run at the same
 *     time on the GPU (different streams, or different host threads) race on
 *     it and must be serialised by the caller.
 */
#define MOE_TAIL_NOALLOC_SCRATCH_BYTES (1u << 20)
int moe_tail_latent_up_noalloc(const void* latent, const void* gamma, float eps, const void* w_up,
                               const void* shared, int tp_s, int b, int tp, int L, int H, void* out,
                               void* stream);

/*
 * Kernel form of a call (no counterpart on the pages: a choice between
 * kernels of this library that compute the same bits).  Some calls have more
 * than one kernel form; the library picks one per call from the sizes unless
 * a form is pinned here.  Every form of a call gives bit for bit the same
 * outputs, so a pin only changes speed; it exists for tests that run every
 * form and for measurements.  The setting is process-wide (all devices and
 * host threads) and applies to calls made after it returns.
 *   call MOE_TAIL_FORM_EP      (moe_tail_ep_finalize, _flags):
 *        1 token-resident kernel (a token's routes held in registers),
 *        2 route-parallel kernel (route groups of a CTA, products in shared memory)
 *   call MOE_TAIL_FORM_TP      (moe_tail_tp_finalize, _flags):
 *        1 staged kernel (route rows streamed into a shared-memory ring),
 *        2 route-parallel kernel
 *   call MOE_TAIL_FORM_LATENT  (moe_tail_latent_up, _flags, _noalloc):
 *        MOE_TAIL_FORM_LATENT_ONE_KERNEL (1): the latent tail as one kernel
 *        wherever the sizes allow (b <= 32, L <= 8192, tp within the ring),
 *        the norm and the up-projection as two kernels elsewhere;
 *        2: always the two kernels
 *   form 0 (every call): the library's choice (the default).
 * Returns MOE_TAIL_EINVAL for an unknown call or form, else MOE_TAIL_OK.
 */
enum { MOE_TAIL_FORM_EP = 0, MOE_TAIL_FORM_TP = 1, MOE_TAIL_FORM_LATENT = 2 };
#define MOE_TAIL_FORM_LATENT_ONE_KERNEL 1
int moe_tail_set_kernel_form(int call, int form);

/* Workspace bytes of moe_tail_latent_up (which = 0, dim = L) or
 * moe_shared_expert (which = 1, dim = I) at b tokens; 0 for bad arguments. */
size_t moe_tail_workspace_bytes(int which, int b, int dim);

/* Static text for a moe_tail_status value. */
const char* moe_tail_status_str(int status);

/* Reads and clears the device error word of the calling thread's current
 * device (synchronises with it).  *bits receives the bits raised since the
 * last read: 1 operand stage never arrived, 2 stage never released,
 * 4 accumulator never completed, 8 drain after abort failed.  Returns
 * MOE_TAIL_OK or MOE_TAIL_ECUDA. */
int moe_tail_take_device_error(unsigned int* bits);

/* Failure-detection self-test (no counterpart on the pages).  Every wait
 * inside these kernels is bounded in time: when one expires the kernel sets a
 * bit in the device error word, finishes what it started and returns, instead
 * of hanging or trapping.  This call exercises that path: it launches one
 * thread that waits, with the same bounded wait, on a barrier nothing arrives
 * at, for limit_us microseconds (1..1000000).  Afterwards
 * moe_tail_take_device_error() reports 1 (an operand stage never arrived)
 * and the device stays usable.
 * Returns MOE_TAIL_EINVAL for a limit out of range, MOE_TAIL_ECUDA if the
 * launch fails. */
int moe_tail_selftest_wait_timeout(unsigned int limit_us, void* stream);

/* Failure-detection test hook (no counterpart on the pages): the limit of
 * the operand-stage waits -- the GEMM kernels' tensor-core issuer waiting for
 * a stage of weights and tokens, the staged expert-TP finalize kernel's
 * threads waiting for a stage of route rows -- for calls made after it
 * returns (process-wide), in nanoseconds (1: give up at the first such
 * wait, whether or not the stage has landed); 0 restores the default (0.5 s).
 * Only those waits change.  The waits that guard memory a CTA is about to
 * release keep their full limit: the copies still in flight when a call
 * aborts, and the tensor-core work issued before it, so an expired short wait
 * aborts the call cleanly -- the kernel raises bit 1 of the device error word,
 * issues nothing more, waits for what it started, frees its tensor memory and
 * returns; that call's outputs are then undefined.  A limit shorter than a
 * memory trip makes calls fail: it exists for tests of the abort path.
 * Returns MOE_TAIL_EINVAL for a limit above 1 s. */
int moe_tail_set_stage_wait_limit(unsigned long long limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TAIL_H */
