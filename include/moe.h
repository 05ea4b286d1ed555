/*
 * moe.h -- C ABI of the single-GPU MoE dispatch / experts / combine path for
 * GB300 (sm_103a).
 *
 * What the path computes is defined by two pages:
 *   [HEP] "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)" -- Changelog and
 *         the review of dispatch(): top-k indices become a multihot
 *         routing_map with fp32 probs, dispatch returns tokens_per_expert and
 *         pads each expert's rows to pad_multiple, and the number of permuted
 *         rows is tokens_per_expert.sum().
 *   [DEP] "Add the deepep expert-parallel implementation
 *         (huggingface/transformers #49638)" -- What this adds: Expanded
 *         layout (each (token, expert) pair has its own row; rows are grouped
 *         per expert and carry the pair's weight, which the experts apply;
 *         the combine adds rows without weights); Eager vs captured (either
 *         the exact row count is read back to the host, or a buffer sized
 *         for any routing is used without a sync, its unused rows zero and
 *         owned by a sentinel expert that is never computed); Custom ops and
 *         Training (the combine's gradient is a dispatch along the same
 *         layout; the routing weights get gradients through the combine);
 *         Usage (the hidden size must be a multiple of 256).
 *
 * Conventions for every entry point:
 *   - Pointers named in a signature are DEVICE pointers unless the comment
 *     says "host".  The caller owns all memory; the library allocates no
 *     device memory, keeps no state between calls and holds no handles.  Row
 *     buffers hold `capacity` rows.  One exception, host-side only:
 *     host-synced moe_dispatch keeps 16 bytes of mapped pinned host memory per
 *     device, allocated on its first call and kept until the process exits.
 *     The count kernel writes the row totals and the status word straight
 *     into it.
 *   - bf16 tensors are passed as raw bit patterns (moe_bf16), row-major,
 *     with the last dimension contiguous and rows packed (no row stride).
 *     Every pointer must be 16-byte aligned.
 *   - Every call is asynchronous and ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream), except moe_dispatch in host-synced
 *     mode, which waits on the host once, for the row counts: everything
 *     queued on `stream` before the call has completed when it returns.
 *   - Every call validates its arguments on the host and returns a
 *     moe_status; it never aborts the process.  moe_last_error() gives a
 *     human-readable detail of the last failure on the calling thread.
 *   - Errors found on the device (an expert index outside [-1, E), a
 *     capacity overflow, a bounded wait that ran out) are OR-ed into the
 *     caller's device status word as MOE_DEVERR_* bits; kernels never trap.
 *     The caller zeroes the word before first use and reads it when it
 *     chooses (host-synced moe_dispatch reads it at its sync).
 *   - Shapes: H % 256 == 0, I % 128 == 0, 1 <= K <= min(E, 127),
 *     E <= 1024 with E % 4 == 0, pad_multiple >= 1, T >= 0, and
 *     T*K + E*(pad_multiple-1) < 2^31.  The device must be compute capability 10.3.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* raw bfloat16 bit pattern            */
typedef struct CUstream_st* moe_stream_t;  /* the same type as cudaStream_t       */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, misalignment     */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* H % 256, I % 128, K > 127, E > 1024 ...        */
  MOE_ERR_CAPACITY = 3,           /* the layout needs more rows than `capacity`     */
  MOE_ERR_BAD_INDEX = 4,          /* an expert index outside [-1, E) was seen       */
  MOE_ERR_TIMEOUT = 5,            /* a bounded device-side wait ran out             */
  MOE_ERR_DEVICE = 6,             /* the current device is not compute cap. 10.3    */
  MOE_ERR_CUDA = 7                /* a CUDA runtime / driver call failed            */
} moe_status;

/* Bits of the device status word (int32, OR-ed by kernels). */
#define MOE_DEVERR_BAD_INDEX 1
#define MOE_DEVERR_CAPACITY  2
#define MOE_DEVERR_TIMEOUT   4
/* Set only by the bounds-checked build of the library (moe_build_flags() has
 * MOE_BUILD_BOUNDS_CHECKS): a kernel found an index it derived from the
 * layout outside its buffer and skipped the access. */
#define MOE_DEVERR_BOUNDS    8

/* Name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status status);

/* Detail of the last failing call on this thread (thread-local, static storage). */
MOE_API const char* moe_last_error(void);

/* MOE_OK if the current CUDA device is compute capability 10.3, else MOE_ERR_DEVICE. */
MOE_API moe_status moe_device_check(void);

/* How this copy of the library was built: MOE_BUILD_BOUNDS_CHECKS when its
 * kernels check the indices they derive from the layout against their
 * buffers (the debugging build, compiled with MOE_DEBUG_BOUNDS; results are
 * the same as the normal build's, MOE_DEVERR_BOUNDS flags a failed check). */
#define MOE_BUILD_BOUNDS_CHECKS 1u
MOE_API uint32_t moe_build_flags(void);

/* Rows a sync-free buffer needs so that no routing can overflow it:
 * T*K (every slot valid) + E*(pad_multiple-1) (every group padded).
 * [DEP] Eager vs captured: the sync-free buffer is sized for the worst case. */
MOE_API int64_t moe_worst_case_rows(int32_t T, int32_t E, int32_t K, int32_t pad_multiple);

/*
 * The expanded layout of one forward + backward: the "handle" that
 * [HEP]'s hybrid_ep_dispatch returns, made explicit as caller-owned device
 * buffers ([DEP] Custom ops: the handle is passed as tensors).  Written by
 * moe_dispatch, read by every later call.  All pointers are device pointers.
 */
typedef struct moe_layout {
  int32_t T, E, K, pad_multiple;
  int64_t capacity;            /* C: rows in every row buffer below                  */
  int32_t* tokens_per_expert;  /* [E]    exact number of tokens routed to each expert */
  int32_t* offsets;            /* [E+1]  start row of each expert's group; groups are
                                           padded to a multiple of pad_multiple       */
  int32_t* totals;             /* [2]    R = offsets[E] rows used, N = valid rows     */
  int32_t* row_token;          /* [C]    token of each row; -1 on pad / spare rows    */
  int32_t* row_expert;         /* [C]    expert of each row; E (the sentinel) on pad /
                                           spare rows                                  */
  float*   row_weight;         /* [C]    fp32 routing weight of the row's slot; 0 on
                                           pad / spare rows                            */
  int32_t* token_row;          /* [T*K]  each token's rows in ascending expert order,
                                           then -1                                     */
  int32_t* status;             /* [1]    device status word (MOE_DEVERR_* bits)        */
  void*    workspace;          /* moe_layout_workspace_bytes(T, E) bytes of scratch   */
} moe_layout;

/* Bytes of scratch moe_dispatch needs in moe_layout.workspace (256-byte aligned). */
MOE_API moe_status moe_layout_workspace_bytes(int32_t T, int32_t E, size_t* bytes);

/*
 * r0. The router in front of the path: per token, a softmax over the E
 * logits, the K most probable experts, and their probabilities renormalised
 * to sum to one.  The pages begin the path at its output (top-k indices and
 * fp32 weights; [HEP] Changelog); the three steps are the workload's router
 * recipe.
 *   logits       [T, E] fp32, finite (a NaN counts as -inf; a token whose
 *                chosen logits are all -inf gets NaN weights).
 *   topk_idx     [T, K] int64 (out): experts in descending probability; equal
 *                logits are ordered by ascending expert index.
 *   topk_probs   [T, K] fp32  (out): the renormalised weights, which equal the
 *                softmax of the K chosen logits.
 *   routing_map, probs, winner_slot: NULL, or all three given: then the call
 *                also writes the multihot outputs of moe_route_to_multihot
 *                for these top-k choices (16-byte aligned), in the same
 *                kernel.
 * Errors: MOE_ERR_UNSUPPORTED_SHAPE unless E % 4 == 0, E <= 1024 and
 * 1 <= K <= min(E, 127); MOE_ERR_INVALID_ARG for NULL or misaligned buffers.
 * Every output is caller-owned device memory; nothing is allocated.
 */
MOE_API moe_status moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t K,
                                   int64_t* topk_idx, float* topk_probs, uint8_t* routing_map,
                                   float* probs, int8_t* winner_slot, moe_stream_t stream);

/*
 * r0 backward.  grad_logits [T, E] fp32 (out, 16-byte aligned):
 *   w_j * (g_j - sum_k w_k g_k) at each chosen expert j (w = topk_probs,
 *   g = grad_topk_probs), 0 at the others -- the chain rule through the
 *   softmax of the chosen logits; the selection passes no gradient.
 */
MOE_API moe_status moe_router_topk_backward(const float* grad_topk_probs, const float* topk_probs,
                                            const int64_t* topk_idx, int32_t T, int32_t E,
                                            int32_t K, float* grad_logits, moe_stream_t stream);

/*
 * a1. Top-k -> multihot.  [HEP] Changelog (the HybridEP preprocessing turns
 * top-k indices into multihot routing metadata) and the review of dispatch()
 * (probs are fp32).
 *   topk_idx     [T, K] int64: expert of each slot, -1 = no expert (dropped).
 *   topk_probs   [T, K] fp32:  the slot's routing weight.
 *   routing_map  [T, E] uint8 (out): 1 where token t is routed to expert e.
 *   probs        [T, E] fp32  (out): the weight of that pair, 0 elsewhere.
 *   winner_slot  [T, E] int8  (out): the slot k that set the pair, -1 elsewhere.
 *   status       [1] int32 device status word.
 * Slots are taken in order k = 0..K-1, so when one token names the same
 * expert twice the pair is set once and the last such slot's prob wins.  An
 * index outside [-1, E) sets MOE_DEVERR_BAD_INDEX and is treated as -1.
 */
MOE_API moe_status moe_route_to_multihot(const int64_t* topk_idx, const float* topk_probs,
                                 int32_t T, int32_t K, int32_t E,
                                 uint8_t* routing_map, float* probs, int8_t* winner_slot,
                                 int32_t* status, moe_stream_t stream);

/*
 * a2-a4. Counts, padded offsets, the expanded layout, and the row gather.
 * [HEP] review of dispatch(): tokens_per_expert, pad_multiple, the number of
 * permuted rows; [DEP] Expanded layout; Eager vs captured.
 *   x            [T, H] bf16 tokens.
 *   routing_map, probs: as written by moe_route_to_multihot.
 *   L            layout to fill (its pointers and sizes are read on the host).
 *   x_disp       [C, H] bf16 (out): x_disp[r] = x[row_token[r]] bit for bit;
 *                pad and spare rows are zero.
 *   rows_host    HOST int64[2] or NULL.
 *     non-NULL = host-synced (eager) mode: the call waits until the count
 *       kernel has published the counts to the host (it may still be
 *       finishing), writes rows_host[0] = R (rows used) and
 *       rows_host[1] = N (valid rows), returns MOE_ERR_BAD_INDEX if the
 *       status word has MOE_DEVERR_BAD_INDEX, or MOE_ERR_CAPACITY (before
 *       writing any row) if R > capacity.
 *     NULL = sync-free mode: capacity must be >= moe_worst_case_rows(...)
 *       (checked on the host, else MOE_ERR_CAPACITY); nothing is read back,
 *       rows R..C-1 become spare rows (zero, sentinel expert), and the call
 *       can be captured in a CUDA graph.
 * Within an expert's group the rows are in ascending token order.
 */
MOE_API moe_status moe_dispatch(const moe_bf16* x, const uint8_t* routing_map, const float* probs,
                        int32_t H, const moe_layout* L, moe_bf16* x_disp,
                        int64_t* rows_host, moe_stream_t stream);

/*
 * a1-a4 in one call: moe_route_to_multihot followed by moe_dispatch, from the
 * top-k choices.  [HEP] Changelog (top-k indices become multihot routing
 * data) and the passages of moe_dispatch.
 *   topk_idx, topk_probs: [T, K] int64 / fp32, as for moe_route_to_multihot
 *                (an index outside [-1, E) sets MOE_DEVERR_BAD_INDEX and
 *                counts as -1).
 *   routing_map, probs, winner_slot: [T, E] (out, required, 16-byte
 *                aligned): the multihot outputs of moe_route_to_multihot, for
 *                the backward.
 *   x, L, x_disp, rows_host, stream: as for moe_dispatch, with the same
 *                modes, results and errors.
 * Layers of more than 8 chunks of 32 tokens run all of it as one cooperative
 * kernel (the multihot rows, counts, offsets, placement and row copies);
 * smaller ones as the multihot kernel followed by moe_dispatch's kernels.
 */
MOE_API moe_status moe_dispatch_topk(const moe_bf16* x, const int64_t* topk_idx,
                                     const float* topk_probs, int32_t H, const moe_layout* L,
                                     uint8_t* routing_map, float* probs, int8_t* winner_slot,
                                     moe_bf16* x_disp, int64_t* rows_host, moe_stream_t stream);

/*
 * a2-a3 alone: the layout of moe_dispatch (counts, offsets, totals, row
 * metadata, with the pad and spare rows' sentinel metadata) without copying
 * any rows -- for moe_grouped_experts_gather, which reads the tokens itself.
 * Modes, rows_host and errors as in moe_dispatch.
 */
MOE_API moe_status moe_dispatch_layout(const uint8_t* routing_map, const float* probs,
                                       const moe_layout* L, int64_t* rows_host,
                                       moe_stream_t stream);

/*
 * a4 in FP8 ([DEP] What this adds, scope note: FP8 dispatch, half the
 * dispatch bytes, is the named follow-up).  As moe_dispatch, but the rows are
 * float8 e4m3 codes with one fp32 scale per row:
 *   x_disp_q     [C, H] uint8 (out): e4m3(x[t] / s_t) for row r of token t,
 *                rounded to nearest even, saturated at +-448.
 *   x_disp_scale [C] fp32 (out): s_t = amax(|x[t]|) / 448 (1 for a zero row);
 *                pad and spare rows get zero codes and scale 0.
 * The division and the amax are fp32, so the codes are exact functions of x.
 * Arguments, modes and errors are otherwise those of moe_dispatch.
 */
MOE_API moe_status moe_dispatch_fp8(const moe_bf16* x, const uint8_t* routing_map,
                                    const float* probs, int32_t H, const moe_layout* L,
                                    uint8_t* x_disp_q, float* x_disp_scale, int64_t* rows_host,
                                    moe_stream_t stream);

/*
 * a1-a4 in one call with FP8 rows: moe_route_to_multihot followed by
 * moe_dispatch_fp8, from the top-k choices.  The passages of both.
 *   topk_idx, topk_probs, routing_map, probs, winner_slot: as for
 *                moe_dispatch_topk.
 *   x, L, x_disp_q, x_disp_scale, rows_host, stream: as for
 *                moe_dispatch_fp8, with the same modes, results and errors.
 * Layers of more than 8 chunks of 32 tokens run all of it as one cooperative
 * kernel (the multihot rows, counts, offsets, placement, the e4m3 codes and
 * scales); smaller ones as the multihot kernel followed by moe_dispatch_fp8's
 * kernels.
 */
MOE_API moe_status moe_dispatch_topk_fp8(const moe_bf16* x, const int64_t* topk_idx,
                                         const float* topk_probs, int32_t H, const moe_layout* L,
                                         uint8_t* routing_map, float* probs, int8_t* winner_slot,
                                         uint8_t* x_disp_q, float* x_disp_scale, int64_t* rows_host,
                                         moe_stream_t stream);

/*
 * Rowwise e4m3 quantization of a bf16 matrix [rows, cols] (cols a multiple
 * of 256, src and codes 16-byte aligned), with the rule of moe_dispatch_fp8:
 * codes [rows, cols] uint8 and scales [rows] fp32 (out).  For the gate/up
 * weight W1 [E, 2I, H] this is one scale per output channel (rows = E * 2I).
 */
MOE_API moe_status moe_quantize_fp8(const moe_bf16* src, int64_t rows, int32_t cols,
                                    uint8_t* codes, float* scales, moe_stream_t stream);

/*
 * moe_dispatch without caller-provided scratch.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory -- for example a plugin inside an inference engine
 * that owns the whole device pool and passes a layer only its declared
 * inputs and outputs, or a serving loop that must not call cudaMalloc
 * because it can synchronise the device.
 *
 * Arguments, results and errors are those of moe_dispatch, except that
 * L->workspace is ignored (it may be NULL): the per-chunk expert masks and
 * start rows live in a static device array inside the library,
 * 2 * MOE_STATIC_SCRATCH_INTS int32 (2 MiB, plus 33 KiB for the kernel's
 * barrier words and count copies) per GPU, held from library load until the
 * process exits.
 *   - Limit: E * ceil(T / 32) <= MOE_STATIC_SCRATCH_INTS (E = 128 allows
 *     T <= 65536); larger sizes return MOE_ERR_UNSUPPORTED_SHAPE before any
 *     work is queued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress), and so does the first call after a device
 *     reset.  Make that call before any stream capture: made while `stream`
 *     is being captured it returns MOE_ERR_INVALID_ARG and queues nothing.
 *   - All calls share the one array and it keeps the last call's contents
 *     (every counter a call reads is written earlier in that call, so nothing
 *     needs clearing).  A call uses the array until its work on `stream` has
 *     completed -- a host-synced call too, which returns once the row counts
 *     are known, while its kernels may still be reading the array.  Calls
 *     whose work overlaps on the GPU -- on different streams, or from
 *     different host threads -- race on it: order each call after the
 *     previous call's stream work (one shared stream, or an event).
 *   - No device memory is allocated or freed.
 */
#define MOE_STATIC_SCRATCH_INTS 262144
MOE_API moe_status moe_dispatch_static_scratch(const moe_bf16* x, const uint8_t* routing_map,
                                               const float* probs, int32_t H,
                                               const moe_layout* L, moe_bf16* x_disp,
                                               int64_t* rows_host, moe_stream_t stream);

/*
 * a5. Grouped SwiGLU experts that apply the routing weight.  [DEP] Expanded
 * layout (the experts apply the routing weights); Benchmarks (bf16 grouped GEMMs).
 *   x_disp  [C, H] bf16 rows (moe_dispatch's output).
 *   W1      [E, 2I, H] bf16: per expert, rows 0..I-1 gate, rows I..2I-1 up.
 *   W2      [E, H, I] bf16: per expert, the down projection.
 *   h       [C, I] bf16 (out, required): h = bf16(silu(x Wg^T) * (x Wu^T)).
 *   y_disp  [C, H] bf16 (out): y = bf16(w_r * (h W2^T)), fp32 accumulation.
 *   o_save  [C, H] bf16 (out, nullable): bf16(h W2^T), the pre-weight output
 *           the routing-weight gradient needs.
 *   gu_save [C, 2I] bf16 (out, nullable): bf16 of the gate and up
 *           pre-activations, which the expert backward needs.
 * Above 64 rows per expert on average (T*K > 64*E) each expert's rows are
 * computed in chunks of up to 256 on CTA pairs; smaller layers in 128-row
 * tiles, one CTA each.  The valid rows are written.  When gu_save is given
 * (training), the pad rows of each expert's group are written too (with
 * 128-row tiles, those the tiles cover), and come out as zeros in h, y, o_save
 * and gu_save because moe_dispatch leaves x_disp's pad rows zero and their
 * weight is 0; without gu_save they are not touched.  Spare rows (R..C-1) are
 * never written.  The row counts are read on the device, so the call never
 * synchronises and can be captured.
 * On CTA pairs an eager call takes one of 16 slots of row-chunk readiness
 * counters (static device memory of the library, 2 x 128 KiB per GPU), so
 * that the down projection can start on a chunk as soon as its h is written;
 * a call being captured into a graph takes none and waits for the whole
 * gate/up launch instead.  Calls on one stream are ordered; more than 16 such
 * calls in flight at once on different streams would share a slot, so order
 * them (one stream, or events).
 */
MOE_API moe_status moe_grouped_experts(const moe_bf16* x_disp, const moe_layout* L,
                               int32_t H, int32_t I,
                               const moe_bf16* W1, const moe_bf16* W2,
                               moe_bf16* h, moe_bf16* y_disp,
                               moe_bf16* o_save, moe_bf16* gu_save,
                               moe_stream_t stream);

/*
 * a4 fused into a5 ([DEP] Expanded layout: the experts see their own rows):
 * as moe_grouped_experts, but the gate/up GEMM gathers its A rows straight
 * from the tokens, row r being x[row_token[r]] (zeros where row_token is -1),
 * so no x_disp is written or read.  x [T, H] bf16; L from moe_dispatch_layout
 * (or moe_dispatch).  The outputs equal moe_grouped_experts' on the x_disp
 * moe_dispatch would have written, bit for bit.
 */
MOE_API moe_status moe_grouped_experts_gather(const moe_bf16* x, const moe_layout* L, int32_t H,
                                              int32_t I, const moe_bf16* W1, const moe_bf16* W2,
                                              moe_bf16* h, moe_bf16* y_disp, moe_bf16* o_save,
                                              moe_bf16* gu_save, moe_stream_t stream);

/*
 * a5 with the gate/up GEMM on e4m3 operands: x_disp_q / x_disp_scale from
 * moe_dispatch_fp8 and W1_q [E, 2I, H] uint8 / W1_scale [E * 2I] fp32 from
 * moe_quantize_fp8.  The tensor cores multiply the codes exactly
 * (tcgen05.mma kind::f8f6f4, fp32 accumulation); the epilogue multiplies by
 * row scale x channel scale, then applies the SwiGLU.  The down projection,
 * W2 and the outputs h and y are bf16, as in moe_grouped_experts.  Inference
 * only (no saved operands for the backward).  Shapes and errors as in
 * moe_grouped_experts.
 */
MOE_API moe_status moe_grouped_experts_fp8(const uint8_t* x_disp_q, const float* x_disp_scale,
                                           const moe_layout* L, int32_t H, int32_t I,
                                           const uint8_t* W1_q, const float* W1_scale,
                                           const moe_bf16* W2, moe_bf16* h, moe_bf16* y_disp,
                                           moe_stream_t stream);

/*
 * a6. Combine: out[t] = bf16(sum over t's rows of fp32(y_disp[row])), adding
 * in ascending expert order from +0.0 in fp32, one final rounding; no weights
 * ([DEP] Expanded layout: the combine is a plain sum).  A token with no rows
 * gets +0.  Pad and spare rows are never read.
 *   y_disp [C, H] bf16; out [T, H] bf16 (out).
 */
MOE_API moe_status moe_combine(const moe_bf16* y_disp, const moe_layout* L, int32_t H,
                       moe_bf16* out, moe_stream_t stream);

/*
 * a7 + a8. Combine backward and the routing-weight gradient.  [DEP] Training:
 * the combine's backward dispatches along the forward layout, and the
 * weight gradients go back through the combine.
 *   grad_out [T, H] bf16: dL/d out.
 *   o_save   [C, H] bf16 (nullable): moe_grouped_experts' o_save.
 *   grad_y   [C, H] bf16 (out): grad_y[r] = grad_out[row_token[r]] bit for
 *            bit; zero on pad / spare rows.
 *   grad_w   [C] fp32 (out, nullable; needs o_save): grad_w[r] =
 *            sum_h grad_y[r,h] * o[r,h] in fp32; zero on pad / spare rows.
 */
MOE_API moe_status moe_combine_backward(const moe_bf16* grad_out, const moe_bf16* o_save,
                                const moe_layout* L, int32_t H,
                                moe_bf16* grad_y, float* grad_w, moe_stream_t stream);

/*
 * a7 + a8 with the routing weight applied: as moe_combine_backward, but each
 * valid row receives G_o[r] = bf16(row_weight[r] * grad_out[row_token[r]])
 * -- the gradient with respect to the experts' pre-weight output o, since
 * y = w_r * o ([DEP] Expanded layout: the experts apply the weights;
 * Training) -- instead of grad_y; pad and spare rows are zero.  grad_w is
 * still the dot of the unscaled gradient with o_save, as in
 * moe_combine_backward.  Feed G_o to moe_grouped_experts_backward_scaled,
 * which then skips its own scaling pass (one read and one write of [C, H]
 * fewer).  Arguments and errors as in moe_combine_backward.
 */
MOE_API moe_status moe_combine_backward_scaled(const moe_bf16* grad_out, const moe_bf16* o_save,
                                               const moe_layout* L, int32_t H, moe_bf16* g_o,
                                               float* grad_w, moe_stream_t stream);

/*
 * a10 + the weight-gradient scatter.  [DEP] Training (both the tokens and
 * the routing weights receive gradients).
 *   grad_x_disp [C, H] bf16: dL/d x_disp.
 *   grad_x      [T, H] bf16 (out): the combine applied to grad_x_disp (same
 *               order and rounding as moe_combine).
 *   grad_w      [C] fp32 (nullable) and grad_probs [T, E] fp32 (out,
 *               nullable): grad_probs[t, e] = grad_w[row of (t, e)], 0 where
 *               t is not routed to e.
 */
MOE_API moe_status moe_dispatch_backward(const moe_bf16* grad_x_disp, const float* grad_w,
                                 const moe_layout* L, int32_t H,
                                 moe_bf16* grad_x, float* grad_probs, moe_stream_t stream);

/*
 * Multihot backward: grad_topk_probs[t, k] = grad_probs[t, topk_idx[t, k]]
 * when slot k is valid and is the slot that set the pair (winner_slot), else 0.
 *   grad_probs [T, E] fp32, topk_idx [T, K] int64, winner_slot [T, E] int8;
 *   grad_topk_probs [T, K] fp32 (out).
 */
MOE_API moe_status moe_route_to_multihot_backward(const float* grad_probs, const int64_t* topk_idx,
                                          const int8_t* winner_slot,
                                          int32_t T, int32_t K, int32_t E,
                                          float* grad_topk_probs, moe_stream_t stream);

/*
 * a9. Expert backward: the dgrad and wgrad of the SwiGLU experts.  [DEP]
 * Training (both the tokens and the routing weights receive gradients; the
 * routing-weight part is moe_combine_backward's grad_w).  With
 * G_o = w_r * grad_y (y = w_r * o moves the weight onto the gradient):
 *   dW2[e] = sum_r G_o[r]^T h[r];  G_h = G_o W2[e];
 *   G_g = G_h * u * silu'(g),  G_u = G_h * silu(g)  (g, u: gate / up pre-activations);
 *   dW1[e] = sum_r [G_g | G_u][r]^T x_disp[r];  grad_x_disp = [G_g | G_u] W1[e].
 *   grad_y [C, H] bf16 (moe_combine_backward's output); x_disp [C, H], h [C, I]
 *     and gu_save [C, 2I] bf16 from the forward (gu_save is required here).
 *   W1, W2: as in moe_grouped_experts.
 *   grad_x_disp [C, H] bf16 (out): written on the valid rows and the pad
 *     rows inside each expert's tiles (zeros there).
 *   dW1 [E, 2I, H], dW2 [E, H, I] fp32 (out): fully overwritten, fp32
 *     accumulation; an expert with no rows gets zeros.
 *   workspace: moe_experts_backward_workspace_bytes(capacity, H, I) bytes,
 *     caller-owned scratch.  On return it holds the backward GEMMs' bf16
 *     operands on the valid rows: G_o [C, H] from the workspace's first
 *     256-byte boundary, then [G_g | G_u] [C, 2I] from the next 256-byte
 *     boundary after C*H*2 bytes.
 * Row counts are read on the device: no host sync.  When pad_multiple is a
 * multiple of 64, the pad rows of x_disp, h and gu_save must be zero, as
 * moe_dispatch and moe_grouped_experts (with gu_save) leave them: the weight
 * gradients then read them instead of masking the last partial 64-row block
 * of each expert.
 */
MOE_API moe_status moe_experts_backward_workspace_bytes(int64_t capacity, int32_t H, int32_t I,
                                                        size_t* bytes);
MOE_API moe_status moe_grouped_experts_backward(const moe_bf16* grad_y, const moe_bf16* x_disp,
                                                const moe_bf16* h, const moe_bf16* gu_save,
                                                const moe_layout* L, int32_t H, int32_t I,
                                                const moe_bf16* W1, const moe_bf16* W2,
                                                moe_bf16* grad_x_disp, float* dW1, float* dW2,
                                                void* workspace, moe_stream_t stream);

/*
 * a9 from G_o: moe_grouped_experts_backward with g_o [C, H] bf16 (written by
 * moe_combine_backward_scaled) in place of grad_y; the routing weight is
 * already applied, so no scaling pass runs and the workspace's G_o region is
 * not written.  Arguments, outputs and errors otherwise as in
 * moe_grouped_experts_backward.
 */
MOE_API moe_status moe_grouped_experts_backward_scaled(const moe_bf16* g_o, const moe_bf16* x_disp,
                                                       const moe_bf16* h, const moe_bf16* gu_save,
                                                       const moe_layout* L, int32_t H, int32_t I,
                                                       const moe_bf16* W1, const moe_bf16* W2,
                                                       moe_bf16* grad_x_disp, float* dW1, float* dW2,
                                                       void* workspace, moe_stream_t stream);

/*
 * Failure-detection self-test.  Runs one CTA whose wait on an mbarrier can
 * never complete, using the bounded-wait helper of the pipelined kernels with
 * a limit of limit_ns (0 < limit_ns <= 1 s).  The wait gives up, the kernel
 * ORs MOE_DEVERR_TIMEOUT into *status (device) and, if waited_ns (device,
 * nullable) is given, stores how long it waited; then it returns normally.
 * Asynchronous on `stream`.
 */
MOE_API moe_status moe_selftest_wait_timeout(int32_t* status, int64_t limit_ns, uint64_t* waited_ns,
                                             moe_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MOE_GB300_H */
