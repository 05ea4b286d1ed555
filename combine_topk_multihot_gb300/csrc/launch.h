// Internal launchers (host side).  The public C ABI in moe.h validates the
// arguments and calls these; they only size grids and launch.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

int sm_count();  // SMs of the current device (cached)

// Launches `kernel` so that it may start while the previous kernel in the
// stream is still running (programmatic dependent launch); the kernel itself
// waits for that kernel's results with griddep_wait().
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// Tensor map of a row-major bf16 matrix [rows, cols] (cols contiguous) read as
// boxes of box_rows x 64 columns with the 128-byte swizzle; reads past the
// last row return zeros.  False if the driver entry point is missing or the
// encoding is rejected.
bool make_tma_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);

// The same for a row-major 8-bit matrix, read as boxes of box_rows x 128
// columns (128 bytes) with the 128-byte swizzle.
bool make_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

// Tensor maps whose boxes carry 128 columns of K as two 64-column sub-tiles
// (128-byte swizzle; sub-tile j follows sub-tile j - 1 in shared memory), so
// one TMA operation moves a whole 128-wide K step:
//   * the gate/up weights W1 [E, 2I, H] (bf16): 64 features x {gate, up} x
//     128 columns of one expert, interleaved -- sub-tile row 2j is gate row
//     f + j, row 2j + 1 up row f + j (H % 128 == 0);
//   * a row-major bf16 matrix [rows, cols]: box_rows rows x 128 columns
//     (cols % 128 == 0); reads past the last row return zeros.
bool make_tma_w1_gate_up_k128(CUtensorMap* map, const void* W1, uint64_t E, uint64_t I, uint64_t H);
bool make_tma_rows_k128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Tensor map for TMA stores of 32-row x 32-column bf16 boxes (64-byte rows)
// into a row-major [rows, cols] matrix.  The shared-memory box is 64-byte
// swizzled: the 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
// (see staged_chunk), so a warp writing one row per lane spreads over all
// shared-memory banks.
bool make_tma_store_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);
// The same for 32-row x 16-column bf16 boxes (32-byte rows, no swizzle).
bool make_tma_store_2d_bf16_16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);
// The same for fp32: 32-row x 16-column boxes (64-byte rows).
bool make_tma_store_2d_f32(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols);

// Unique id of the calling thread's current CUDA context; false when there is
// none yet or the driver does not say.  The device addresses of the library's
// static arrays are cached per device and looked up again when it changes
// (a device reset loads the module into a new context).
bool current_context_id(unsigned long long* id);

// Records `text` as this thread's moe_last_error() and returns `st`.
moe_status set_last_error(moe_status st, const char* text);

// Tokens per chunk of the layout's histogram / placement passes.
constexpr int LAYOUT_CHUNK = 32;

inline int64_t layout_chunks(int32_t T) { return (T + LAYOUT_CHUNK - 1) / LAYOUT_CHUNK; }

cudaError_t launch_multihot(const int64_t* topk_idx, const float* topk_probs, int T, int K, int E,
                            uint8_t* routing_map, float* probs, int8_t* winner, int* status,
                            cudaStream_t s);
// Router: softmax -> top-K -> renormalise per token; with routing_map also
// the multihot outputs (probs and winner then non-NULL too).
cudaError_t launch_router_topk(const float* logits, int T, int K, int E, int64_t* topk_idx,
                               float* topk_probs, uint8_t* routing_map, float* probs,
                               int8_t* winner, cudaStream_t s);
cudaError_t launch_router_topk_backward(const float* grad_w, const float* w,
                                        const int64_t* topk_idx, int T, int K, int E,
                                        float* grad_logits, cudaStream_t s);
cudaError_t launch_multihot_backward(const float* grad_probs, const int64_t* topk_idx,
                                     const int8_t* winner, int T, int K, int E, float* grad_topk,
                                     cudaStream_t s);

// Bytes of per-chunk expert counters at the start of the layout workspace
// (E * chunks int32, rounded up to 256); the grid barrier's counter follows.
inline size_t layout_counter_bytes(int32_t T, int32_t E) {
  const size_t b = static_cast<size_t>(layout_chunks(T)) * E * sizeof(int32_t);
  return (b + 255) / 256 * 256;
}

// Counts, padded offsets and the stable placement of every (token, expert)
// pair, in one launch.  workspace: layout_counter_bytes(T, E) + 256 bytes.
// Placement is skipped when the rows do not fit (R > capacity); the status
// word then has MOE_DEVERR_CAPACITY.
// readback (may be NULL): device address of 3 ints of host-mapped memory
// that receive N and the status word, then R (written last, after a system
// fence), as soon as the offsets are known.
// rows_done (may be NULL): when the layout runs as one CTA and the
// dispatch's row pass is small, that CTA also does the row pass (x -> x_disp,
// or only the pad and spare rows' metadata when x_disp is NULL) and sets
// *rows_done; otherwise *rows_done is false and the caller runs the row pass.
cudaError_t launch_layout(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                          void* workspace, cudaStream_t s, int* readback = nullptr,
                          const uint16_t* x = nullptr, uint16_t* x_disp = nullptr, int H = 0,
                          bool* rows_done = nullptr);
// Workspace of the dispatch (moe_layout.workspace): per (expert, chunk) a
// token mask and a start row, then the fused kernel's grid-barrier words,
// then 8 copies of the per-expert counts.
constexpr size_t FUSED_BARRIER_BYTES = 1280;
inline size_t dispatch_workspace_bytes(int32_t T, int32_t E) {
  const size_t rep = (static_cast<size_t>(8) * E * sizeof(int32_t) + 255) / 256 * 256;
  return 2 * layout_counter_bytes(T, E) + FUSED_BARRIER_BYTES + rep;
}

// a1-a4 in one cooperative launch for layers of more than 8 chunks: counts,
// offsets, placement, the pad and spare rows, and (x_disp non-NULL) the row
// copies.  Input the multihot map (_map) or the top-k choices (_topk, which
// also writes routing_map / probs / winner).  workspace: L.workspace, which
// holds dispatch_workspace_bytes(T, E).  readback as in launch_layout.
bool dispatch_fused_fits(const moe_layout& L);
cudaError_t launch_dispatch_fused_map(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                                      int H, const uint16_t* x, uint16_t* x_disp, int* readback,
                                      cudaStream_t s);
// The same from a multihot map, with the rows as e4m3 codes and one fp32
// scale per row (x_q [capacity, H], x_scale [capacity]).
cudaError_t launch_dispatch_fused_map_fp8(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                                          int H, const uint16_t* x, uint8_t* x_q, float* x_scale, int* readback,
                                          cudaStream_t s);
cudaError_t launch_dispatch_fused_topk(const int64_t* topk_idx, const float* topk_probs,
                                       uint8_t* routing_map, float* probs, int8_t* winner,
                                       const moe_layout& L, int H, const uint16_t* x, uint16_t* x_disp,
                                       int* readback, cudaStream_t s);
cudaError_t launch_dispatch_fused_topk_fp8(const int64_t* topk_idx, const float* topk_probs,
                                           uint8_t* routing_map, float* probs, int8_t* winner,
                                           const moe_layout& L, int H, const uint16_t* x, uint8_t* x_q,
                                           float* x_scale, int* readback, cudaStream_t s);
// Rows of the expanded layout from token rows (a4: x -> x_disp, plus the pad /
// spare rows' metadata when from_offsets); also the combine backward (a7)
// with the optional routing-weight gradient (a8).  Each token row is read
// once and scattered to the token's rows; pad / spare rows are zeroed.
// With scale (combine backward only) each row gets bf16(row_weight * src).
cudaError_t launch_row_gather(const uint16_t* src, const moe_layout& L, int H, uint16_t* dst,
                              bool write_row_meta, const uint16_t* o_save, float* grad_w,
                              cudaStream_t s, bool scale = false);
// Per-token ordered sum of rows (a6 / a10), optional grad_probs scatter.
cudaError_t launch_combine(const uint16_t* rows, const moe_layout& L, int H, uint16_t* out,
                           const float* grad_w, float* grad_probs, cudaStream_t s);

// tcgen05 grouped GEMMs of the experts (a5).
cudaError_t launch_experts_forward(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                   const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                   uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                   cudaStream_t s);

// a5 (bf16) on CTA pairs with each expert's rows on the MMA's N side, for
// layers with rows for every SM: the accumulator is W[e] x_disp^T, tiles of
// 256 weight rows by up to 256 expert rows in multiples of 16.
cudaError_t launch_experts_forward_pair(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                        const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                        uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                        cudaStream_t s);

// a5 on the CUDA cores for layers with at most 4 rows per expert (T <= 4)
// and nothing saved for a backward: weight streaming with warp dot products.
bool gemv_experts_fits(const moe_layout& L, int H, int I, bool saves);
// With gather, x_disp is the tokens x and row r of A is x[row_token[r]].
cudaError_t launch_experts_forward_gemv(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                        const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                        uint16_t* y, cudaStream_t s, bool gather = false);
// a4 fused into a5: GEMM1's producer gathers the A rows from x by row_token
// (zero rows for pad and spare rows); no x_disp is written or read.
cudaError_t launch_experts_forward_gather(const uint16_t* x, const moe_layout& L, int H, int I,
                                          const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                          uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                          cudaStream_t s);

// FP8: a4 with e4m3 rows (one fp32 scale per row; pad and spare rows zero
// codes, scale 0, sentinel metadata), and rowwise e4m3 quantization of a
// bf16 matrix (cols % 256 == 0).
cudaError_t launch_row_gather_fp8(const uint16_t* x, const moe_layout& L, int H, uint8_t* x_q,
                                  float* x_scale, cudaStream_t s);
cudaError_t launch_quantize_rows_fp8(const uint16_t* src, long long rows, int cols, uint8_t* codes,
                                     float* scales, cudaStream_t s);
// a5 with the gate/up GEMM on e4m3 operands (scales applied in its epilogue);
// the down projection stays bf16.
cudaError_t launch_experts_forward_fp8(const uint8_t* x_q, const float* x_scale,
                                       const moe_layout& L, int H, int I, const uint8_t* W1_q,
                                       const float* W1_scale, const uint16_t* W2, uint16_t* h,
                                       uint16_t* y, cudaStream_t s);

// tcgen05 grouped GEMMs of the expert backward (a9); workspace holds G_o [C, H]
// and G_gu [C, 2I] (bf16).
size_t experts_backward_workspace(long long capacity, int H, int I);
cudaError_t launch_experts_backward(const uint16_t* grad_y, const uint16_t* x_disp,
                                    const uint16_t* h, const uint16_t* gu_save, const moe_layout& L,
                                    int H, int I, const uint16_t* W1, const uint16_t* W2,
                                    uint16_t* grad_x_disp, float* dW1, float* dW2, void* workspace,
                                    cudaStream_t s, bool g_o_given = false);

}  // namespace moe
