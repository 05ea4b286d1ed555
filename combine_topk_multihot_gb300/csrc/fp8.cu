// FP8 dispatch (a4 with e4m3 rows) and rowwise e4m3 quantization.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds, scope note: FP8 dispatch -- half the dispatch bytes
// for FP8 recipes -- is the named follow-up.  Format: e4m3 values with one
// fp32 scale per row, scale = amax(|row|) / 448 (1 for an all-zero row), code
// = e4m3(v / scale) rounded to nearest even and saturated at +-448.  The
// division is an IEEE fp32 division, so a code is the same on any machine.
//
// A warp owns a row of H values: lane l holds the 8-value vectors l, l + 32,
// ...  A first pass finds the row's amax (warp max), a second re-reads the
// row (now in L1), converts it and stores 8 codes per vector.

#include "common.cuh"
#include "fp8_quant.cuh"
#include "launch.h"

namespace moe {

namespace {

// a4 in e4m3.  Items [0, T): tokens -- the token's row is quantized once and
// its codes and scale written to each of its rows.  Items [T, T + C): rows --
// a pad or spare row (found from offsets and counts) gets zero codes, scale
// 0 and the sentinel metadata (token -1, expert E, weight 0).
__global__ void __launch_bounds__(256) row_scatter_fp8_kernel(
    const uint16_t* __restrict__ x, int T, int K, int H, int E, long long C,
    const int* __restrict__ token_row, const int* __restrict__ offsets,
    const int* __restrict__ counts, int* __restrict__ row_token, int* __restrict__ row_expert,
    float* __restrict__ row_weight, uint8_t* __restrict__ x_q, float* __restrict__ x_scale) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int s_meta[];  // offsets [E + 1], counts [E]
  int* s_off = s_meta;
  int* s_cnt = s_meta + E + 1;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = counts[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;
  const long long items = T + C;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int R = s_off[E];
  if (R > C) return;  // the layout placed nothing: the rows do not fit
  for (long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += nwarps) {
    if (it < T) {
      const long long t = it;
      const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
      const float scale = row_scale(src, V, lane);
      for (int j0 = 0; j0 < K; j0 += 32) {
        const int r_ld = j0 + lane < K ? __ldcg(token_row + t * K + j0 + lane) : -1;
        const int r_lane = r_ld < C ? r_ld : -1;
        const uint32_t rows = __ballot_sync(FULL_MASK, r_lane >= 0);
        if (r_lane >= 0) x_scale[r_lane] = scale;
        for (int v = 0; v < V; ++v) {
          const uint2 c = quantize8(__ldg(src + lane + 32 * v), scale);
          for (uint32_t m = rows; m; m &= m - 1u) {
            const int r = __shfl_sync(FULL_MASK, r_lane, __ffs(m) - 1);
            reinterpret_cast<uint2*>(x_q + static_cast<long long>(r) * H)[lane + 32 * v] = c;
          }
        }
      }
    } else {
      const long long r = it - T;
      bool pad = true;
      if (r < R) {
        int lo = 0, hi = E;  // s_off[lo] <= r < s_off[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_off[mid] <= r) lo = mid; else hi = mid;
        }
        pad = r - s_off[lo] >= s_cnt[lo];
      }
      if (!pad) continue;
      if (lane == 0) {
        row_token[r] = -1;
        row_expert[r] = E;
        row_weight[r] = 0.f;
        x_scale[r] = 0.f;
      }
      uint2* d = reinterpret_cast<uint2*>(x_q + r * H);
      for (int v = 0; v < V; ++v) d[lane + 32 * v] = make_uint2(0, 0);
    }
  }
}

// Rowwise e4m3 of a bf16 matrix [rows, cols], one warp per row.
__global__ void __launch_bounds__(256) quantize_rows_fp8_kernel(const uint16_t* __restrict__ src,
                                                                long long rows, int cols,
                                                                uint8_t* __restrict__ codes,
                                                                float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int V = cols >> 8;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += nwarps) {
    const uint4* s = reinterpret_cast<const uint4*>(src + r * cols);
    const float scale = row_scale(s, V, lane);
    uint2* d = reinterpret_cast<uint2*>(codes + r * cols);
    for (int v = 0; v < V; ++v) d[lane + 32 * v] = quantize8(__ldg(s + lane + 32 * v), scale);
    if (lane == 0) scales[r] = scale;
  }
}

}  // namespace

cudaError_t launch_row_gather_fp8(const uint16_t* x, const moe_layout& L, int H, uint8_t* x_q,
                                  float* x_scale, cudaStream_t s) {
  const long long C = L.capacity;
  const long long items = static_cast<long long>(L.T) + C;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (items + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  const size_t smem = (2 * L.E + 1) * sizeof(int);
  return launch_dependent(row_scatter_fp8_kernel, blocks, threads, smem, s, x, L.T, L.K, H, L.E, C,
                          L.token_row, L.offsets, L.tokens_per_expert, L.row_token, L.row_expert,
                          L.row_weight, x_q, x_scale);
}

cudaError_t launch_quantize_rows_fp8(const uint16_t* src, long long rows, int cols, uint8_t* codes,
                                     float* scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (rows + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  quantize_rows_fp8_kernel<<<blocks, threads, 0, s>>>(src, rows, cols, codes, scales);
  return cudaGetLastError();
}

}  // namespace moe
