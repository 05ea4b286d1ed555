// a5 for decode-sized layers: the SwiGLU experts on the CUDA cores.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)": Expanded layout -- an expert computes only its own rows and the
// routing weight scales each row's output inside the expert step; Benchmarks
// -- decode runs one to a few hundred tokens per step.
//
// With at most four rows per expert (T <= 4: a token names an expert at
// most once), the expert step reads each weight once and does at most four
// FMAs with it, so it is a stream over the active experts' weights.  A
// 128-row tensor-core tile would carry 124 empty rows and, with only a few
// experts active, too few tiles to keep every SM streaming.  Here the work is
// (active expert, column slice) items spread over a grid of up to 8 CTAs per
// SM (4 resident at a time; the CTAs loop when there are more items):
//   step 1: 8 h columns = 8 gate + 8 up rows of W1, h = bf16(silu(g) * u);
//   step 2: 32 y columns = 32 rows of W2, y = bf16(w_row * o).
// A warp takes 2 (step 1: gate and up) or 4 (step 2) weight rows and issues
// their 16-byte loads together, multiplies them by the expert's rows (held in
// shared memory) and reduces with shuffles.  Accumulation is fp32; h is rounded to bf16 between the steps, as
// in the tensor-core path.

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int GEMV_ROWS = 4;       // rows per expert this path takes
constexpr int GEMV_THREADS = 256;  // 8 warps
// Four CTAs per SM (64 registers a thread): with 2.5 waves of 2 CTAs per SM
// before, each wave paid the list, A-row and weight round trips again.  A
// warp now loads 4 (gate/up) or 2 (down) 16-byte vectors per lane and row in
// one round instead of 8 or 4: decode T = 1, the two kernels under graph
// replay went from 24.3 to 21.8 us.
constexpr int GEMV_CTAS_PER_SM = 4;
constexpr int S1_COLS = 8;         // h columns per step-1 item (1 per warp)
constexpr int S2_COLS = 32;        // y columns per step-2 item (4 per warp)

struct GemvArgs {
  const int* counts;       // [E]
  const int* offsets;      // [E + 1]
  const float* row_weight; // [C]
  int E, H, I;
  const uint16_t* a;       // step 1: x_disp [C, H] (or x [T, H], see row_token); step 2: h [C, I]
  const int* row_token;    // step 1 with the dispatch fused: row r of A is x[row_token[r]]
  const uint16_t* w;       // step 1: W1 [E, 2I, H]; step 2: W2 [E, H, I]
  uint16_t* out;           // step 1: h [C, I];      step 2: y [C, H]
};

// acc[w][r] = sum_k a[r, k] * W[w][k] for NR weight rows W[w] = wbase + w *
// wstride and the n (<= 4) rows of a in shared memory (K bf16 each, K % 8 ==
// 0); lane-partial sums reduced over the warp.  Lane l takes the 16-byte
// vectors l, l + 32, ... of a row; each chunk issues the loads of all NR rows
// (CH vectors each) before using them, so a short row costs one round trip.
template <int NR, int CH>
__device__ __forceinline__ void warp_dot(const uint16_t* __restrict__ wbase, long long wstride,
                                         const uint4* s_a, int K, int n, int lane,
                                         float (&acc)[NR][GEMV_ROWS]) {
#pragma unroll
  for (int w = 0; w < NR; ++w)
#pragma unroll
    for (int r = 0; r < GEMV_ROWS; ++r) acc[w][r] = 0.f;
  const int NV = K >> 3;  // 16-byte vectors per row
  for (int q0 = 0; q0 < NV; q0 += CH * 32) {
    uint4 wv[NR][CH];
#pragma unroll
    for (int w = 0; w < NR; ++w) {
      const uint4* w4 = reinterpret_cast<const uint4*>(wbase + w * wstride);
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int q = q0 + lane + 32 * i;
        if (q < NV) wv[w][i] = __ldg(w4 + q);
      }
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int q = q0 + lane + 32 * i;
      if (q >= NV) continue;
#pragma unroll
      for (int r = 0; r < GEMV_ROWS; ++r) {
        if (r >= n) continue;
        const uint4 av = s_a[r * NV + q];
        const uint32_t aq[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int w = 0; w < NR; ++w) {
          const uint32_t wq[4] = {wv[w][i].x, wv[w][i].y, wv[w][i].z, wv[w][i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[w][r] = fmaf(bf16_lo(aq[k]), bf16_lo(wq[k]), acc[w][r]);
            acc[w][r] = fmaf(bf16_hi(aq[k]), bf16_hi(wq[k]), acc[w][r]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int w = 0; w < NR; ++w)
#pragma unroll
    for (int r = 0; r < GEMV_ROWS; ++r)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[w][r] += __shfl_xor_sync(FULL_MASK, acc[w][r], o);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int STEP>
__global__ void __launch_bounds__(GEMV_THREADS, GEMV_CTAS_PER_SM) gemv_experts_kernel(GemvArgs args) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = STEP == 1 ? args.H : args.I;
  uint4* s_a = reinterpret_cast<uint4*>(smem);                                  // [4][K] bf16
  int* s_list = reinterpret_cast<int*>(smem + GEMV_ROWS * K * 2);               // [E]
  __shared__ int s_nact;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = args.E;
  // the experts with rows, in ascending order
  if (warp == 0) {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool act = e < E && args.counts[e] > 0;
      const uint32_t m = __ballot_sync(FULL_MASK, act);
      if (act) s_list[base + __popc(m & ((1u << lane) - 1u))] = e;
      base += __popc(m);
    }
    if (lane == 0) s_nact = base;
  }
  __syncthreads();
  const int slices = STEP == 1 ? args.I / S1_COLS : args.H / S2_COLS;
  const int items = s_nact * slices;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int e = s_list[it / slices];
    const int j = it - (it / slices) * slices;
    const int n = min(args.counts[e], GEMV_ROWS);
    const long long r0 = args.offsets[e];
    // the expert's rows of A into shared memory
    const int NV = K >> 3;
    for (int i = threadIdx.x; i < n * NV; i += GEMV_THREADS) {
      const int r = i / NV;
      const long long src_row = args.row_token ? __ldg(args.row_token + r0 + r) : r0 + r;
      s_a[i] = __ldg(reinterpret_cast<const uint4*>(args.a + src_row * K) + (i - r * NV));
    }
    __syncthreads();
    if (STEP == 1) {
      // warp: h column c -> W1 rows c (gate) and I + c (up), in one pass
      const int c = j * S1_COLS + warp;
      const uint16_t* w1 = args.w + static_cast<long long>(e) * 2 * args.I * K;
      float gu[2][GEMV_ROWS];
      warp_dot<2, 4>(w1 + static_cast<long long>(c) * K, static_cast<long long>(args.I) * K, s_a, K, n,
                     lane, gu);
      if (lane < n) {
        float gv = gu[0][0], uv = gu[1][0];
#pragma unroll
        for (int r = 1; r < GEMV_ROWS; ++r)
          if (lane == r) {
            gv = gu[0][r];
            uv = gu[1][r];
          }
        const float hv = gv / (1.0f + __expf(-gv)) * uv;
        args.out[(r0 + lane) * args.I + c] = to_bf16_bits(hv);
      }
    } else {
      // warp: y columns c0 .. c0 + 3 -> W2 rows c0 .. c0 + 3, in one pass
      const int c0 = j * S2_COLS + warp * 4;
      const uint16_t* w2 = args.w + static_cast<long long>(e) * args.H * K;
      float o[4][GEMV_ROWS];
      warp_dot<4, 2>(w2 + static_cast<long long>(c0) * K, K, s_a, K, n, lane, o);
      if (lane < n) {
        const float wgt = args.row_weight[r0 + lane];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float ov = o[cc][0];
#pragma unroll
          for (int r = 1; r < GEMV_ROWS; ++r)
            if (lane == r) ov = o[cc][r];
          args.out[(r0 + lane) * args.H + c0 + cc] = to_bf16_bits(wgt * ov);
        }
      }
    }
    __syncthreads();  // before the next item overwrites s_a
  }
}

}  // namespace

bool gemv_experts_fits(const moe_layout& L, int H, int I, bool saves) {
  // the expert's rows of A and the active-expert list in 48 KiB of shared memory
  const size_t smem = static_cast<size_t>(GEMV_ROWS) * (H > I ? H : I) * 2 +
                      static_cast<size_t>(L.E) * sizeof(int);
  return !saves && L.T <= GEMV_ROWS && I % S1_COLS == 0 && H % S2_COLS == 0 && smem <= 48 * 1024;
}

cudaError_t launch_experts_forward_gemv(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                        const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                        uint16_t* y, cudaStream_t s, bool gather) {
  GemvArgs a{};
  a.counts = L.tokens_per_expert;
  a.offsets = L.offsets;
  a.row_weight = L.row_weight;
  a.E = L.E;
  a.H = H;
  a.I = I;
  // at most min(E, T*K) experts have rows
  const long long pairs = static_cast<long long>(L.T) * L.K;
  const long long active = pairs < L.E ? pairs : L.E;
  const long long cap = 8LL * sm_count();
  a.a = x_disp;
  a.row_token = gather ? L.row_token : nullptr;
  a.w = W1;
  a.out = h;
  long long items = active * (I / S1_COLS);
  int grid = static_cast<int>(items < cap ? (items > 0 ? items : 1) : cap);
  size_t smem = static_cast<size_t>(GEMV_ROWS) * H * 2 + static_cast<size_t>(L.E) * sizeof(int);
  cudaError_t err = launch_dependent(gemv_experts_kernel<1>, grid, GEMV_THREADS, smem, s, a);
  if (err != cudaSuccess) return err;
  a.a = h;
  a.row_token = nullptr;
  a.w = W2;
  a.out = y;
  items = active * (H / S2_COLS);
  grid = static_cast<int>(items < cap ? (items > 0 ? items : 1) : cap);
  smem = static_cast<size_t>(GEMV_ROWS) * I * 2 + static_cast<size_t>(L.E) * sizeof(int);
  return launch_dependent(gemv_experts_kernel<2>, grid, GEMV_THREADS, smem, s, a);
}

}  // namespace moe
