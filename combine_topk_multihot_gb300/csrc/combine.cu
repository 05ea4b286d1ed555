// a6 / a10: combine -- each token's rows summed back into place, no weights.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds, Expanded layout: the routing weights are applied
// inside the experts, so the combine is a plain sum.  It runs in fp32 from +0.0 over
// the token's rows in ascending expert order (token_row order), with one
// rounding to bf16 at the end, so the result is independent of scheduling.
// Training: the dispatch's backward is this same sum on the gradient rows;
// the routing-weight gradient of each row is scattered to grad_probs[t, e].

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

template <int KW>
__device__ __forceinline__ int pick4(const int (&a)[KW], int j) {
  if constexpr (KW == 1) return a[0];
  else return j == 0 ? a[0] : j == 1 ? a[1] : j == 2 ? a[2] : a[3];
}

__device__ __forceinline__ void acc_add(float (&acc)[8], const uint4& v) {
  acc[0] += bf16_lo(v.x);
  acc[1] += bf16_hi(v.x);
  acc[2] += bf16_lo(v.y);
  acc[3] += bf16_hi(v.y);
  acc[4] += bf16_lo(v.z);
  acc[5] += bf16_hi(v.z);
  acc[6] += bf16_lo(v.w);
  acc[7] += bf16_hi(v.w);
}

__device__ __forceinline__ uint4 acc_pack(const float (&acc)[8]) {
  return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                    pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

// One warp per (token, 512-byte column chunk): lane l sums the 16-byte vector
// at column chunk v of each of the token's rows.  All of the token's rows
// (up to 8 at a time) are loaded before they are added, in row order, so an
// item costs one memory round trip; T * H/256 items keep every SM busy even
// at small T.  With SCATTER, the warp of chunk 0 also writes the token's
// grad_probs row.  KW: 32-slot words of a token's row list (1 for K <= 32,
// else 4).
template <bool SCATTER, int KW>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const int* __restrict__ token_row, int T,
                                                      int K, int H, uint16_t* __restrict__ out,
                                                      const int* __restrict__ row_expert,
                                                      const float* __restrict__ grad_w,
                                                      float* __restrict__ grad_probs, int E,
                                                      long long C, int* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;  // 512-byte chunks per row
  const long long items = static_cast<long long>(T) * V;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  // The token_row entries of the warp's next item are loaded while the
  // current item's rows are, so that an item costs one memory round trip
  // rather than two (its row list, then its rows).
  auto load_rows_of = [&](long long item, int (&dst)[KW]) {
    const long long tt = item / V;
#pragma unroll
    for (int jj = 0; jj < KW; ++jj) {
      const int k = lane + 32 * jj;
      dst[jj] = item < items && k < K ? __ldg(token_row + tt * K + k) : -1;
    }
  };
  long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int tr_next[KW];
  load_rows_of(it, tr_next);
  for (; it < items; it += nwarps) {
    const long long t = it / V;
    const int v = static_cast<int>(it - t * V);
    int tr[KW];
    int n = 0;
#pragma unroll
    for (int jj = 0; jj < KW; ++jj) {
      tr[jj] = tr_next[jj];
      if (!MOE_IN_BOUNDS(tr[jj] < C, status)) tr[jj] = -1;
      n += __popc(__ballot_sync(FULL_MASK, tr[jj] >= 0));
    }
    load_rows_of(it + nwarps, tr_next);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < n; j0 += 8) {
      uint4 b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + i;
        const int r = __shfl_sync(FULL_MASK, pick4<KW>(tr, j >> 5), j & 31);
        if (j < n)
          b[i] = __ldg(reinterpret_cast<const uint4*>(rows + static_cast<long long>(r) * H) + lane + 32 * v);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (j0 + i < n) acc_add(acc, b[i]);
    }
    reinterpret_cast<uint4*>(out + t * H)[lane + 32 * v] = acc_pack(acc);
    if (SCATTER && grad_probs && v == 0) {
      float* gp = grad_probs + t * E;
      for (int e = lane * 4; e < E; e += 128)
        *reinterpret_cast<float4*>(gp + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      __syncwarp();
#pragma unroll
      for (int jj = 0; jj < KW; ++jj) {
        const int r = tr[jj];
        if (r >= 0 && MOE_IN_BOUNDS(row_expert[r] >= 0 && row_expert[r] < E, status))
          gp[row_expert[r]] = grad_w ? grad_w[r] : 0.f;
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* rows, const moe_layout& L, int H, uint16_t* out,
                           const float* grad_w, float* grad_probs, cudaStream_t s) {
  if (L.T == 0) return cudaSuccess;
  const int threads = 256;
  const long long items = static_cast<long long>(L.T) * (H >> 8);
  const long long need = (items + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  const long long C = static_cast<long long>(L.capacity);
  if (grad_probs) {
    if (L.K <= 32)
      combine_kernel<true, 1><<<blocks, threads, 0, s>>>(rows, L.token_row, L.T, L.K, H, out, L.row_expert, grad_w,
                                                         grad_probs, L.E, C, L.status);
    else
      combine_kernel<true, 4><<<blocks, threads, 0, s>>>(rows, L.token_row, L.T, L.K, H, out, L.row_expert, grad_w,
                                                         grad_probs, L.E, C, L.status);
    return cudaGetLastError();
  }
  const int* no_expert = nullptr;
  const float* no_grad_w = nullptr;
  float* no_grad_probs = nullptr;
  if (L.K <= 32)
    return launch_dependent(combine_kernel<false, 1>, blocks, threads, 0, s, rows, L.token_row, L.T, L.K, H, out,
                            no_expert, no_grad_w, no_grad_probs, L.E, C, L.status);
  return launch_dependent(combine_kernel<false, 4>, blocks, threads, 0, s, rows, L.token_row, L.T, L.K, H, out,
                          no_expert, no_grad_w, no_grad_probs, L.E, C, L.status);
}

}  // namespace moe
