// a1: top-k -> multihot routing map, and its backward; and the router in
// front of it (logits -> top-k), alone or fused with the multihot.
//
// "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)", Changelog: the HybridEP
// preprocessing turns top-k indices into multihot routing metadata (a
// routing_map and per-(token, expert) probs); review of dispatch(): the probs
// are fp32.  Duplicated expert indices inside one token are set once, the
// last slot's prob winning (slots are taken in order).

#include "common.cuh"
#include "coop.cuh"
#include "launch.h"

namespace moe {

namespace {

// One warp per token: the K slot indices are loaded by the lanes and the row
// is written by write_multihot_row.
__global__ void __launch_bounds__(256) multihot_kernel(const int64_t* __restrict__ topk_idx,
                                                       const float* __restrict__ topk_probs,
                                                       int T, int K, int E,
                                                       uint8_t* __restrict__ routing_map,
                                                       float* __restrict__ probs,
                                                       int8_t* __restrict__ winner,
                                                       int* __restrict__ status) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_block;
  for (long long t = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
       t < T; t += nwarps) {
    int ek[4];
    float pk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = lane + 32 * j;
      ek[j] = -1;
      pk[j] = 0.f;
      if (k < K) {
        long long v = topk_idx[t * K + k];
        if (v < -1 || v >= E) {
          report(status, MOE_DEVERR_BAD_INDEX);
          v = -1;
        }
        ek[j] = static_cast<int>(v);
        pk[j] = topk_probs[t * K + k];
      }
    }
    write_multihot_row(t, ek, pk, K, E, lane, routing_map, probs, winner);
  }
}

// The router in front of the path: softmax over the E logits, the K most
// probable experts, their probabilities renormalised to sum to one.  The
// softmax's normaliser cancels in the renormalisation, so the weights are the
// softmax of the K chosen logits alone: w_k = exp(l_k - l_0) / sum_j
// exp(l_j - l_0), l_0 the largest.
// One warp per token.  Lane l holds logits l, l + 32, ... (up to 32 in
// registers); K rounds of a warp argmax pick the experts in descending order,
// equal logits by ascending index (a NaN logit counts as -inf).  Slot k lands
// in lane k % 32, register k / 32, which is the layout write_multihot_row
// takes, so with MULTIHOT the same warp also writes the token's multihot row.
template <bool MULTIHOT>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int K, int E,
                                                          int64_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_probs,
                                                          uint8_t* __restrict__ routing_map,
                                                          float* __restrict__ probs,
                                                          int8_t* __restrict__ winner) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_block;
  const int J = (E + 31) >> 5;  // logits per lane
  for (long long t = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
       t < T; t += nwarps) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = lane + 32 * j;
      float x = -INFINITY;
      if (j < J && e < E) {
        x = logits[t * E + e];
        if (x != x) x = -INFINITY;
      }
      v[j] = x;
    }
    uint32_t taken = 0;
    int ek[4] = {-1, -1, -1, -1};
    float lk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int k = 0; k < K; ++k) {
      // this lane's best untaken logit
      float bv = -INFINITY;
      int bj = -1;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < J && !((taken >> j) & 1u) && (bj < 0 || v[j] > bv)) {
          bv = v[j];
          bj = j;
        }
      }
      int be = bj >= 0 ? lane + 32 * bj : 0x7fffffff;
      if (bj >= 0 && be >= E) be = 0x7fffffff;  // padding slots never win
      // warp argmax: larger value, then smaller expert index
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, bv, o);
        const int oe = __shfl_xor_sync(FULL_MASK, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane && be < E) taken |= 1u << (be >> 5);
      if ((k & 31) == lane) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if ((k >> 5) == j) {
            ek[j] = be;
            lk[j] = bv;
          }
        }
      }
    }
    // weights: softmax of the chosen logits, relative to the largest (slot 0)
    const float l0 = __shfl_sync(FULL_MASK, lk[0], 0);
    float ex[4], part = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ex[j] = (lane + 32 * j < K) ? expf(lk[j] - l0) : 0.f;
      part += ex[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL_MASK, part, o);
    float pk[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = lane + 32 * j;
      pk[j] = ex[j] / part;
      if (k < K) {
        topk_idx[t * K + k] = ek[j];
        topk_probs[t * K + k] = pk[j];
      }
    }
    if (MULTIHOT) write_multihot_row(t, ek, pk, K, E, lane, routing_map, probs, winner);
  }
}

// dL/dlogits for the router: w_j (g_j - sum_k w_k g_k) at the chosen experts,
// zero elsewhere.  One warp per token: the row is zeroed with 16-byte stores,
// then the K values are written.
__global__ void __launch_bounds__(256) router_topk_backward_kernel(
    const float* __restrict__ grad_w, const float* __restrict__ w,
    const int64_t* __restrict__ topk_idx, int T, int K, int E, float* __restrict__ grad_logits) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_block;
  for (long long t = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
       t < T; t += nwarps) {
    float gk[4], wk[4], dot = 0.f;
    int ek[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = lane + 32 * j;
      gk[j] = k < K ? grad_w[t * K + k] : 0.f;
      wk[j] = k < K ? w[t * K + k] : 0.f;
      ek[j] = k < K ? static_cast<int>(topk_idx[t * K + k]) : -1;
      dot = fmaf(wk[j], gk[j], dot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(FULL_MASK, dot, o);
    float4* row = reinterpret_cast<float4*>(grad_logits + t * E);
    for (int i = lane; i < (E >> 2); i += 32) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (ek[j] >= 0 && ek[j] < E) grad_logits[t * E + ek[j]] = wk[j] * (gk[j] - dot);
  }
}

// grad_topk[t, k] = grad_probs[t, e] if slot k is valid and set the pair (t, e).
__global__ void multihot_backward_kernel(const float* __restrict__ grad_probs,
                                         const int64_t* __restrict__ topk_idx,
                                         const int8_t* __restrict__ winner, int T, int K, int E,
                                         float* __restrict__ grad_topk) {
  const long long n = static_cast<long long>(T) * K;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / K;
    const int k = static_cast<int>(i - t * K);
    const long long e = topk_idx[i];
    float g = 0.f;
    if (e >= 0 && e < E && winner[t * E + e] == k) g = grad_probs[t * E + e];
    grad_topk[i] = g;
  }
}

}  // namespace

cudaError_t launch_multihot(const int64_t* topk_idx, const float* topk_probs, int T, int K, int E,
                            uint8_t* routing_map, float* probs, int8_t* winner, int* status,
                            cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks_needed = (static_cast<long long>(T) + 7) / 8;
  const int blocks = static_cast<int>(blocks_needed < 8LL * sm_count() ? blocks_needed : 8LL * sm_count());
  return launch_dependent(multihot_kernel, blocks, threads, 0, s, topk_idx, topk_probs, T, K, E,
                          routing_map, probs, winner, status);
}

cudaError_t launch_router_topk(const float* logits, int T, int K, int E, int64_t* topk_idx,
                               float* topk_probs, uint8_t* routing_map, float* probs,
                               int8_t* winner, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks_needed = (static_cast<long long>(T) + 7) / 8;
  const int blocks = static_cast<int>(blocks_needed < 8LL * sm_count() ? blocks_needed : 8LL * sm_count());
  if (routing_map)
    return launch_dependent(router_topk_kernel<true>, blocks, threads, 0, s, logits, T, K, E,
                            topk_idx, topk_probs, routing_map, probs, winner);
  return launch_dependent(router_topk_kernel<false>, blocks, threads, 0, s, logits, T, K, E, topk_idx,
                          topk_probs, static_cast<uint8_t*>(nullptr), static_cast<float*>(nullptr),
                          static_cast<int8_t*>(nullptr));
}

cudaError_t launch_router_topk_backward(const float* grad_w, const float* w,
                                        const int64_t* topk_idx, int T, int K, int E,
                                        float* grad_logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks_needed = (static_cast<long long>(T) + 7) / 8;
  const int blocks = static_cast<int>(blocks_needed < 8LL * sm_count() ? blocks_needed : 8LL * sm_count());
  router_topk_backward_kernel<<<blocks, threads, 0, s>>>(grad_w, w, topk_idx, T, K, E, grad_logits);
  return cudaGetLastError();
}

cudaError_t launch_multihot_backward(const float* grad_probs, const int64_t* topk_idx,
                                     const int8_t* winner, int T, int K, int E, float* grad_topk,
                                     cudaStream_t s) {
  const long long n = static_cast<long long>(T) * K;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  multihot_backward_kernel<<<blocks, threads, 0, s>>>(grad_probs, topk_idx, winner, T, K, E,
                                                      grad_topk);
  return cudaGetLastError();
}

}  // namespace moe
