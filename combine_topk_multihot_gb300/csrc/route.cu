// a1: top-k -> multihot routing map, and its backward.
//
// "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)", Changelog: the HybridEP
// preprocessing turns top-k indices into multihot routing metadata (a
// routing_map and per-(token, expert) probs); review of dispatch(): the probs
// are fp32.  Duplicated expert indices inside one token are set once, the
// last slot's prob winning (slots are taken in order).

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

// One warp per token.  Lane l owns experts [e0 + 4l, e0 + 4l + 4) of each
// 128-expert stripe, so each warp writes 128 bytes of routing_map, 512 bytes
// of probs and 128 bytes of winner_slot per stripe with 4/16/4-byte stores.
// The K slot indices are held by the lanes (slot k in lane k % 32, register
// k / 32) and broadcast with shuffles in slot order.
__global__ void __launch_bounds__(256) multihot_kernel(const int64_t* __restrict__ topk_idx,
                                                       const float* __restrict__ topk_probs,
                                                       int T, int K, int E,
                                                       uint8_t* __restrict__ routing_map,
                                                       float* __restrict__ probs,
                                                       int8_t* __restrict__ winner,
                                                       int* __restrict__ status) {
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
    for (int e0 = 0; e0 < E; e0 += 128) {
      const int eb = e0 + 4 * lane;
      uint32_t m = 0, w = 0xffffffffu;  // 4 bytes each; winner -1 = 0xff
      float pr[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k = 0; k < K; ++k) {
        const int j = k >> 5;
        const int src_e = j == 0 ? ek[0] : j == 1 ? ek[1] : j == 2 ? ek[2] : ek[3];
        const float src_p = j == 0 ? pk[0] : j == 1 ? pk[1] : j == 2 ? pk[2] : pk[3];
        const int e = __shfl_sync(FULL_MASK, src_e, k & 31);
        const float p = __shfl_sync(FULL_MASK, src_p, k & 31);
        const unsigned d = static_cast<unsigned>(e - eb);
        if (e >= 0 && d < 4u) {
          m |= 1u << (8 * d);
          w = (w & ~(0xffu << (8 * d))) | (static_cast<uint32_t>(k) << (8 * d));
          pr[0] = d == 0 ? p : pr[0];
          pr[1] = d == 1 ? p : pr[1];
          pr[2] = d == 2 ? p : pr[2];
          pr[3] = d == 3 ? p : pr[3];
        }
      }
      if (eb < E) {  // E % 4 == 0, so the 4 experts are all in range
        const long long o = t * E + eb;
        *reinterpret_cast<uint32_t*>(routing_map + o) = m;
        *reinterpret_cast<uint32_t*>(winner + o) = w;
        *reinterpret_cast<float4*>(probs + o) = make_float4(pr[0], pr[1], pr[2], pr[3]);
      }
    }
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
  multihot_kernel<<<blocks, threads, 0, s>>>(topk_idx, topk_probs, T, K, E, routing_map, probs,
                                             winner, status);
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
