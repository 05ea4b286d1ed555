// Device helpers shared by the layout, dispatch and multihot kernels: warp and
// block scans, the bounded grid barrier of a cooperative launch, and the
// writer of one token's multihot row.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Block-wide exclusive scan of one value per thread (blockDim.x a multiple of
// 32, at most 1024); returns the exclusive prefix and writes the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int incl = warp_inclusive_scan(v, lane);
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nwarps ? s_warp[lane] : 0;
    const int wi = warp_inclusive_scan(w, lane);
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int excl = incl - v + s_warp[warp];
  *total = s_warp[32];
  return excl;
}

// A relaxed gpu-scope load: it reads the value in L2 but, unlike an acquire,
// orders nothing, so a spin on it leaves the SM's L1 and memory pipeline to
// the other CTAs on the SM.  A spin ends with one fence (the acquire).
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch (every CTA is resident).  The
// counter is zeroed before the launch and each CTA adds one per barrier, so
// barrier n is passed once it reads n * gridDim.x.  The wait is bounded: after
// WAIT_LIMIT_NS it reports MOE_DEVERR_TIMEOUT and returns false, and the
// caller's CTA stops.  Data written before the barrier by other CTAs is read
// after it with ld.global.cg (L2), never through this SM's L1.
static __device__ bool grid_barrier(unsigned* ctr, unsigned target, int* status, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    int ok = 1;
    const unsigned long long t0 = global_timer_ns();
    while (ld_relaxed_gpu(ctr) < target) {
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        report(status, MOE_DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();  // the acquire of everything written before the barrier
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Words of the replicated grid barrier: an arrival counter, then REP release
// flags, each in its own 128-byte line, so that the waiting CTAs poll REP
// different lines instead of one.
constexpr int BARRIER_REP = 8;
constexpr int BARRIER_WORDS = 32 * (1 + BARRIER_REP);  // 1152 bytes, zeroed before the launch

// Grid-wide barrier number n (1, 2, ...) of a cooperative launch.  Each CTA
// adds one to the counter; the CTA whose addition completes barrier n (the
// counter reaching n * gridDim.x) sets every release flag to n, and the others
// wait for flag (blockIdx.x % REP) to reach n.  Bounded like grid_barrier.
static __device__ bool grid_barrier_rep(unsigned* words, unsigned n, int* status, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(words, 1u);
    int ok = 1;
    if (old == n * gridDim.x - 1) {
      __threadfence();  // one fence, then the flags: a release of everything before it
      for (int i = 0; i < BARRIER_REP; ++i) reinterpret_cast<volatile unsigned*>(words)[32 * (1 + i)] = n;
    } else {
      const unsigned* flag = words + 32 * (1 + (blockIdx.x % BARRIER_REP));
      const unsigned long long t0 = global_timer_ns();
      while (ld_relaxed_gpu(flag) < n) {
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
          report(status, MOE_DEVERR_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(100);
      }
    }
    __threadfence();  // the acquire of everything written before the barrier
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Writes token t's multihot row (routing_map, probs, winner_slot) from its K
// slots, held by the warp as slot k in lane k % 32, register k / 32 (-1 =
// no expert).  Lane l owns experts [e0 + 4l, e0 + 4l + 4) of each 128-expert
// stripe, so the warp writes 128 bytes of routing_map, 512 bytes of probs and
// 128 bytes of winner_slot per stripe with 4/16/4-byte stores.  Slots are
// visited in order, so a duplicated expert keeps the last slot's prob.
__device__ __forceinline__ void write_multihot_row(long long t, const int (&ek)[4],
                                                   const float (&pk)[4], int K, int E, int lane,
                                                   uint8_t* __restrict__ routing_map,
                                                   float* __restrict__ probs,
                                                   int8_t* __restrict__ winner) {
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

}  // namespace moe
