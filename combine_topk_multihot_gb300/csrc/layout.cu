// a2-a4 and a7-a8: per-expert counts and padded offsets, the expanded layout,
// and the row gathers that fill it.
//
// "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)", review of dispatch():
// dispatch returns tokens_per_expert, pads each expert's rows to pad_multiple,
// and the number of permuted rows is tokens_per_expert.sum().
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds: Expanded layout -- each (token, expert) pair has
// its own row, rows are grouped per expert and carry the pair's weight; Eager
// vs captured -- the unused rows of the sync-free buffer hold zeros and carry
// the sentinel expert id; Training -- the combine's gradient is gathered with
// the same layout as the forward dispatch.
//
// The layout is built without atomics on the output order: a chunked
// histogram (shared-memory counters), one scan block over (expert, chunk),
// and a placement pass in which the thread of expert e walks the chunk's
// tokens in order, so rows inside a group are in ascending token order and
// the result does not depend on scheduling.

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

// Per-chunk, per-expert counts.  The chunk's routing_map bytes are read as
// coalesced 32-bit words; only set bytes touch the shared counters.
__global__ void __launch_bounds__(256) layout_count_kernel(const uint8_t* __restrict__ map, int T,
                                                           int E, int chunks,
                                                           int* __restrict__ chunk_counts) {
  extern __shared__ int s_cnt[];  // [E]
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
  const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), T - t0));
  const int E4 = E >> 2;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(map + t0 * E);
  const int nw = nt * E4;
  for (int i = threadIdx.x; i < nw; i += blockDim.x) {
    const uint32_t v = words[i];
    if (v) {
      const int eb = (i % E4) * 4;
#pragma unroll
      for (int d = 0; d < 4; ++d)
        if ((v >> (8 * d)) & 0xffu) atomicAdd(&s_cnt[eb + d], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<long long>(e) * chunks + c] = s_cnt[e];
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One block of 1024 threads.  Turns the [E][chunks] counts into each chunk's
// exclusive start inside its expert's group (in place), then scans the padded
// group sizes over the experts: offsets[e], offsets[E] = R, and N = sum counts.
__global__ void __launch_bounds__(1024) layout_scan_kernel(int* __restrict__ chunk_counts, int E,
                                                           int chunks, int P, long long capacity,
                                                           int* __restrict__ tokens_per_expert,
                                                           int* __restrict__ offsets,
                                                           int* __restrict__ totals,
                                                           int* __restrict__ status) {
  __shared__ int s_count[1024];
  __shared__ int s_wsum[32], s_wcnt[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // One warp per expert; lane l owns the contiguous chunks [l*per, (l+1)*per):
  // a batched load pass for its sum, one warp scan of the sums, then a
  // batched pass that writes the exclusive starts.
  const int per = (chunks + 31) >> 5;
  for (int e = warp; e < E; e += 32) {
    int* row = chunk_counts + static_cast<long long>(e) * chunks;
    const int c0 = min(chunks, lane * per), c1 = min(chunks, c0 + per);
    int sum = 0;
    for (int c = c0; c < c1; c += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = c + i < c1 ? row[c + i] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += v[i];
    }
    const int incl = warp_inclusive_scan(sum, lane);
    int run = incl - sum;
    for (int c = c0; c < c1; c += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = c + i < c1 ? row[c + i] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c + i < c1) row[c + i] = run;
        run += v[i];
      }
    }
    const int total = __shfl_sync(FULL_MASK, incl, 31);
    if (lane == 0) s_count[e] = total;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int cnt = e < E ? s_count[e] : 0;
  const int padded = e < E ? ((cnt + P - 1) / P) * P : 0;
  int v = warp_inclusive_scan(padded, lane);
  int n = warp_inclusive_scan(cnt, lane);
  if (lane == 31) {
    s_wsum[warp] = v;
    s_wcnt[warp] = n;
  }
  __syncthreads();
  if (warp == 0) {
    const int a = s_wsum[lane], b = s_wcnt[lane];
    const int ia = warp_inclusive_scan(a, lane), ib = warp_inclusive_scan(b, lane);
    s_wsum[lane] = ia - a;
    s_wcnt[lane] = ib - b;
  }
  __syncthreads();
  v += s_wsum[warp];
  n += s_wcnt[warp];
  if (e < E) {
    offsets[e] = v - padded;
    tokens_per_expert[e] = cnt;
  }
  if (e == E - 1) {
    offsets[E] = v;
    totals[0] = v;
    totals[1] = n;
    if (v > capacity) report(status, MOE_DEVERR_CAPACITY);
  }
}

// Stable placement.  A chunk is 32 tokens, so the tokens of the chunk that go
// to expert e form one 32-bit mask, and a pair's rank inside its expert's
// group is (the chunk's start in the group) + popcount(mask below the token).
// The chunk's map is staged in shared memory and turned into both bit
// matrices: experts per token (ballots) and tokens per expert (a transpose of
// it); then one warp per token places the token's pairs, lane l taking the
// experts l, l+32, ...  A pair's position j in token_row is the popcount of the
// token's expert mask below it.
__global__ void __launch_bounds__(256) layout_place_kernel(
    const uint8_t* __restrict__ map, const float* __restrict__ probs, int T, int E, int K,
    int chunks, const int* __restrict__ chunk_base, const int* __restrict__ offsets,
    long long capacity, int* __restrict__ row_token, int* __restrict__ row_expert,
    float* __restrict__ row_weight, int* __restrict__ token_row, int* __restrict__ status) {
  static_assert(LAYOUT_CHUNK == 32, "one 32-bit token mask per expert");
  extern __shared__ __align__(16) uint8_t smem[];
  const int c = blockIdx.x;
  const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
  const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), T - t0));
  const int E4 = E >> 2, EW = (E + 31) >> 5;
  uint32_t* s_map32 = reinterpret_cast<uint32_t*>(smem);     // [32][E] bytes
  uint32_t* s_emask = s_map32 + LAYOUT_CHUNK * E4;             // [32][EW]: experts of each token
  uint32_t* s_tmask = s_emask + LAYOUT_CHUNK * EW;             // [E]: tokens of each expert
  int* s_base = reinterpret_cast<int*>(s_tmask + E);           // [E]: first row of this chunk's pairs
  const uint8_t* s_map = smem;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(map + t0 * E);
  for (int i = threadIdx.x; i < nt * E4; i += blockDim.x) s_map32[i] = words[i];
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    s_base[e] = offsets[e] + chunk_base[static_cast<long long>(e) * chunks + c];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int tl = warp; tl < LAYOUT_CHUNK; tl += nwarps) {
    for (int seg = 0; seg < EW; ++seg) {
      const int e = seg * 32 + lane;
      const bool b = tl < nt && e < E && s_map[tl * E + e] != 0;
      const uint32_t m = __ballot_sync(FULL_MASK, b);
      if (lane == 0) s_emask[tl * EW + seg] = m;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int seg = e >> 5, bit = e & 31;
    uint32_t m = 0;
#pragma unroll 8
    for (int tl = 0; tl < LAYOUT_CHUNK; ++tl) m |= ((s_emask[tl * EW + seg] >> bit) & 1u) << tl;
    s_tmask[e] = m;
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int tl = warp; tl < nt; tl += nwarps) {
    const long long t = t0 + tl;
    const uint32_t below_t = (1u << tl) - 1u;
    int j_base = 0;
    for (int seg = 0; seg < EW; ++seg) {
      const uint32_t em = s_emask[tl * EW + seg];
      const int e = seg * 32 + lane;
      if ((em >> lane) & 1u) {
        const long long row = static_cast<long long>(s_base[e]) + __popc(s_tmask[e] & below_t);
        const int j = j_base + __popc(em & lt);
        if (row < capacity && j < K) {
          row_token[row] = static_cast<int>(t);
          row_expert[row] = e;
          row_weight[row] = probs[t * E + e];
          token_row[t * K + j] = static_cast<int>(row);
        } else {
          report(status, row < capacity ? MOE_DEVERR_BAD_INDEX : MOE_DEVERR_CAPACITY);
        }
      }
      j_base += __popc(em);
    }
    for (int j = j_base + lane; j < K; j += 32) token_row[t * K + j] = -1;
  }
}

// Row gather, one warp per row, each lane moving H/256 16-byte vectors.
//   FROM_OFFSETS: decide valid / pad / spare from offsets and counts (dispatch,
//     where the pad rows' metadata is written here), else from row_token (the
//     combine backward, after dispatch wrote every row's metadata).
//   DOT: also grad_w[r] = <src[t], o_save[r]> in fp32 (routing-weight gradient).
template <bool FROM_OFFSETS, bool DOT>
__global__ void __launch_bounds__(256) row_gather_kernel(
    const uint16_t* __restrict__ src, int H, int E, long long C, const int* __restrict__ offsets,
    const int* __restrict__ counts, int* __restrict__ row_token, int* __restrict__ row_expert,
    float* __restrict__ row_weight, uint16_t* __restrict__ dst, const uint16_t* __restrict__ o_save,
    float* __restrict__ grad_w) {
  extern __shared__ int s_meta[];  // offsets [E+1], counts [E]
  int* s_off = s_meta;
  int* s_cnt = s_meta + E + 1;
  if (FROM_OFFSETS) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = counts[i];
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;  // 16-byte vectors per lane
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int R = FROM_OFFSETS ? s_off[E] : 0;
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < C; r += nwarps) {
    int t = -1;
    if (FROM_OFFSETS) {
      if (r < R) {
        int lo = 0, hi = E;  // s_off[lo] <= r < s_off[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_off[mid] <= r) lo = mid; else hi = mid;
        }
        if (r - s_off[lo] < s_cnt[lo]) t = row_token[r];
      }
      if (t < 0 && lane == 0) {
        row_token[r] = -1;
        row_expert[r] = E;
        row_weight[r] = 0.f;
      }
    } else {
      t = row_token[r];
    }
    uint4* d = reinterpret_cast<uint4*>(dst + r * H);
    float dot = 0.f;
    if (t >= 0) {
      const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<long long>(t) * H);
      const uint4* o = DOT ? reinterpret_cast<const uint4*>(o_save + r * H) : nullptr;
      for (int v0 = 0; v0 < V; v0 += 8) {
        uint4 buf[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (v0 + i < V) buf[i] = __ldg(s + lane + 32 * (v0 + i));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (v0 + i < V) d[lane + 32 * (v0 + i)] = buf[i];
        if (DOT) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (v0 + i < V) {
              const uint4 ov = __ldg(o + lane + 32 * (v0 + i));
              const uint32_t g[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
              const uint32_t q[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                dot = fmaf(bf16_lo(g[k]), bf16_lo(q[k]), dot);
                dot = fmaf(bf16_hi(g[k]), bf16_hi(q[k]), dot);
              }
            }
          }
        }
      }
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = 0; v < V; ++v) d[lane + 32 * v] = z;
    }
    if (DOT) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(FULL_MASK, dot, o);
      if (lane == 0) grad_w[r] = t >= 0 ? dot : 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_layout_counts(const uint8_t* routing_map, const moe_layout& L,
                                 int* chunk_counts, cudaStream_t s) {
  const int chunks = static_cast<int>(layout_chunks(L.T));
  if (chunks > 0) {
    layout_count_kernel<<<chunks, 256, L.E * sizeof(int), s>>>(routing_map, L.T, L.E, chunks,
                                                                chunk_counts);
  }
  layout_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, L.E, chunks, L.pad_multiple, L.capacity,
                                        L.tokens_per_expert, L.offsets, L.totals, L.status);
  return cudaGetLastError();
}

cudaError_t launch_layout_place(const uint8_t* routing_map, const float* probs,
                                const moe_layout& L, const int* chunk_base, cudaStream_t s) {
  const int chunks = static_cast<int>(layout_chunks(L.T));
  if (chunks == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(LAYOUT_CHUNK) * L.E +
                      static_cast<size_t>(LAYOUT_CHUNK) * ((L.E + 31) / 32) * sizeof(uint32_t) +
                      static_cast<size_t>(L.E) * (sizeof(uint32_t) + sizeof(int));
  layout_place_kernel<<<chunks, 256, smem, s>>>(routing_map, probs, L.T, L.E, L.K, chunks,
                                                chunk_base, L.offsets, L.capacity, L.row_token,
                                                L.row_expert, L.row_weight, L.token_row, L.status);
  return cudaGetLastError();
}

cudaError_t launch_row_gather(const uint16_t* src, const moe_layout& L, int H, uint16_t* dst,
                              bool from_offsets, const uint16_t* o_save, float* grad_w,
                              cudaStream_t s) {
  const long long C = L.capacity;
  if (C == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (C + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  const size_t smem = from_offsets ? (2 * L.E + 1) * sizeof(int) : 0;
  if (from_offsets) {
    row_gather_kernel<true, false><<<blocks, threads, smem, s>>>(
        src, H, L.E, C, L.offsets, L.tokens_per_expert, L.row_token, L.row_expert, L.row_weight,
        dst, nullptr, nullptr);
  } else if (grad_w) {
    row_gather_kernel<false, true><<<blocks, threads, 0, s>>>(
        src, H, L.E, C, nullptr, nullptr, L.row_token, nullptr, nullptr, dst, o_save, grad_w);
  } else {
    row_gather_kernel<false, false><<<blocks, threads, 0, s>>>(
        src, H, L.E, C, nullptr, nullptr, L.row_token, nullptr, nullptr, dst, nullptr, nullptr);
  }
  return cudaGetLastError();
}

}  // namespace moe
