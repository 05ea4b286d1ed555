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

// One CTA per expert: the expert's per-chunk counts become each chunk's
// exclusive start inside the expert's group (in place), and the total is the
// expert's token count.  Thread i owns a contiguous run of chunks.
__global__ void __launch_bounds__(256) layout_expert_scan_kernel(int* __restrict__ chunk_counts,
                                                                 int chunks,
                                                                 int* __restrict__ tokens_per_expert) {
  __shared__ int s_warp[33];
  const int e = blockIdx.x;
  int* row = chunk_counts + static_cast<long long>(e) * chunks;
  const int per = (chunks + blockDim.x - 1) / blockDim.x;
  const int c0 = min(chunks, static_cast<int>(threadIdx.x) * per), c1 = min(chunks, c0 + per);
  int sum = 0;
  for (int c = c0; c < c1; c += 8) {
    int v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = c + i < c1 ? row[c + i] : 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += v[i];
  }
  int total;
  int run = block_exclusive_scan(sum, s_warp, &total);
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
  if (threadIdx.x == 0) tokens_per_expert[e] = total;
}

// One CTA of 1024 threads: offsets[e] = exclusive prefix of the counts padded
// to multiples of P; offsets[E] = R = totals[0]; totals[1] = N.
__global__ void __launch_bounds__(1024) layout_offsets_kernel(const int* __restrict__ tokens_per_expert,
                                                              int E, int P, long long capacity,
                                                              int* __restrict__ offsets,
                                                              int* __restrict__ totals,
                                                              int* __restrict__ status) {
  __shared__ int s_warp[33];
  const int e = threadIdx.x;
  const int cnt = e < E ? tokens_per_expert[e] : 0;
  const int padded = e < E ? ((cnt + P - 1) / P) * P : 0;
  int R, N;
  const int excl = block_exclusive_scan(padded, s_warp, &R);
  __syncthreads();
  block_exclusive_scan(cnt, s_warp, &N);
  if (e < E) offsets[e] = excl;
  if (e == 0) {
    offsets[E] = R;
    totals[0] = R;
    totals[1] = N;
    if (R > capacity) report(status, MOE_DEVERR_CAPACITY);
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

// Dispatch (and the combine's backward) as a scatter, one warp per item.
//   Items [0, T) are tokens: the warp reads the token's source row once from
//   memory -- later passes over it hit L1 -- and writes it to each of the
//   token's rows (token_row).  Reading each token once matters when [T, H]
//   no longer fits in L2: a per-row gather would fetch it K times from DRAM.
//   With DOT it also forms grad_w[r] = <src[t], o_save[r]> in fp32.
//   Items [T, T + C) are rows: a pad or spare row is zeroed (and grad_w = 0).
//   With META the row's validity comes from offsets / counts and the pad and
//   spare rows get their metadata here (token -1, the sentinel expert, weight
//   0); without it, from row_token (the combine's backward, after dispatch).
template <bool META, bool DOT>
__global__ void __launch_bounds__(256) row_scatter_kernel(
    const uint16_t* __restrict__ src, int T, int K, int H, int E, long long C,
    const int* __restrict__ token_row, const int* __restrict__ offsets,
    const int* __restrict__ counts, int* __restrict__ row_token, int* __restrict__ row_expert,
    float* __restrict__ row_weight, uint16_t* __restrict__ dst, const uint16_t* __restrict__ o_save,
    float* __restrict__ grad_w) {
  extern __shared__ int s_meta[];  // META: offsets [E+1], counts [E]
  int* s_off = s_meta;
  int* s_cnt = s_meta + E + 1;
  if (META) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = counts[i];
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;  // 16-byte vectors per lane
  const long long items = T + C;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int R = META ? s_off[E] : 0;
  for (long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += nwarps) {
    if (it < T) {
      const long long t = it;
      const uint4* s = reinterpret_cast<const uint4*>(src + t * H);
      for (int j = 0; j < K; ++j) {
        const int r = __ldg(token_row + t * K + j);
        if (r < 0) break;
        uint4* d = reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * H);
        const uint4* o = DOT ? reinterpret_cast<const uint4*>(o_save + static_cast<long long>(r) * H) : nullptr;
        float dot = 0.f;
        for (int v0 = 0; v0 < V; v0 += 8) {
          uint4 buf[8], ob[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (v0 + i < V) {
              buf[i] = __ldg(s + lane + 32 * (v0 + i));
              if (DOT) ob[i] = __ldg(o + lane + 32 * (v0 + i));
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (v0 + i < V) {
              d[lane + 32 * (v0 + i)] = buf[i];
              if (DOT) {
                const uint32_t g[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
                const uint32_t q[4] = {ob[i].x, ob[i].y, ob[i].z, ob[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  dot = fmaf(bf16_lo(g[k]), bf16_lo(q[k]), dot);
                  dot = fmaf(bf16_hi(g[k]), bf16_hi(q[k]), dot);
                }
              }
            }
          }
        }
        if (DOT) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(FULL_MASK, dot, off);
          if (lane == 0) grad_w[r] = dot;
        }
      }
    } else {
      const long long r = it - T;
      bool pad;
      if (META) {
        pad = true;
        if (r < R) {
          int lo = 0, hi = E;  // s_off[lo] <= r < s_off[hi]
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= r) lo = mid; else hi = mid;
          }
          pad = r - s_off[lo] >= s_cnt[lo];
        }
      } else {
        pad = __ldg(row_token + r) < 0;
      }
      if (!pad) continue;
      if (lane == 0) {
        if (META) {
          row_token[r] = -1;
          row_expert[r] = E;
          row_weight[r] = 0.f;
        }
        if (DOT) grad_w[r] = 0.f;
      }
      uint4* d = reinterpret_cast<uint4*>(dst + r * H);
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = 0; v < V; ++v) d[lane + 32 * v] = z;
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
  if (chunks > 0) layout_expert_scan_kernel<<<L.E, 256, 0, s>>>(chunk_counts, chunks, L.tokens_per_expert);
  else cudaMemsetAsync(L.tokens_per_expert, 0, L.E * sizeof(int), s);
  layout_offsets_kernel<<<1, 1024, 0, s>>>(L.tokens_per_expert, L.E, L.pad_multiple, L.capacity,
                                           L.offsets, L.totals, L.status);
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
  const long long items = static_cast<long long>(L.T) + C;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (items + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  if (from_offsets) {
    const size_t smem = (2 * L.E + 1) * sizeof(int);
    row_scatter_kernel<true, false><<<blocks, threads, smem, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, L.offsets, L.tokens_per_expert, L.row_token,
        L.row_expert, L.row_weight, dst, nullptr, nullptr);
  } else if (grad_w) {
    row_scatter_kernel<false, true><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, nullptr,
        dst, o_save, grad_w);
  } else {
    row_scatter_kernel<false, false><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, nullptr,
        dst, nullptr, nullptr);
  }
  return cudaGetLastError();
}

}  // namespace moe
