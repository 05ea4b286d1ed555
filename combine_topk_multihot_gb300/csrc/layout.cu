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
// The layout is built without atomics on the output order: per 32-token chunk
// each expert's count, a scan over the chunks of each expert, padded offsets,
// and a placement pass that ranks each (token, expert) pair inside its chunk
// by a popcount of the expert's token mask, so rows inside a group are in
// ascending token order and the result does not depend on scheduling.  Large
// layers run this as one cooperative launch with two bounded grid barriers;
// layers of up to 8 chunks as one CTA per chunk that each count every chunk,
// with no barrier.  For a host-synced caller the kernel also hands R, N and
// the status word to the host through mapped memory as soon as the offsets are
// known, and places nothing when the rows do not fit.

#include "common.cuh"
#include "coop.cuh"
#include "launch.h"

namespace moe {

namespace {

// The single-CTA layout also does the dispatch's row pass when it has at most
// this many items (tokens + rows) and moves at most this many bytes.
constexpr long long LAYOUT_FUSED_ITEMS = 64;
// Layers of at most this many 32-token chunks take the barrier-free layout
// (decode T = 256, 8 chunks: 21.1 -> 12.7 us under graph replay; at 32 chunks
// the cooperative kernel was faster).
constexpr int LAYOUT_REDUNDANT_CHUNKS = 8;
constexpr long long LAYOUT_FUSED_BYTES = 256 * 1024;

enum LayoutMode : int {
  LAYOUT_ALL = 0,    // counts, scans, offsets and placement: one cooperative launch
  LAYOUT_SINGLE = 3, // up to 8 chunks, one CTA per chunk: each counts every chunk, then
                     // places its own (no grid barrier; one CTA may also do the row pass)
};

struct LayoutArgs {
  const uint8_t* map;
  const float* probs;
  int T, E, K, P, chunks;
  long long capacity;
  int* chunk_counts;  // [E][chunks]: counts, then in place each chunk's start in its expert's group
  unsigned* barrier;  // zeroed before a cooperative launch
  int* tokens_per_expert;
  int* offsets;
  int* totals;
  int* row_token;
  int* row_expert;
  float* row_weight;
  int* token_row;
  int* status;
  int* readback;  // {R, N, status} in host-mapped memory (host-synced callers), or NULL
  // LAYOUT_SINGLE with rows: the CTA also does the dispatch's row pass (the
  // copies into x_disp when it is not NULL, and the pad and spare rows)
  bool rows;
  const uint16_t* x;
  uint16_t* x_disp;
  int H;
};

// Dispatch (and the combine's backward) as a scatter, one warp per item.
//   Items [0, T) are tokens: the warp reads the token's source row once from
//   memory -- later passes over it hit L1 -- and writes it to each of the
//   token's rows (token_row).  Reading each token once matters when [T, H]
//   no longer fits in L2: a per-row gather would fetch it K times from DRAM.
//   With DOT it also forms grad_w[r] = <src[t], o_save[r]> in fp32.  With
//   SCALE the row gets bf16(row_weight[r] * src[t]) instead of src[t] (the
//   combine's backward handing the experts dL/do = w dL/dy directly; the dot
//   uses the unscaled src).
//   Items [T, T + C) are rows: a pad or spare row is zeroed (and grad_w = 0).
//   With META the row's validity comes from offsets / counts and the pad and
//   spare rows get their metadata here (token -1, the sentinel expert, weight
//   0); without it, from row_token (the combine's backward, after dispatch).
// This is one warp's share: items first, first + stride, ...  With META,
// s_off / s_cnt are the offsets and counts (shared memory, or global memory
// this CTA wrote before a barrier).
template <bool META, bool DOT, bool SCALE = false>
__device__ __forceinline__ void scatter_items(
    long long first, long long stride, const uint16_t* __restrict__ src, int T, int K, int H, int E,
    long long C, const int* __restrict__ token_row, const int* s_off, const int* s_cnt,
    int* __restrict__ row_token, int* __restrict__ row_expert, float* __restrict__ row_weight,
    uint16_t* __restrict__ dst, const uint16_t* __restrict__ o_save, float* __restrict__ grad_w,
    int* status = nullptr) {
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;  // 16-byte vectors per lane
  const long long items = T + C;
  const int R = META ? s_off[E] : 0;
  if (META && R > C) return;  // the layout placed nothing: the rows do not fit
  for (long long it = first; it < items; it += stride) {
    if (it < T) {
      if (META && dst == nullptr) continue;  // the layout alone: no rows to copy
      const long long t = it;
      const uint4* s = reinterpret_cast<const uint4*>(src + t * H);
      // The token's rows, 32 slots per load (a token's valid slots come first).
      int r_lane = -1;
      for (int j = 0; j < K; ++j) {
        // (L2 load: the layout kernel itself may have just written token_row)
        if ((j & 31) == 0) r_lane = j + lane < K ? __ldcg(token_row + t * K + j + lane) : -1;
        const int r = __shfl_sync(FULL_MASK, r_lane, j & 31);
        if (r < 0 || !MOE_IN_BOUNDS(r < C, status) || r >= C) break;
        uint4* d = reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * H);
        const uint4* o = DOT ? reinterpret_cast<const uint4*>(o_save + static_cast<long long>(r) * H) : nullptr;
        const float w = SCALE ? __ldg(row_weight + r) : 0.f;
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
              if (SCALE) {
                const uint4 a = buf[i];
                d[lane + 32 * (v0 + i)] = make_uint4(pack_bf16x2(w * bf16_lo(a.x), w * bf16_hi(a.x)),
                                                     pack_bf16x2(w * bf16_lo(a.y), w * bf16_hi(a.y)),
                                                     pack_bf16x2(w * bf16_lo(a.z), w * bf16_hi(a.z)),
                                                     pack_bf16x2(w * bf16_lo(a.w), w * bf16_hi(a.w)));
              } else {
                d[lane + 32 * (v0 + i)] = buf[i];
              }
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
      if (dst == nullptr) continue;
      uint4* d = reinterpret_cast<uint4*>(dst + r * H);
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = 0; v < V; ++v) d[lane + 32 * v] = z;
    }
  }
}

// a2 + a3 in one kernel.  A chunk is 32 tokens.
//   1. Per chunk, each expert's token count (the chunk's routing_map bytes are
//      staged in shared memory; thread e counts column e).
//   -- grid barrier --
//   2. One warp per expert turns the expert's per-chunk counts into each
//      chunk's exclusive start inside the expert's group (in place, 32 chunks
//      per coalesced step); the total is tokens_per_expert[e].
//   -- grid barrier --
//   3. Every CTA forms the padded offsets itself (a block scan over E);
//      CTA 0 also writes offsets, totals and the capacity check.
//   4. Stable placement per chunk: the tokens of the chunk that go to expert
//      e form one 32-bit mask, so a pair's rank in its group is (the chunk's
//      start) + popcount(mask below the token).  Ballots turn the staged map
//      into experts-per-token masks, a transpose gives tokens-per-expert, and
//      one thread per (token, slot j) places the token's j-th expert (the
//      j-th set bit of its expert mask), so all of a chunk's loads and
//      stores are in flight together.
// Rows inside a group come out in ascending token order and nothing depends
// on scheduling: no atomics decide a position.
template <int MODE>
__global__ void __launch_bounds__(256) layout_kernel(LayoutArgs a) {
  static_assert(LAYOUT_CHUNK == 32, "one 32-bit token mask per expert");
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_warp[33];
  __shared__ int s_ok;
  const int E = a.E, E4 = E >> 2, EW = (E + 31) >> 5;
  uint32_t* s_map32 = reinterpret_cast<uint32_t*>(smem);             // [32][E] bytes
  const uint8_t* s_map = smem;
  uint32_t* s_tmask = s_map32;                                         // [E], over the map once read
  int* s_base = reinterpret_cast<int*>(s_map32 + E);                   // [E], likewise
  uint32_t* s_emask = s_map32 + LAYOUT_CHUNK * E4;                     // [32][EW]
  int* s_off = reinterpret_cast<int*>(s_emask + LAYOUT_CHUNK * EW);    // [E + 1]
  int* s_tot = s_off + E + 1;  // LAYOUT_SINGLE: [E] each expert's count
  int* s_cc = s_tot + E;       // LAYOUT_SINGLE: [chunks][E] counts, then each chunk's start
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

  if constexpr (MODE == LAYOUT_ALL) {
    // 1. this CTA's chunks, staged in shared memory; thread e counts column e
    for (int c = blockIdx.x; c < a.chunks; c += gridDim.x) {
      const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
      const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), a.T - t0));
      const uint32_t* words = reinterpret_cast<const uint32_t*>(a.map + t0 * E);
      for (int i = threadIdx.x; i < nt * E4; i += blockDim.x) s_map32[i] = words[i];
      __syncthreads();
      for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n = 0;
        for (int tl = 0; tl < nt; ++tl) n += s_map[tl * E + e] != 0;
        a.chunk_counts[static_cast<long long>(e) * a.chunks + c] = n;
      }
      __syncthreads();
    }
  } else {
    // 1. every CTA counts every chunk (no grid barrier needed): warp w takes
    // chunks w, w + 8, ..., lane l the 4-expert words l, l + 32, ... of each
    // token row.  A word's four map bytes become four 0/1 bytes and the 32
    // token rows of a chunk are summed bytewise (at most 32: no carry), all
    // 32 loads in flight together.  One thread owns each (chunk, expert) count.
    const uint32_t* map32 = reinterpret_cast<const uint32_t*>(a.map);
    for (int c = warp; c < a.chunks; c += nwarps) {
      const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
      const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), a.T - t0));
      for (int w4 = lane; w4 < E4; w4 += 32) {
        uint32_t wd[LAYOUT_CHUNK];
#pragma unroll
        for (int tl = 0; tl < LAYOUT_CHUNK; ++tl)
          wd[tl] = tl < nt ? __ldg(map32 + (t0 + tl) * E4 + w4) : 0u;
        uint32_t sum = 0;
#pragma unroll
        for (int tl = 0; tl < LAYOUT_CHUNK; ++tl) {
          uint32_t b = wd[tl] | (wd[tl] >> 4);  // bit 0 of each byte: the byte is nonzero
          b |= b >> 2;
          b |= b >> 1;
          sum += b & 0x01010101u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) s_cc[c * E + 4 * w4 + k] = (sum >> (8 * k)) & 0xffu;
      }
    }
    __syncthreads();
  }
  if constexpr (MODE == LAYOUT_SINGLE) {
    // one CTA: each expert's per-chunk starts and total, in shared memory
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = 0;
      for (int c = 0; c < a.chunks; ++c) {
        const int v = s_cc[c * E + e];
        s_cc[c * E + e] = run;
        run += v;
      }
      s_tot[e] = run;
      if (blockIdx.x == 0) a.tokens_per_expert[e] = run;
    }
    __syncthreads();
  } else {
    if (!grid_barrier(a.barrier, gridDim.x, a.status, &s_ok)) return;
    for (int e = blockIdx.x * nwarps + warp; e < E; e += gridDim.x * nwarps) {
      int* row = a.chunk_counts + static_cast<long long>(e) * a.chunks;
      int run = 0;
      // 8 coalesced steps of 32 chunks per batch: the loads of a batch are
      // issued together, then scanned in order
      for (int b0 = 0; b0 < a.chunks; b0 += 8 * 32) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = b0 + 32 * i + lane;
          v[i] = c < a.chunks ? __ldcg(row + c) : 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = b0 + 32 * i + lane;
          const int incl = warp_inclusive_scan(v[i], lane);
          if (c < a.chunks) row[c] = run + incl - v[i];
          run += __shfl_sync(FULL_MASK, incl, 31);
        }
      }
      if (lane == 0) a.tokens_per_expert[e] = run;
    }
    if (!grid_barrier(a.barrier, 2 * gridDim.x, a.status, &s_ok)) return;
  }

  // Padded offsets; thread i owns experts 4i .. 4i + 3 (E <= 4 * blockDim.x).
  {
    int cnt[4], pad[4], psum = 0, nsum = 0;
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const int e = 4 * threadIdx.x + d;
      if constexpr (MODE == LAYOUT_SINGLE)
        cnt[d] = e < E ? s_tot[e] : 0;
      else
        cnt[d] = e < E ? __ldcg(a.tokens_per_expert + e) : 0;
      pad[d] = ((cnt[d] + a.P - 1) / a.P) * a.P;
      psum += pad[d];
      nsum += cnt[d];
    }
    int R;
    int excl = block_exclusive_scan(psum, s_warp, &R);
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const int e = 4 * threadIdx.x + d;
      if (e < E) s_off[e] = excl;
      excl += pad[d];
    }
    if (threadIdx.x == 0) s_off[E] = R;
    if (blockIdx.x == 0) {
      __syncthreads();
      int N;
      block_exclusive_scan(nsum, s_warp, &N);
      for (int e = threadIdx.x; e <= E; e += blockDim.x) a.offsets[e] = s_off[e];
      if (threadIdx.x == 0) {
        a.totals[0] = R;
        a.totals[1] = N;
        if (R > a.capacity) report(a.status, MOE_DEVERR_CAPACITY);
        if (a.readback) {  // for the host-synced caller, without a copy engine
          // R goes last, after a system-scope fence: the host waits for it and
          // then reads the other two
          volatile int* rb = a.readback;
          rb[1] = N;
          rb[2] = *reinterpret_cast<volatile int*>(a.status);
          __threadfence_system();
          rb[0] = R;
        }
      }
    }
    __syncthreads();
  }
  // 4. Placement, only when the rows fit: with R > capacity nothing is
  // written (the host-synced caller then reports the capacity error).
  if (s_off[E] <= a.capacity) {
    for (int c = blockIdx.x; c < a.chunks; c += gridDim.x) {
      const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
      const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), a.T - t0));
      const uint32_t* words = reinterpret_cast<const uint32_t*>(a.map + t0 * E);
      for (int i = threadIdx.x; i < nt * E4; i += blockDim.x) s_map32[i] = words[i];
      __syncthreads();
      for (int tl = warp; tl < LAYOUT_CHUNK; tl += nwarps) {
        for (int seg = 0; seg < EW; ++seg) {
          const int e = seg * 32 + lane;
          const bool b = tl < nt && e < E && s_map[tl * E + e] != 0;
          const uint32_t m = __ballot_sync(FULL_MASK, b);
          if (lane == 0) s_emask[tl * EW + seg] = m;
        }
      }
      __syncthreads();  // the map's space now holds s_tmask and s_base
      for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int seg = e >> 5, bit = e & 31;
        uint32_t m = 0;
  #pragma unroll 8
        for (int tl = 0; tl < LAYOUT_CHUNK; ++tl) m |= ((s_emask[tl * EW + seg] >> bit) & 1u) << tl;
        s_tmask[e] = m;
        if constexpr (MODE == LAYOUT_SINGLE)
          s_base[e] = s_off[e] + s_cc[c * E + e];
        else
          s_base[e] = s_off[e] + __ldcg(a.chunk_counts + static_cast<long long>(e) * a.chunks + c);
      }
      __syncthreads();
      // One thread per (token, slot j): slot j of a token is the token's j-th
      // expert in ascending order.  Every load of the chunk is issued at once.
      for (int i = threadIdx.x; i < nt * a.K; i += blockDim.x) {
        const int tl = i / a.K, j = i - tl * a.K;
        const long long t = t0 + tl;
        const uint32_t* em = s_emask + tl * EW;
        int seg = 0, below = 0, n = __popc(em[0]);
        while (below + n <= j && seg + 1 < EW) {
          below += n;
          n = __popc(em[++seg]);
        }
        int row_out = -1;
        if (below + n > j) {
          uint32_t m = em[seg];
          for (int k = j - below; k > 0; --k) m &= m - 1u;  // drop the lower set bits
          const int e = seg * 32 + __ffs(m) - 1;
          const long long row = static_cast<long long>(s_base[e]) + __popc(s_tmask[e] & ((1u << tl) - 1u));
          if (row < a.capacity) {
            a.row_token[row] = static_cast<int>(t);
            a.row_expert[row] = e;
            a.row_weight[row] = __ldg(a.probs + t * E + e);
            row_out = static_cast<int>(row);
          } else {
            report(a.status, MOE_DEVERR_CAPACITY);
          }
        }
        a.token_row[t * a.K + j] = row_out;
        if (j == 0) {  // more experts than slots: a routing_map that no top-k could make
          int total = 0;
          for (int w = 0; w < EW; ++w) total += __popc(em[w]);
          if (total > a.K) report(a.status, MOE_DEVERR_BAD_INDEX);
        }
      }
      __syncthreads();  // before the next chunk overwrites the shared arrays
    }
  }
  if constexpr (MODE == LAYOUT_SINGLE) {
    if (a.rows && s_off[E] <= a.capacity) {
      // every row of the layout is placed (the barrier above): the row pass,
      // one warp per item, with the offsets in shared memory and the counts
      // this CTA wrote
      scatter_items<true, false>(warp, nwarps, a.x, static_cast<int>(a.T), a.K, a.H, E, a.capacity,
                                 a.token_row, s_off, a.tokens_per_expert, a.row_token, a.row_expert,
                                 a.row_weight, a.x_disp, nullptr, nullptr, a.status);
    }
  }
}

// The scatter as a kernel: offsets and counts staged in shared memory, then
// one warp per item over the grid.
template <bool META, bool DOT, bool SCALE = false>
__global__ void __launch_bounds__(256) row_scatter_kernel(
    const uint16_t* __restrict__ src, int T, int K, int H, int E, long long C,
    const int* __restrict__ token_row, const int* __restrict__ offsets,
    const int* __restrict__ counts, int* __restrict__ row_token, int* __restrict__ row_expert,
    float* __restrict__ row_weight, uint16_t* __restrict__ dst, const uint16_t* __restrict__ o_save,
    float* __restrict__ grad_w, int* status) {
  griddep_launch_dependents();
  griddep_wait();
  extern __shared__ int s_meta[];  // META: offsets [E+1], counts [E]
  int* s_off = s_meta;
  int* s_cnt = s_meta + E + 1;
  if (META) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = counts[i];
    __syncthreads();
  }
  scatter_items<META, DOT, SCALE>(static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5),
                           static_cast<long long>(gridDim.x) * (blockDim.x >> 5), src, T, K, H, E, C,
                           token_row, s_off, s_cnt, row_token, row_expert, row_weight, dst, o_save,
                           grad_w, status);
}

}  // namespace

namespace {

size_t layout_smem_bytes(int E) {
  return static_cast<size_t>(LAYOUT_CHUNK) * E +
         static_cast<size_t>(LAYOUT_CHUNK) * ((E + 31) / 32) * sizeof(uint32_t) +
         static_cast<size_t>(2 * E + 1) * sizeof(int);
}

// CTAs of layout_kernel<MODE> resident at once on the current device with
// `smem` bytes of dynamic shared memory (the last answer is kept per thread).
template <int MODE>
int layout_resident_ctas(size_t smem) {
  static thread_local int last_dev = -1;
  static thread_local size_t last_smem = 0;
  static thread_local int last_ctas = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev == last_dev && smem == last_smem) return last_ctas;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layout_kernel<MODE>, 256, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  last_dev = dev;
  last_smem = smem;
  last_ctas = per_sm * sm_count();
  return last_ctas;
}

template <int MODE>
cudaError_t launch_layout_mode(const LayoutArgs& a, size_t smem, cudaStream_t s) {
  if (MODE == LAYOUT_SINGLE) {
    // one CTA per chunk (one CTA in all when it also does the row pass)
    const int grid = a.rows || a.chunks < 1 ? 1 : a.chunks;
    return launch_dependent(layout_kernel<MODE>, grid, 256,
                            smem + static_cast<size_t>(a.chunks) * a.E * sizeof(int), s, a);
  }
  cudaError_t err = cudaMemsetAsync(a.barrier, 0, sizeof(unsigned), s);
  if (err != cudaSuccess) return err;
  // Enough CTAs for one chunk each (phases 1 and 4) and one warp per expert
  // (phase 2), but never more than can be resident at once.
  const int want = a.chunks > (a.E + 7) / 8 ? a.chunks : (a.E + 7) / 8;
  const int resident = layout_resident_ctas<MODE>(smem);
  const int grid = want < resident ? want : resident;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, layout_kernel<MODE>, a);
}

}  // namespace

cudaError_t launch_layout(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                          void* workspace, cudaStream_t s, int* readback, const uint16_t* x,
                          uint16_t* x_disp, int H, bool* rows_done) {
  LayoutArgs a;
  a.readback = readback;
  a.rows = false;
  a.x = x;
  a.x_disp = x_disp;
  a.H = H;
  if (rows_done) *rows_done = false;
  a.map = routing_map;
  a.probs = probs;
  a.T = L.T;
  a.E = L.E;
  a.K = L.K;
  a.P = L.pad_multiple;
  a.chunks = static_cast<int>(layout_chunks(L.T));
  a.capacity = L.capacity;
  a.chunk_counts = static_cast<int*>(workspace);
  a.barrier = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) +
                                          layout_counter_bytes(L.T, L.E));
  a.tokens_per_expert = L.tokens_per_expert;
  a.offsets = L.offsets;
  a.totals = L.totals;
  a.row_token = L.row_token;
  a.row_expert = L.row_expert;
  a.row_weight = L.row_weight;
  a.token_row = L.token_row;
  a.status = L.status;
  const size_t smem = layout_smem_bytes(L.E);
  // Up to LAYOUT_REDUNDANT_CHUNKS chunks (T <= 256): one CTA per chunk, each
  // counting every chunk itself, so there is no grid barrier, no memset and
  // no cooperative launch, and the kernel takes part in programmatic
  // dependent launch.  Larger layers use the cooperative kernel.
  if (a.chunks <= LAYOUT_REDUNDANT_CHUNKS &&
      smem + static_cast<size_t>(a.chunks) * a.E * sizeof(int) <= 48 * 1024) {
    // A decode-sized row pass (a few rows of a few KB, one or two chunks)
    // costs a single CTA less than a launch of its own.
    const long long items = L.T + L.capacity;
    const long long bytes = x_disp ? items * H * 2 : 0;
    if (rows_done && a.chunks <= 2 && items <= LAYOUT_FUSED_ITEMS && bytes <= LAYOUT_FUSED_BYTES) {
      a.rows = true;
      *rows_done = true;
    }
    return launch_layout_mode<LAYOUT_SINGLE>(a, smem, s);
  }
  return launch_layout_mode<LAYOUT_ALL>(a, smem, s);
}

cudaError_t launch_row_gather(const uint16_t* src, const moe_layout& L, int H, uint16_t* dst,
                              bool from_offsets, const uint16_t* o_save, float* grad_w,
                              cudaStream_t s, bool scale) {
  const long long C = L.capacity;
  const long long items = static_cast<long long>(L.T) + C;
  if (items == 0) return cudaSuccess;
  const int threads = 256;
  const long long need = (items + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
  if (from_offsets) {
    const size_t smem = (2 * L.E + 1) * sizeof(int);
    return launch_dependent(row_scatter_kernel<true, false>, blocks, threads, smem, s, src, L.T, L.K,
                            H, L.E, C, L.token_row, L.offsets, L.tokens_per_expert, L.row_token,
                            L.row_expert, L.row_weight, dst, static_cast<const uint16_t*>(nullptr),
                            static_cast<float*>(nullptr), L.status);
  } else if (grad_w && scale) {
    row_scatter_kernel<false, true, true><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, L.row_weight,
        dst, o_save, grad_w, L.status);
  } else if (scale) {
    row_scatter_kernel<false, false, true><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, L.row_weight,
        dst, nullptr, nullptr, L.status);
  } else if (grad_w) {
    row_scatter_kernel<false, true><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, nullptr,
        dst, o_save, grad_w, L.status);
  } else {
    row_scatter_kernel<false, false><<<blocks, threads, 0, s>>>(
        src, L.T, L.K, H, L.E, C, L.token_row, nullptr, nullptr, L.row_token, nullptr, nullptr,
        dst, nullptr, nullptr, L.status);
  }
  return cudaGetLastError();
}

}  // namespace moe
