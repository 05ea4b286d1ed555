// a1-a4 in one cooperative launch: from the top-k choices (or the multihot
// routing map) to the expanded layout with every row copied, as bf16 or (the
// FP8 dispatch) as e4m3 codes with one scale per row.
//
// "feat: add hybridep (NVIDIA-NeMo/Automodel #1333)", Changelog: top-k indices
// become multihot routing data (a routing_map and fp32 per-(token, expert)
// probs); review of dispatch(): tokens_per_expert, rows padded per expert to
// pad_multiple, the permuted-row total as the sum of the counts.
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds: Expanded layout (one row per (token, expert) pair,
// grouped by expert, carrying the pair's weight); Eager vs captured (the exact
// row count read back to the host, or a worst-case buffer whose unused rows
// are zero and belong to the sentinel expert).
//
// One launch, every CTA resident, two bounded grid barriers:
//   A. Per 32-token chunk, each expert's 32-bit token mask (shared-memory
//      atomics).
//   -- barrier --
//   B. One warp per expert: each chunk's start inside the expert's group (an
//      exclusive scan of the masks' popcounts) and the expert's count.
//   -- barrier --
//   C. Every CTA forms the padded offsets and each expert's pad-row prefix
//      (block scans); CTA 0 writes offsets and totals and hands R, N and the
//      status word to a host-synced caller through mapped memory.
//   D. Items: the T tokens, then the C - N pad and spare rows, one warp each.
//      A token's warp starts copying the token's x row into its 4 KiB
//      shared-memory slot (cp.async), then (from the top-k choices, after
//      writing the token's multihot row: routing_map, probs, winner_slot)
//      finds its experts in ascending order, places each pair
//      at offsets[e] + start[e][chunk] + popcount(mask below the token) and
//      writes the rows' metadata and token_row while the copy lands; one lane
//      then hands each of the token's rows to the TMA engine as a bulk copy
//      (cp.async.bulk shared -> global), so a warp issues a few instructions
//      per row.  A pad or spare row is a bulk copy of a zeroed slot and gets
//      the sentinel metadata.
// The two barriers release the CTAs through replicated flags and phase B
// publishes each count in replicated copies, so the 600-odd CTAs do not all
// poll or read one L2 line.  Nothing is loaded ahead for phase D: in-kernel
// %globaltimer stamps at T = 4096 showed that loading each warp's first x row
// before barrier 1 (16.8 MB at once) stretched phase A from about 2 to 12 us,
// because it fills the memory pipeline of the SMs whose CTAs are still in
// phase A.  The multihot rows are written in phase D for the same reason: as
// stores in phase A, whose new L2 lines wait for the write-back of the
// previous kernel's dirty lines, they added about 6 us to it.
// No atomic decides a position, so the result does not depend on scheduling,
// and rows inside a group are in ascending token order.  When the rows do not
// fit (R > capacity) phase D writes nothing.

#include "common.cuh"
#include "coop.cuh"
#include "fp8_quant.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int FD_THREADS = 256;
constexpr int FD_WARPS = FD_THREADS / 32;
constexpr int FD_PF = 8;         // 16-byte vectors per lane of one 4 KiB piece of a row
constexpr int FD_MAX_K = 128;    // slots of the per-warp row list (K <= 127)
constexpr int FD_SLOT = 32 * FD_PF * 16;  // bytes of a warp's staging slot (4 KiB)
constexpr int FD_REP = BARRIER_REP;       // copies of each count, one per group of CTAs
static_assert(BARRIER_WORDS * 4 <= FUSED_BARRIER_BYTES, "barrier words fit their workspace region");

__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}

enum FusedInput : int { IN_MAP = 0, IN_TOPK = 1 };

struct FusedArgs {
  const uint16_t* x;         // [T, H]; NULL: the layout alone, no rows copied
  const uint8_t* map;        // [T, E] (IN_MAP)
  const float* probs;        // [T, E] (IN_MAP)
  const int64_t* topk_idx;   // [T, K] (IN_TOPK)
  const float* topk_probs;   // [T, K] (IN_TOPK)
  uint8_t* map_out;          // [T, E] multihot outputs (IN_TOPK)
  float* probs_out;
  int8_t* winner_out;
  int T, E, K, P, H, chunks;
  long long capacity;
  uint32_t* masks;    // [E][chunks] token mask of each chunk
  int* starts;        // [E][chunks] the chunk's first row inside the expert's group
  unsigned* barrier;  // BARRIER_WORDS, zeroed before the launch
  int* counts_rep;    // [FD_REP][E] copies of tokens_per_expert
  int* tokens_per_expert;
  int* offsets;
  int* totals;
  int* row_token;
  int* row_expert;
  float* row_weight;
  int* token_row;
  int* status;
  int* readback;      // {R, N, status} in host-mapped memory, or NULL
  uint16_t* x_disp;
  uint8_t* x_q;       // FP8 rows: e4m3 codes [C, H] and one fp32 scale per row [C]
  float* x_scale;
};

// Token t's K slots, slot k in lane k % 32, register k / 32 (-1 = none); an
// index outside [-1, E) counts as -1 and, with report_bad, sets the status bit.
__device__ __forceinline__ void load_slots(const FusedArgs& a, long long t, int lane, int (&ek)[4],
                                           float (&pk)[4], bool report_bad) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = lane + 32 * j;
    ek[j] = -1;
    pk[j] = 0.f;
    if (k < a.K) {
      long long v = __ldg(a.topk_idx + t * a.K + k);
      if (v < -1 || v >= a.E) {
        if (report_bad) report(a.status, MOE_DEVERR_BAD_INDEX);
        v = -1;
      }
      ek[j] = static_cast<int>(v);
      pk[j] = __ldg(a.topk_probs + t * a.K + k);
    }
  }
}

__device__ __forceinline__ int pick(const int (&v)[4], int j) {
  return j == 0 ? v[0] : j == 1 ? v[1] : j == 2 ? v[2] : v[3];
}

// The row of pair (t, e): offsets[e] + the chunk's start in e's group + the
// number of the chunk's earlier tokens routed to e.
__device__ __forceinline__ int pair_row(const FusedArgs& a, const int* s_off, long long t, int e) {
  const long long c = t >> 5;
  const int tl = static_cast<int>(t & 31);
  const long long i = static_cast<long long>(e) * a.chunks + c;
  const uint32_t m = __ldcg(a.masks + i);
  return s_off[e] + __ldcg(a.starts + i) + __popc(m & ((1u << tl) - 1u));
}

// FP8: the rows are written as e4m3 codes with one scale per row (the
// rowwise format of fp8_quant.cuh) to x_q / x_scale instead of bf16 to x_disp.
template <int IN, bool FP8>
__global__ void __launch_bounds__(FD_THREADS, 4) dispatch_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(128) uint8_t fd_smem[];
  __shared__ int s_warp[33];
  __shared__ int s_ok;
  const int E = a.E, K = a.K;
  // The next kernel (the experts, launched for programmatic dependent launch)
  // may be scheduled now: it sets up on the SMs this grid frees and waits for
  // the whole grid's completion before it reads any of its outputs.  This
  // kernel itself follows a memset in stream order, so it waits for nothing.
  griddep_launch_dependents();
  // staging slots first (16-byte aligned for the bulk copies), then the tables
  uint8_t* s_slots = fd_smem;                                            // [FD_WARPS][FD_SLOT]
  uint8_t* s_zero = fd_smem + FD_WARPS * FD_SLOT;                        // [FD_SLOT] zeros
  uint32_t* s_tmask = reinterpret_cast<uint32_t*>(s_zero + FD_SLOT);     // [E]
  int* s_off = reinterpret_cast<int*>(s_tmask + E);                      // [E + 1]
  int* s_cnt = s_off + E + 1;                                            // [E]
  int* s_pad = s_cnt + E;                                                // [E + 1] pad rows before e
  int* s_rows = s_pad + E + 1;                                           // [FD_WARPS][FD_MAX_K]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gwarp = static_cast<long long>(blockIdx.x) * FD_WARPS + warp;
  const long long gwarps = static_cast<long long>(gridDim.x) * FD_WARPS;
  const int V = a.H >> 8;  // 16-byte vectors per lane of one row

  if (FP8 ? a.x_q != nullptr : a.x_disp != nullptr) {  // the zero slot of the pad and spare rows
    for (int i = threadIdx.x; i < FD_SLOT / 16; i += FD_THREADS)
      reinterpret_cast<uint4*>(s_zero)[i] = make_uint4(0, 0, 0, 0);
    fence_async_shared();
  }

  // ---- A. per chunk, each expert's token mask
  for (int c = blockIdx.x; c < a.chunks; c += gridDim.x) {
    const long long t0 = static_cast<long long>(c) * LAYOUT_CHUNK;
    const int nt = static_cast<int>(min(static_cast<long long>(LAYOUT_CHUNK), a.T - t0));
    for (int e = threadIdx.x; e < E; e += FD_THREADS) s_tmask[e] = 0u;
    __syncthreads();
    if constexpr (IN == IN_MAP) {
      const int E4 = E >> 2;
      const uint32_t* words = reinterpret_cast<const uint32_t*>(a.map + t0 * E);
      for (int i = threadIdx.x; i < nt * E4; i += FD_THREADS) {
        const uint32_t w = __ldg(words + i);
        if (w == 0u) continue;
        const int tl = i / E4, e0 = 4 * (i - tl * E4);
#pragma unroll
        for (int d = 0; d < 4; ++d)
          if ((w >> (8 * d)) & 0xffu) atomicOr(s_tmask + e0 + d, 1u << tl);
      }
    } else if (K <= 32) {
      // the warp's four tokens (warp, warp + 8, ...): every slot load issued at once
      int em[4];
      float pm[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tl = warp + FD_WARPS * m;
        em[m] = -1;
        pm[m] = 0.f;
        if (tl < nt && lane < K) {
          const long long o = (t0 + tl) * K + lane;
          long long v = __ldg(a.topk_idx + o);
          pm[m] = __ldg(a.topk_probs + o);
          if (v < -1 || v >= E) {
            report(a.status, MOE_DEVERR_BAD_INDEX);
            v = -1;
          }
          em[m] = static_cast<int>(v);
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tl = warp + FD_WARPS * m;
        if (tl < nt && em[m] >= 0) atomicOr(s_tmask + em[m], 1u << tl);
      }
    } else {
      for (int tl = warp; tl < nt; tl += FD_WARPS) {
        int ek[4];
        float pk[4];
        load_slots(a, t0 + tl, lane, ek, pk, true);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (ek[j] >= 0) atomicOr(s_tmask + ek[j], 1u << tl);
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += FD_THREADS)
      a.masks[static_cast<long long>(e) * a.chunks + c] = s_tmask[e];
    __syncthreads();  // before the next chunk clears s_tmask
  }

  if (!grid_barrier_rep(a.barrier, 1, a.status, &s_ok)) return;

  // ---- B. per expert, each chunk's start in the group and the count
  for (long long e = gwarp; e < E; e += gwarps) {
    const uint32_t* mrow = a.masks + e * a.chunks;
    int* srow = a.starts + e * a.chunks;
    int run = 0;
    // 8 coalesced steps of 32 chunks per batch: the loads are issued together
    for (int b0 = 0; b0 < a.chunks; b0 += 8 * 32) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = b0 + 32 * i + lane;
        v[i] = c < a.chunks ? __popc(__ldcg(mrow + c)) : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = b0 + 32 * i + lane;
        const int incl = warp_inclusive_scan(v[i], lane);
        if (c < a.chunks) srow[c] = run + incl - v[i];
        run += __shfl_sync(FULL_MASK, incl, 31);
      }
    }
    if (lane == 0) a.tokens_per_expert[e] = run;
    if (lane < FD_REP) a.counts_rep[lane * E + e] = run;
  }
  if (!grid_barrier_rep(a.barrier, 2, a.status, &s_ok)) return;

  // ---- C. padded offsets and pad-row prefixes; thread i owns experts 4i .. 4i + 3
  int R, pad_total;
  {
    const int* counts = a.counts_rep + (blockIdx.x % FD_REP) * E;
    int cnt[4], padded[4], psum = 0, qsum = 0;
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const int e = 4 * threadIdx.x + d;
      cnt[d] = e < E ? __ldcg(counts + e) : 0;
      padded[d] = ((cnt[d] + a.P - 1) / a.P) * a.P;
      psum += padded[d];
      qsum += padded[d] - cnt[d];
    }
    int off = block_exclusive_scan(psum, s_warp, &R);
    __syncthreads();  // s_warp is reused by the second scan
    int pre = block_exclusive_scan(qsum, s_warp, &pad_total);
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      const int e = 4 * threadIdx.x + d;
      if (e < E) {
        s_off[e] = off;
        s_cnt[e] = cnt[d];
        s_pad[e] = pre;
      }
      off += padded[d];
      pre += padded[d] - cnt[d];
    }
    if (threadIdx.x == 0) {
      s_off[E] = R;
      s_pad[E] = pad_total;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int e = threadIdx.x; e <= E; e += FD_THREADS) a.offsets[e] = s_off[e];
      if (threadIdx.x == 0) {
        const int N = R - pad_total;
        a.totals[0] = R;
        a.totals[1] = N;
        if (R > a.capacity) report(a.status, MOE_DEVERR_CAPACITY);
        if (a.readback) {  // R last, after a system-scope fence: the host waits for it
          volatile int* rb = a.readback;
          rb[1] = N;
          rb[2] = *reinterpret_cast<volatile int*>(a.status);
          __threadfence_system();
          rb[0] = R;
        }
      }
    }
  }
  if (R > a.capacity) return;  // the rows do not fit: nothing is placed

  // ---- D. tokens, then pad and spare rows
  const long long C = a.capacity;
  const long long N = R - pad_total;
  const long long items = a.T + (C - N);
  int* rows = s_rows + warp * FD_MAX_K;
  const uint32_t slot = smem_u32(s_slots + warp * FD_SLOT);
  const uint32_t zero = smem_u32(s_zero);
  const long long row_bytes = 2LL * a.H;
  for (long long it = gwarp; it < items; it += gwarps) {
    if (it < a.T) {
      const long long t = it;
      // the first 4 KiB of x[t] start into the warp's slot now (cp.async, no
      // registers held) and land while the token's rows are placed below
      const uint4* src = a.x ? reinterpret_cast<const uint4*>(a.x + t * a.H) : nullptr;
      if (!FP8 && src) {
        if (lane == 0) tma_store_wait_read<0>();  // the slot's previous copies have read it
        __syncwarp();
        const int nv = min(FD_PF, V);
#pragma unroll
        for (int i = 0; i < FD_PF; ++i)
          if (i < nv) cp_async_16(slot + 16 * (lane + 32 * i), src + lane + 32 * i, 16u);
        cp_async_commit();
      }
      int n = 0;  // the token's rows, in ascending expert order, go to rows[0 .. n)
      if constexpr (IN == IN_MAP) {
        const int E4 = E >> 2;
        const uint32_t* mrow = reinterpret_cast<const uint32_t*>(a.map + t * E);
        for (int s0 = 0; s0 < E4; s0 += 32) {
          const int w4 = s0 + lane;
          const uint32_t w = w4 < E4 ? __ldg(mrow + w4) : 0u;
          int bits = 0;
#pragma unroll
          for (int d = 0; d < 4; ++d) bits |= ((w >> (8 * d)) & 0xffu) ? (1 << d) : 0;
          const int cnt = __popc(bits);
          const int incl = warp_inclusive_scan(cnt, lane);
          int j = n + incl - cnt;
#pragma unroll
          for (int d = 0; d < 4; ++d) {
            if (!((bits >> d) & 1)) continue;
            const int e = 4 * w4 + d;
            if (j < K) {
              const int r = pair_row(a, s_off, t, e);
              rows[j] = r;
              a.token_row[t * K + j] = r;
              if (MOE_IN_BOUNDS(r >= 0 && r < C, a.status) && r < C) {
                a.row_token[r] = static_cast<int>(t);
                a.row_expert[r] = e;
                a.row_weight[r] = __ldg(a.probs + t * E + e);
              }
            } else {
              report(a.status, MOE_DEVERR_BAD_INDEX);  // more experts than slots
            }
            ++j;
          }
          n += __shfl_sync(FULL_MASK, incl, 31);
        }
        n = min(n, K);
      } else {
        int ek[4];
        float pk[4];
        load_slots(a, t, lane, ek, pk, false);
        // the token's multihot row, for the backward (nothing in this kernel reads it)
        write_multihot_row(t, ek, pk, K, E, lane, a.map_out, a.probs_out, a.winner_out);
        // A slot is its expert's winner unless a later slot names the same expert.
        bool win[4] = {ek[0] >= 0, ek[1] >= 0, ek[2] >= 0, ek[3] >= 0};
        for (int k2 = 0; k2 < K; ++k2) {
          const int e2 = __shfl_sync(FULL_MASK, pick(ek, k2 >> 5), k2 & 31);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (k2 > lane + 32 * j && e2 == ek[j]) win[j] = false;
        }
        // rank of a winner = winners with a smaller expert
        int rank[4] = {0, 0, 0, 0};
        for (int k2 = 0; k2 < K; ++k2) {
          const int jj = k2 >> 5;
          const int e2 = __shfl_sync(FULL_MASK, pick(ek, jj), k2 & 31);
          const int w2 = __shfl_sync(FULL_MASK, (jj == 0 ? win[0] : jj == 1 ? win[1] : jj == 2 ? win[2] : win[3]) ? 1 : 0,
                                     k2 & 31);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (w2 && e2 < ek[j]) ++rank[j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          n += __popc(__ballot_sync(FULL_MASK, win[j]));
          if (win[j]) {
            const int r = pair_row(a, s_off, t, ek[j]);
            rows[rank[j]] = r;
            a.token_row[t * K + rank[j]] = r;
            if (MOE_IN_BOUNDS(r >= 0 && r < C && rank[j] < K, a.status) && r < C) {
              a.row_token[r] = static_cast<int>(t);
              a.row_expert[r] = ek[j];
              a.row_weight[r] = pk[j];
            }
          }
        }
      }
      for (int j = n + lane; j < K; j += 32) a.token_row[t * K + j] = -1;
      __syncwarp();
      if (a.x == nullptr) continue;
      if constexpr (FP8) {
        // the token's codes, quantized once with the row's scale, 2 KiB at a
        // time into the warp's slot, one lane bulk-copying them to every row
        const float scale = row_scale(src, V, lane);
        for (int j = lane; j < n; j += 32) {
          const int r = rows[j];
          if (r >= 0 && r < C) a.x_scale[r] = scale;
        }
        for (int v0 = 0; v0 < V; v0 += FD_PF) {
          const int nv = min(FD_PF, V - v0);
          if (lane == 0) tma_store_wait_read<0>();  // the slot's previous copies have read it
          __syncwarp();
#pragma unroll
          for (int i = 0; i < FD_PF; ++i)
            if (i < nv) {
              const uint2 c = quantize8(__ldg(src + lane + 32 * (v0 + i)), scale);
              asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(slot + 8 * (lane + 32 * i)), "r"(c.x), "r"(c.y)
                           : "memory");
            }
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            for (int j = 0; j < n; ++j) {
              const int r = rows[j];
              if (r < 0 || r >= C) continue;
              bulk_store(a.x_q + r * a.H + 256LL * v0, slot, 256u * nv);
            }
            tma_store_commit();
          }
        }
        continue;
      }
      // x[t] into each of the token's rows, 4 KiB at a time: the lanes put the
      // piece into the warp's slot (the first one is already on its way), one
      // lane bulk-copies it to every row
      for (int v0 = 0; v0 < V; v0 += FD_PF) {
        const int nv = min(FD_PF, V - v0);
        if (v0 == 0) {
          cp_async_wait_all();
        } else {
          uint4 xr[FD_PF];
#pragma unroll
          for (int i = 0; i < FD_PF; ++i)
            if (i < nv) xr[i] = __ldg(src + lane + 32 * (v0 + i));
          if (lane == 0) tma_store_wait_read<0>();  // the slot's previous copies have read it
          __syncwarp();
#pragma unroll
          for (int i = 0; i < FD_PF; ++i)
            if (i < nv)
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(slot + 16 * (lane + 32 * i)),
                           "r"(xr[i].x), "r"(xr[i].y), "r"(xr[i].z), "r"(xr[i].w)
                           : "memory");
        }
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          for (int j = 0; j < n; ++j) {
            const int r = rows[j];
            if (r < 0 || r >= C) continue;
            bulk_store(reinterpret_cast<uint8_t*>(a.x_disp) + r * row_bytes + 512LL * v0, slot, 512u * nv);
          }
          tma_store_commit();
        }
      }
    } else {
      // pad item p: a pad row of some expert's group, or a spare row after R
      const long long p = it - a.T;
      long long r;
      if (p < pad_total) {
        int lo = 0, hi = E;  // s_pad[lo] <= p < s_pad[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_pad[mid] <= p) lo = mid; else hi = mid;
        }
        r = s_off[lo] + s_cnt[lo] + (p - s_pad[lo]);
      } else {
        r = R + (p - pad_total);
      }
      if (lane != 0 || !MOE_IN_BOUNDS(r >= 0 && r < C, a.status) || r >= C) continue;
      a.row_token[r] = -1;
      a.row_expert[r] = E;
      a.row_weight[r] = 0.f;
      if constexpr (FP8) {
        if (a.x_q == nullptr) continue;
        a.x_scale[r] = 0.f;  // zero codes, scale 0
        for (int v0 = 0; v0 < V; v0 += FD_PF)
          bulk_store(a.x_q + r * a.H + 256LL * v0, zero, 256u * min(FD_PF, V - v0));
      } else {
        if (a.x_disp == nullptr) continue;
        for (int v0 = 0; v0 < V; v0 += FD_PF)
          bulk_store(reinterpret_cast<uint8_t*>(a.x_disp) + r * row_bytes + 512LL * v0, zero,
                     512u * min(FD_PF, V - v0));
      }
      tma_store_commit();
    }
  }
  if (lane == 0) tma_store_wait_all();  // every bulk copy done before the CTA exits
  __syncwarp();
}

size_t fused_smem_bytes(int E) {
  return static_cast<size_t>(FD_WARPS + 1) * FD_SLOT + (static_cast<size_t>(4) * E + 2) * sizeof(int) +
         static_cast<size_t>(FD_WARPS) * FD_MAX_K * sizeof(int);
}

// CTAs of dispatch_fused_kernel<IN, FP8> resident at once on the current
// device (the last answer is kept per thread).
template <int IN, bool FP8>
int fused_resident_ctas(size_t smem) {
  static thread_local int last_dev = -1;
  static thread_local size_t last_smem = 0;
  static thread_local int last_ctas = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev == last_dev && smem == last_smem) return last_ctas;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_fused_kernel<IN, FP8>, FD_THREADS, smem) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  last_dev = dev;
  last_smem = smem;
  last_ctas = per_sm * sm_count();
  return last_ctas;
}

template <int IN, bool FP8 = false>
cudaError_t launch_fused(FusedArgs& a, void* workspace, cudaStream_t s) {
  const size_t cb = layout_counter_bytes(a.T, a.E);
  char* ws = static_cast<char*>(workspace);
  a.masks = reinterpret_cast<uint32_t*>(ws);
  a.starts = reinterpret_cast<int*>(ws + cb);
  a.barrier = reinterpret_cast<unsigned*>(ws + 2 * cb);
  a.counts_rep = reinterpret_cast<int*>(ws + 2 * cb + FUSED_BARRIER_BYTES);
  cudaError_t err = cudaMemsetAsync(a.barrier, 0, BARRIER_WORDS * sizeof(unsigned), s);
  if (err != cudaSuccess) return err;
  const size_t smem = fused_smem_bytes(a.E);
  static bool configured[64] = {};  // one table per instantiation
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(dispatch_fused_kernel<IN, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(fused_smem_bytes(1024)));
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  // phase D has T + (C - N) warp items, and N is at most T * K; a CTA per 8
  // of them, at most every resident CTA (more CTAs than the work needs only
  // make the two grid barriers slower: decode T = 1024 took 38.9 us with all
  // 608 resident CTAs)
  const long long tk = static_cast<long long>(a.T) * a.K;
  const long long items = a.T + (a.capacity > tk ? a.capacity - tk : 0);
  const long long want = (items + FD_WARPS - 1) / FD_WARPS;
  const int resident = fused_resident_ctas<IN, FP8>(smem);
  const int grid = static_cast<int>(want < resident ? (want > a.chunks ? want : a.chunks) : resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid > 0 ? grid : 1);
  cfg.blockDim = dim3(FD_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dispatch_fused_kernel<IN, FP8>, a);
}

void fill_common(FusedArgs& a, const moe_layout& L, int H, const uint16_t* x, uint16_t* x_disp,
                 int* readback) {
  a.x = x_disp ? x : nullptr;
  a.x_disp = x_disp;
  a.T = L.T;
  a.E = L.E;
  a.K = L.K;
  a.P = L.pad_multiple;
  a.H = H;
  a.chunks = static_cast<int>(layout_chunks(L.T));
  a.capacity = L.capacity;
  a.tokens_per_expert = L.tokens_per_expert;
  a.offsets = L.offsets;
  a.totals = L.totals;
  a.row_token = L.row_token;
  a.row_expert = L.row_expert;
  a.row_weight = L.row_weight;
  a.token_row = L.token_row;
  a.status = L.status;
  a.readback = readback;
}

}  // namespace

bool dispatch_fused_fits(const moe_layout& L) {
  // the cooperative launch is for layers of more than 8 chunks (smaller ones
  // take the barrier-free layout) whose per-CTA arrays fit shared memory
  return layout_chunks(L.T) > 8 && fused_smem_bytes(L.E) <= fused_smem_bytes(1024);
}

cudaError_t launch_dispatch_fused_map(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                                      int H, const uint16_t* x, uint16_t* x_disp, int* readback,
                                      cudaStream_t s) {
  FusedArgs a = {};
  fill_common(a, L, H, x, x_disp, readback);
  a.map = routing_map;
  a.probs = probs;
  return launch_fused<IN_MAP>(a, L.workspace, s);
}

cudaError_t launch_dispatch_fused_map_fp8(const uint8_t* routing_map, const float* probs, const moe_layout& L,
                                          int H, const uint16_t* x, uint8_t* x_q, float* x_scale, int* readback,
                                          cudaStream_t s) {
  FusedArgs a = {};
  fill_common(a, L, H, x, nullptr, readback);
  a.x = x;
  a.x_q = x_q;
  a.x_scale = x_scale;
  a.map = routing_map;
  a.probs = probs;
  return launch_fused<IN_MAP, true>(a, L.workspace, s);
}

cudaError_t launch_dispatch_fused_topk(const int64_t* topk_idx, const float* topk_probs,
                                       uint8_t* routing_map, float* probs, int8_t* winner,
                                       const moe_layout& L, int H, const uint16_t* x, uint16_t* x_disp,
                                       int* readback, cudaStream_t s) {
  FusedArgs a = {};
  fill_common(a, L, H, x, x_disp, readback);
  a.topk_idx = topk_idx;
  a.topk_probs = topk_probs;
  a.map_out = routing_map;
  a.probs_out = probs;
  a.winner_out = winner;
  return launch_fused<IN_TOPK>(a, L.workspace, s);
}

cudaError_t launch_dispatch_fused_topk_fp8(const int64_t* topk_idx, const float* topk_probs,
                                           uint8_t* routing_map, float* probs, int8_t* winner,
                                           const moe_layout& L, int H, const uint16_t* x, uint8_t* x_q,
                                           float* x_scale, int* readback, cudaStream_t s) {
  FusedArgs a = {};
  fill_common(a, L, H, x, nullptr, readback);
  a.x = x;
  a.x_q = x_q;
  a.x_scale = x_scale;
  a.topk_idx = topk_idx;
  a.topk_probs = topk_probs;
  a.map_out = routing_map;
  a.probs_out = probs;
  a.winner_out = winner;
  return launch_fused<IN_TOPK, true>(a, L.workspace, s);
}

}  // namespace moe
