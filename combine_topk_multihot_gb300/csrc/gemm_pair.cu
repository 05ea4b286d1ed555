// a5: the SwiGLU experts' two grouped GEMMs on CTA pairs, with each expert's
// rows on the N side of the tensor-core MMA.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", Expanded layout: an expert multiplies only the rows routed to it,
// and the routing weight scales each row's output inside the expert step.
//
//   GEMM1 (per expert e, over its rows):  [g | u] = x_disp W1[e]^T,
//          h = bf16(silu(g) * u)                  (optionally g, u saved)
//   GEMM2:  o = h W2[e]^T,  y = bf16(w_row * o)   (optionally o saved)
//
// The tensor cores compute the transposed products, acc = W[e] x^T: one
// accumulator column per expert row.  A tile is 256 weight rows (the MMA's
// M, 128 in each CTA of a pair) by one chunk of the expert's rows (the MMA's
// N: up to 256, a multiple of 16, half of them loaded by each CTA).  An
// expert's rows are cut into chunks of 256 and a last chunk of the rest, so
// a tile covers fewer than 16 rows past the ones it owns.  With the rows on
// the M side, as in the other expert kernels, a tile is 256 rows, and an
// expert of 257 rows costs two full tiles: at about 256 rows per expert that
// is half again the MMA work.  (Cutting the rows into equal chunks instead,
// e.g. 2 x 144 for 272 rows, was slower: MMAs with N between 128 and 256
// ran below the rate of N = 256.)
//
// GEMM1 loads the gate and up rows of W1 interleaved (a 5-D tensor map):
// weight row 2j of a CTA's 128 is gate row f + j and row 2j + 1 is up row
// f + j.  Lanes 2j and 2j + 1 of tensor memory then hold the gate and up
// values of one h column, and the SwiGLU pairs them with one shuffle.
//
// Roles (one CTA per SM, clusters of two, persistent over a tile list built
// on the device from the counts and offsets, so no host sync is needed):
//   * warp 0 issues the TMA loads of both operands into a ring of 64 KiB
//     stages of 128 K columns (weights 32 KiB, expert rows up to 32 KiB),
//     completing on the even CTA's barrier;
//   * warp 1 of the even CTA issues the pair's tcgen05.mma (cta_group::2);
//   * warps 2-9 are the epilogue: two warps per 32-lane quarter of tensor
//     memory, taking alternate 32-column chunks.  An epilogue thread holds
//     one output column for 32 expert rows, and each store instruction of a
//     warp writes whole row segments (64 bytes in GEMM2, 32 in GEMM1);
//   * two 256-column accumulators let the epilogue of one tile overlap the
//     MMAs of the next;
//   * every wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT and the CTA
//     drains its in-flight work, frees tensor memory and exits.
// Rows written: each expert's valid rows, plus (when g, u are saved for the
// backward) the pad rows of its group, which come out zero from the zero pad
// rows of x_disp.  Spare rows are never written.

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

// Readiness of h per row chunk (an expert's 256-row chunk), so that the down
// launch can start a tile as soon as the gate/up tiles of its chunk are
// written rather than when the whole gate/up launch has finished: each
// gate/up epilogue warp adds one to its tile's chunk once its stores of the
// tile have completed, and the down launch's producer waits for the count of
// all the chunk's gate/up tiles.  16 slots rotate between launch pairs (a
// launch pair's down launch clears its slot as its last CTA finishes, so a
// slot is clean for its next use 16 launch pairs later).  2 x 128 KiB of
// device memory per GPU, held from library load until the process exits.
constexpr int HR_SLOTS = 16;
constexpr int HR_CAP = 2048;  // row chunks per layer
static __device__ __align__(128) int g_h_ready[HR_SLOTS][HR_CAP];
static __device__ unsigned int g_h_done[HR_SLOTS];

namespace {

constexpr int BK = 64;                           // bf16 elements per 128-byte swizzled row
constexpr int KSUB = 2;                          // 64-column sub-tiles per stage (K = 128)
constexpr int UMMA_K = 16;                       // K per tcgen05.mma for 16-bit inputs
constexpr int MAX_N = 256;                       // expert rows per tile
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS);
constexpr int MAX_STAGES = 8;
constexpr int SMEM_LIMIT = 232448;
constexpr int W_SUB = 128 * BK * 2;              // a CTA's 128 weight rows x 64 columns
constexpr int W_BYTES = KSUB * W_SUB;            // ... x 128 columns: one stage
constexpr int R_BYTES = KSUB * (MAX_N / 2) * BK * 2;  // its up to 128 expert rows x 128 columns
constexpr int STAGE_BYTES = W_BYTES + R_BYTES;
constexpr int TMEM_COLS = 2 * MAX_N;             // double-buffered accumulator
constexpr int STAGING_PER_WARP = 4096;           // epilogue staging for TMA stores
constexpr int STAGING_BYTES = EPI_WARPS * STAGING_PER_WARP;

enum Epilogue { EPI_SWIGLU = 0, EPI_WEIGHTED = 1 };

struct PairArgs {
  const int* counts;       // [E] rows of each expert
  const int* offsets;      // [E+1] group start rows
  const float* row_weight; // [C]
  int E;
  int k_blocks;            // contraction length / BK
  int n_fblocks;           // 256-row weight blocks per expert
  int w_rows_per_expert;   // GEMM2: rows of W2 per expert (H)
  uint16_t* out0;          // GEMM1: h [C, I]     GEMM2: y [C, H]
  int ld0;
  uint16_t* out1;          // GEMM1: gu_save [C, 2I] (nullable)   GEMM2: o_save [C, H] (nullable)
  int ld1;
  int I;                   // GEMM1: offset of the up half in gu_save
  int write_pad;           // also cover the pad rows of each expert's group
  int* status;
  int* ready;              // per row chunk: h-ready signals (NULL: the down launch waits for the whole gate/up launch)
  unsigned int* done;      // the down launch's finished CTAs; the last one clears `ready`
  int ready_target;        // signals that make a chunk ready: gate/up tiles per chunk x 16 epilogue warps
};

// Barriers and scalars; the per-expert tables (offsets [E+1], counts [E],
// tile prefix [E+1]) follow it in shared memory.
struct Smem {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int last;  // the down launch's last CTA (it clears the readiness counters)
};

constexpr size_t smem_bytes(int stages, int E) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(stages) * STAGE_BYTES + STAGING_BYTES + sizeof(Smem) +
         static_cast<size_t>(3 * E + 2) * sizeof(int);
}

struct Tile {
  int e, fb;   // expert, 256-row weight block
  int row0;    // first expert row of the chunk (row of the expanded layout)
  int rows;    // expert rows of the chunk
  int n;       // MMA N: rows rounded up to 16
  int chunk;   // the chunk's index among all experts' chunks
};

// Rows an expert's tiles cover: its valid rows, or its whole padded group.
__device__ __forceinline__ int covered_rows(const int* s_off, const int* s_cnt, int e, int write_pad) {
  return write_pad ? s_off[e + 1] - s_off[e] : s_cnt[e];
}

__device__ __forceinline__ int chunks_of(int n) { return (n + MAX_N - 1) / MAX_N; }

__device__ __forceinline__ Tile decode_tile(const int* s_off, const int* s_cnt, const int* s_pre, int E,
                                            int n_fb, int write_pad, int tile) {
  int lo = 0, hi = E;  // s_pre[lo] <= tile < s_pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pre[mid] <= tile) lo = mid; else hi = mid;
  }
  const int ne = covered_rows(s_off, s_cnt, lo, write_pad);
  const int local = tile - s_pre[lo];
  const int chunk = local / n_fb;
  Tile t;
  t.e = lo;
  t.fb = local - chunk * n_fb;
  t.row0 = s_off[lo] + chunk * MAX_N;
  t.chunk = s_pre[lo] / n_fb + chunk;
  t.rows = ne - chunk * MAX_N < MAX_N ? ne - chunk * MAX_N : MAX_N;
  t.n = (t.rows + 15) & ~15;
  return t;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Tensor maps of the expert rows with boxes of 32, 64, 96 and 128 rows.
struct RowMaps {
  const CUtensorMap* box[4];
};

// The loads of one tile: for each 128-column K step, wait for a free stage,
// then load the CTA's 128 weight rows and its ROWS expert rows, all
// completing on the even CTA's barrier, which expects both CTAs' bytes.  Each
// operand comes as one TMA box of two 64-column sub-tiles: a CTA's TMA engine
// takes a roughly fixed time per box, so 32 KiB boxes stream twice as fast
// from L2 as 16 KiB ones (a probe: 134 against 71 GB/s per SM).  The rows box
// is ROWS rounded up to 32 (the MMA reads only the first ROWS; the rest are
// the next rows of the layout, or zeros past its end).  ROWS is a template
// argument so that the issue sequence has a constant shape (with the box
// choice made at run time the same loads ran about a quarter slower).
// Transaction bytes of one stage of a tile with N expert rows, both CTAs.
__device__ __forceinline__ uint32_t stage_tx(int n) {
  const int box = (n / 2 + 31) / 32 * 32;
  return 2u * static_cast<uint32_t>(W_BYTES + KSUB * box * BK * 2);
}

// The weight box of one stage (the CTA's 128 weight rows, 128 columns of K).
template <int EPI>
__device__ __forceinline__ void load_weights(const CUtensorMap* tmW, const Tile& t, uint32_t rank, int w_rows_per_expert,
                                             uint32_t w_dst, int kb, uint32_t full0) {
  const int w_row = EPI == EPI_SWIGLU ? t.fb * 128 + static_cast<int>(rank) * 64
                                      : t.e * w_rows_per_expert + t.fb * 256 + static_cast<int>(rank) * 128;
  if constexpr (EPI == EPI_SWIGLU)
    tma_load_5d_pair(w_dst, tmW, 0, 0, w_row, t.e, kb * KSUB, full0);
  else
    tma_load_3d_pair(w_dst, tmW, 0, w_row, kb * KSUB, full0);
}

// pre: the leading stages of this tile whose weight box (and the stage's
// expected bytes) were issued already; only their rows remain.
template <int ROWS, int EPI, int STAGES>
__device__ __forceinline__ bool load_tile(const CUtensorMap* tmW, const RowMaps& rm, const Tile& t, uint32_t rank,
                                          uint32_t tiles_u32, Smem& s, int k_blocks, int w_rows_per_expert,
                                          int& stage, uint32_t& phase, long long& issued,
                                          volatile int* abort_flag, int pre) {
  constexpr int BOX = (ROWS + 31) / 32 * 32;
  constexpr uint32_t TX = 2u * static_cast<uint32_t>(W_BYTES + KSUB * BOX * BK * 2);
  const int r0 = t.row0 + static_cast<int>(rank) * ROWS;
  for (int kb = 0; kb < k_blocks; ++kb) {
    const uint32_t full = smem_u32(&s.full[stage]);
    const uint32_t full0 = mapa_shared(full, 0);
    const uint32_t w_dst = tiles_u32 + stage * STAGE_BYTES;
    const uint32_t r_dst = w_dst + W_BYTES;
    if (kb >= pre) {
      if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort_flag)) return false;
      if (rank == 0) mbar_arrive_expect_tx(full, TX);
      load_weights<EPI>(tmW, t, rank, w_rows_per_expert, w_dst, kb, full0);
    }
    tma_load_3d_pair(r_dst, rm.box[BOX / 32 - 1], 0, r0, kb * KSUB, full0);
    ++issued;
    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
  }
  return true;
}

template <int EPI, int STAGES>
__device__ __forceinline__ bool load_tile_n(const CUtensorMap* tmW, const RowMaps& rm, const Tile& t, uint32_t rank,
                                            uint32_t tiles_u32, Smem& s, int k_blocks, int w_rows_per_expert,
                                            int& stage, uint32_t& phase, long long& issued,
                                            volatile int* abort_flag, int pre) {
#define MOE_LOAD_N(NN)                                                                                     \
  case NN / 16:                                                                                            \
    return load_tile<NN / 2, EPI, STAGES>(tmW, rm, t, rank, tiles_u32, s, k_blocks, w_rows_per_expert, stage, \
                                          phase, issued, abort_flag, pre);
  switch (t.n >> 4) {
    MOE_LOAD_N(16) MOE_LOAD_N(32) MOE_LOAD_N(48) MOE_LOAD_N(64) MOE_LOAD_N(80) MOE_LOAD_N(96)
    MOE_LOAD_N(112) MOE_LOAD_N(128) MOE_LOAD_N(144) MOE_LOAD_N(160) MOE_LOAD_N(176) MOE_LOAD_N(192)
    MOE_LOAD_N(208) MOE_LOAD_N(224) MOE_LOAD_N(240) MOE_LOAD_N(256)
    default: return false;
  }
#undef MOE_LOAD_N
}

// The MMAs of one tile: for each K step, wait for its stage, issue the
// pair's MMAs of 256 x N x 16 along each sub-tile's 128-byte rows, free the
// stage.  N is a template argument so that the instruction descriptor is a
// compile-time constant (and so is the rows box's sub-tile stride).
template <int N, int STAGES>
__device__ __forceinline__ bool mma_tile(uint32_t d_tmem, uint32_t tiles_u32, Smem& s, int k_blocks,
                                         int& stage, uint32_t& phase, volatile int* abort_flag) {
  constexpr uint32_t IDESC = idesc_bf16_f32(2 * 128, N);
  constexpr int R_SUB = (N / 2 + 31) / 32 * 32 * BK * 2;  // bytes of one sub-tile of the rows box
  for (int kb = 0; kb < k_blocks; ++kb) {
    if (!mbar_wait(smem_u32(&s.full[stage]), phase, abort_flag)) return false;
    tc_fence_after();
    const uint32_t w_addr = tiles_u32 + stage * STAGE_BYTES;
#pragma unroll
    for (int j = 0; j < KSUB; ++j) {
      const uint64_t a_desc = sdesc_k_sw128(w_addr + j * W_SUB);
      const uint64_t b_desc = sdesc_k_sw128(w_addr + W_BYTES + j * R_SUB);
#pragma unroll
      for (int kk = 0; kk < BK / UMMA_K; ++kk)  // 32 bytes along K per step
        tc_mma_bf16_pair(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, IDESC, (kb | j | kk) != 0);
    }
    tc_commit_pair(smem_u32(&s.empty[stage]));  // frees the stage in both CTAs
    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
  }
  return true;
}

template <int STAGES>
__device__ __forceinline__ bool mma_tile_n(int n, uint32_t d_tmem, uint32_t tiles_u32, Smem& s, int k_blocks,
                                           int& stage, uint32_t& phase, volatile int* abort_flag) {
#define MOE_MMA_N(NN) \
  case NN / 16: return mma_tile<NN, STAGES>(d_tmem, tiles_u32, s, k_blocks, stage, phase, abort_flag);
  switch (n >> 4) {
    MOE_MMA_N(16) MOE_MMA_N(32) MOE_MMA_N(48) MOE_MMA_N(64) MOE_MMA_N(80) MOE_MMA_N(96)
    MOE_MMA_N(112) MOE_MMA_N(128) MOE_MMA_N(144) MOE_MMA_N(160) MOE_MMA_N(176) MOE_MMA_N(192)
    MOE_MMA_N(208) MOE_MMA_N(224) MOE_MMA_N(240) MOE_MMA_N(256)
    default: return false;
  }
#undef MOE_MMA_N
}

// Waits until *counter reaches target (acquire at GPU scope).  Bounded like
// every wait of the kernel: false (and the CTA's abort flag raised) if it
// runs past the limit or another role of the CTA has given up.
__device__ __forceinline__ bool wait_ready(const int* counter, int target, volatile int* abort_flag) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ld_acquire_gpu(counter) >= target) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int EPI, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmW,    // weights
                     const __grid_constant__ CUtensorMap tmR32,   // expert rows: boxes of 32,
                     const __grid_constant__ CUtensorMap tmR64,   //   64,
                     const __grid_constant__ CUtensorMap tmR96,   //   96
                     const __grid_constant__ CUtensorMap tmR128,  //   and 128 rows
                     const __grid_constant__ CUtensorMap tmS0,    // stores: h or y
                     const __grid_constant__ CUtensorMap tmS1,    //   gu_save or o_save
                     const PairArgs args) {
  static_assert(STAGES <= MAX_STAGES, "barrier slots");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(tiles + STAGES * STAGE_BYTES + STAGING_BYTES);
  int* s_off = reinterpret_cast<int*>(&s + 1);  // [E+1]
  int* s_cnt = s_off + args.E + 1;              // [E]
  int* s_pre = s_cnt + args.E;                  // [E+1] tile prefix
  const uint32_t tiles_u32 = smem_u32(tiles);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const uint32_t rank = cluster_ctarank();  // the even CTA of a pair issues the MMAs
  const int tile0 = static_cast<int>(blockIdx.x >> 1);
  const int tstep = static_cast<int>(gridDim.x >> 1);

  // ---- set-up: barriers, tensor memory, the device-side tile list
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      // an accumulator is free once the epilogue warps of both CTAs have read it
      mbar_init(smem_u32(&s.tempty[i]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(&s.drain), 1);
    s.abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmR32);
    tma_prefetch_desc(&tmR64);
    tma_prefetch_desc(&tmR96);
    tma_prefetch_desc(&tmR128);
    tma_prefetch_desc(&tmS0);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(&s.tmem_base), TMEM_COLS);
  // Launch order.  Each launch lets its dependents start only once its own
  // wait has returned, so a running down-projection CTA implies that the
  // dispatch, two launches back, has completed.  The gate/up launch waits here
  // for the dispatch (the layout and the rows).  The down-projection launch
  // reads the layout now and waits for the gate/up launch's h only in its
  // producer, after it has issued its first stages' weight boxes, so its
  // set-up and first weight loads overlap the gate/up launch's last tiles.
  if constexpr (EPI == EPI_SWIGLU) {
    griddep_wait();
    griddep_launch_dependents();
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = args.offsets[e];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = args.counts[e];
  __syncthreads();
  if (warp == 0) {  // exclusive scan of per-expert tile counts
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int n = e < E ? chunks_of(covered_rows(s_off, s_cnt, e, args.write_pad)) * args.n_fblocks : 0;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) s_pre[e] = running + incl - n;
      running += __shfl_sync(FULL_MASK, incl, 31);
    }
    if (lane == 0) {
      s_pre[E] = running;
      s.total_tiles = running;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();

  const int total = s.total_tiles;
  const uint32_t tmem_base = s.tmem_base;
  volatile int* abort_flag = &s.abort;

  if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      const RowMaps rm{{&tmR32, &tmR64, &tmR96, &tmR128}};
      int pre = 0;  // leading stages of the first tile whose weights are already on their way
      const bool fine = EPI == EPI_WEIGHTED && args.ready != nullptr;
      if constexpr (EPI == EPI_WEIGHTED) {
        if (tile0 < total) {
          const Tile t = decode_tile(s_off, s_cnt, s_pre, E, args.n_fblocks, args.write_pad, tile0);
          pre = args.k_blocks < STAGES ? args.k_blocks : STAGES;
          for (int kb = 0; kb < pre; ++kb) {  // fresh stages: nothing to wait for
            const uint32_t full = smem_u32(&s.full[kb]);
            if (rank == 0) mbar_arrive_expect_tx(full, stage_tx(t.n));
            load_weights<EPI>(&tmW, t, rank, args.w_rows_per_expert, tiles_u32 + kb * STAGE_BYTES, kb,
                              mapa_shared(full, 0));
          }
        }
        if (!fine) griddep_wait();  // h comes from the gate/up launch
        griddep_launch_dependents();
      }
      for (int tile = tile0; tile < total && ok; tile += tstep) {
        const Tile t = decode_tile(s_off, s_cnt, s_pre, E, args.n_fblocks, args.write_pad, tile);
        if (fine) {
          // this chunk's h rows are written (bounded wait), then read them with TMA
          if (!wait_ready(args.ready + t.chunk, args.ready_target, abort_flag)) { ok = false; break; }
          fence_proxy_async_global();
        }
        // this CTA loads t.n / 2 expert rows (a multiple of 8): rows t.row0 + rank * t.n / 2 on
        ok = load_tile_n<EPI, STAGES>(&tmW, rm, t, rank, tiles_u32, s, args.k_blocks, args.w_rows_per_expert,
                                      stage, phase, issued, abort_flag, tile == tile0 ? pre : 0);
      }
      if (!ok && rank == 0) {
        // drain: wait for the loads of the last (up to STAGES) issued stages
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
          mbar_wait_drain(smem_u32(&s.full[stage]), phase);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (the even CTA) =================
    if (lane == 0 && rank != 0) {
      // the odd CTA issues nothing; it waits until the even CTA's last MMAs,
      // which write its tensor memory, have completed
      if (!mbar_wait_drain(smem_u32(&s.drain), 0)) *abort_flag = 1;
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = tile0; tile < total && ok; tile += tstep, ++local) {
        const Tile t = decode_tile(s_off, s_cnt, s_pre, E, args.n_fblocks, args.write_pad, tile);
        const int buf = local & 1;
        const uint32_t use = (local >> 1) & 1;
        if (!mbar_wait(smem_u32(&s.tempty[buf]), use ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        ok = mma_tile_n<STAGES>(t.n, tmem_base + buf * MAX_N, tiles_u32, s, args.k_blocks, stage, phase,
                                abort_flag);
        if (ok) tc_commit_pair(smem_u32(&s.tfull[buf]));
      }
      // every MMA issued has finished before anyone frees tensor or shared memory
      tc_commit_pair(smem_u32(&s.drain));
      if (!mbar_wait_drain(smem_u32(&s.drain), 0)) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ================= epilogue: warps 2..9 =================
    // lane quarter q = warp % 4 of tensor memory; column chunks alternate
    // between the two warps of a quarter.  A chunk whose 32 rows are all the
    // tile's goes out as TMA stores of boxes staged in this warp's 4 KiB of
    // shared memory (slots of one chunk's boxes, recycled once their stores
    // have read them); the rows of a partial chunk are stored directly.
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const bool save = args.out1 != nullptr;
    const uint32_t staging = tiles_u32 + STAGES * STAGE_BYTES + (warp - 2) * STAGING_PER_WARP;
    const int slot_bytes = EPI == EPI_SWIGLU ? (save ? 3072 : 1024) : (save ? 4096 : 2048);
    const int n_slots = STAGING_PER_WARP / slot_bytes;  // 4 or 1 (GEMM1), 2 or 1 (GEMM2)
    uint32_t n_staged = 0;
    int local = 0;
    for (int tile = tile0; tile < total; tile += tstep, ++local) {
      const Tile t = decode_tile(s_off, s_cnt, s_pre, E, args.n_fblocks, args.write_pad, tile);
      const int buf = local & 1;
      const uint32_t use = (local >> 1) & 1;
      // every lane waits, then the warp leaves together if any lane's wait ran
      // out: lanes leaving one by one would strand the others at the
      // warp-wide instructions below
      const bool ready = mbar_wait(smem_u32(&s.tfull[buf]), use, abort_flag);
      if (!__all_sync(FULL_MASK, ready)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * MAX_N + (static_cast<uint32_t>(q * 32) << 16);
      const int n_chunks = (t.n + 31) >> 5;
#pragma unroll 1
      for (int ch = hf; ch < n_chunks; ch += 2) {
        const int c = ch * 32;
        const int valid = t.rows - c;  // expert rows in this chunk (at least 1)
        const long long row = static_cast<long long>(t.row0) + c;
        const bool full = valid >= 32;
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(tb + c, v);
        tmem_ld_wait();
        uint32_t slot = 0;
        if (full) {
          slot = staging + (n_staged % n_slots) * slot_bytes;
          if (lane == 0) {  // the slot's earlier boxes have been read by their stores
            if (n_slots == 1) tma_store_wait_read<0>();
            else if (n_slots == 2) tma_store_wait_read<1>();
            else tma_store_wait_read<3>();
          }
          __syncwarp();
        }
        if constexpr (EPI == EPI_SWIGLU) {
          // lane 2j: gate of h column col0 + j for the chunk's 32 rows; lane 2j + 1: its up
          const bool up = lane & 1;
          const int j = lane >> 1;
          const int col0 = t.fb * 128 + static_cast<int>(rank) * 64 + q * 16;
          if (save) {
            if (full) {
              // g box at slot + 1024 (gate lanes), u box at slot + 2048 (up
              // lanes, one row ahead so that the two halves of the warp use
              // different banks)
              const uint32_t base = slot + (up ? 2048 : 1024) + 2 * j;
#pragma unroll
              for (int r = 0; r < 32; ++r) {
                const uint32_t val = up ? v[(r + 1) & 31] : v[r];
                const int rr = up ? ((r + 1) & 31) : r;
                st_shared_b16(base + 32 * rr, bf16_bits(__uint_as_float(val)));
              }
            } else {
              uint16_t* dst = args.out1 + row * args.ld1 + (up ? args.I : 0) + col0 + j;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < valid) dst[static_cast<long long>(i) * args.ld1] = bf16_bits(__uint_as_float(v[i]));
            }
          }
          // the gate lane takes rows 0..15 of the chunk, the up lane rows 16..31
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float mine_other = __uint_as_float(up ? v[i] : v[16 + i]);
            const float theirs = __shfl_xor_sync(FULL_MASK, mine_other, 1);
            const float g = up ? theirs : __uint_as_float(v[i]);
            const float u = up ? __uint_as_float(v[16 + i]) : theirs;
            hv[i] = silu(g) * u;
          }
          const int rb = up ? 16 : 0;
          if (full) {
            // h box at slot (32 rows x 16 columns); the up lanes go one row ahead
            const uint32_t base = slot + 2 * j;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float val = up ? hv[(i + 1) & 15] : hv[i];
              const int rr = up ? 16 + ((i + 1) & 15) : i;
              st_shared_b16(base + 32 * rr, bf16_bits(val));
            }
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmS0, slot, col0, static_cast<int>(row));
              if (save) {
                tma_store_2d(&tmS1, slot + 1024, col0, static_cast<int>(row));
                tma_store_2d(&tmS1, slot + 2048, args.I + col0, static_cast<int>(row));
              }
              tma_store_commit();
            }
            ++n_staged;
          } else {
            uint16_t* dst = args.out0 + (row + rb) * args.ld0 + col0 + j;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (rb + i < valid) dst[static_cast<long long>(i) * args.ld0] = bf16_bits(hv[i]);
          }
        } else {
          // lane l: y column col0 + l for the chunk's 32 rows; lane pairs trade
          // values so that each holds two adjacent columns of one row
          const bool odd = lane & 1;
          const int col0 = t.fb * 256 + static_cast<int>(rank) * 128 + q * 32;
          const float wl = lane < valid ? args.row_weight[row + lane] : 0.f;
          // pair value i of this lane: row 2i + odd, columns (lane & ~1, +1), as
          // w * o (y) and o (o_save)
          auto pair = [&](int i, uint32_t& yw, uint32_t& ow) {
            const float give = __uint_as_float(odd ? v[2 * i] : v[2 * i + 1]);
            const float got = __shfl_xor_sync(FULL_MASK, give, 1);
            const float w = __shfl_sync(FULL_MASK, wl, 2 * i + (odd ? 1 : 0));
            const float lo = odd ? got : __uint_as_float(v[2 * i]);
            const float hi = odd ? __uint_as_float(v[2 * i + 1]) : got;
            yw = pack_bf16x2(w * lo, w * hi);
            ow = pack_bf16x2(lo, hi);
          };
          if (full) {
            // y box at slot, o box at slot + 2048: 32 rows x 32 columns, with
            // the 64-byte swizzle of the store tensor maps (16-byte chunk c of
            // row r at chunk c ^ ((r >> 1) & 3))
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t yw, ow;
              pair(i, yw, ow);
              const int r = 2 * i + (odd ? 1 : 0);
              const uint32_t off = static_cast<uint32_t>(r * 64 + (((lane >> 3) ^ (i & 3)) << 4) + ((lane & 6) << 1));
              st_shared_b32(slot + off, yw);
              if (save) st_shared_b32(slot + 2048 + off, ow);
            }
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmS0, slot, col0, static_cast<int>(row));
              if (save) tma_store_2d(&tmS1, slot + 2048, col0, static_cast<int>(row));
              tma_store_commit();
            }
            ++n_staged;
          } else {
            uint32_t* dst0 = reinterpret_cast<uint32_t*>(args.out0 + row * args.ld0 + col0 + (lane & ~1));
            uint32_t* dst1 =
                save ? reinterpret_cast<uint32_t*>(args.out1 + row * args.ld1 + col0 + (lane & ~1)) : nullptr;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t yw, ow;
              pair(i, yw, ow);
              const int r = 2 * i + (odd ? 1 : 0);
              if (r < valid) {
                dst0[static_cast<long long>(r) * (args.ld0 >> 1)] = yw;
                if (save) dst1[static_cast<long long>(r) * (args.ld1 >> 1)] = ow;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // hand the accumulator back to the MMA issuer (its barrier is in the even
      // CTA) without waiting for this warp's global stores to complete
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&s.tempty[buf]), 0));
      if constexpr (EPI == EPI_SWIGLU) {
        if (args.ready != nullptr) {
          // this warp's part of the tile's h is in memory: its bulk stores have
          // completed, and the lanes' direct stores are ordered before lane 0's
          // release by the warp barrier above
          if (lane == 0) {
            tma_store_wait_all();
            fence_proxy_async_global();
            red_release_gpu_add(args.ready + t.chunk, 1);
          }
          __syncwarp();
        }
      }
    }
    if (lane == 0) tma_store_wait_all();  // every store done before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA frees its tensor memory or leaves while the pair's MMAs,
  // loads or barrier signals may still reach it
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && s.abort) report(args.status, MOE_DEVERR_TIMEOUT);
  if constexpr (EPI == EPI_WEIGHTED) {
    if (args.ready != nullptr) {
      // the last CTA of the down launch (every CTA has read its counters by
      // now) clears the slot's counters for their next use
      if (threadIdx.x == 0) {
        __threadfence();
        s.last = atomicAdd(args.done, 1u) == gridDim.x - 1;
      }
      __syncthreads();
      if (s.last) {
        const int n_chunks = total / args.n_fblocks;
        for (int i = threadIdx.x; i < n_chunks; i += blockDim.x) args.ready[i] = 0;
        if (threadIdx.x == 0) *args.done = 0u;
        __threadfence();
      }
    }
  }
}

// ---------------------------------------------------------------- host side

template <int EPI, int STAGES>
cudaError_t launch_stages(const CUtensorMap& w, const CUtensorMap (&r)[4], const CUtensorMap& st0,
                          const CUtensorMap& st1, const PairArgs& args, cudaStream_t s) {
  auto kernel = pair_gemm_kernel<EPI, STAGES>;
  static bool configured[64] = {};
  static int grid_cache[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const bool cacheable = dev >= 0 && dev < 64;
  if (!cacheable || !configured[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (err != cudaSuccess) return err;
    if (cacheable) configured[dev] = true;
  }
  const size_t smem = smem_bytes(STAGES, args.E);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // persistent grid: as many pairs as can be resident at once (a pair needs
  // two free SMs of one GPC), at most one CTA per SM
  int grid = cacheable ? grid_cache[dev] : 0;
  if (grid == 0) {
    cfg.gridDim = dim3(sm_count() & ~1);
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
      clusters = sm_count() / 2;
    grid = 2 * (clusters < sm_count() / 2 ? clusters : sm_count() / 2);
    if (grid < 2) grid = 2;
    if (cacheable) grid_cache[dev] = grid;
  }
  cfg.gridDim = dim3(grid);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, w, r[0], r[1], r[2], r[3], st0, st1, args);
}

// Three 64 KiB stages when they fit beside the staging and the per-expert
// tables, else two (E above about 150).
template <int EPI>
cudaError_t launch_pair_gemm(const CUtensorMap& w, const CUtensorMap (&r)[4], const CUtensorMap& st0,
                             const CUtensorMap& st1, const PairArgs& args, cudaStream_t s) {
  if (smem_bytes(3, args.E) <= static_cast<size_t>(SMEM_LIMIT))
    return launch_stages<EPI, 3>(w, r, st0, st1, args, s);
  return launch_stages<EPI, 2>(w, r, st0, st1, args, s);
}

std::mutex g_ready_mu;
int* g_ready_ptr[64];
unsigned int* g_done_ptr[64];
unsigned long long g_ready_ctx[64];
std::atomic<unsigned int> g_ready_next{0};

// A slot of readiness counters on the current device, or false.  A launch
// pair that is being captured into a graph goes without (the down launch then
// waits for the whole gate/up launch): a graph would keep the slot it was
// captured with for every replay, while eager launch pairs on other streams
// go on rotating through all the slots.  The counters' device address is
// looked up on the first use on each device (and again after a device reset).
bool ready_counters(cudaStream_t stream, int** ready, unsigned int** done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return false;
  }
  unsigned long long ctx = 0;
  const bool known_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_ready_mu);
  if (g_ready_ptr[dev] == nullptr || !known_ctx || g_ready_ctx[dev] != ctx) {
    void* r = nullptr;
    void* d = nullptr;
    if (cudaGetSymbolAddress(&r, g_h_ready) != cudaSuccess || cudaGetSymbolAddress(&d, g_h_done) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    g_ready_ptr[dev] = static_cast<int*>(r);
    g_done_ptr[dev] = static_cast<unsigned int*>(d);
    g_ready_ctx[dev] = ctx;
  }
  const unsigned int slot = g_ready_next.fetch_add(1u) % HR_SLOTS;
  *ready = g_ready_ptr[dev] + static_cast<size_t>(slot) * HR_CAP;
  *done = g_done_ptr[dev] + slot;
  return true;
}

bool row_maps(CUtensorMap (&r)[4], const void* base, uint64_t rows, uint64_t cols) {
  const uint32_t boxes[4] = {32, 64, 96, 128};
  for (int i = 0; i < 4; ++i)
    if (!make_tma_rows_k128(&r[i], base, rows, cols, boxes[i])) return false;
  return true;
}

}  // namespace

cudaError_t launch_experts_forward_pair(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                        const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                        uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                        cudaStream_t s) {
  if (L.capacity == 0) return cudaSuccess;
  const uint64_t C = static_cast<uint64_t>(L.capacity);
  CUtensorMap mW1, mW2, mX[4], mH[4], sH, sGU, sY, sO;
  if (!make_tma_w1_gate_up_k128(&mW1, W1, L.E, I, H) ||
      !make_tma_rows_k128(&mW2, W2, static_cast<uint64_t>(L.E) * H, I, 128) || !row_maps(mX, x_disp, C, H) ||
      !row_maps(mH, h, C, I) || !make_tma_store_2d_bf16_16(&sH, h, C, I) ||
      !make_tma_store_2d_bf16(&sY, y, C, H))
    return cudaErrorInvalidValue;
  sGU = sH;  // unused unless g, u are saved
  sO = sY;   // unused unless o is saved
  if ((gu_save && !make_tma_store_2d_bf16_16(&sGU, gu_save, C, 2 * static_cast<uint64_t>(I))) ||
      (o_save && !make_tma_store_2d_bf16(&sO, o_save, C, H)))
    return cudaErrorInvalidValue;

  PairArgs g1{};
  g1.counts = L.tokens_per_expert;
  g1.offsets = L.offsets;
  g1.row_weight = L.row_weight;
  g1.E = L.E;
  g1.k_blocks = H / (KSUB * BK);
  g1.n_fblocks = I / 128;  // a 256-row block of W1 is 128 gate and 128 up rows
  g1.w_rows_per_expert = 2 * I;
  g1.out0 = h;
  g1.ld0 = I;
  g1.out1 = gu_save;
  g1.ld1 = 2 * I;
  g1.I = I;
  g1.write_pad = gu_save != nullptr;  // training: the backward reads the pad rows
  g1.status = L.status;
  // readiness counters when the layer's row chunks fit a slot (at most one
  // chunk per expert more than its rows / 256)
  const long long rows_bound = static_cast<long long>(L.T) * L.K +
                               (g1.write_pad ? static_cast<long long>(L.E) * (L.pad_multiple - 1) : 0);
  if (rows_bound / MAX_N + L.E + 1 <= HR_CAP && !ready_counters(s, &g1.ready, &g1.done)) {
    g1.ready = nullptr;
    g1.done = nullptr;
  }
  g1.ready_target = (I / 128) * 2 * EPI_WARPS;
  cudaError_t err = launch_pair_gemm<EPI_SWIGLU>(mW1, mX, sH, sGU, g1, s);
  if (err != cudaSuccess) return err;

  PairArgs g2 = g1;
  g2.k_blocks = I / (KSUB * BK);
  g2.n_fblocks = H / 256;
  g2.w_rows_per_expert = H;
  g2.out0 = y;
  g2.ld0 = H;
  g2.out1 = o_save;
  g2.ld1 = H;
  err = launch_pair_gemm<EPI_WEIGHTED>(mW2, mH, sY, sO, g2, s);
  if (err != cudaSuccess && g2.ready != nullptr) {
    // the down launch, which clears the slot, did not start: clear it here
    // so that its next use does not see this use's signals
    cudaMemsetAsync(g2.ready, 0, sizeof(int) * HR_CAP, s);
    cudaMemsetAsync(g2.done, 0, sizeof(unsigned int), s);
  }
  return err;
}

}  // namespace moe
