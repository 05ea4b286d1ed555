// a5: the SwiGLU experts as two grouped GEMMs on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)": Expanded layout -- an expert computes only the rows routed to it,
// and the routing weight scales each row's output inside the expert step;
// Eager vs captured -- unused rows carry the sentinel expert id and are never
// computed; Benchmarks -- the experts are bf16 grouped GEMMs.  The SwiGLU form (gate, up, down) is the expert of the Qwen3-MoE
// layer shapes benchmarked there.
//
//   GEMM1 (per expert e, over its rows):  [g | u] = x_disp W1[e]^T,
//          epilogue h = bf16(silu(g) * u)            (optionally g, u saved)
//   GEMM2:  o = h W2[e]^T,  epilogue y = bf16(w_row * o)   (optionally o saved)
//
// This kernel takes the layers the CTA-pair kernel (gemm_pair.cu) does not:
// bf16 layers averaging at most 64 rows per expert (or with too few rows for
// every SM, in 64-column tiles), e4m3 gate/up operands, and the A rows
// gathered straight from the tokens.
//
// Design (one CTA per SM, persistent):
//   * the tile list is built on the device from tokens_per_expert / offsets,
//     so no host sync is needed and the launch can be graph-captured; an
//     expert's rows are covered by ceil(count / 128) tiles; only the valid
//     rows are written, plus -- when the gate/up values are saved for the
//     backward -- the pad rows of the expert's group (the tiles then cover
//     the whole padded group), which come out as zeros (x_disp's pad rows
//     are zero) and let the backward skip masking them; spare rows are never
//     written;
//   * warp 0 issues TMA loads into a 4-stage (3 for large E) shared-memory
//     ring (128-byte swizzle), warp 1 owns the tensor memory and issues
//     tcgen05.mma (128 x 256 x 16 per instruction), warps 2-9 are the
//     epilogue: two warps per 32-lane quarter of tensor memory, each taking
//     half of the tile's columns, so the epilogue keeps up with the MMAs;
//   * two 256-column fp32 accumulators in tensor memory let the epilogue of
//     one tile overlap the MMAs of the next;
//   * every wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT and the CTA
//     drains its in-flight work, frees tensor memory and exits.

#include <cstdio>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int BM = 128;          // rows per tile (tensor-memory lanes)
constexpr int BK = 64;           // bf16 elements per 128-byte swizzled row (128 for e4m3)
constexpr int UMMA_K = 16;       // K per tcgen05.mma for 16-bit inputs
constexpr int EPI_WARPS = 8;                   // two per TMEM lane quarter
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS);
// The gathered-A kernel adds three producer warps (10..12) to warp 0: each of
// the four copies 32 rows of the A tile, one row per lane.
constexpr int GATHER_WARPS = 4;
constexpr int NUM_THREADS_GATHER = NUM_THREADS + 32 * (GATHER_WARPS - 1);
constexpr int MAX_STAGES = 16;                 // barrier slots (the ring uses up to this many)
constexpr int SMEM_LIMIT = 232448;             // dynamic shared memory per CTA

// Tile shape.  BN (accumulator columns) is 256 in general, and 64 when the
// layer has too few rows to give every SM a 256-column tile (decode), so
// that four times as many CTAs stream the weights.  A_ROWS is how many rows
// of A a stage loads: 128, or 32 when no tile can have more than 32 rows to
// store.  The MMA always reads 128 rows; with A_ROWS = 32 the other 96 are
// whatever bytes follow in shared memory and only feed accumulator rows that
// are never stored.  The smaller A slot leaves room for more stages, i.e.
// more weight bytes in flight per SM, which is what bounds a decode step.
enum OperandKind { OPS_BF16 = 0, OPS_E4M3 = 1 };

template <int BN, int A_ROWS>
struct Fwd {
  static constexpr int A_BYTES = A_ROWS * BK * 2;        // 16 KiB at A_ROWS = 128
  static constexpr int B_BYTES = BN * BK * 2;            // 32 KiB at BN = 256
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KiB at BN = 256, A_ROWS = 128
  static constexpr int TMEM_COLS = 2 * BN;               // double-buffered accumulator
  // ring depth (one less when the per-expert tables of a large E need the room)
  static constexpr int STAGES = BN == 256 ? 4 : (A_ROWS == 128 ? 8 : 16);
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static constexpr uint32_t IDESC_E4M3 = idesc_e4m3_f32(BM, BN);
};

enum Epilogue { EPI_SWIGLU = 0, EPI_WEIGHTED = 1 };

struct GemmArgs {
  const int* counts;       // [E] rows of each expert
  const int* offsets;      // [E+1] group start rows
  const float* row_weight; // [C]
  int E;
  int k_blocks;            // contraction length / BK
  int n_tiles;             // N tiles per expert
  int b_rows_per_expert;   // rows of B per expert (2I or H)
  int b_tile_step;         // B row step per N tile (128 for GEMM1, 256 for GEMM2)
  int b_second_off;        // row offset of the second 128-row B box (I or 128)
  uint16_t* out0;          // GEMM1: h [C, I]     GEMM2: y [C, H]
  int ld0;
  uint16_t* out1;          // GEMM1: gu_save [C, 2I] (nullable)   GEMM2: o_save [C, H] (nullable)
  int ld1;
  int I;                   // GEMM1: offset of the up half in gu_save
  int write_pad;           // also write the pad rows of each expert's group (zeros)
  int* status;
  const float* a_scale;    // e4m3 GEMM1: [C] scale of each A row
  const float* b_scale;    // e4m3 GEMM1: [E * 2I] scale of each W1 row (output channel)
  const uint16_t* x;       // gathered GEMM1: the tokens [T, H]; A row r is x[row_token[r]]
  const int* row_token;    //   (a zero row where row_token is -1)
  long long capacity;
  int H;
};

// Barriers and scalars; the per-expert tables (offsets [E+1], counts [E],
// tile_prefix [E+1]) follow it in shared memory, sized by E.
struct Smem {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
};

// Epilogue staging for TMA stores: per epilogue warp, two 32 x 32 bf16 boxes.
constexpr int STAGING_BYTES = EPI_WARPS * 2 * 32 * 64;

constexpr size_t smem_bytes(int stages, int stage_bytes, int E) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(stages) * stage_bytes + STAGING_BYTES +
         sizeof(Smem) + static_cast<size_t>(3 * E + 2) * sizeof(int);
}

struct Tile {
  int e, mt, nt;
};

__device__ __forceinline__ Tile decode_tile(const int* tile_prefix, int E, int n_tiles, int tile) {
  int lo = 0, hi = E;  // tile_prefix[lo] <= tile < tile_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - tile_prefix[lo];
  Tile t;
  t.e = lo;
  t.mt = local / n_tiles;
  t.nt = local - t.mt * n_tiles;
  return t;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

template <int EPI, int BN, int A_ROWS, int STAGES, int OPS, bool GATHER>
__global__ void __launch_bounds__(GATHER ? NUM_THREADS_GATHER : NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  static_assert(STAGES <= MAX_STAGES, "barrier slots");
  using F = Fwd<BN, A_ROWS>;
  constexpr int A_BYTES = F::A_BYTES;
  constexpr int B_BYTES = F::B_BYTES;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int TMEM_COLS = F::TMEM_COLS;
  constexpr uint32_t IDESC = OPS == OPS_E4M3 ? F::IDESC_E4M3 : F::IDESC;
  constexpr int BKE = OPS == OPS_E4M3 ? 128 : BK;   // K elements per 128-byte row of a stage
  static_assert(OPS == OPS_BF16 || EPI == EPI_SWIGLU, "e4m3 operands only in the gate/up GEMM");
  static_assert(!GATHER || (OPS == OPS_BF16 && EPI == EPI_SWIGLU && A_ROWS == BM),
                "the gathered A is the bf16 gate/up GEMM's, 128 rows per stage");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(tiles + STAGES * STAGE_BYTES + STAGING_BYTES);
  int* s_off = reinterpret_cast<int*>(&s + 1);  // [E+1]
  int* s_cnt = s_off + args.E + 1;              // [E]
  int* s_pre = s_cnt + args.E;                  // [E+1] tile prefix
  const uint32_t tiles_u32 = smem_u32(tiles);
  const uint32_t staging_u32 = tiles_u32 + STAGES * STAGE_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  griddep_launch_dependents();

  // ---- set-up: barriers, tensor memory, the device-side tile list
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // gathered A: the cp.async arrivals of the producer lanes + the TMA expect_tx of B
      mbar_init(smem_u32(&s.full[i]), GATHER ? 32 * GATHER_WARPS + 1 : 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      // a pair's accumulator is free once the epilogue warps of both CTAs have read it
      mbar_init(smem_u32(&s.tempty[i]), EPI_WARPS);
    }
    mbar_init(smem_u32(&s.drain), 1);
    s.abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) tmem_alloc(smem_u32(&s.tmem_base), TMEM_COLS);
  griddep_wait();  // the layout, the dispatched rows (and h) come from earlier kernels
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = args.offsets[e];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = args.counts[e];
  __syncthreads();
  if (warp == 0) {  // exclusive scan of per-expert tile counts
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      // rows an expert's tiles cover: its valid rows, or with the pad rows
      // written (training) its whole padded group
      const int rows_e = e < E ? (args.write_pad ? s_off[e + 1] - s_off[e] : s_cnt[e]) : 0;
      const int n = ((rows_e + BM - 1) / BM) * args.n_tiles;
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
  tc_fence_after();

  const int total = s.total_tiles;
  const uint32_t tmem_base = s.tmem_base;
  volatile int* abort_flag = &s.abort;

  if (GATHER && (warp == 0 || warp >= 2 + EPI_WARPS)) {
    // ================= producers, A gathered from the tokens =================
    // Producer warp pw (warp 0, then 10..12) copies rows 32 pw .. 32 pw + 31 of
    // the A tile, lane l row 32 pw + l, with 16-byte cp.async into the
    // positions the 128-byte swizzle gives them (chunk c of row r at r * 128 +
    // ((c ^ (r & 7)) * 16)); warp 0's lane 0 also loads B by TMA.
    const int pw = warp == 0 ? 0 : warp - (1 + EPI_WARPS);
    const int row = 32 * pw + lane;
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = decode_tile(s_pre, E, args.n_tiles, tile);
      const long long r = static_cast<long long>(s_off[t.e]) + t.mt * BM + row;
      const int b_row = t.e * args.b_rows_per_expert + t.nt * args.b_tile_step;
      const int tk = r < args.capacity ? __ldg(args.row_token + r) : -1;
      const uint16_t* src = tk >= 0 ? args.x + static_cast<long long>(tk) * args.H : args.x;
      const uint32_t nbytes = tk >= 0 ? 16u : 0u;  // a zero row where there is no token
      for (int kb = 0; kb < args.k_blocks; ++kb) {
        int wok = 1;
        if (lane == 0) wok = mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort_flag);
        if (!__shfl_sync(FULL_MASK, wok, 0)) { ok = false; break; }
        const uint32_t full = smem_u32(&s.full[stage]);
        const uint32_t a_dst = tiles_u32 + stage * STAGE_BYTES;
        const uint32_t b_dst = a_dst + A_BYTES;
        if (pw == 0 && lane == 0) {
          mbar_arrive_expect_tx(full, B_BYTES);
          tma_load_2d(b_dst, &tmB, kb * BKE, b_row, full);
          tma_load_2d(b_dst + B_BYTES / 2, &tmB, kb * BKE, b_row + args.b_second_off, full);
        }
        const uint16_t* src_k = tk >= 0 ? src + kb * BK : src;
        const uint32_t row_dst = a_dst + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          cp_async_16(row_dst + ((c ^ (row & 7)) << 4), src_k + (tk >= 0 ? c * 8 : 0), nbytes);
        cp_async_mbar_arrive_noinc(full);
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && pw == 0 && lane == 0) {
      for (int i = 0; i < STAGES && i < issued; ++i) {
        if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
        mbar_wait_drain(smem_u32(&s.full[stage]), phase);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(s_pre, E, args.n_tiles, tile);
        const int a_row = s_off[t.e] + t.mt * BM;
        const int b_row = t.e * args.b_rows_per_expert + t.nt * args.b_tile_step;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t full = smem_u32(&s.full[stage]);
          const uint32_t a_dst = tiles_u32 + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          mbar_arrive_expect_tx(full, STAGE_BYTES);
          tma_load_2d(a_dst, &tmA, kb * BKE, a_row, full);
          tma_load_2d(b_dst, &tmB, kb * BKE, b_row, full);
          tma_load_2d(b_dst + B_BYTES / 2, &tmB, kb * BKE, b_row + args.b_second_off, full);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // drain: wait for the loads of the last (up to STAGES) issued stages
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
          mbar_wait_drain(smem_u32(&s.full[stage]), phase);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (local >> 1) & 1;
        if (!mbar_wait(smem_u32(&s.tempty[buf]), use ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait(smem_u32(&s.full[stage]), phase, abort_flag)) { ok = false; break; }
          if constexpr (GATHER) fence_proxy_async_shared();  // A arrived through cp.async
          tc_fence_after();
          const uint32_t a_addr = tiles_u32 + stage * STAGE_BYTES;
          const uint64_t a_desc = sdesc_k_sw128(a_addr);
          const uint64_t b_desc = sdesc_k_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // advance along K inside the 128-byte swizzled row: 32 bytes per step
            // (16 bf16 or 32 e4m3 elements)
            if constexpr (OPS == OPS_E4M3)
              tc_mma_e4m3(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, IDESC, (kb | kk) != 0);
            else
              tc_mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, IDESC, (kb | kk) != 0);
          }
          tc_commit(smem_u32(&s.empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc_commit(smem_u32(&s.tfull[buf]));
      }
      // make sure every MMA this thread issued has finished before anyone
      // frees tensor memory or shared memory
      tc_commit(smem_u32(&s.drain));
      if (!mbar_wait_drain(smem_u32(&s.drain), 0)) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..5 -> TMEM lanes 32*(warp%4)) =================
    // warps 2..9: lane quarter q = warp % 4 of TMEM, column half (warp - 2) / 4
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r_in_tile = q * 32 + lane;
    int local = 0;
    // Staged TMA store of one 32-row x 32-column bf16 box: each lane writes its
    // row (64 bytes, swizzled) into one of the warp's two staging buffers, then
    // lane 0 stores the box.  Used only when all 32 rows of the warp are valid.
    const uint32_t my_staging = staging_u32 + (warp - 2) * 2 * 2048;  // two 2 KiB boxes
    uint32_t n_staged = 0;
    int warp_row0 = 0;
    auto store_staged = [&](const uint32_t (&v)[16], int col) {
      const uint32_t buf = my_staging + (n_staged & 1) * 2048;
      if (lane == 0) tma_store_wait_read<1>();
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i)
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(buf + staged_chunk(lane, i)), "r"(v[4 * i]),
                     "r"(v[4 * i + 1]), "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                     : "memory");
      fence_async_shared();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&tmOut, buf, col, warp_row0);
        tma_store_commit();
      }
      ++n_staged;
    };
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const Tile t = decode_tile(s_pre, E, args.n_tiles, tile);
      const int buf = local & 1;
      const uint32_t use = (local >> 1) & 1;
      // every lane waits, then the warp leaves together if any lane's wait ran
      // out: lanes leaving one by one would strand the others at the
      // warp-wide instructions below
      const bool ready = mbar_wait(smem_u32(&s.tfull[buf]), use, abort_flag);
      if (!__all_sync(FULL_MASK, ready)) break;
      tc_fence_after();
      const int group_row = t.mt * BM + r_in_tile;
      // rows written: the valid rows, plus (write_pad) the pad rows of the
      // expert's group, which come out zero from the zero pad rows of x_disp
      const bool valid = group_row < (args.write_pad ? s_off[t.e + 1] - s_off[t.e] : s_cnt[t.e]);
      const bool full_warp = __all_sync(FULL_MASK, valid);
      const long long row = static_cast<long long>(s_off[t.e]) + group_row;
      warp_row0 = s_off[t.e] + t.mt * BM + q * 32;
      const uint32_t tb = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (EPI == EPI_SWIGLU) {
        // columns [0, BN/2) gate, [BN/2, BN) up, for h columns nt*BN/2 + [0, BN/2);
        // each column half of the epilogue takes half of them (at BN = 64
        // there are only 32: the first half takes them)
        constexpr int H_COLS = BN / 2;
        constexpr int PER_HALF = H_COLS >= 64 ? H_COLS / 2 : H_COLS;
        const int col0 = t.nt * H_COLS;
        const int c_end = (half + 1) * PER_HALF < H_COLS ? (half + 1) * PER_HALF : H_COLS;
#pragma unroll 1
        for (int c = half * PER_HALF; c < c_end; c += 32) {
          uint32_t g[32], u[32];
          __syncwarp();
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + BN / 2 + c, u);
          tmem_ld_wait();
          if constexpr (OPS == OPS_E4M3) {
            // acc * scale(row) * scale(channel); lane i holds channel i's scales
            const long long bs = static_cast<long long>(t.e) * args.b_rows_per_expert + col0 + c + lane;
            const float sg = __ldg(args.b_scale + bs);
            const float su = __ldg(args.b_scale + bs + args.b_second_off);
            const float sa = valid ? __ldg(args.a_scale + row) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __float_as_uint(__uint_as_float(g[i]) * (sa * __shfl_sync(FULL_MASK, sg, i)));
              u[i] = __float_as_uint(__uint_as_float(u[i]) * (sa * __shfl_sync(FULL_MASK, su, i)));
            }
          }
          if (valid) {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              hv[i] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
            }
            if (!full_warp) {
              uint4* dst = reinterpret_cast<uint4*>(args.out0 + row * args.ld0 + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
            } else {
              store_staged(hv, col0 + c);
            }
            if (args.out1) {
              uint4* dg = reinterpret_cast<uint4*>(args.out1 + row * args.ld1 + col0 + c);
              uint4* du = reinterpret_cast<uint4*>(args.out1 + row * args.ld1 + args.I + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                dg[i] = make_uint4(pack_bf16x2(__uint_as_float(g[8 * i + 0]), __uint_as_float(g[8 * i + 1])),
                                   pack_bf16x2(__uint_as_float(g[8 * i + 2]), __uint_as_float(g[8 * i + 3])),
                                   pack_bf16x2(__uint_as_float(g[8 * i + 4]), __uint_as_float(g[8 * i + 5])),
                                   pack_bf16x2(__uint_as_float(g[8 * i + 6]), __uint_as_float(g[8 * i + 7])));
                du[i] = make_uint4(pack_bf16x2(__uint_as_float(u[8 * i + 0]), __uint_as_float(u[8 * i + 1])),
                                   pack_bf16x2(__uint_as_float(u[8 * i + 2]), __uint_as_float(u[8 * i + 3])),
                                   pack_bf16x2(__uint_as_float(u[8 * i + 4]), __uint_as_float(u[8 * i + 5])),
                                   pack_bf16x2(__uint_as_float(u[8 * i + 6]), __uint_as_float(u[8 * i + 7])));
              }
            }
          }
        }
      } else {
        const int col0 = t.nt * BN;
        const float w = valid ? args.row_weight[row] : 0.f;
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          uint32_t o[32];
          __syncwarp();
          tmem_ld32(tb + c, o);
          tmem_ld_wait();
          if (valid) {
            uint32_t yv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              yv[i] = pack_bf16x2(w * __uint_as_float(o[2 * i]), w * __uint_as_float(o[2 * i + 1]));
            if (!full_warp) {
              uint4* dst = reinterpret_cast<uint4*>(args.out0 + row * args.ld0 + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(yv[4 * i], yv[4 * i + 1], yv[4 * i + 2], yv[4 * i + 3]);
            } else {
              store_staged(yv, col0 + c);
            }
            if (args.out1) {
              uint4* dso = reinterpret_cast<uint4*>(args.out1 + row * args.ld1 + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float f[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(o[8 * i + k]);
                dso[i] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.tempty[buf]));
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && s.abort) report(args.status, MOE_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------- host side

template <int EPI, int BN, int A_ROWS, int STAGES, int OPS, bool GATHER>
cudaError_t launch_gemm_stages(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                               const GemmArgs& args, cudaStream_t s) {
  auto kernel = grouped_gemm_kernel<EPI, BN, A_ROWS, STAGES, OPS, GATHER>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const size_t smem = smem_bytes(STAGES, Fwd<BN, A_ROWS>::STAGE_BYTES, args.E);
  return launch_dependent(kernel, sm_count(), GATHER ? NUM_THREADS_GATHER : NUM_THREADS, smem, s, a, b, out,
                          args);
}

// The ring depth of Fwd when it fits beside the staging and the per-expert
// tables, else one stage less (E above about 200).
template <int EPI, int BN, int A_ROWS, int OPS = OPS_BF16, bool GATHER = false>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                        const GemmArgs& args, cudaStream_t s) {
  using F = Fwd<BN, A_ROWS>;
  if (smem_bytes(F::STAGES, F::STAGE_BYTES, args.E) <= static_cast<size_t>(SMEM_LIMIT))
    return launch_gemm_stages<EPI, BN, A_ROWS, F::STAGES, OPS, GATHER>(a, b, out, args, s);
  return launch_gemm_stages<EPI, BN, A_ROWS, F::STAGES - 1, OPS, GATHER>(a, b, out, args, s);
}

// GEMM1 reads A (x_disp rows) and B (W1) as bf16, or as e4m3 codes with
// fp32 scales per A row and per W1 row, or (GATHER) A straight from the
// tokens x by row_token; GEMM2 is bf16.
template <int BN, int A_ROWS, int OPS, bool GATHER = false>
cudaError_t experts_forward(const void* x_disp, const float* x_scale, const moe_layout& L, int H,
                            int I, const void* W1, const float* W1_scale, const uint16_t* W2,
                            uint16_t* h, uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                            cudaStream_t s) {
  const uint64_t C = static_cast<uint64_t>(L.capacity);
  const uint64_t w1_rows = static_cast<uint64_t>(L.E) * 2 * I;
  // B is loaded as two boxes of BN/2 rows: the gate and up rows (GEMM1) or
  // the two halves of the tile's output columns (GEMM2).
  CUtensorMap mA1, mB1, mA2, mB2, mH, mY;
  const bool maps1 = OPS == OPS_E4M3
                         ? make_tma_2d_u8(&mA1, x_disp, C, H, A_ROWS) &&
                               make_tma_2d_u8(&mB1, W1, w1_rows, H, BN / 2)
                         : (GATHER || make_tma_2d_bf16(&mA1, x_disp, C, H, A_ROWS)) &&
                               make_tma_2d_bf16(&mB1, W1, w1_rows, H, BN / 2);
  if (GATHER) mA1 = mB1;  // unused: the producer gathers A with cp.async
  if (!maps1 || !make_tma_2d_bf16(&mA2, h, C, I, A_ROWS) ||
      !make_tma_2d_bf16(&mB2, W2, static_cast<uint64_t>(L.E) * H, I, BN / 2) ||
      !make_tma_store_2d_bf16(&mH, h, C, I) || !make_tma_store_2d_bf16(&mY, y, C, H))
    return cudaErrorInvalidValue;

  GemmArgs g1{};
  g1.counts = L.tokens_per_expert;
  g1.offsets = L.offsets;
  g1.row_weight = L.row_weight;
  g1.E = L.E;
  g1.k_blocks = H / (OPS == OPS_E4M3 ? 128 : BK);
  g1.n_tiles = I / (BN / 2);
  g1.b_rows_per_expert = 2 * I;
  g1.b_tile_step = BN / 2;
  g1.b_second_off = I;
  g1.out0 = h;
  g1.ld0 = I;
  g1.out1 = gu_save;
  g1.ld1 = 2 * I;
  g1.I = I;
  g1.write_pad = gu_save != nullptr;  // training: the backward reads the pad rows
  g1.status = L.status;
  g1.a_scale = x_scale;
  g1.b_scale = W1_scale;
  g1.x = static_cast<const uint16_t*>(x_disp);  // GATHER: the tokens
  g1.row_token = L.row_token;
  g1.capacity = L.capacity;
  g1.H = H;
  cudaError_t err = launch_gemm<EPI_SWIGLU, BN, A_ROWS, OPS, GATHER>(mA1, mB1, mH, g1, s);
  if (err != cudaSuccess) return err;

  GemmArgs g2 = g1;
  g2.k_blocks = I / BK;
  g2.n_tiles = H / BN;
  g2.b_rows_per_expert = H;
  g2.b_tile_step = BN;
  g2.b_second_off = BN / 2;
  g2.out0 = y;
  g2.ld0 = H;
  g2.out1 = o_save;
  g2.ld1 = H;
  g2.a_scale = nullptr;
  g2.b_scale = nullptr;
  return launch_gemm<EPI_WEIGHTED, BN, A_ROWS, OPS_BF16, false>(mA2, mB2, mY, g2, s);
}

// The tile shape for a layer (all from host-known sizes, so the sync-free
// path needs no row counts).  At most min(E, T*K) experts have rows; when
// even one 128-row tile per such expert at BN = 256 leaves SMs idle, take
// 64-column tiles.  An expert has at most T rows (one per token); with the
// pad rows written (training) its group is T rounded up to pad_multiple.
enum class Shape { kWide, kNarrow, kNarrowShortA };

Shape pick_shape(const moe_layout& L, int I, bool write_pad) {
  const long long pairs = static_cast<long long>(L.T) * L.K;
  const long long active = pairs < L.E ? pairs : L.E;
  if (active * (I / 128) >= sm_count()) return Shape::kWide;
  const long long P = L.pad_multiple;
  const long long stored = write_pad ? (L.T + P - 1) / P * P : L.T;
  return stored <= 32 ? Shape::kNarrowShortA : Shape::kNarrow;
}

// Which kernel takes a bf16 layer with rows for every SM (from host-known
// sizes, so the sync-free path needs no row counts): at most 64 rows per
// expert on average, one CTA per tile -- the step is a weight stream, and a
// CTA's four 48 KiB stages hold 128 KiB of weights in flight per SM where a
// pair's stages hold 96 KiB (decode T = 256: 206 against 215 us); otherwise
// CTA pairs with the expert rows on the MMA's N side (gemm_pair.cu).  (CTA
// pairs with the rows on the M side, 256-row tiles, ran slower at every
// size: 301 against 296 us at T = 4096, 830 against 809 us at T = 16384.)
bool wide_single_cta(const moe_layout& L) {
  const long long pairs = static_cast<long long>(L.T) * L.K;
  return pairs <= 64LL * L.E;
}

template <int OPS>
cudaError_t experts_forward_any(const void* x_disp, const float* x_scale, const moe_layout& L,
                                int H, int I, const void* W1, const float* W1_scale,
                                const uint16_t* W2, uint16_t* h, uint16_t* y, uint16_t* o_save,
                                uint16_t* gu_save, cudaStream_t s) {
  switch (pick_shape(L, I, gu_save != nullptr)) {
    case Shape::kWide:
      if constexpr (OPS == OPS_BF16) {
        if (!wide_single_cta(L))
          return launch_experts_forward_pair(static_cast<const uint16_t*>(x_disp), L, H, I,
                                             static_cast<const uint16_t*>(W1), W2, h, y, o_save, gu_save, s);
        return experts_forward<256, 128, OPS>(x_disp, x_scale, L, H, I, W1, W1_scale, W2, h, y, o_save,
                                              gu_save, s);
      } else
        return experts_forward<256, 128, OPS>(x_disp, x_scale, L, H, I, W1, W1_scale, W2, h, y,
                                              o_save, gu_save, s);
    case Shape::kNarrow:
      return experts_forward<64, 128, OPS>(x_disp, x_scale, L, H, I, W1, W1_scale, W2, h, y,
                                           o_save, gu_save, s);
    case Shape::kNarrowShortA:
      return experts_forward<64, 32, OPS>(x_disp, x_scale, L, H, I, W1, W1_scale, W2, h, y,
                                          o_save, gu_save, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_experts_forward(const uint16_t* x_disp, const moe_layout& L, int H, int I,
                                   const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                   uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                   cudaStream_t s) {
  if (L.capacity == 0) return cudaSuccess;
  if (gemv_experts_fits(L, H, I, o_save || gu_save))
    return launch_experts_forward_gemv(x_disp, L, H, I, W1, W2, h, y, s);
  return experts_forward_any<OPS_BF16>(x_disp, nullptr, L, H, I, W1, nullptr, W2, h, y, o_save,
                                       gu_save, s);
}

cudaError_t launch_experts_forward_gather(const uint16_t* x, const moe_layout& L, int H, int I,
                                          const uint16_t* W1, const uint16_t* W2, uint16_t* h,
                                          uint16_t* y, uint16_t* o_save, uint16_t* gu_save,
                                          cudaStream_t s) {
  if (L.capacity == 0) return cudaSuccess;
  if (gemv_experts_fits(L, H, I, o_save || gu_save))
    return launch_experts_forward_gemv(x, L, H, I, W1, W2, h, y, s, /*gather=*/true);
  if (pick_shape(L, I, gu_save != nullptr) == Shape::kWide)
    return experts_forward<256, 128, OPS_BF16, true>(x, nullptr, L, H, I, W1, nullptr, W2, h, y,
                                                     o_save, gu_save, s);
  return experts_forward<64, 128, OPS_BF16, true>(x, nullptr, L, H, I, W1, nullptr, W2, h, y, o_save,
                                                  gu_save, s);
}

cudaError_t launch_experts_forward_fp8(const uint8_t* x_q, const float* x_scale,
                                       const moe_layout& L, int H, int I, const uint8_t* W1_q,
                                       const float* W1_scale, const uint16_t* W2, uint16_t* h,
                                       uint16_t* y, cudaStream_t s) {
  if (L.capacity == 0) return cudaSuccess;
  return experts_forward_any<OPS_E4M3>(x_q, x_scale, L, H, I, W1_q, W1_scale, W2, h, y, nullptr,
                                       nullptr, s);
}

}  // namespace moe
