// a9: the backward of the SwiGLU experts on the tensor cores.
//
// "Add the deepep expert-parallel implementation (huggingface/transformers
// #49638)", What this adds, Training: gradients flow back to the tokens (and,
// through the combine, to the routing weights).  With G_o = w_r * grad_y (the
// routing weight moves onto the gradient, because y = w_r * o):
//
//   dgrad1:  G_h  = G_o W2[e]            [n x H] . [H x I]    epilogue: SwiGLU'
//            G_g  = G_h * u * silu'(g),  G_u = G_h * silu(g)  -> G_gu [n x 2I]
//   dgrad2:  grad_x_disp = G_gu W1[e]    [n x 2I] . [2I x H]
//   wgrad2:  dW2[e] = G_o^T h            [H x n] . [n x I]     (fp32 out)
//   wgrad1:  dW1[e] = G_gu^T x_disp      [2I x n] . [n x H]    (fp32 out)
//
// The forward kernel's structure is kept (persistent CTAs, a TMA producer
// warp, an MMA warp owning two 256-column TMEM accumulators, four epilogue
// warps, bounded waits), with two generalisations:
//   * MN-major operands.  The weights in dgrad and both operands of wgrad are
//     contiguous along M or N rather than K.  They are loaded as 64 x 64 TMA
//     boxes (64 MN elements = one 128-byte swizzled line per K index) and
//     described to tcgen05.mma as MN-major: 64-wide MN blocks 8 KiB apart
//     (leading byte offset), 8-deep K groups 1 KiB apart (stride byte offset),
//     and the instruction descriptor's transpose bit set for that operand.
//   * K over an expert's rows (wgrad).  Each tile's contraction runs over the
//     rows of one expert, so the last 64-row block may reach past them.  When
//     the groups are padded to a multiple of 64 rows those are the expert's
//     own pad rows, zero in every operand; otherwise the MMA warp zeroes those
//     K lines of both operands in shared memory before issuing the MMAs.  An
//     expert with no rows gets zero weight gradients.

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int EPI_WARPS = 8;              // two per TMEM lane quarter
constexpr int NUM_THREADS = 32 * (2 + EPI_WARPS);
constexpr int SMEM_LIMIT = 232448;
constexpr int A_BYTES = BM * BK * 2;      // 16 KiB
constexpr int MN_BOX_BYTES = 64 * BK * 2; // 8 KiB: 64 MN x 64 K, MN-major
constexpr int TMEM_COLS = 512;

enum BwdEpilogue { EPI_DSWIGLU = 0, EPI_BF16 = 1, EPI_F32 = 2 };

template <int BN>
struct Cfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int MAX_STAGES = BN == 256 ? 4 : 6;
};

struct BwdArgs {
  const int* counts;         // [E]
  const int* offsets;        // [E+1]
  int E;
  int k_blocks;              // M-grouped: contraction length / 64
  int m_tiles;               // K-grouped: M extent / 128
  int n_tiles;               // N tiles per expert
  int b_rows_per_expert;     // M-grouped: rows of B's 2-D view per expert
  int m_total, n_total;      // K-grouped: output extents per expert
  uint16_t* out_bf16;        // dgrad outputs [C, ld_out]
  int ld_out;
  const uint16_t* gu;        // EPI_DSWIGLU: gate / up pre-activations [C, 2I]
  int I;
  float* out_f32;            // K-grouped: [E, m_total, n_total]
  int zero_tail;             // K-grouped: zero the K lines past an expert's count
  int* status;
  long long capacity;        // rows of the row buffers (bounds-checked builds)
};

// Barriers and scalars; the per-expert tables (offsets [E+1], counts [E],
// tile_prefix [E+1]) follow it in shared memory, sized by E.
struct Smem {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
};

// Epilogue staging for TMA stores: 4 KiB per epilogue warp (two boxes of
// 32 rows x 64 bytes: 32 bf16 or 16 fp32 columns).
constexpr int STAGING_BYTES = EPI_WARPS * 4096;

template <int BN, bool PAIR = false>
constexpr size_t smem_bytes(int stages, int E) {
  return 1024 + static_cast<size_t>(stages) * (PAIR ? A_BYTES + Cfg<BN>::B_BYTES / 2 : Cfg<BN>::STAGE_BYTES) +
         STAGING_BYTES + sizeof(Smem) + static_cast<size_t>(3 * E + 2) * sizeof(int);
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(sbo >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

struct Tile {
  int e, mt, nt;
};

__device__ __forceinline__ Tile decode(const int* tile_prefix, int E, int n_tiles, int tile) {
  int lo = 0, hi = E;
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

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
  return __shfl_sync(FULL_MASK, ok, 0) != 0;
}

// GROUP_K = false: tiles are (expert, 128-row block of its rows, N block),
//   A is K-major (rows of the expert), B is MN-major (the expert's weight).
// GROUP_K = true: tiles are (expert, M block, N block); both operands are
//   MN-major slices of the expert's rows, the contraction runs over the rows.
// PAIR: clusters of two CTAs, tiles of 256 M rows (the expert's rows, or the
//   M extent of a weight gradient): each CTA loads its own 128 of them and
//   one half (128) of the tile's N columns, the even CTA issues cta_group::2
//   MMAs for the pair, each CTA's epilogue takes its own 128 rows (as in the
//   forward kernel's pairs).  Used with 256-column tiles and no K-line
//   masking, so that neither CTA touches shared memory the other's MMAs read.
template <bool GROUP_K, int BN, int EPI, int STAGES, bool PAIR = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const BwdArgs args) {
  static_assert(!PAIR || BN == 256, "CTA pairs take 256-column tiles");
  constexpr int B_BYTES = PAIR ? Cfg<BN>::B_BYTES / 2 : Cfg<BN>::B_BYTES;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int RB = PAIR ? 2 * BM : BM;  // M rows of a tile
  constexpr int B_BOXES = (PAIR ? BN / 2 : BN) / 64;
  constexpr uint32_t IDESC = idesc_bf16_f32(RB, BN) | (GROUP_K ? (1u << 15) : 0u) | (1u << 16);
  // K-major A: 8-row groups 1 KiB apart, next 16-wide K slice 32 bytes on.
  // MN-major A / B: 64-wide MN blocks 8 KiB apart, 8-deep K groups 1 KiB
  // apart, next 16-deep K slice two groups (2 KiB) on.
  constexpr uint32_t A_LBO = GROUP_K ? MN_BOX_BYTES : 16;
  constexpr uint32_t A_STEP = GROUP_K ? 2048 : 32;
  constexpr uint32_t B_LBO = MN_BOX_BYTES;
  constexpr uint32_t B_STEP = 2048;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Smem& s = *reinterpret_cast<Smem*>(tiles + STAGES * STAGE_BYTES + STAGING_BYTES);
  int* s_off = reinterpret_cast<int*>(&s + 1);  // [E+1]
  int* s_cnt = s_off + args.E + 1;              // [E]
  int* s_pre = s_cnt + args.E;                  // [E+1]
  const uint32_t tiles_u32 = smem_u32(tiles);
  const uint32_t staging_u32 = tiles_u32 + STAGES * STAGE_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // the even CTA of a pair issues the MMAs
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      mbar_init(smem_u32(&s.tempty[i]), PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    mbar_init(smem_u32(&s.drain), 1);
    s.abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(smem_u32(&s.tmem_base), TMEM_COLS);
    else
      tmem_alloc(smem_u32(&s.tmem_base), TMEM_COLS);
  }
  for (int e = threadIdx.x; e <= E; e += NUM_THREADS) s_off[e] = args.offsets[e];
  for (int e = threadIdx.x; e < E; e += NUM_THREADS) s_cnt[e] = args.counts[e];
  __syncthreads();
  if (warp == 0) {
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int n = 0;
      if (e < E) n = GROUP_K ? args.m_tiles * args.n_tiles : ((s_cnt[e] + RB - 1) / RB) * args.n_tiles;
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
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();

  const int total = s.total_tiles;
  const uint32_t tmem_base = s.tmem_base;
  volatile int* abort_flag = &s.abort;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = tile0; tile < total && ok; tile += tstep) {
        const Tile t = decode(s_pre, E, args.n_tiles, tile);
        const int kbs = GROUP_K ? (s_cnt[t.e] + BK - 1) / BK : args.k_blocks;
        const int m0 = t.mt * RB + static_cast<int>(rank) * BM;         // this CTA's M rows
        const int n0 = t.nt * BN + static_cast<int>(rank) * (BN / 2);   // (pair) this CTA's N half
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t full = smem_u32(&s.full[stage]);
          const uint32_t a_dst = tiles_u32 + stage * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          if constexpr (PAIR) {
            // both CTAs' loads complete on the even CTA's barrier, which expects them all
            const uint32_t full0 = mapa_shared(full, 0);
            if (rank == 0) mbar_arrive_expect_tx(full, 2 * STAGE_BYTES);
            // an MN-major operand's 64-wide blocks come as one 3-D box (64
            // columns x 64 K lines x 2 blocks, the blocks 8 KiB apart in shared
            // memory): one TMA operation instead of two
            static_assert(B_BOXES == 2, "the pair's N half is two 64-wide blocks");
            if (GROUP_K) {
              const int k_row = s_off[t.e] + kb * BK;
              tma_load_3d_pair(a_dst, &tmA, 0, k_row, m0 / 64, full0);
              tma_load_3d_pair(b_dst, &tmB, 0, k_row, n0 / 64, full0);
            } else {
              tma_load_2d_pair(a_dst, &tmA, kb * BK, s_off[t.e] + m0, full0);
              const int k_row = t.e * args.b_rows_per_expert + kb * BK;
              tma_load_3d_pair(b_dst, &tmB, 0, k_row, n0 / 64, full0);
            }
          } else {
            mbar_arrive_expect_tx(full, STAGE_BYTES);
            if (GROUP_K) {
              const int k_row = s_off[t.e] + kb * BK;
              tma_load_2d(a_dst, &tmA, t.mt * BM, k_row, full);
              tma_load_2d(a_dst + MN_BOX_BYTES, &tmA, t.mt * BM + 64, k_row, full);
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(b_dst + j * MN_BOX_BYTES, &tmB, t.nt * BN + 64 * j, k_row, full);
            } else {
              tma_load_2d(a_dst, &tmA, kb * BK, s_off[t.e] + t.mt * BM, full);
              const int k_row = t.e * args.b_rows_per_expert + kb * BK;
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(b_dst + j * MN_BOX_BYTES, &tmB, t.nt * BN + 64 * j, k_row, full);
            }
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && (!PAIR || rank == 0)) {
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
          mbar_wait_drain(smem_u32(&s.full[stage]), phase);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && PAIR && rank != 0) {
    // ================= the odd CTA of a pair: no MMAs; wait for the even CTA's last ones =================
    if (lane == 0 && !mbar_wait_drain(smem_u32(&s.drain), 0)) *abort_flag = 1;
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA warp (lane 0 issues; the warp zeroes tail K lines) =================
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int tile = tile0; tile < total && ok; tile += tstep, ++local) {
      const Tile t = decode(s_pre, E, args.n_tiles, tile);
      const int count = s_cnt[t.e];
      const int kbs = GROUP_K ? (count + BK - 1) / BK : args.k_blocks;
      const int buf = local & 1;
      const uint32_t use = (local >> 1) & 1;
      if (!wait_warp(smem_u32(&s.tempty[buf]), use ^ 1u, abort_flag, lane)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (int kb = 0; kb < kbs; ++kb) {
        if (!wait_warp(smem_u32(&s.full[stage]), phase, abort_flag, lane)) { ok = false; break; }
        const uint32_t a_addr = tiles_u32 + stage * STAGE_BYTES;
        if (GROUP_K) {
          const int valid = count - kb * BK;
          if (valid < BK && args.zero_tail) {
            // zero K lines [valid, 64) of the two A boxes and the BN/64 B boxes
            const int lines = BK - valid;
            const int per_box = lines * 8;  // 16-byte chunks
            const int nbox = 2 + BN / 64;
            for (int i = lane; i < nbox * per_box; i += 32) {
              const int box = i / per_box;
              const int rem = i - box * per_box;
              const int line = valid + (rem >> 3);
              const uint32_t box_base = box < 2 ? a_addr + box * MN_BOX_BYTES
                                                : a_addr + A_BYTES + (box - 2) * MN_BOX_BYTES;
              const uint32_t addr = box_base + line * 128 + (rem & 7) * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t a_desc = sdesc_sw128(a_addr + kk * A_STEP, A_LBO, 1024);
            const uint64_t b_desc = sdesc_sw128(b_addr + kk * B_STEP, B_LBO, 1024);
            if constexpr (PAIR)
              tc_mma_bf16_pair(d_tmem, a_desc, b_desc, IDESC, (kb | kk) != 0);
            else
              tc_mma_bf16(d_tmem, a_desc, b_desc, IDESC, (kb | kk) != 0);
          }
          if constexpr (PAIR)
            tc_commit_pair(smem_u32(&s.empty[stage]));
          else
            tc_commit(smem_u32(&s.empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok && lane == 0) {
        if constexpr (PAIR)
          tc_commit_pair(smem_u32(&s.tfull[buf]));
        else
          tc_commit(smem_u32(&s.tfull[buf]));
      }
      __syncwarp();
    }
    if (lane == 0) {
      if constexpr (PAIR)
        tc_commit_pair(smem_u32(&s.drain));
      else
        tc_commit(smem_u32(&s.drain));
      if (!mbar_wait_drain(smem_u32(&s.drain), 0)) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..9) =================
    // Warp w reads TMEM lane quarter w % 4 and takes column half (w - 2) / 4
    // of each tile.  A warp whose 32 rows are all written stores 32-row boxes
    // through TMA; a warp with rows past the group stores its rows directly.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r_in_tile = q * 32 + lane;
    StagedStore st{staging_u32 + (warp - 2) * 4096, 0u, lane};
    int local = 0;
    for (int tile = tile0; tile < total; tile += tstep, ++local) {
      const Tile t = decode(s_pre, E, args.n_tiles, tile);
      const int buf = local & 1;
      const uint32_t use = (local >> 1) & 1;
      // every lane waits, then the warp leaves together if any lane's wait ran out
      const bool ready = mbar_wait(smem_u32(&s.tfull[buf]), use, abort_flag);
      if (!__all_sync(FULL_MASK, ready)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (GROUP_K) {
        // dW rows of expert e: rows (e * m_total + m) of the [E * m_total, n_total] output
        const int out_row0 = t.e * args.m_total + t.mt * RB + static_cast<int>(rank) * BM + q * 32;
        const bool empty = s_cnt[t.e] == 0;
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          uint32_t v[32];
          __syncwarp();
          if (!empty) {
            tmem_ld32(tb + c, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          st.box(&tmOut, v, t.nt * BN + c, out_row0);
          st.box(&tmOut, v + 16, t.nt * BN + c + 16, out_row0);
        }
      } else {
        // rows written: the expert's group (valid and pad rows) inside the tile
        const int group_row = t.mt * RB + static_cast<int>(rank) * BM + r_in_tile;
        const bool valid = group_row < s_off[t.e + 1] - s_off[t.e];
        const bool full_warp = __all_sync(FULL_MASK, valid);
        const long long row = static_cast<long long>(s_off[t.e]) + group_row;
        const int warp_row0 = s_off[t.e] + t.mt * RB + static_cast<int>(rank) * BM + q * 32;
        const int col0 = t.nt * BN;
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
          if (!__any_sync(FULL_MASK, valid)) continue;
          if (EPI == EPI_DSWIGLU) {
            uint32_t og[16], ou[16];
            uint4 g4[4], u4[4];
            const uint4* gp = reinterpret_cast<const uint4*>(args.gu + row * (2 * args.I) + col0 + c);
            const uint4* up = reinterpret_cast<const uint4*>(args.gu + row * (2 * args.I) + args.I + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              g4[i] = valid ? gp[i] : make_uint4(0, 0, 0, 0);
              u4[i] = valid ? up[i] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t gw[4] = {g4[i].x, g4[i].y, g4[i].z, g4[i].w};
              const uint32_t uw[4] = {u4[i].x, u4[i].y, u4[i].z, u4[i].w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float rg[2], ru[2];
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                  const float g = hlf ? bf16_hi(gw[k]) : bf16_lo(gw[k]);
                  const float u = hlf ? bf16_hi(uw[k]) : bf16_lo(uw[k]);
                  const float gh = __uint_as_float(v[8 * i + 2 * k + hlf]);
                  const float sg = 1.0f / (1.0f + __expf(-g));
                  const float dsilu = sg * (1.0f + g * (1.0f - sg));
                  rg[hlf] = gh * u * dsilu;
                  ru[hlf] = gh * g * sg;
                }
                og[4 * i + k] = pack_bf16x2(rg[0], rg[1]);
                ou[4 * i + k] = pack_bf16x2(ru[0], ru[1]);
              }
            }
            if (full_warp) {
              st.box(&tmOut, og, col0 + c, warp_row0);
              st.box(&tmOut, ou, args.I + col0 + c, warp_row0);
            } else if (valid) {
              uint4* dg = reinterpret_cast<uint4*>(args.out_bf16 + row * args.ld_out + col0 + c);
              uint4* du = reinterpret_cast<uint4*>(args.out_bf16 + row * args.ld_out + args.I + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                dg[i] = make_uint4(og[4 * i], og[4 * i + 1], og[4 * i + 2], og[4 * i + 3]);
                du[i] = make_uint4(ou[4 * i], ou[4 * i + 1], ou[4 * i + 2], ou[4 * i + 3]);
              }
            }
          } else {
            uint32_t ov[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              ov[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            if (full_warp) {
              st.box(&tmOut, ov, col0 + c, warp_row0);
            } else if (valid) {
              uint4* d4 = reinterpret_cast<uint4*>(args.out_bf16 + row * args.ld_out + col0 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(mapa_shared(smem_u32(&s.tempty[buf]), 0));  // the MMA issuer's barrier
        else
          mbar_arrive(smem_u32(&s.tempty[buf]));
      }
    }
    st.finish();
  }

  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA frees its tensor memory or leaves while the pair's
  // MMAs, loads or barrier signals may still reach it
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && s.abort) report(args.status, MOE_DEVERR_TIMEOUT);
}

// G_o[r] = bf16(w_r * grad_y[r]) on the valid rows and 0 on the pad rows
// (rows below R = totals[0] with no token); one warp per row.
__global__ void __launch_bounds__(256) scale_rows_kernel(const uint16_t* __restrict__ grad_y,
                                                         const int* __restrict__ row_token,
                                                         const float* __restrict__ row_weight,
                                                         const int* __restrict__ totals,
                                                         long long C, int H,
                                                         uint16_t* __restrict__ g_o) {
  const long long R = totals[0];
  const int lane = threadIdx.x & 31;
  const int V = H >> 8;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < C && r < R; r += nwarps) {
    uint4* dst = reinterpret_cast<uint4*>(g_o + r * H);
    if (row_token[r] < 0) {
      for (int v = lane; v < 32 * V; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const float w = row_weight[r];
    const uint4* src = reinterpret_cast<const uint4*>(grad_y + r * H);
    for (int v = lane; v < 32 * V; v += 32) {
      const uint4 a = __ldg(src + v);
      dst[v] = make_uint4(pack_bf16x2(w * bf16_lo(a.x), w * bf16_hi(a.x)),
                          pack_bf16x2(w * bf16_lo(a.y), w * bf16_hi(a.y)),
                          pack_bf16x2(w * bf16_lo(a.z), w * bf16_hi(a.z)),
                          pack_bf16x2(w * bf16_lo(a.w), w * bf16_hi(a.w)));
    }
  }
}

template <bool GROUP_K, int BN, int EPI, int STAGES, bool PAIR = false>
cudaError_t launch_bwd_stages(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                              const BwdArgs& args, cudaStream_t s) {
  auto kernel = bwd_gemm_kernel<GROUP_K, BN, EPI, STAGES, PAIR>;
  static bool configured[64] = {};
  static int pair_grid[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const size_t smem = smem_bytes<BN, PAIR>(STAGES, args.E);
  if constexpr (!PAIR) {
    kernel<<<sm_count(), NUM_THREADS, smem, s>>>(a, b, out, args);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many pairs as can be resident at once (a pair needs two
    // free SMs of one GPC), at most one CTA per SM
    int grid = dev >= 0 && dev < 64 ? pair_grid[dev] : 0;
    if (grid == 0) {
      cfg.gridDim = dim3(sm_count() & ~1);
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
        clusters = sm_count() / 2;
      grid = 2 * (clusters < sm_count() / 2 ? clusters : sm_count() / 2);
      if (dev >= 0 && dev < 64) pair_grid[dev] = grid;
    }
    cfg.gridDim = dim3(grid);
    return cudaLaunchKernelEx(&cfg, kernel, a, b, out, args);
  }
}

// The deepest ring that fits beside the staging and the per-expert tables
// (a pair's 32 KiB stages: six; 48 KiB stages: four).
template <bool GROUP_K, int BN, int EPI, bool PAIR = false>
cudaError_t launch_bwd(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                       const BwdArgs& args, cudaStream_t s) {
  constexpr int MS = PAIR ? 6 : Cfg<BN>::MAX_STAGES;
  if (smem_bytes<BN, PAIR>(MS, args.E) <= static_cast<size_t>(SMEM_LIMIT))
    return launch_bwd_stages<GROUP_K, BN, EPI, MS, PAIR>(a, b, out, args, s);
  return launch_bwd_stages<GROUP_K, BN, EPI, MS - 1, PAIR>(a, b, out, args, s);
}

// 256-column tiles where N allows, on CTA pairs when the layer has rows for
// them (pair): the M-grouped dgrads always, the K-grouped wgrads when M is a
// multiple of 256 and no K lines need masking.
// a3 / b3: the operands' maps for the pair kernel, whose MN-major operands
// load two 64-wide blocks per box (make_tma_rows_k128 with 64-line boxes).
template <bool GROUP_K, int EPI>
cudaError_t launch_bwd_bn(int n_total, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a3,
                          const CUtensorMap& b3, const CUtensorMap& out, BwdArgs args, cudaStream_t s,
                          bool pair) {
  if (n_total % 256 == 0) {
    args.n_tiles = n_total / 256;
    if (pair && (!GROUP_K || (args.m_total % 256 == 0 && !args.zero_tail))) {
      if (GROUP_K) args.m_tiles = args.m_total / 256;
      return launch_bwd<GROUP_K, 256, EPI, true>(a3, b3, out, args, s);
    }
    return launch_bwd<GROUP_K, 256, EPI>(a, b, out, args, s);
  }
  args.n_tiles = n_total / 128;
  return launch_bwd<GROUP_K, 128, EPI>(a, b, out, args, s);
}

}  // namespace

size_t experts_backward_workspace(long long capacity, int H, int I) {
  const size_t go = static_cast<size_t>(capacity) * H * 2;
  const size_t gu = static_cast<size_t>(capacity) * 2 * I * 2;
  return ((go + 255) / 256) * 256 + ((gu + 255) / 256) * 256 + 256;
}

cudaError_t launch_experts_backward(const uint16_t* grad_y, const uint16_t* x_disp,
                                    const uint16_t* h, const uint16_t* gu_save, const moe_layout& L,
                                    int H, int I, const uint16_t* W1, const uint16_t* W2,
                                    uint16_t* grad_x_disp, float* dW1, float* dW2, void* workspace,
                                    cudaStream_t s, bool g_o_given) {
  const long long C = L.capacity;
  const int E = L.E;
  uintptr_t ws = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255);
  // g_o_given: grad_y already holds G_o = bf16(w * grad_y) (the scaled combine
  // backward wrote it), so the scaling pass is skipped
  uint16_t* g_o = g_o_given ? const_cast<uint16_t*>(grad_y) : reinterpret_cast<uint16_t*>(ws);
  uint16_t* g_gu = reinterpret_cast<uint16_t*>(ws + ((static_cast<size_t>(C) * H * 2 + 255) / 256) * 256);

  if (C > 0 && !g_o_given) {
    const long long need = (C + 7) / 8;
    const int blocks = static_cast<int>(need < 8LL * sm_count() ? need : 8LL * sm_count());
    scale_rows_kernel<<<blocks, 256, 0, s>>>(grad_y, L.row_token, L.row_weight, L.totals, C, H, g_o);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }

  // CTA pairs for layers with rows for every SM, as in the forward: at least
  // as many experts' 256-column tiles as SMs
  const long long pairs_rows = static_cast<long long>(L.T) * L.K;
  const bool pair = (pairs_rows < E ? pairs_rows : E) * (I / 128) >= sm_count();
  BwdArgs base{};
  base.capacity = C;
  base.counts = L.tokens_per_expert;
  base.offsets = L.offsets;
  base.E = E;
  base.status = L.status;
  base.I = I;
  cudaError_t err = cudaSuccess;

  if (C > 0) {
    // dgrad1: G_gu = SwiGLU'(G_o W2)
    CUtensorMap mA, mB, mB3, mO;
    if (!make_tma_2d_bf16(&mA, g_o, C, H, 128) ||
        !make_tma_2d_bf16(&mB, W2, static_cast<uint64_t>(E) * H, I, 64) ||
        !make_tma_rows_k128(&mB3, W2, static_cast<uint64_t>(E) * H, I, 64) ||
        !make_tma_store_2d_bf16(&mO, g_gu, C, 2 * I))
      return cudaErrorInvalidValue;
    BwdArgs a = base;
    a.k_blocks = H / BK;
    a.b_rows_per_expert = H;
    a.out_bf16 = g_gu;
    a.ld_out = 2 * I;
    a.gu = gu_save;
    err = launch_bwd_bn<false, EPI_DSWIGLU>(I, mA, mB, mA, mB3, mO, a, s, pair);
    if (err != cudaSuccess) return err;

    // dgrad2: grad_x_disp = G_gu W1
    if (!make_tma_2d_bf16(&mA, g_gu, C, 2 * I, 128) ||
        !make_tma_2d_bf16(&mB, W1, static_cast<uint64_t>(E) * 2 * I, H, 64) ||
        !make_tma_rows_k128(&mB3, W1, static_cast<uint64_t>(E) * 2 * I, H, 64) ||
        !make_tma_store_2d_bf16(&mO, grad_x_disp, C, H))
      return cudaErrorInvalidValue;
    a = base;
    a.k_blocks = 2 * I / BK;
    a.b_rows_per_expert = 2 * I;
    a.out_bf16 = grad_x_disp;
    a.ld_out = H;
    err = launch_bwd_bn<false, EPI_BF16>(H, mA, mB, mA, mB3, mO, a, s, pair);
    if (err != cudaSuccess) return err;
  }

  // wgrad2: dW2[e] = G_o^T h     (M = H, N = I, K = the expert's rows)
  {
    CUtensorMap mA, mB, mA3, mB3, mO;
    const uint64_t rows = C > 0 ? static_cast<uint64_t>(C) : 1;
    const void* a_src = C > 0 ? static_cast<const void*>(g_o) : static_cast<const void*>(dW2);
    const void* b_src = C > 0 ? static_cast<const void*>(h) : static_cast<const void*>(dW2);
    if (!make_tma_2d_bf16(&mA, a_src, rows, H, 64) || !make_tma_2d_bf16(&mB, b_src, rows, I, 64) ||
        !make_tma_rows_k128(&mA3, a_src, rows, H, 64) || !make_tma_rows_k128(&mB3, b_src, rows, I, 64) ||
        !make_tma_store_2d_f32(&mO, dW2, static_cast<uint64_t>(E) * H, I))
      return cudaErrorInvalidValue;
    BwdArgs a = base;
    a.m_tiles = H / BM;
    // With groups padded to a multiple of 64 rows, an expert's last K block
    // holds only its own pad rows, which are zero in every operand (x_disp by
    // the dispatch, h and the gate/up values by the forward, G_o and G_gu
    // here); otherwise the lines past the count are zeroed in shared memory.
    a.zero_tail = (L.pad_multiple % BK) != 0;
    a.m_total = H;
    a.n_total = I;
    a.out_f32 = dW2;
    err = launch_bwd_bn<true, EPI_F32>(I, mA, mB, mA3, mB3, mO, a, s, pair);
    if (err != cudaSuccess) return err;
  }
  // wgrad1: dW1[e] = G_gu^T x_disp   (M = 2I, N = H)
  {
    CUtensorMap mA, mB, mA3, mB3, mO;
    const uint64_t rows = C > 0 ? static_cast<uint64_t>(C) : 1;
    const void* a_src = C > 0 ? static_cast<const void*>(g_gu) : static_cast<const void*>(dW1);
    const void* b_src = C > 0 ? static_cast<const void*>(x_disp) : static_cast<const void*>(dW1);
    if (!make_tma_2d_bf16(&mA, a_src, rows, 2 * I, 64) || !make_tma_2d_bf16(&mB, b_src, rows, H, 64) ||
        !make_tma_rows_k128(&mA3, a_src, rows, 2 * I, 64) || !make_tma_rows_k128(&mB3, b_src, rows, H, 64) ||
        !make_tma_store_2d_f32(&mO, dW1, static_cast<uint64_t>(E) * 2 * I, H))
      return cudaErrorInvalidValue;
    BwdArgs a = base;
    a.m_tiles = 2 * I / BM;
    // With groups padded to a multiple of 64 rows, an expert's last K block
    // holds only its own pad rows, which are zero in every operand (x_disp by
    // the dispatch, h and the gate/up values by the forward, G_o and G_gu
    // here); otherwise the lines past the count are zeroed in shared memory.
    a.zero_tail = (L.pad_multiple % BK) != 0;
    a.m_total = 2 * I;
    a.n_total = H;
    a.out_f32 = dW1;
    err = launch_bwd_bn<true, EPI_F32>(H, mA, mB, mA3, mB3, mO, a, s, pair);
  }
  return err;
}

}  // namespace moe
