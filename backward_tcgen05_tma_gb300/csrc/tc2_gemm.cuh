// tc2_gemm.cuh -- the tensor-core GEMM on SM pairs (tcgen05 cta_group::2).
//
// A cluster of two CTAs on the two SMs of a TPC computes 256 x 256 output
// tiles with one tcgen05.mma.cta_group::2 M=256 N=256 K=16 per step, issued
// by the even CTA.  Each CTA's shared memory holds its own 128 rows of A and
// its own half (128 of the 256 columns) of B, loaded by its own TMA; each
// CTA's TMEM holds its 128 rows of the accumulator.  Per SM and k-block that
// is 32 KB of operands instead of the 48 KB of a 128 x 256 single-SM tile for
// the same tensor-core work, which relieves the shared-memory port that both
// TMA writes and MMA operand reads go through.
//
// Roles, per CTA (10 warps as in tc_gemm.cuh):
//   warp 0      TMA producer (both CTAs): waits for its own ring slot to be
//               free (the MMA's commit reaches both CTAs), loads its halves,
//               and counts the bytes on the even CTA's "full" barrier;
//   warp 1      both CTAs allocate TMEM for the pair; the even CTA issues the
//               MMAs and commits to both CTAs' "empty" / "accumulator full"
//               barriers;
//   warps 2..9  epilogue of this CTA's 128 rows (the epilogues of
//               tc_gemm.cuh, or the TMA dG/dU form below); one arrival per
//               warp on the even CTA's "accumulator empty" barrier.
// Tiles (and the stream-K shares of the hybrid) are handed out per cluster.
#pragma once

#include "tc_gemm.cuh"

namespace swiglu {

constexpr int TC2_BM = 256;  // output rows per tile (128 per CTA)
constexpr int TC2_BN = 256;

// The TMA form of the dG/dU epilogue: each epilogue warp streams its 32 x 32
// chunks of G and U through GU_SLOTS shared-memory slots (G box, then U box).
// Two slots leave room for five ring stages; three slots (loads two chunks
// ahead, four stages) measured 3% slower at D = 1024 and D = 2048.
constexpr int GU_SLOTS = 2;
constexpr int GU_SLOT_BYTES = 4096;
constexpr int GU_CHUNKS = TC2_BN / 64;  // 32-column chunks per warp and tile

// GU: the epilogue is the TMA dG/dU form (G/U slots and their barriers
// instead of the 2 KB store-staging buffers).
// BN: tile columns, 256 (two 256-column accumulators, the epilogue of one
// tile overlapping the next tile's main loop) or 512 (one accumulator of all
// 512 TMEM columns: each A k-block feeds twice the columns, for the long
// contractions whose main loop dwarfs the epilogue).  Each CTA holds BN / 2
// columns of B per stage, as BN / 256 chunks of 128.
template <int STAGES, bool GU = false, int BN = TC2_BN>
struct Tc2Smem {
  static constexpr int A_BYTES = 128 * TC_BK * 2;       // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * TC_BK * 2;  // this CTA's BN / 2 columns of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;  // 8 warps x 2 KB store staging
  static constexpr int GU_OFFSET = EPI_OFFSET + (GU ? 0 : 8 * 2048);  // 8 warps x GU_SLOTS slots
  static constexpr int BAR_OFFSET = GU_OFFSET + (GU ? 8 * GU_SLOTS * GU_SLOT_BYTES : 0);
  // barriers: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain,
  // then (GU) one per G/U slot
  static constexpr int GU_BAR = 2 * STAGES + 5;
  static constexpr int NUM_BARS = GU_BAR + (GU ? 8 * GU_SLOTS : 0);
  static constexpr int MISC_OFFSET = BAR_OFFSET + NUM_BARS * 8;  // tmem slot, abort, last
  static constexpr int TOTAL = MISC_OFFSET + 16;
  static constexpr int DYN_BYTES = TOTAL + 1024;
  static constexpr int NACC = BN > 256 ? 1 : 2;  // accumulators in TMEM
  static constexpr int TMEM_COLS = NACC * BN;
};

// Backward SwiGLU epilogue (the math of EpiDSwiGLUT) with its G/U traffic on
// TMA: per warp, G and U arrive in 32 x 32 boxes (64-byte swizzle, so that
// each lane reads its row without bank conflicts) GU_SLOTS - 1 chunks ahead
// -- across tiles too, when the next tile is taken whole -- and dG, dU are
// written back into the same slot and leave by TMA store.  The tensor maps
// bound both directions at M rows and H columns (ragged tiles need no
// checks), and no register holds a prefetched chunk.  With a short
// contraction (K = D <= 2048) the epilogue bounds this GEMM and its loads,
// issued one chunk ahead from registers, were latency-bound.
struct EpiDSwiGLUTma {
  static constexpr bool TMA_GU = true;
  // the kernel's tensor maps tmG (G [M][H] within the saved rows, row stride
  // 3H, box 32 x 32) and tmU (U, the same at column offset H) carry G and U
  struct Params {
    float gate_mul, down_mul;
  };
};

template <class E, class = void>
struct epi_tma_gu {
  static constexpr bool value = false;
};
template <class E>
struct epi_tma_gu<E, decltype((void)E::TMA_GU)> {
  static constexpr bool value = E::TMA_GU;
};

// Wait until at most n of this thread's committed bulk groups still read
// shared memory (n clamped to the GU_SLOTS - 1 the pipeline can need).
__device__ __forceinline__ void bulk_wait_group_read_n(int n) {
  static_assert(GU_SLOTS <= 4, "bulk_wait_group_read_n covers up to 3 pending groups");
  if (n <= 0)
    bulk_wait_group_read<0>();
  else if (n == 1)
    bulk_wait_group_read<1>();
  else if (n == 2)
    bulk_wait_group_read<2>();
  else
    bulk_wait_group_read<3>();
}

// One epilogue warp's stream of G/U jobs: job k (one 32 x 32 chunk) uses
// slot k % GU_SLOTS and that slot's barrier phase (k / GU_SLOTS) & 1.  Each
// job commits one bulk group of stores (empty when nothing is stored), so
// group k belongs to job k.  The issue cursor walks the chunks of a tile
// (row0, col0), then of the next tile if it is known to run its epilogue.
struct GuPipe {
  uint32_t slot0, bar0;      // slot 0's shared address and barrier
  uint32_t issued, done;     // jobs whose loads were issued / whose stores were issued
  int cur_row0, cur_col0, cur_c;  // next job to issue: chunk cur_c (GU_CHUNKS: none)
  int nxt_row0, nxt_col0;
  bool nxt;

  // Issue jobs up to index kmax (lane 0 issues; every lane keeps the count).
  __device__ __forceinline__ void issue_upto(uint32_t kmax, const CUtensorMap* gm,
                                             const CUtensorMap* um, int lane) {
    while (issued <= kmax && cur_c < GU_CHUNKS) {
      const uint32_t b = issued % GU_SLOTS;
      if (lane == 0 && issued >= (uint32_t)GU_SLOTS) {
        // the slot's previous job, issued - GU_SLOTS, must have finished
        // reading its dG/dU out of the slot; the groups committed after its
        // own (done - 1 - (issued - GU_SLOTS) of them) may still be reading
        const int prev = (int)issued - GU_SLOTS;
        if (prev < (int)done) bulk_wait_group_read_n((int)done - 1 - prev);
      }
      if (lane == 0) {
        const uint32_t bar = bar0 + 8u * b, dst = slot0 + GU_SLOT_BYTES * b;
        mbar_arrive_expect_tx(bar, GU_SLOT_BYTES);
        tma_load_2d(dst, gm, bar, cur_col0 + cur_c * 32, cur_row0);
        tma_load_2d(dst + 2048, um, bar, cur_col0 + cur_c * 32, cur_row0);
      }
      ++issued;
      if (++cur_c == GU_CHUNKS && nxt) {
        cur_row0 = nxt_row0;
        cur_col0 = nxt_col0;
        cur_c = 0;
        nxt = false;
      }
    }
  }
};

// One tile's dG/dU for this warp's 32 rows (from row0) and GU_CHUNKS chunks
// (from column col0; TMEM columns from tacc) of the M x H matrices.  nxt:
// the next tile of this CTA, if taken whole (its epilogue certainly runs),
// whose first chunks may be loaded during this one.  Loads of boxes outside
// the matrices read zeros; stores of boxes wholly outside are not issued.
// Returns false if a wait ran out.
template <bool BF16>
__device__ __forceinline__ bool dgu_tma_tile(GuPipe& gp, const CUtensorMap* gm,
                                             const CUtensorMap* um, const EpiDSwiGLUTma::Params& p,
                                             uint32_t tacc, int row0, int col0, int M, int H,
                                             bool nxt, int nrow0, int ncol0, int lane,
                                             uint8_t* slots, uint64_t wl, volatile int* abort_flag,
                                             int* err) {
  if (gp.cur_c == GU_CHUNKS) {  // nothing of this tile issued ahead
    gp.cur_row0 = row0;
    gp.cur_col0 = col0;
    gp.cur_c = 0;
  }
  gp.nxt = nxt;
  gp.nxt_row0 = nrow0;
  gp.nxt_col0 = ncol0;
  const int sw = (lane >> 1) & 3;  // 64-byte swizzle: 16-byte unit q of row r at q ^ ((r / 2) % 4)
#pragma unroll 1
  for (int c = 0; c < GU_CHUNKS; ++c) {
    const uint32_t k = gp.done;
    gp.issue_upto(k + GU_SLOTS - 2, gm, um, lane);  // this chunk (and any ahead) on its way
    const uint32_t b = k % GU_SLOTS;
    const int ok = mbar_wait_bounded(gp.bar0 + 8u * b, (k / GU_SLOTS) & 1u, wl, abort_flag, err);
    if (!__all_sync(0xffffffffu, ok)) return false;
    uint8_t* gs = slots + GU_SLOT_BYTES * b + lane * 64;
    uint8_t* us = gs + 2048;
    uint4 vg[4], vu[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      vg[q] = *reinterpret_cast<const uint4*>(gs + ((q ^ sw) << 4));
      vu[q] = *reinterpret_cast<const uint4*>(us + ((q ^ sw) << 4));
    }
    uint32_t r[32];
    tmem_ld_32x32b_x32(tacc + c * 32, r);
    tmem_ld_wait();
    uint32_t odg[16], odu[16];
    dswiglu_32<BF16>(vg, vu, r, p.gate_mul, p.down_mul, odg, odu);
    // GU_SLOTS - 1 chunks ahead, into the slot whose stores left one chunk ago
    gp.issue_upto(k + GU_SLOTS - 1, gm, um, lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      *reinterpret_cast<uint4*>(gs + ((q ^ sw) << 4)) =
          make_uint4(odg[4 * q], odg[4 * q + 1], odg[4 * q + 2], odg[4 * q + 3]);
      *reinterpret_cast<uint4*>(us + ((q ^ sw) << 4)) =
          make_uint4(odu[4 * q], odu[4 * q + 1], odu[4 * q + 2], odu[4 * q + 3]);
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      const uint32_t src = gp.slot0 + GU_SLOT_BYTES * b;
      if (row0 < M && col0 + c * 32 < H) {
        tma_store_2d(gm, src, col0 + c * 32, row0);
        tma_store_2d(um, src + 2048, col0 + c * 32, row0);
      }
      bulk_commit_group();  // (an empty group when nothing was stored)
    }
    ++gp.done;
  }
  return true;
}

template <int STAGES, int A_MODE, int B_MODE, bool BF16, class Epi, int BN = TC2_BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const TcShape s,
                    const typename Epi::Params ep, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmU) {
  constexpr bool TMA_GU = epi_tma_gu<Epi>::value;
  using L = Tc2Smem<STAGES, TMA_GU, BN>;
  static_assert(BN == 256 || (BN == 512 && !TMA_GU && B_MODE != LOAD_GATEUP),
                "512-column tiles serve the plain-store GEMMs");
  constexpr int NACC = L::NACC;
  constexpr int MMA_N = BN > 256 ? 256 : BN;  // columns per tcgen05.mma
  constexpr int NCH = BN / 256;               // B chunks (of 128 columns per CTA) per stage
  static_assert(L::TOTAL + 1024 <= 232448, "shared memory plan exceeds 227 KB");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFFSET;
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (STAGES + i); };
  auto accf_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto acce_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFFSET);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the MMAs
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {  // (the second pair is unused with one accumulator)
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), 16);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    if constexpr (TMA_GU)
      for (int i = 0; i < 8 * GU_SLOTS; ++i) mbar_init(bar0 + 8u * (L::GU_BAR + i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_cg2(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish_cg2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = s.m_tiles * s.n_tiles;
  const int64_t sk_total = (int64_t)s.sk_tiles * s.k_blocks;
  const int cl = (int)(blockIdx.x >> 1);
  const int64_t ncl = gridDim.x >> 1;
  auto segs = [&]() {
    return TcSegIter{sk_start(cl, sk_total, ncl), sk_start(cl + 1, sk_total, ncl), s.k_blocks,
                     s.sk_tiles + cl, num_tiles, (int)ncl};
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      bool skip_once = s.inject_stall != 0 && leader;
      TcSegIter it = segs();
      int tile, kb0, nkb;
      bool whole;
      while (ok && it.next(tile, kb0, nkb, whole)) {
        int mt, nt;
        tc_tile_coords(tile, s, mt, nt);
        const int m0 = mt * TC2_BM + (int)rank * 128;  // this CTA's rows of A
        // this CTA's columns of B: in chunk j, nt * BN + j * 256 + rank * 128
        const int nb = nt * BN + (int)rank * 128;
        for (int kb = kb0; kb < kb0 + nkb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s.wait_limit_ns, abort_flag, s.err)) {
            ok = false;
            break;
          }
          if (skip_once) {
            skip_once = false;  // fault injection: this stage never fills
          } else {
            const uint32_t sa = sbase + stage * L::STAGE_BYTES;
            const uint32_t sb = sa + L::A_BYTES;
            const uint32_t fb = mapa_shared(full_bar(stage), 0);
            const int k0 = kb * TC_BK;
            if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * L::STAGE_BYTES);
            if (A_MODE == LOAD_KMAJOR) {
              tma_load_2d_cg2(sa, &tmA, fb, k0, m0);
            } else {
              tma_load_2d_cg2(sa, &tmA, fb, m0, k0);
              tma_load_2d_cg2(sa + 8192, &tmA, fb, m0 + 64, k0);
            }
            if (B_MODE == LOAD_GATEUP) {
              // the even CTA brings the Wg rows, the odd one the Wu rows
              tma_load_3d_cg2(sb, &tmB, fb, k0, nt * (BN / 2), (int)rank);
            } else {
#pragma unroll
              for (int j = 0; j < NCH; ++j) {
                const uint32_t sbj = sb + j * 16384;
                if (B_MODE == LOAD_KMAJOR) {
                  tma_load_2d_cg2(sbj, &tmB, fb, k0, nb + j * 256);
                } else {
                  tma_load_2d_cg2(sbj, &tmB, fb, nb + j * 256, k0);
                  tma_load_2d_cg2(sbj + 8192, &tmB, fb, nb + j * 256 + 64, k0);
                }
              }
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // unwinding: the copies counted on this CTA's barriers land first
        for (int i = 0; i < STAGES; ++i)
          if (issued_mask & (1u << i))
            mbar_wait_bounded(full_bar(i), (issued_parity >> i) & 1u, s.wait_limit_ns, nullptr,
                              s.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc =
          make_idesc_f16(BF16, A_MODE == LOAD_MNMAJOR, B_MODE == LOAD_MNMAJOR, TC2_BM, MMA_N);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      TcSegIter it = segs();
      int tile, kb0, nkb;
      bool whole;
      while (ok && it.next(tile, kb0, nkb, whole)) {
        if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, s.wait_limit_ns, abort_flag, s.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, s.wait_limit_ns, abort_flag, s.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * L::STAGE_BYTES;
          const uint32_t sb = sa + L::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / TC_UMMA_K; ++kk) {
            const uint64_t ad = (A_MODE == LOAD_MNMAJOR)
                                    ? make_sw128_desc(sa + kk * 2048, 8192, 1024)
                                    : make_sw128_desc(sa + kk * 32, 16, 1024);
#pragma unroll
            for (int j = 0; j < NCH; ++j) {  // chunk j: accumulator columns j*256..
              const uint32_t sbj = sb + j * 16384;
              const uint64_t bd = (B_MODE == LOAD_MNMAJOR)
                                      ? make_sw128_desc(sbj + kk * 2048, 8192, 1024)
                                      : make_sw128_desc(sbj + kk * 32, 16, 1024);
              umma_f16_ss_cg2(d_tmem + j * MMA_N, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit_cg2_mc(empty_bar(stage), 0x3);  // frees the slot in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_cg2_mc(accf_bar(acc), 0x3);  // accumulator complete in both CTAs
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit_cg2_mc(drain_bar, 0x1);
      mbar_wait_bounded(drain_bar, 0, s.wait_limit_ns, nullptr, s.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // column half of the tile
    const int row = quarter * 32 + lane;
    const int e = threadIdx.x - 64;  // 0..255 among the epilogue threads
    constexpr int CH = BN / 64;      // 32-column chunks per half
    int acc = 0;
    uint32_t acc_phase = 0;
    int seg = 0;  // shared segments done (= partial slot index)
    GuPipe gp;    // TMA dG/dU epilogue: this warp's G/U job stream
    gp.slot0 = sbase + L::GU_OFFSET + (warp - 2) * GU_SLOTS * GU_SLOT_BYTES;
    gp.bar0 = bar0 + 8u * (L::GU_BAR + (warp - 2) * GU_SLOTS);
    gp.issued = gp.done = 0;
    gp.cur_c = GU_CHUNKS;
    gp.nxt = false;
    int gu_ok = 1;
    TcSegIter it = segs();
    int tile, kb0, nkb;
    bool whole;
    while (it.next(tile, kb0, nkb, whole)) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(accf_bar(acc), acc_phase, s.wait_limit_ns, abort_flag, s.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!tc_epi_bar_and(ok && gu_ok)) break;
      tc_fence_after();
      int mt, nt;
      tc_tile_coords(tile, s, mt, nt);
      const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      int run_epi = whole ? 1 : 0;
      if (!whole) {
        // this CTA's 128 rows of the partial tile -> its slot, in TMEM order
        float4* slot = reinterpret_cast<float4*>(
            s.part + ((size_t)blockIdx.x * s.seg_max + seg) * (size_t)(TC_BM * BN));
        const bool slot_ok = SWIGLU_CHECK(seg < s.seg_max, s.err) &&
                             SWIGLU_CHECK_PTR(s.dbg, slot, (int64_t)TC_BM * BN * 4, s.err);
#pragma unroll 1
        for (int c = half * CH; c < (half + 1) * CH; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (slot_ok)
              slot[((c * 4 + quarter) * 8 + g) * 32 + lane] =
                  make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                              __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        }
        __threadfence();
        ++seg;
        // clusters sharing this tile; each CTA half of the tile has its own counter
        const int c_first = sk_owner((int64_t)tile * s.k_blocks, sk_total, ncl);
        const int c_last = sk_owner((int64_t)(tile + 1) * s.k_blocks - 1, sk_total, ncl);
        tc_epi_bar();
        if (e == 0) {
          int last = 0;
          if (!*abort_flag)
            last = SWIGLU_CHECK(2 * tile + rank < 2 * s.sk_tiles, s.err) &&
                   atomicAdd(s.counters + 2 * tile + rank, 1) == c_last - c_first;
          *last_flag = last;
        }
        tc_epi_bar();
        run_epi = *last_flag;
        if (run_epi) {
          __threadfence();
#pragma unroll 1
          for (int c = half * CH; c < (half + 1) * CH; ++c) {
            uint32_t own[32];
            tmem_ld_32x32b_x32(tacc + c * 32, own);
            tmem_ld_wait();
            float sum[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
#pragma unroll 1
            for (int pc = c_first; pc <= c_last; ++pc) {
              if (pc == cl) {
#pragma unroll
                for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(own[i]);
              } else {
                const int j = tile - (int)(sk_start(pc, sk_total, ncl) / s.k_blocks);
                const float4* ps = reinterpret_cast<const float4*>(
                    s.part + ((size_t)(2 * pc + rank) * s.seg_max + j) * (size_t)(TC_BM * BN));
                const bool ps_ok =
                    SWIGLU_CHECK(j >= 0 && j < s.seg_max, s.err) &&
                    SWIGLU_CHECK_PTR(s.dbg, ps, (int64_t)TC_BM * BN * 4, s.err);
                float4 v[8];
#pragma unroll
                for (int g = 0; g < 8; ++g)
                  v[g] = ps_ok ? __ldcg(ps + ((c * 4 + quarter) * 8 + g) * 32 + lane)
                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  sum[4 * g] += v[g].x;
                  sum[4 * g + 1] += v[g].y;
                  sum[4 * g + 2] += v[g].z;
                  sum[4 * g + 3] += v[g].w;
                }
              }
            }
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(sum[i]);
            tmem_st_32x32b_x32(tacc + c * 32, w);
          }
          tmem_st_wait();
          // ready for the next launch
          if (e == 0 && SWIGLU_CHECK(2 * tile + rank < 2 * s.sk_tiles, s.err))
            s.counters[2 * tile + rank] = 0;
          tc_fence_before();
          tc_epi_bar();
          tc_fence_after();
        }
      }
      if (run_epi) {
        if constexpr (TMA_GU) {
          // the next segment, when whole, certainly runs its epilogue next
          TcSegIter pk = it;
          int t2, kb2, nkb2, mt2 = 0, nt2 = 0;
          bool w2 = false;
          const bool nx = pk.next(t2, kb2, nkb2, w2) && w2;
          if (nx) tc_tile_coords(t2, s, mt2, nt2);
          const int rq = (int)rank * 128 + quarter * 32;
          gu_ok = dgu_tma_tile<BF16>(gp, &tmG, &tmU, ep, tacc + half * CH * 32, mt * TC2_BM + rq,
                                     nt * BN + half * (BN / 2), s.M, s.N, nx, mt2 * TC2_BM + rq,
                                     nt2 * BN + half * (BN / 2), lane,
                                     smem + L::GU_OFFSET + (warp - 2) * GU_SLOTS * GU_SLOT_BYTES,
                                     s.wait_limit_ns, abort_flag, s.err)
                      ? 1
                      : 0;
        } else {
          Epi::template run<BN, BF16>(ep, s, tacc, mt * TC2_BM + (int)rank * 128, nt, row, half,
                                      smem + L::EPI_OFFSET + (warp - 2) * 2048);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (TMA_GU) {
      if (lane == 0) {
        // loads issued ahead but never used (the loop ended early) land
        // before the CTA exits; the dG/dU stores complete
        for (uint32_t k = gp.done; k < gp.issued; ++k)
          mbar_wait_bounded(gp.bar0 + 8u * (k % GU_SLOTS), (k / GU_SLOTS) & 1u, s.wait_limit_ns,
                            nullptr, s.err);
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair frees its TMEM together, after both are done
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_cg2(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace swiglu
