// ng_gemm.cuh -- the no-grad forward for a handful of tokens (M <= 64), where
// the work is bound by streaming the weights from HBM, not by the tensor core.
//
// Swap-AB: 128 weight rows take the MMA's M dimension and the (padded) tokens
// its N dimension (NT = 16, 32, 48 or 64), so one tcgen05.mma M=128 x N=NT x K=16
// consumes 4 KB of weights.  The weight stream is spread evenly over every
// SM by a stream-K decomposition: the tiles' k-blocks are laid end to end
// (tile-major) and each persistent CTA (one per SM) takes one contiguous
// range of that sequence, so every CTA streams the same number of bytes and
// its TMA ring never drains between tiles.  A range cuts a tile into
// segments; each segment's fp32 partial tile goes to the workspace (slot =
// CTA x segment index), two TMEM accumulators let the epilogue of one segment
// overlap the MMAs of the next, and the last CTA of a tile to finish (per-tile
// arrival counter) sums the tile's partials in CTA order -- deterministic --
// and applies the epilogue:
//   gate/up: tile = 64 hidden units; rows 0..63 are Wg rows, 64..127 the Wu
//            rows of the same units (one 3-D TMA box), so the partial sums of
//            G and U meet in one CTA: A = rnd(SiLU(g) * u) -> A [M, H];
//   down:    tile = 128 output features of Wd; Y = rnd(sum) -> Y [M, D].
// When there are at least as many tiles as CTAs the split is a hybrid: the
// first tiles (tiles mod CTAs of them) are shared stream-K style and every CTA
// streams its share of those first, so their reductions happen mid-kernel;
// then each CTA takes whole tiles, whose epilogue writes the output straight
// from TMEM (no partial, no counter, no reduction at the end of the kernel).
// No CTA ever waits for another CTA: a segment that is not last moves on.
// The down kernel is launched as a programmatic dependent of the gate/up
// kernel: its CTAs start streaming Wd into the ring while gate/up drains, and
// wait (griddepcontrol.wait) only before touching anything gate/up writes.
//
// Packed weights (PACKED): the weight boxes were laid out once, ahead of the
// calls, as contiguous 16 KB blocks in the order the stream-K split consumes
// them (tile-major, k-blocks within a tile), each already in the 128-byte
// swizzled form the TMA box load would produce in shared memory.  A CTA's
// range is then one contiguous region of the packed buffer, fetched with
// plain bulk copies instead of 128-byte rows scattered over the weight
// matrix; the shared-memory contents, and so the results, are the same.
#pragma once

#include "tc_gemm.cuh"

namespace swiglu {

struct NgArgs {
  int M;            // tokens (<= NT)
  int rows;         // gate/up: H (hidden units); down: D (output features)
  int kb_tile;      // k-blocks of 64 in one tile's contraction
  int tiles;
  int sk_tiles;     // tiles [0, sk_tiles) are shared stream-K; the rest are whole,
                    //   (tiles - sk_tiles) / gridDim.x per CTA
  int seg_max;      // partial slots per CTA (>= stream-K segments of any CTA)
  float* part;      // [gridDim.x * seg_max][128][NT] fp32 partial tiles
  int* counters;    // [tiles] arrival counters, zero at launch
  int* zero_ptr;    // block 0 zeroes zero_ptr[0 .. zero_count): the other
  int zero_count;   //   kernel's counters (after the dependency wait)
  int clear_err;    // block 0 clears the error word at start (first kernel of a call)
  int dependent;    // launched as a programmatic dependent of the gate/up kernel
  int ctas;         // CTAs that share the work (the grid, or fewer in a fused phase)
  void* out;        // A [M, ld_out] or Y [M, ld_out]
  int64_t ld_out;
  uint64_t wait_limit_ns;
  int* err;
  float scale = 1.0f;  // gate/up: gate multiplier (SiLU(scale g) u); down: Y = scale y
  const uint8_t* wpack = nullptr;  // PACKED: this GEMM's boxes, box (tile, kb) at
                                   //   (tile * kb_tile + kb) * 16 KB
#ifdef SWIGLU_DEBUG
  DbgWin dbg;       // buffers the kernel may touch by plain accesses: out, workspace
#endif
};

// out[m, col] = rnd(v) (one element of A or Y); debug builds check the address
// against the launch's windows.
template <bool BF16>
__device__ __forceinline__ void ng_put(const NgArgs& a, int m, int col, float v) {
  if (BF16) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.out) + (int64_t)m * a.ld_out + col;
    if (SWIGLU_CHECK_PTR(a.dbg, o, 2, a.err)) *o = __float2bfloat16_rn(v);
  } else {
    __half* o = reinterpret_cast<__half*>(a.out) + (int64_t)m * a.ld_out + col;
    if (SWIGLU_CHECK_PTR(a.dbg, o, 2, a.err)) *o = __float2half_rn(v);
  }
}

template <int NT, int RING_KB = 110>
struct NgSmem {
  static constexpr int W_BYTES = 128 * 64 * 2;  // 16 KB of weights per k-block
  static constexpr int X_BYTES = NT * 64 * 2;   // the tokens' k-block
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int USTAGE_BYTES = 64 * NT * 4;  // U rows of a whole gate/up tile
  // ~110 KB of ring (5 stages at 16 and 32 tokens, 4 at 64): single L2-flushed
  // calls at D = 4096, H = 11008 measured 62.1 vs 64.2 us (1-16 tokens) and
  // 68.2 vs 74.4 us (32 tokens) against a ~200 KB ring, with the same bits;
  // the extra bytes in flight only queued behind the other SMs' requests.
  // (Two CTAs per SM -- this ring with registers capped so that the down
  // kernel's CTAs sit beside gate/up's from the start -- was slower still.)
  static constexpr int STAGES_FIT = (RING_KB * 1024 - USTAGE_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 4 ? 4 : STAGES_FIT;
  static constexpr int USTAGE_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFFSET = USTAGE_OFFSET + USTAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, acc_full[2], acc_empty[2], drain
  static constexpr int MISC_OFFSET = BAR_OFFSET + NUM_BARS * 8;
  static constexpr int TOTAL = MISC_OFFSET + 16;
  static constexpr int DYN_BYTES = TOTAL + 1024;
  // two accumulators, allocated as a power of two of at least 32 columns
  static constexpr int TMEM_COLS = 2 * NT <= 32 ? 32 : (2 * NT <= 64 ? 64 : (2 * NT <= 128 ? 128 : 256));
};

// Token rows the two-kernel form loads per k-block: M rounded up to the
// 8-row swizzle atom, at most NT.  The MMA still reads NT rows; rows past
// these hold whatever the ring slot held before, and only feed accumulator
// columns of tokens >= M, which no epilogue stores (a column depends on its
// own token row alone), so the stored outputs are the same bits.
__host__ __device__ inline int ng_x_rows(int NT, int M) {
  const int r = (M + 7) & ~7;
  return r < NT ? r : NT;
}

// Named barrier 1 over the 128 epilogue threads (warps 2..5).
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Stream-K partition: CTA c owns global k-blocks [ng_start(c), ng_start(c+1)).
__device__ __forceinline__ int64_t ng_start(int64_t c, int64_t total, int64_t ctas) {
  return c * total / ctas;
}

// This CTA's sequence of segments: its stream-K range first, then its whole
// tiles.
struct NgSegIter {
  int64_t x, x_end;   // stream-K k-block range still to cover
  int dp, dp_count;   // whole tiles taken / to take
  int kb_tile, sk_tiles, cta, ctas;
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& nkb, bool& whole) {
    if (x < x_end) {
      tile = (int)(x / kb_tile);
      kb0 = (int)(x - (int64_t)tile * kb_tile);
      nkb = (int)min((int64_t)(kb_tile - kb0), x_end - x);
      x += nkb;
      whole = false;
      return true;
    }
    if (dp < dp_count) {
      tile = sk_tiles + cta + dp * ctas;
      kb0 = 0;
      nkb = kb_tile;
      ++dp;
      whole = true;
      return true;
    }
    return false;
  }
};

// The CTA whose range holds global k-block x.
__device__ __forceinline__ int ng_owner(int64_t x, int64_t total, int64_t ctas) {
  int64_t c = x * ctas / total;
  while (c + 1 < ctas && ng_start(c + 1, total, ctas) <= x) ++c;
  while (c > 0 && ng_start(c, total, ctas) > x) --c;
  return (int)c;
}

// Same barrier, returning the AND of v over the 128 threads, so that every
// epilogue warp takes the same branch afterwards.
__device__ __forceinline__ int epi_bar_and(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}

// Epilogue building blocks, run by the 128 epilogue threads (warps 2..5;
// TMEM lane quarter = warp & 3, lane = weight row of the tile).  ``tacc`` is
// the accumulator's TMEM address (lane 0), ``acce`` the barrier that hands it
// back to the MMA warp.

// A whole tile's output straight from TMEM.  gate/up: rows 0..63 hold G and
// rows 64..127 U of the same 64 hidden units, met through ``ustage``.
template <int NT, bool GATE_UP, bool BF16>
__device__ __forceinline__ void ng_store_whole(const NgArgs& a, int tile, uint32_t tacc,
                                               uint32_t acce, float* ustage) {
  const int row = (threadIdx.x & 96) + (threadIdx.x & 31);  // (warp & 3) * 32 + lane
  tc_fence_after();
  const uint32_t taddr = tacc + ((uint32_t)(row & 96) << 16);
  float v[NT];
#pragma unroll
  for (int c = 0; c < NT; c += 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr + c, r);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 16; ++q) v[c + q] = __uint_as_float(r[q]);
  }
  tc_fence_before();
  mbar_arrive(acce);
  if (GATE_UP) {
    // rows 64..127 (U) hand their values to rows 0..63 (G) of the same unit
    if (row >= 64) {
#pragma unroll
      for (int n = 0; n < NT; n += 4)
        *reinterpret_cast<float4*>(ustage + (row - 64) * NT + n) =
            make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
    }
    epi_bar_sync();
    const int j = tile * 64 + row;
    if (row < 64 && j < a.rows) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (n < a.M) ng_put<BF16>(a, n, j, silu_f32(a.scale * v[n]) * ustage[row * NT + n]);
      }
    }
    epi_bar_sync();  // ustage is free again
  } else {
    const int d = tile * 128 + row;
    if (d < a.rows) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (n < a.M) ng_put<BF16>(a, n, d, a.scale * v[n]);
      }
    }
  }
}

// The accumulator as an fp32 partial tile [128][NT] at ``dst`` (the stores
// skipped when ``ok`` is false: a debug check failed).  Callers publish it
// with one release after a barrier over the 128 threads.
template <int NT>
__device__ __forceinline__ void ng_store_partial(float* dst, uint32_t tacc, uint32_t acce,
                                                 bool ok = true) {
  const int row = (threadIdx.x & 96) + (threadIdx.x & 31);
  tc_fence_after();
  float* drow = dst + (size_t)row * NT;
  const uint32_t taddr = tacc + ((uint32_t)(row & 96) << 16);
#pragma unroll
  for (int c = 0; c < NT; c += 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr + c, r);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (ok)
        reinterpret_cast<float4*>(drow + c)[q] =
            make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                        __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
  }
  tc_fence_before();
  mbar_arrive(acce);  // accumulator free for a later unit
}

// Sums the n partial tiles part_of(0), ..., part_of(n-1) in that order and
// writes the tile's output (gate/up: A = rnd(SiLU(g) * u); down: Y = rnd(y)).
template <int NT, bool GATE_UP, bool BF16, class PartOf>
__device__ __forceinline__ void ng_reduce_store(const NgArgs& a, int tile, int n, PartOf part_of) {
  // partials loaded per batch (the down tiles' per-thread share is half the
  // gate/up pair's)
  constexpr int RB = GATE_UP ? (NT <= 16 ? 4 : (NT <= 32 ? 2 : 1)) : (NT <= 16 ? 8 : (NT <= 32 ? 4 : 2));
  const int e = threadIdx.x - 64;  // 0..127 among the epilogue threads
  if (GATE_UP) {
    // thread e: hidden unit tile*64 + (e & 63), tokens [h*NT/2, (h+1)*NT/2)
    const int jr = e & 63, h = e >> 6;
    const int j = tile * 64 + jr;
    float g[NT / 2], uu[NT / 2];
#pragma unroll
    for (int q = 0; q < NT / 2; ++q) g[q] = uu[q] = 0.0f;
    for (int i0 = 0; i0 < n; i0 += RB) {
      // issue the loads of up to RB partials, then add them in order
      float4 vg[RB][NT / 8], vu[RB][NT / 8];
#pragma unroll
      for (int q = 0; q < RB; ++q)
        if (i0 + q < n) {
          const float* pb = part_of(i0 + q);
          const bool pok = SWIGLU_CHECK_PTR(a.dbg, pb, 128 * NT * 4, a.err);
#pragma unroll
          for (int k = 0; k < NT / 8; ++k) {
            vg[q][k] = pok ? __ldcg(reinterpret_cast<const float4*>(pb + jr * NT + h * (NT / 2)) + k)
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            vu[q][k] = pok ? __ldcg(reinterpret_cast<const float4*>(pb + (64 + jr) * NT + h * (NT / 2)) + k)
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          }
        }
#pragma unroll
      for (int q = 0; q < RB; ++q)
        if (i0 + q < n) {
#pragma unroll
          for (int k = 0; k < NT / 8; ++k) {
            g[4 * k] += vg[q][k].x; g[4 * k + 1] += vg[q][k].y;
            g[4 * k + 2] += vg[q][k].z; g[4 * k + 3] += vg[q][k].w;
            uu[4 * k] += vu[q][k].x; uu[4 * k + 1] += vu[q][k].y;
            uu[4 * k + 2] += vu[q][k].z; uu[4 * k + 3] += vu[q][k].w;
          }
        }
    }
    if (j < a.rows) {
#pragma unroll
      for (int q = 0; q < NT / 2; ++q) {
        const int m = h * (NT / 2) + q;
        if (m < a.M) ng_put<BF16>(a, m, j, silu_f32(a.scale * g[q]) * uu[q]);
      }
    }
  } else {
    // thread e: output feature tile*128 + e, all tokens
    const int d = tile * 128 + e;
    float y[NT];
#pragma unroll
    for (int q = 0; q < NT; ++q) y[q] = 0.0f;
    for (int i0 = 0; i0 < n; i0 += RB) {
      float4 v[RB][NT / 4];
#pragma unroll
      for (int q = 0; q < RB; ++q)
        if (i0 + q < n) {
          const float* pt = part_of(i0 + q);
          const bool pok = SWIGLU_CHECK_PTR(a.dbg, pt, 128 * NT * 4, a.err);
          const float* pb = pt + e * NT;
#pragma unroll
          for (int k = 0; k < NT / 4; ++k)
            v[q][k] = pok ? __ldcg(reinterpret_cast<const float4*>(pb) + k)
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
      for (int q = 0; q < RB; ++q)
        if (i0 + q < n) {
#pragma unroll
          for (int k = 0; k < NT / 4; ++k) {
            y[4 * k] += v[q][k].x; y[4 * k + 1] += v[q][k].y;
            y[4 * k + 2] += v[q][k].z; y[4 * k + 3] += v[q][k].w;
          }
        }
    }
    if (d < a.rows) {
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        if (q < a.M) ng_put<BF16>(a, q, d, a.scale * y[q]);
      }
    }
  }
}

// One segment's epilogue in the stream-K split: a whole tile's output from
// TMEM; else this CTA's partial to the workspace, and the tile's last
// contributor (per-tile arrival counter) sums the partials in CTA order and
// writes the output.  Returns true when this CTA wrote the tile's output.
template <int NT, bool GATE_UP, bool BF16>
__device__ __forceinline__ bool ng_epilogue_segment(const NgArgs& a, int tile, bool whole, int seg,
                                                    uint32_t tacc, uint32_t acce, int64_t total,
                                                    int64_t ctas, float* ustage,
                                                    volatile int* abort_flag,
                                                    volatile int* last_flag) {
  if (whole) {
    ng_store_whole<NT, GATE_UP, BF16>(a, tile, tacc, acce, ustage);
    return true;
  }
  float* const dst = a.part + ((size_t)blockIdx.x * a.seg_max + seg) * 128 * NT;
  ng_store_partial<NT>(dst, tacc, acce,
                       SWIGLU_CHECK(seg < a.seg_max, a.err) &&
                           SWIGLU_CHECK_PTR(a.dbg, dst, 128 * NT * 4, a.err));
  // CTAs sharing this tile: owners of its first and last k-block
  const int c_first = ng_owner((int64_t)tile * a.kb_tile, total, ctas);
  const int c_last = ng_owner((int64_t)(tile + 1) * a.kb_tile - 1, total, ctas);
  const int nparts = c_last - c_first + 1;
  const int e = threadIdx.x - 64;
  epi_bar_sync();
  if (e == 0) {
    int last = 0;
    __threadfence();  // the 128 threads' partial stores before the count
    if (!*abort_flag)
      last = SWIGLU_CHECK(tile < a.tiles, a.err) && atomicAdd(a.counters + tile, 1) == nparts - 1;
    *last_flag = last;
  }
  epi_bar_sync();
  const int last = *last_flag;
  if (last) {
    __threadfence();
    // partial of CTA c for this tile: its segment index is tile - (first tile of c)
    ng_reduce_store<NT, GATE_UP, BF16>(a, tile, nparts, [&](int i) -> const float* {
      const int c = c_first + i;
      const int j = tile - (int)(ng_start(c, total, ctas) / a.kb_tile);
      return SWIGLU_CHECK(j >= 0 && j < a.seg_max, a.err)
                 ? a.part + ((size_t)c * a.seg_max + j) * 128 * NT
                 : nullptr;
    });
    if (e == 0 && SWIGLU_CHECK(tile < a.tiles, a.err)) a.counters[tile] = 0;  // next call
  }
  return last != 0;
}

constexpr int NG_THREADS = 192;  // producer warp, MMA warp, 4 epilogue warps

template <int NT, bool GATE_UP, bool BF16, bool PACKED = false>
__global__ void __launch_bounds__(NG_THREADS, 1)
    ng_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const NgArgs a) {
  using L = NgSmem<NT>;
  static_assert(NT == 16 || NT == 32 || NT == 48 || NT == 64, "NT must be 16, 32, 48 or 64");
  static_assert(L::TOTAL + 1024 <= 232448, "shared memory plan exceeds 227 KB");
  constexpr int TILE_ROWS = GATE_UP ? 64 : 128;  // output rows (hidden units / features) per tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFFSET;
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (L::STAGES + i); };
  auto accf_bar = [&](int i) { return bar0 + 8u * (2 * L::STAGES + i); };
  auto acce_bar = [&](int i) { return bar0 + 8u * (2 * L::STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * L::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFFSET);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (blockIdx.x == 0 && a.clear_err && threadIdx.x == 0) *a.err = 0;
  if (!a.dependent) {
    if (blockIdx.x == 0 &&
        SWIGLU_CHECK_PTR(a.dbg, a.zero_ptr, 4 * (int64_t)a.zero_count, a.err))
      for (int i = threadIdx.x; i < a.zero_count; i += blockDim.x) a.zero_ptr[i] = 0;
    pdl_launch_dependents();  // the down kernel may begin its prologue
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (!PACKED) tma_prefetch_desc(&tmW);  // (with packed weights tmW is unused)
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int64_t total = (int64_t)a.sk_tiles * a.kb_tile;  // stream-K k-blocks
  const int64_t ctas = gridDim.x;
  const int64_t x_begin = ng_start(blockIdx.x, total, ctas);
  const int64_t x_end = ng_start(blockIdx.x + 1, total, ctas);
  const int dp_count = (a.tiles - a.sk_tiles) / gridDim.x;
  auto segs = [&]() {
    return NgSegIter{x_begin, x_end, 0, dp_count, a.kb_tile, a.sk_tiles, (int)blockIdx.x,
                     (int)gridDim.x};
  };

  // the weight box (tile, k-block kb) into the ring slot at ``slot``
  auto load_w = [&](uint32_t slot, uint32_t bar, int tile, int kb) {
    if (PACKED)
      bulk_load(slot, a.wpack + ((size_t)tile * a.kb_tile + kb) * L::W_BYTES, L::W_BYTES, bar);
    else if (GATE_UP)
      tma_load_3d(slot, &tmW, bar, kb * TC_BK, tile * TILE_ROWS, 0);
    else
      tma_load_2d(slot, &tmW, bar, kb * TC_BK, tile * TILE_ROWS);
  };

  // bytes per ring slot: the weight box and the token rows actually loaded
  const uint32_t stage_tx = L::W_BYTES + (uint32_t)ng_x_rows(NT, a.M) * 128u;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      // A dependent launch first fills the ring with weights only (they do not
      // depend on the previous kernel), then waits, then adds the activations.
      int pending_x = 0;  // ring slots holding weights whose activation load is deferred
      int32_t pending_k0[L::STAGES];
      if (a.dependent) {
        NgSegIter it = segs();
        int tile, kb0, nkb;
        bool whole;
        while (pending_x < L::STAGES && it.next(tile, kb0, nkb, whole)) {
          for (int i = 0; i < nkb && pending_x < L::STAGES; ++i) {
            const int k0 = (kb0 + i) * TC_BK;
            const uint32_t sw = sbase + pending_x * L::STAGE_BYTES;
            mbar_arrive_expect_tx(full_bar(pending_x), stage_tx);
            load_w(sw, full_bar(pending_x), tile, kb0 + i);
            pending_k0[pending_x] = k0;
            issued_mask |= 1u << pending_x;
            ++pending_x;
          }
        }
        pdl_wait();
        if (blockIdx.x == 0 &&
            SWIGLU_CHECK_PTR(a.dbg, a.zero_ptr, 4 * (int64_t)a.zero_count, a.err))
          for (int i = 0; i < a.zero_count; ++i) a.zero_ptr[i] = 0;
        for (int i = 0; i < pending_x; ++i)
          tma_load_2d(sbase + i * L::STAGE_BYTES + L::W_BYTES, &tmX, full_bar(i), pending_k0[i], 0);
      }
      int skip = pending_x;  // k-blocks already issued above
      NgSegIter it = segs();
      int tile, kb0, nkb;
      bool whole;
      while (ok && it.next(tile, kb0, nkb, whole)) {
        for (int i = 0; i < nkb; ++i) {
          if (skip > 0) {
            --skip;
            if (++stage == L::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, a.wait_limit_ns, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t sw = sbase + stage * L::STAGE_BYTES;
          const uint32_t sx = sw + L::W_BYTES;
          const int k0 = (kb0 + i) * TC_BK;
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          load_w(sw, full_bar(stage), tile, kb0 + i);
          tma_load_2d(sx, &tmX, full_bar(stage), k0, 0);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == L::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int i = 0; i < L::STAGES; ++i)
          if (issued_mask & (1u << i))
            mbar_wait_bounded(full_bar(i), (issued_parity >> i) & 1u, a.wait_limit_ns, nullptr,
                              a.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_f16(BF16, false, false, 128, NT);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      NgSegIter it = segs();
      int tile, kb0, nkb;
      bool whole;
      while (ok && it.next(tile, kb0, nkb, whole)) {
        if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, a.wait_limit_ns, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * NT;
        for (int i = 0; i < nkb; ++i) {
          if (!mbar_wait_bounded(full_bar(stage), phase, a.wait_limit_ns, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = sbase + stage * L::STAGE_BYTES;
          const uint32_t sx = sw + L::W_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / TC_UMMA_K; ++kk)
            umma_f16_ss(d_tmem, make_sw128_desc(sw + kk * 32, 16, 1024),
                        make_sw128_desc(sx + kk * 32, 16, 1024), idesc, (i | kk) != 0 ? 1u : 0u);
          umma_commit(empty_bar(stage));
          if (++stage == L::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, a.wait_limit_ns, nullptr, a.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    int acc = 0;
    uint32_t acc_phase = 0;
    int seg = 0;
    NgSegIter it = segs();
    int tile, kb0, nkb;
    bool whole;
    float* ustage = reinterpret_cast<float*>(smem + L::USTAGE_OFFSET);
    for (; it.next(tile, kb0, nkb, whole); ++seg) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(accf_bar(acc), acc_phase, a.wait_limit_ns, abort_flag, a.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!epi_bar_and(ok)) break;  // all four epilogue warps leave together
      ng_epilogue_segment<NT, GATE_UP, BF16>(a, tile, whole, seg, tmem_base + acc * NT,
                                             acce_bar(acc), total, ctas, ustage, abort_flag,
                                             last_flag);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace swiglu
