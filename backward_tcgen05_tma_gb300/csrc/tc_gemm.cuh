// tc_gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with
// the SwiGLU-MLP epilogues.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]      (fp32 accumulation in TMEM)
//
// Each operand is read from global memory by TMA into 128-byte-swizzled
// shared-memory tiles, either K-major (K contiguous in memory) or MN-major (M
// or N contiguous); the tensor core reads both layouts natively, so no
// operand of the MLP's six GEMMs is ever transposed in memory.
//
// CTA = 10 warps, one CTA per SM, persistent over output tiles:
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) k-blocks
//   warp 1      owns TMEM (allocates 2 x BN columns) and issues tcgen05.mma
//   warps 2..9  epilogue: TMEM -> registers -> fused elementwise -> global;
//               warps w and w + 4 share TMEM lane quarter (w % 4) and split
//               the tile's columns in two halves
// Two TMEM accumulators alternate between tiles, so the epilogue of tile i
// overlaps the main loop of tile i + 1.  Every wait is bounded (see
// mbar_wait_bounded); a stuck pipeline records an error and the CTA unwinds.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace swiglu {

constexpr int TC_BM = 128;       // tile rows (MMA M)
constexpr int TC_BK = 64;        // k-block: 64 16-bit elements = one 128-byte swizzle row
constexpr int TC_THREADS = 320;  // 10 warps
constexpr int TC_EPI_THREADS = 256;  // warps 2..9
constexpr int TC_UMMA_K = 16;    // K of one kind::f16 MMA

enum LoadMode : int {
  LOAD_KMAJOR = 0,   // operand rows are contiguous along K: one box {64, rows}
  LOAD_MNMAJOR = 1,  // operand is stored [K][MN]: boxes {64 MN, 64 K}, one per 64-wide chunk
  LOAD_GATEUP = 2    // Wgu viewed as [2][H][D]: one 3-D box {64, rows/2, 2} = Wg rows then Wu rows
};

struct TcShape {
  int M, N, K;           // GEMM problem (N counts hidden units for the gate/up GEMM)
  int m_tiles, n_tiles;  // output tiles
  int k_blocks;          // ceil(K / 64)
  int group_m;           // rasterisation: m tiles per group
  uint64_t wait_limit_ns;
  int* err;              // device error word (workspace)
  int inject_stall;      // test hook: producer skips stage 0 of its first tile
  // Stream-K hybrid (sk_tiles = 0: every tile whole, round-robin).  Tiles
  // [0, sk_tiles) of the raster order are shared: their k-blocks, laid end to
  // end, are split evenly over the CTAs, which stream their share first; the
  // remaining tiles are taken whole, round-robin.  A shared tile's segments
  // leave fp32 partial tiles in `part` (slot = CTA x segment); the last CTA to
  // finish a shared tile (counter) sums them in CTA order into its TMEM
  // accumulator and runs the epilogue.
  int sk_tiles;
  int seg_max;     // partial slots per CTA
  float* part;     // [gridDim.x * seg_max][128 * BN] fp32 in TMEM order
  int* counters;   // [sk_tiles], zero at launch; each reducer re-zeroes its own
#ifdef SWIGLU_DEBUG
  DbgWin dbg;      // buffers the epilogue may touch: its output(s) and the workspace
#endif
};

// Stream-K partition of `total` shared k-blocks: CTA c owns
// [sk_start(c), sk_start(c + 1)).
__device__ __forceinline__ int64_t sk_start(int64_t c, int64_t total, int64_t ctas) {
  return c * total / ctas;
}

// The CTA whose stream-K range holds shared k-block x.
__device__ __forceinline__ int sk_owner(int64_t x, int64_t total, int64_t ctas) {
  int64_t c = x * ctas / total;
  while (c + 1 < ctas && sk_start(c + 1, total, ctas) <= x) ++c;
  while (c > 0 && sk_start(c, total, ctas) > x) --c;
  return (int)c;
}

// One CTA's work: its stream-K range over the shared tiles, then its whole
// tiles (sk_tiles + blockIdx.x, + gridDim.x, ...).
struct TcSegIter {
  int64_t x, x_end;  // shared k-blocks still to cover
  int kb_tile;
  int t, tiles, step;
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& nkb, bool& whole) {
    if (x < x_end) {
      tile = (int)(x / kb_tile);
      kb0 = (int)(x - (int64_t)tile * kb_tile);
      nkb = (int)min((int64_t)(kb_tile - kb0), x_end - x);
      x += nkb;
      whole = false;
      return true;
    }
    if (t < tiles) {
      tile = t;
      kb0 = 0;
      nkb = kb_tile;
      t += step;
      whole = true;
      return true;
    }
    return false;
  }
};

// Named barrier 1 over the 256 epilogue threads; the AND form returns the
// same decision to every one of them.
__device__ __forceinline__ void tc_epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ int tc_epi_bar_and(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}

// Tile order: groups of group_m m-tiles, m fastest inside a group, so the CTAs
// running at one time share a few A row-blocks and B column-blocks in L2.
__device__ __forceinline__ void tc_tile_coords(int t, const TcShape& s, int& mt, int& nt) {
  const int per_group = s.group_m * s.n_tiles;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gm0 = g * s.group_m;
  const int gh = min(s.group_m, s.m_tiles - gm0);
  mt = gm0 + r % gh;
  nt = r / gh;
}

// ---------------------------------------------------------------------------
// Epilogues.  Each is called by the 256 epilogue threads of a CTA for one
// output tile; thread `row` (0..127) owns output row m0 + row and reads its
// TMEM lane, over column half `half` (0 or 1) of the tile.  `tacc` is the
// TMEM address of this warp's lane quarter at the accumulator's first column.
// ---------------------------------------------------------------------------
template <bool BF16>
struct Pack;
template <>
struct Pack<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ uint32_t two(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(h);
  }
};
template <>
struct Pack<false> {
  using T = __half;
  static __device__ __forceinline__ uint32_t two(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
};

// Coalesced store of one 32 x 32 tile of 16-bit values held row-per-thread
// (lane l owns row l: 16 packed words = 64 bytes).  The warp transposes it
// through a 2 KB shared buffer and then writes 8 rows x 64 contiguous bytes
// per instruction, so every 32-byte sector is written whole (row-per-thread
// 16-byte stores leave sectors half-written and cost read-modify-write
// traffic).  The buffer's 16-byte chunks are XOR-swizzled by (row / 2) % 4,
// which keeps both the row writes and the column reads free of bank
// conflicts.  row_ptr(r) is row r's destination for this chunk (or nullptr
// when the row is outside the matrix); chunk_ok(q) says whether 8-column
// group q lies inside it.
// Debug builds: row_ptr wrapped so that the bytes each row access touches
// (the 16-byte groups chunk_ok admits, a prefix of the row's 64) are checked
// against the launch's windows; a row that fails is skipped.  Release
// builds: row_ptr itself.
template <class RowPtr, class ChunkOk>
__device__ __forceinline__ auto checked_rows(const TcShape& s, RowPtr row_ptr, ChunkOk chunk_ok) {
#ifdef SWIGLU_DEBUG
  return [=, &s](int r) -> decltype(row_ptr(0)) {
    auto p = row_ptr(r);
    if (p == nullptr) return p;
    int nq = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) nq += chunk_ok(q) ? 1 : 0;
    return nq == 0 || SWIGLU_CHECK_PTR(s.dbg, p, nq * 16, s.err) ? p : nullptr;
  };
#else
  (void)s;
  (void)chunk_ok;
  return row_ptr;
#endif
}

template <class RowPtr, class ChunkOk>
__device__ __forceinline__ void warp_store_tile(uint8_t* buf, const uint32_t (&v)[16], int lane,
                                                RowPtr row_ptr, ChunkOk chunk_ok) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int pc = c ^ ((lane >> 1) & 3);
    *reinterpret_cast<uint4*>(buf + lane * 64 + pc * 16) =
        make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  }
  __syncwarp();
  const int q = lane & 3;
  const bool qok = chunk_ok(q);
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int r = pass * 8 + (lane >> 2);
    const int pc = q ^ ((r >> 1) & 3);
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 64 + pc * 16);
    uint8_t* dst = row_ptr(r);
    if (dst != nullptr && qok) *reinterpret_cast<uint4*>(dst + q * 16) = w;
  }
  __syncwarp();
}

// The inverse: a 32 x 32 tile of 16-bit values read with coalesced loads (8
// rows x 64 contiguous bytes per instruction) and handed to its rows' lanes
// through the same swizzled 2 KB buffer.  Split in two so the loads of the
// next tile can be in flight while the current one is used:
// warp_load_issue (global -> w, zero outside the matrix) and
// warp_load_finish (w -> the lane's own row, 16 packed words).
template <class RowPtr, class ChunkOk>
__device__ __forceinline__ void warp_load_issue(uint4 (&w)[4], int lane, RowPtr row_ptr,
                                                ChunkOk chunk_ok) {
  const int q = lane & 3;
  const bool qok = chunk_ok(q);
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const uint8_t* src = row_ptr(pass * 8 + (lane >> 2));
    w[pass] = (src != nullptr && qok) ? *reinterpret_cast<const uint4*>(src + q * 16)
                                      : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ void warp_load_finish(uint8_t* buf, const uint4 (&w)[4], int lane,
                                                 uint4 (&row)[4]) {
  const int q = lane & 3;
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int r = pass * 8 + (lane >> 2);
    *reinterpret_cast<uint4*>(buf + r * 64 + (q ^ ((r >> 1) & 3)) * 16) = w[pass];
  }
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c)
    row[c] = *reinterpret_cast<const uint4*>(buf + lane * 64 + (c ^ ((lane >> 1) & 3)) * 16);
  __syncwarp();
}

// e^x for x <= 0, from the identity e^x = 2^(x log2 e) on the
// special-function unit (ex2.approx.f32, without .ftz: subnormal results are
// kept, so e^x stays nonzero down to x = -103).
__device__ __forceinline__ float exp_nonpos_f32(float x) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x * 1.44269504088896341f));
  return r;
}

// sigma(g) = 1 / (1 + e^-g) in fp32, evaluated through t = e^-|g| in (0, 1],
// which never overflows: sigma = 1 / (1 + t) for g >= 0 and t / (1 + t) for
// g < 0.  (1 / (1 + e^-g) directly would give sigma = 0, SiLU = -0, from
// g = -88.8 on, where the fp32 values are still normal numbers.)  The
// reciprocal is the hardware's approximate one (rcp.approx.f32, about one
// fp32 ulp, far below the bf16/fp16 rounding that follows), measured 5%
// faster per training step than the correctly rounded one at D = 1024, where
// the SiLU epilogues dominate.  SiLU(g) = g * sigma(g).
__device__ __forceinline__ float sigmoid_f32(float g) {
  const float t = exp_nonpos_f32(-fabsf(g));
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(1.0f + t));
  return g >= 0.0f ? r : t * r;
}
__device__ __forceinline__ float silu_f32(float g) { return g * sigmoid_f32(g); }

// Plain store: C[m, n] = rnd(acc).
struct EpiStore {
  struct Params {
    void* out;
    int64_t ld;          // elements
    float scale;         // out = rnd(scale * acc) ...
    int accumulate;      // ... or, if nonzero, rnd(out + scale * acc) (one rounding)
  };
  template <int BN, bool BF16>
  static __device__ __forceinline__ void run(const Params& p, const TcShape& s, uint32_t tacc,
                                             int m0, int nt, int row, int half, uint8_t* buf) {
    using P = Pack<BF16>;
    using T = typename P::T;
    const int lane = row & 31;
    const int mw = m0 + (row & ~31);  // first row of this warp's 32
    const int n0 = nt * BN;
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      const int nc = n0 + c * 32;
      auto rows = [&](int rr) -> uint8_t* {
        const int m = mw + rr;
        return m < s.M ? reinterpret_cast<uint8_t*>(reinterpret_cast<T*>(p.out) +
                                                    (int64_t)m * p.ld + nc)
                       : nullptr;
      };
      auto ok = [&](int q) { return nc + q * 8 + 8 <= s.N; };
      const auto crows = checked_rows(s, rows, ok);
      uint4 old[4];
      if (p.accumulate) {
        uint4 w[4];
        warp_load_issue(w, lane, crows, ok);
        warp_load_finish(buf, w, lane, old);
      }
      uint32_t r[32];
      tmem_ld_32x32b_x32(tacc + c * 32, r);
      tmem_ld_wait();
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float a0 = p.scale * __uint_as_float(r[2 * i]);
        float a1 = p.scale * __uint_as_float(r[2 * i + 1]);
        if (p.accumulate) {
          const float2 o = P::unpack((&old[i >> 2].x)[i & 3]);
          a0 += o.x;
          a1 += o.y;
        }
        v[i] = P::two(a0, a1);
      }
      warp_store_tile(buf, v, lane, crows, ok);
    }
  }
};

// The forward elementwise stage for two adjacent hidden units, from the fp32
// accumulators acc_g = X Wg^T and acc_u = X Wu^T: with g = gate_mul acc_g,
// packed G = rnd(g), U = rnd(acc_u) and A = rnd(SiLU(g) acc_u), A formed from
// the unrounded values and rounded once.
// MUL = false: gate_mul is 1 and its multiply is left out (the same bits).
template <bool BF16, bool MUL = true>
__device__ __forceinline__ void swiglu_pair(float gate_mul, float acc_g0, float acc_g1,
                                            float acc_u0, float acc_u1, uint32_t& a,
                                            uint32_t& g, uint32_t& u) {
  using P = Pack<BF16>;
  const float g0 = MUL ? gate_mul * acc_g0 : acc_g0, g1 = MUL ? gate_mul * acc_g1 : acc_g1;
  a = P::two(silu_f32(g0) * acc_u0, silu_f32(g1) * acc_u1);
  g = P::two(g0, g1);
  u = P::two(acc_u0, acc_u1);
}

// Gate/up epilogue: accumulator columns [0, BN/2) hold X Wg^T for hidden
// units j0 .. j0 + BN/2 - 1 and [BN/2, BN) hold U for the same units.  With
// G = gate_mul * (X Wg^T) (1 for the standard MLP) it stores rnd(G), rnd(U)
// (training) and A = rnd(SiLU(G) * U) from the unrounded fp32 values.  With
// g == nullptr only A is written (no-grad).
struct EpiSwiGLU {
  struct Params {
    void* g;       // G base ([M, ld_gu]); U at u
    void* u;
    int64_t ld_gu;
    void* a;       // A base
    int64_t ld_a;
    float gate_mul;
  };
  template <int BN, bool BF16>
  static __device__ __forceinline__ void run(const Params& p, const TcShape& s, uint32_t tacc,
                                             int m0, int nt, int row, int half, uint8_t* buf) {
    using P = Pack<BF16>;
    using T = typename P::T;
    constexpr int HALF = BN / 2;
    const int lane = row & 31;
    const int mw = m0 + (row & ~31);
    const int j0 = nt * HALF;
    const bool keep_gu = p.g != nullptr;
#pragma unroll 1
    for (int c = half * (HALF / 64); c < (half + 1) * (HALF / 64); ++c) {
      uint32_t rg[32], ru[32];
      tmem_ld_32x32b_x32(tacc + c * 32, rg);
      tmem_ld_32x32b_x32(tacc + HALF + c * 32, ru);
      tmem_ld_wait();
      uint32_t va[16], vg[16], vu[16];
      if (p.gate_mul == 1.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          swiglu_pair<BF16, false>(p.gate_mul, __uint_as_float(rg[2 * i]),
                                   __uint_as_float(rg[2 * i + 1]), __uint_as_float(ru[2 * i]),
                                   __uint_as_float(ru[2 * i + 1]), va[i], vg[i], vu[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          swiglu_pair<BF16>(p.gate_mul, __uint_as_float(rg[2 * i]), __uint_as_float(rg[2 * i + 1]),
                            __uint_as_float(ru[2 * i]), __uint_as_float(ru[2 * i + 1]), va[i],
                            vg[i], vu[i]);
      }
      const int jc = j0 + c * 32;
      auto ok = [&](int q) { return jc + q * 8 + 8 <= s.N; };
      auto dst = [&](void* base, int64_t ld) {
        return [=](int rr) -> uint8_t* {
          const int m = mw + rr;
          return m < s.M ? reinterpret_cast<uint8_t*>(reinterpret_cast<T*>(base) + (int64_t)m * ld + jc)
                         : nullptr;
        };
      };
      warp_store_tile(buf, va, lane, checked_rows(s, dst(p.a, p.ld_a), ok), ok);
      if (keep_gu) {
        warp_store_tile(buf, vg, lane, checked_rows(s, dst(p.g, p.ld_gu), ok), ok);
        warp_store_tile(buf, vu, lane, checked_rows(s, dst(p.u, p.ld_gu), ok), ok);
      }
    }
  }
};

// Backward SwiGLU epilogue: the accumulator is dY Wd for hidden units
// j0 .. j0 + BN - 1; dA = down_mul * (dY Wd) is never stored.  Reads the
// stored G (= gate_mul X Wg^T), U, writes
//   dU = rnd(dA * SiLU(G)),  dG = rnd(dA * U * SiLU'(G) * gate_mul)
// over them in place, SiLU'(g) = s (1 + g (1 - s)), s = 1 / (1 + e^-g); dG
// is the gradient with respect to X Wg^T.
//
// G and U are read one 32-column chunk ahead.  DIRECT = false: coalesced
// (8 rows x 64 bytes per instruction) and transposed to each thread's row
// through the warp's shared-memory buffer; DIRECT = true: each thread loads
// its own row's 64 bytes straight into registers, which skips the transpose
// and its shared-memory traffic.  With a short contraction (K = D <= 2048)
// the epilogue bounds this GEMM and the direct form is 13% faster; with a
// long one the tensor core does and the staged form is 3% faster.
// dU = rnd(dA SiLU(g)), dG = rnd(dA u SiLU'(g) gate_mul) for 32 columns of
// one row: g, u packed in vg, vu (8 words of 2 each); r = the accumulator's
// 32 fp32 columns (dA = down_mul r).
template <bool BF16, bool MUL>
__device__ __forceinline__ void dswiglu_32_impl(const uint4 (&vg)[4], const uint4 (&vu)[4],
                                                const uint32_t (&r)[32], float gate_mul,
                                                float down_mul, uint32_t (&odg)[16],
                                                uint32_t (&odu)[16]) {
  using P = Pack<BF16>;
#pragma unroll
  for (int g8 = 0; g8 < 4; ++g8) {
    const uint32_t* pg = &vg[g8].x;
    const uint32_t* pu = &vu[g8].x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 g = P::unpack(pg[e]);
      const float2 u = P::unpack(pu[e]);
      float da0 = __uint_as_float(r[g8 * 8 + 2 * e]);
      float da1 = __uint_as_float(r[g8 * 8 + 2 * e + 1]);
      if constexpr (MUL) {
        da0 *= down_mul;
        da1 *= down_mul;
      }
      const float s0 = sigmoid_f32(g.x);
      const float s1 = sigmoid_f32(g.y);
      float ds0 = s0 * (1.0f + g.x * (1.0f - s0));
      float ds1 = s1 * (1.0f + g.y * (1.0f - s1));
      if constexpr (MUL) {
        ds0 *= gate_mul;
        ds1 *= gate_mul;
      }
      odu[g8 * 4 + e] = P::two(da0 * (g.x * s0), da1 * (g.y * s1));
      odg[g8 * 4 + e] = P::two(da0 * u.x * ds0, da1 * u.y * ds1);
    }
  }
}

// The standard MLP (both multipliers 1) takes a form without the two
// multiplies, the same bits: measured 3.5% faster for the dG/dU kernel at
// B=8 S=8192 D=4096 H=11008, and it leaves that kernel's registers unspilled.
template <bool BF16>
__device__ __forceinline__ void dswiglu_32(const uint4 (&vg)[4], const uint4 (&vu)[4],
                                           const uint32_t (&r)[32], float gate_mul,
                                           float down_mul, uint32_t (&odg)[16],
                                           uint32_t (&odu)[16]) {
  if (gate_mul == 1.0f && down_mul == 1.0f)
    dswiglu_32_impl<BF16, false>(vg, vu, r, gate_mul, down_mul, odg, odu);
  else
    dswiglu_32_impl<BF16, true>(vg, vu, r, gate_mul, down_mul, odg, odu);
}

struct EpiDSwiGLUParams {
  void* g;  // G (becomes dG); U (becomes dU) at u
  void* u;
  int64_t ld;
  float gate_mul, down_mul;
};

template <bool DIRECT>
struct EpiDSwiGLUT {
  using Params = EpiDSwiGLUParams;
  template <int BN, bool BF16>
  static __device__ __forceinline__ void run(const Params& p, const TcShape& s, uint32_t tacc,
                                             int m0, int nt, int row, int half, uint8_t* buf) {
    using P = Pack<BF16>;
    using T = typename P::T;
    const int lane = row & 31;
    const int mw = m0 + (row & ~31);
    const int jt = nt * BN;
    constexpr int CH = BN / 64;  // chunks of 32 columns per half
    const int c0 = half * CH;
    auto rows_of = [&](void* base, int jc) {
      return [=](int rr) -> uint8_t* {
        const int mm = mw + rr;
        return mm < s.M ? reinterpret_cast<uint8_t*>(reinterpret_cast<T*>(base) +
                                                     (int64_t)mm * p.ld + jc)
                        : nullptr;
      };
    };
    // G and U of the next chunk are loaded while this one is used
    uint4 wg[4], wu[4];
    const int mrow = mw + lane;
    auto load_row = [&](uint4 (&w)[4], void* base, int jc) {  // DIRECT: this thread's row
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(base) +
                                                        (int64_t)mrow * p.ld + jc);
      const int ncols = min(32, s.N - jc);  // columns of this chunk inside the matrix
      const bool row_ok =
          mrow < s.M && (ncols <= 0 || SWIGLU_CHECK_PTR(s.dbg, src, 2 * (int64_t)ncols, s.err));
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = (row_ok && jc + q * 8 + 8 <= s.N) ? src[q] : make_uint4(0, 0, 0, 0);
    };
    if constexpr (DIRECT) {
      load_row(wg, p.g, jt + c0 * 32);
      load_row(wu, p.u, jt + c0 * 32);
    } else {
      const int jc = jt + c0 * 32;
      auto ok = [&](int q) { return jc + q * 8 + 8 <= s.N; };
      warp_load_issue(wg, lane, checked_rows(s, rows_of(p.g, jc), ok), ok);
      warp_load_issue(wu, lane, checked_rows(s, rows_of(p.u, jc), ok), ok);
    }
#pragma unroll 1
    for (int c = c0; c < c0 + CH; ++c) {
      uint4 vg[4], vu[4];
      if constexpr (DIRECT) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          vg[q] = wg[q];
          vu[q] = wu[q];
        }
        if (c + 1 < c0 + CH) {
          load_row(wg, p.g, jt + (c + 1) * 32);
          load_row(wu, p.u, jt + (c + 1) * 32);
        }
      } else {
        warp_load_finish(buf, wg, lane, vg);
        warp_load_finish(buf, wu, lane, vu);
        if (c + 1 < c0 + CH) {
          const int jn = jt + (c + 1) * 32;
          auto okn = [&](int q) { return jn + q * 8 + 8 <= s.N; };
          warp_load_issue(wg, lane, checked_rows(s, rows_of(p.g, jn), okn), okn);
          warp_load_issue(wu, lane, checked_rows(s, rows_of(p.u, jn), okn), okn);
        }
      }
      uint32_t r[32];
      tmem_ld_32x32b_x32(tacc + c * 32, r);
      tmem_ld_wait();
      uint32_t odg[16], odu[16];
      dswiglu_32<BF16>(vg, vu, r, p.gate_mul, p.down_mul, odg, odu);
      const int jc = jt + c * 32;
      auto ok = [&](int q) { return jc + q * 8 + 8 <= s.N; };
      warp_store_tile(buf, odg, lane, checked_rows(s, rows_of(p.g, jc), ok), ok);
      warp_store_tile(buf, odu, lane, checked_rows(s, rows_of(p.u, jc), ok), ok);
    }
  }
};

using EpiDSwiGLU = EpiDSwiGLUT<false>;

// ---------------------------------------------------------------------------
// Shared-memory plan
// ---------------------------------------------------------------------------
template <int BN, int STAGES>
struct TcSmem {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * TC_BK * 2;     // 32 KB for BN = 256
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES + 8 * 2048;
  // barriers: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;         // 8 warps x 2 KB store staging
  static constexpr int EPI_BYTES = 8 * 2048;
  static constexpr int MISC_OFFSET = BAR_OFFSET + NUM_BARS * 8;  // tmem slot, abort flag
  static constexpr int TOTAL = MISC_OFFSET + 16;
  static constexpr int DYN_BYTES = TOTAL + 1024;  // slack for 1024-byte alignment
  static constexpr int TMEM_COLS = 2 * BN;        // power of two for BN in {128, 256}
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int BN, int STAGES, int A_MODE, int B_MODE, bool BF16, class Epi>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcShape s, const typename Epi::Params ep) {
  using L = TcSmem<BN, STAGES>;
  static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
  static_assert(L::TOTAL + 1024 <= 232448, "shared memory plan exceeds 227 KB");

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: the 128-byte swizzle pattern repeats every 1024 bytes
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), TC_EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = s.m_tiles * s.n_tiles;
  const int64_t sk_total = (int64_t)s.sk_tiles * s.k_blocks;  // shared k-blocks
  const int64_t ctas = gridDim.x;
  auto segs = [&]() {
    return TcSegIter{sk_start(blockIdx.x, sk_total, ctas), sk_start(blockIdx.x + 1, sk_total, ctas),
                     s.k_blocks, s.sk_tiles + (int)blockIdx.x, num_tiles, (int)gridDim.x};
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // last load per stage
      bool ok = true;
      bool skip_once = s.inject_stall != 0;
      TcSegIter it = segs();
      int tile, kb0, nkb;
      bool whole;
      while (ok && it.next(tile, kb0, nkb, whole)) {
        int mt, nt;
        tc_tile_coords(tile, s, mt, nt);
        const int m0 = mt * TC_BM;
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
            const int k0 = kb * TC_BK;
            mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
            if (A_MODE == LOAD_KMAJOR) {
              tma_load_2d(sa, &tmA, full_bar(stage), k0, m0);
            } else {
#pragma unroll
              for (int c = 0; c < TC_BM / 64; ++c)
                tma_load_2d(sa + c * 8192, &tmA, full_bar(stage), m0 + 64 * c, k0);
            }
            if (B_MODE == LOAD_KMAJOR) {
              tma_load_2d(sb, &tmB, full_bar(stage), k0, nt * BN);
            } else if (B_MODE == LOAD_GATEUP) {
              tma_load_3d(sb, &tmB, full_bar(stage), k0, nt * (BN / 2), 0);
            } else {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(sb + c * 8192, &tmB, full_bar(stage), nt * BN + 64 * c, k0);
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
      if (!ok) {
        // unwinding: let the copies already issued land before the CTA exits
        for (int i = 0; i < STAGES; ++i)
          if (issued_mask & (1u << i))
            mbar_wait_bounded(full_bar(i), (issued_parity >> i) & 1u, s.wait_limit_ns, nullptr,
                              s.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc =
          make_idesc_f16(BF16, A_MODE == LOAD_MNMAJOR, B_MODE == LOAD_MNMAJOR, TC_BM, BN);
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
            const uint64_t bd = (B_MODE == LOAD_MNMAJOR)
                                    ? make_sw128_desc(sb + kk * 2048, 8192, 1024)
                                    : make_sw128_desc(sb + kk * 32, 16, 1024);
            umma_f16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(acc));  // accumulator complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // drain: every MMA this thread issued has completed before TMEM is freed
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, s.wait_limit_ns, nullptr, s.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // column half of the tile
    const int row = quarter * 32 + lane;
    const int e = threadIdx.x - 64;  // 0..255 among the epilogue threads
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 8);
    constexpr int CH = BN / 64;      // 32-column chunks per half
    int acc = 0;
    uint32_t acc_phase = 0;
    int seg = 0;  // shared segments done (= partial slot index)
    TcSegIter it = segs();
    int tile, kb0, nkb;
    bool whole;
    while (it.next(tile, kb0, nkb, whole)) {
      // one lane per warp waits; all eight warps then take the same branch
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(accf_bar(acc), acc_phase, s.wait_limit_ns, abort_flag, s.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!tc_epi_bar_and(ok)) break;
      tc_fence_after();
      int mt, nt;
      tc_tile_coords(tile, s, mt, nt);
      const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      int run_epi = whole ? 1 : 0;
      if (!whole) {
        // partial tile -> this CTA's slot, in TMEM order (coalesced: lanes
        // of a warp write consecutive 16-byte groups)
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
        const int c_first = sk_owner((int64_t)tile * s.k_blocks, sk_total, ctas);
        const int c_last = sk_owner((int64_t)(tile + 1) * s.k_blocks - 1, sk_total, ctas);
        tc_epi_bar();
        if (e == 0) {
          int last = 0;
          if (!*abort_flag)
            last = SWIGLU_CHECK(tile < s.sk_tiles, s.err) &&
                   atomicAdd(s.counters + tile, 1) == c_last - c_first;
          *last_flag = last;
        }
        tc_epi_bar();
        run_epi = *last_flag;
        if (run_epi) {
          // the last CTA: sum every partial of the tile in CTA order (its own
          // straight from TMEM) and put the sum back into its accumulator
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
              if (pc == (int)blockIdx.x) {
#pragma unroll
                for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(own[i]);
              } else {
                const int j = tile - (int)(sk_start(pc, sk_total, ctas) / s.k_blocks);
                const float4* ps = reinterpret_cast<const float4*>(
                    s.part + ((size_t)pc * s.seg_max + j) * (size_t)(TC_BM * BN));
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
          if (e == 0 && SWIGLU_CHECK(tile < s.sk_tiles, s.err)) s.counters[tile] = 0;
          // the epilogue may read columns that another thread summed
          tc_fence_before();
          tc_epi_bar();
          tc_fence_after();
        }
      }
      if (run_epi)
        Epi::template run<BN, BF16>(ep, s, tacc, mt * TC_BM, nt, row, half,
                                    smem + L::EPI_OFFSET + (warp - 2) * 2048);
      tc_fence_before();
      mbar_arrive(acce_bar(acc));
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
