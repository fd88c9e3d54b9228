// swiglu_mlp.cu -- C ABI of the fused SwiGLU MLP (include/swiglu_mlp.h):
// argument validation, TMA tensor-map encoding and kernel launches.
//
// Forward ("[RFC] Full-pipeline SwiGLU MLP with forward/backward
// co-optimization", Liger-Kernel #1347, "Summary"):
//   gate/up   [G | U | A] = X [Wg; Wu]^T with the SwiGLU epilogue
//   down      Y = A Wd^T
// Backward:
//   dGU       dA = dY Wd in TMEM only; epilogue writes dG, dU over G, U
//   dWd       dWd = dY^T A
//   dWgu      [dWg; dWu] = [dG | dU]^T X            (one GEMM)
//   dX        dX = [dG | dU] [Wg; Wu], K = 2H       (one accumulator)
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/swiglu_mlp.h"
#include "ng_fused.cuh"
#include "ng_gemm.cuh"
#include "simt_gemm.cuh"
#include "tc2_gemm.cuh"
#include "tc_gemm.cuh"

using namespace swiglu;

namespace {

constexpr size_t WS_HEADER = 256;  // error word + reserved
constexpr int TC_STAGES = 4;
constexpr int TC_BN = 256;

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

swiglu_status cuda_status(cudaError_t e);

// Debug builds (SWIGLU_DEBUG): the buffers (base, bytes) a launch may touch
// with plain loads and stores, its output first; the kernels check every
// such access against them.  Release builds carry no windows.
using Win = std::pair<const void*, size_t>;

// Test hook (swiglu_mlp_debug_narrow_once): halve the next launch's first
// window, its output buffer.
std::atomic<int> g_narrow_once{0};

#ifdef SWIGLU_DEBUG
DbgWin make_windows(std::initializer_list<Win> wins) {
  DbgWin w = {};
  int i = 0;
  for (const Win& b : wins) {
    if (i == DBG_WINS) break;
    w.lo[i] = reinterpret_cast<uint64_t>(b.first);
    w.hi[i] = w.lo[i] + b.second;
    ++i;
  }
  if (g_narrow_once.exchange(0)) w.hi[0] = w.lo[0] + (w.hi[0] - w.lo[0]) / 2;
  return w;
}
#endif

template <class T>
void set_windows(T& args, std::initializer_list<Win> wins) {
#ifdef SWIGLU_DEBUG
  args.dbg = make_windows(wins);
#else
  (void)args;
  (void)wins;
#endif
}

SimtCheck simt_check(int* err, std::initializer_list<Win> wins) {
  SimtCheck c;
#ifdef SWIGLU_DEBUG
  c.err = err;
  c.win = make_windows(wins);
#else
  (void)err;
  (void)wins;
#endif
  return c;
}

// The multiplier / accumulation options of the _ex entry points (see the
// header); {1, 1, 0} is the standard MLP with gradients overwritten.
struct Opts {
  float gm = 1.0f, dm = 1.0f;
  int acc = 0;
};
std::atomic<int> g_inject_stall{0};  // launches until the injected stall (0: none)

// The stall-injection countdown (swiglu_mlp_inject_stall_once): true for the
// one launch it reaches.
bool take_inject() {
  int v = g_inject_stall.load();
  while (v > 0 && !g_inject_stall.compare_exchange_weak(v, v - 1)) {
  }
  return v == 1;
}
std::atomic<int> g_last_launches{0};
std::atomic<int> g_cta_pairs{1};  // SM pairs (cta_group::2): 0 never, 1 by size, 2 always
std::atomic<int> g_wide_tiles{1};  // 512-column pair tiles for dWd, dWgu, dX: 0 never, 1 by size, 2 always
std::atomic<int> g_ng_fused{0};   // few-token no-grad: fused kernel 0 never, 1 for 33..64 tokens, 2 always
constexpr int TC2_STAGES = 6;

// ---------------------------------------------------------------------------
// optional per-kernel timing: CUDA events bracket each launch on its stream
// ---------------------------------------------------------------------------
enum KernelId : int {
  K_GATE_UP = 0, K_DOWN, K_DGU, K_DWD, K_DWGU, K_DX, K_GATE_UP_NOGRAD, K_DOWN_NOGRAD,
  K_SIMT_GATE_UP, K_SIMT_DOWN, K_SIMT_DGU, K_SIMT_DWD, K_SIMT_DWGU, K_SIMT_DX, K_NG_GATE_UP,
  K_NG_DOWN, K_NG_FUSED, K_COUNT
};
const char* const kKernelNames[K_COUNT] = {
    "gate_up_swiglu", "down_proj", "dgu_inplace", "dwd", "dwgu", "dx", "gate_up_nograd",
    "down_proj_nograd", "simt_gate_up_swiglu", "simt_down_proj", "simt_dgu_inplace", "simt_dwd",
    "simt_dwgu", "simt_dx", "nograd_small_gate_up", "nograd_small_down", "nograd_small_fused"};

struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<int> g_prof_on{0};
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;
double g_prof_ms[K_COUNT];
int64_t g_prof_n[K_COUNT];

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one launch with events when timing is enabled.
struct ProfScope {
  int id;
  cudaStream_t st;
  cudaEvent_t b = nullptr;
  ProfScope(int id_, cudaStream_t st_) : id(id_), st(st_) {
    if (!g_prof_on.load()) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    cudaEvent_t a = prof_event();
    b = prof_event();
    cudaEventRecord(a, st);
    g_prof_pending.push_back(ProfRec{id, a, b});
  }
  ~ProfScope() {
    if (b != nullptr) cudaEventRecord(b, st);
  }
};

// ---------------------------------------------------------------------------
// driver entry point for tensor-map encoding (no link-time libcuda dependency)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// 2-D tiled map over a row-major matrix [outer][inner] (inner contiguous) with
// a row stride in bytes; 128-byte swizzle unless given; out-of-range elements
// read as 0 (and are not written by a store).
bool encode_2d(CUtensorMap* tm, bool bf16, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Wgu [2H][D] seen as [2][H][D]: one box brings rows j0.. of Wg and of Wu
// (depth 2), or of one of them (depth 1: the two CTAs of a pair each bring one).
bool encode_gateup(CUtensorMap* tm, bool bf16, const void* Wgu, uint64_t D, uint64_t H,
                   uint32_t rows, uint32_t depth = 2) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {D, H, 2};
  cuuint64_t strides[2] = {D * 2, H * D * 2};
  cuuint32_t box[3] = {64, rows, depth};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(Wgu), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K-major operand: rows of K elements, box {64, rows_per_tile}.
bool map_kmajor(CUtensorMap* tm, bool bf16, const void* base, int64_t K, int64_t rows, int64_t ld,
                uint32_t box_rows) {
  return encode_2d(tm, bf16, base, (uint64_t)K, (uint64_t)rows, (uint64_t)ld * 2, 64, box_rows);
}

// MN-major operand stored [K][MN]: boxes {64 MN, 64 K}.
bool map_mnmajor(CUtensorMap* tm, bool bf16, const void* base, int64_t MN, int64_t K, int64_t ld) {
  return encode_2d(tm, bf16, base, (uint64_t)MN, (uint64_t)K, (uint64_t)ld * 2, 64, 64);
}

// ---------------------------------------------------------------------------
// stream-K hybrid for the tensor-core kernels
// ---------------------------------------------------------------------------
// Workspace of a training call: [0, 256) header (error word), then the
// shared-tile counters, then the fp32 partial tiles.
constexpr size_t TC_SK_COUNTER_BYTES = 1024;  // up to 256 shared tiles
constexpr int TC_SK_MAX_SMS = 256;

struct TcPlan {
  int grid, sk_tiles, seg_max;
};

// Whole tiles round-robin, unless the last round would leave more than 3% of
// the SMs' time idle: then the (tiles mod SMs) tiles of that round (all of
// them when there are fewer tiles than SMs) are shared stream-K style.  A
// CTA's shared range is at most one tile long, so it meets at most two tiles.
TcPlan tc_plan(int64_t tiles, int64_t kb, int nsm) {
  TcPlan p{(int)(tiles < nsm ? tiles : nsm), 0, 1};
  const int64_t waves = (tiles + nsm - 1) / nsm;
  const double fill = (double)tiles / ((double)waves * nsm);
  if (fill >= 0.97 || kb < 8) return p;
  p.sk_tiles = (int)(tiles >= nsm ? tiles % nsm : tiles);
  const int64_t total = (int64_t)p.sk_tiles * kb;
  p.grid = nsm;
  if (tiles < nsm && total < nsm) p.grid = (int)total;
  const int64_t range = (total + p.grid - 1) / p.grid;
  p.seg_max = (int)((range + kb - 1) / kb) + 1;
  return p;
}

// Bytes of the workspace that must be zero when a training call starts: the
// error word, and the shared-tile counters of the tensor-core kernels.
size_t ws_clear_bytes(swiglu_dtype dt) {
  return dt == SWIGLU_F32_IEEE ? sizeof(int) : WS_HEADER + TC_SK_COUNTER_BYTES;
}

// Workspace bytes left for stream-K partial tiles after the header and the
// tile counters.
size_t part_capacity(size_t ws_bytes) {
  const size_t fixed = WS_HEADER + TC_SK_COUNTER_BYTES;
  return ws_bytes > fixed ? ws_bytes - fixed : 0;
}

size_t tc_part_bytes(const TcPlan& p, int64_t bn = TC_BN) {
  return p.sk_tiles ? (size_t)p.grid * p.seg_max * TC_BM * bn * 4 : 0;
}

// 512-column pair tiles for the weight-gradient and dX GEMMs (use_wide)
constexpr int TC2_WIDE_BN = 512;
constexpr int64_t TC2_WIDE_MIN_K = 16384;

int tc_nsm() {
  const int n = sm_count();
  return n < 1 ? 1 : (n > TC_SK_MAX_SMS ? TC_SK_MAX_SMS : n);
}

// Pairs of SMs that can hold a pair kernel's cluster at once (each TPC
// whose two SMs are both usable), queried once per device.
int tc2_units() {
  static std::mutex mu;
  static int cached[64];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> g(mu);
  if (!done[dev]) {
    int n = 0;
    auto kern = tc2_gemm_kernel<TC2_STAGES, LOAD_KMAJOR, LOAD_KMAJOR, true, EpiStore>;
    constexpr int smem = Tc2Smem<TC2_STAGES>::DYN_BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    const int cap = tc_nsm() / 2;
    cached[dev] = n < cap ? n : cap;
    done[dev] = true;
  }
  return cached[dev];
}

// 512-column pair tiles (one accumulator, no epilogue overlap) for an
// M x N GEMM over K: by size, where the main loop dwarfs a tile's epilogue
// (K >= 16384) and every pair gets at least two whole tiles.  Measured at
// B=8 S=8192 D=4096 H=11008: dWd 3.74 -> 3.61, dWgu 7.46 -> 6.96, dX 7.17
// -> 6.88 ms; at S=4096 D=2048 H=5632 dWgu 0.975 -> 0.897 ms, while dX
// (K = 11264) and dWd (88 tiles for 76 pairs) were slower, which the rule
// leaves on 256-column tiles.
bool use_wide(bool pairs, int64_t M, int64_t N, int64_t K) {
  const int mode = g_wide_tiles.load();
  if (!pairs || mode == 0) return false;
  if (mode == 2) return true;
  const int64_t tiles = ((M + TC2_BM - 1) / TC2_BM) * ((N + TC2_WIDE_BN - 1) / TC2_WIDE_BN);
  return K >= TC2_WIDE_MIN_K && tiles >= 2 * (int64_t)tc2_units();
}

// Whether one GEMM runs on SM pairs.  Measured per kernel on GB300: pairs
// win when the main loop dominates -- long K and several rounds of tiles, or
// the very long K of the weight gradients -- while short-K GEMMs with heavy
// epilogues or few tiles run faster on single SMs (the pair's fixed costs and
// its coupled epilogues are not amortised).
bool use_pairs(int64_t Mg, int64_t N, int64_t n_per_tile, int64_t K) {
  const int mode = g_cta_pairs.load();
  if (mode == 0 || tc2_units() < 1) return false;
  if (mode == 2) return true;
  // pairs once every pair gets at least one of their 256-row tiles and the
  // 256-row tiles add no padding beyond the 128-row ones; measured per GEMM
  // at B=8, S=2048-8192 (D = 1024-4096): as fast or faster on pairs for
  // every GEMM there, including the short contractions (gate/up and dX at
  // D = 1024: 0.151 vs 0.171 and 0.126 vs 0.143 ms); no-grad calls with
  // 65-128 or 384 tokens, whose pair tiles would be partly empty, are 3% and
  // 11% faster on single SMs
  const int64_t pair_tiles = ((Mg + TC2_BM - 1) / TC2_BM) * ((N + n_per_tile - 1) / n_per_tile);
  const bool no_pad = (Mg + TC2_BM - 1) / TC2_BM * TC2_BM == (Mg + TC_BM - 1) / TC_BM * TC_BM;
  const int64_t kb = (K + TC_BK - 1) / TC_BK;
  return (kb >= 16 && no_pad && pair_tiles >= (int64_t)tc2_units()) || kb >= 256;
}

// pairs: tiles of 256 rows handed out per CTA pair (tc2_gemm_kernel).
// Partial-tile bytes a training call needs: its tensor-core GEMMs as
// (GEMM rows, GEMM columns, columns per tile, K).  Without a device the bound
// for any GPU of up to 256 SMs (two slots per CTA).
size_t tc_ws_part_bytes(int64_t M, int64_t D, int64_t H, int op) {
  if (sm_count() < 1) return (size_t)2 * TC_SK_MAX_SMS * TC_BM * TC2_WIDE_BN * 4;
  const int nsm = tc_nsm();
  const int64_t fwd[2][4] = {{M, H, TC_BN / 2, D}, {M, D, TC_BN, H}};
  const int64_t bwd[4][4] = {{D, H, TC_BN, M}, {M, H, TC_BN, D}, {2 * H, D, TC_BN, M},
                             {M, D, TC_BN, 2 * H}};
  size_t best = 0;
  const int n = op == SWIGLU_OP_BWD ? 4 : 2;
  for (int i = 0; i < n; ++i) {
    const int64_t* g = op == SWIGLU_OP_BWD ? bwd[i] : fwd[i];
    const int64_t kb = (g[3] + TC_BK - 1) / TC_BK, nt = (g[1] + g[2] - 1) / g[2];
    // one SM per CTA, or pairs of SMs (two CTAs, so two slots sets per unit)
    const size_t b1 = tc_part_bytes(tc_plan(((g[0] + TC_BM - 1) / TC_BM) * nt, kb, nsm));
    const int units = tc2_units();  // the pair kernel plans with the same count
    const size_t b2 =
        units >= 1 ? 2 * tc_part_bytes(tc_plan(((g[0] + TC2_BM - 1) / TC2_BM) * nt, kb, units)) : 0;
    if (b1 > best) best = b1;
    if (b2 > best) best = b2;
    if (units >= 1 && (op == SWIGLU_OP_BWD ? i != 1 : i == 1)) {
      // the same GEMM on 512-column pair tiles (dWd, dWgu, dX; the down projection)
      const int64_t ntw = (g[1] + TC2_WIDE_BN - 1) / TC2_WIDE_BN;
      const size_t bw = 2 * tc_part_bytes(tc_plan(((g[0] + TC2_BM - 1) / TC2_BM) * ntw, kb, units),
                                          TC2_WIDE_BN);
      if (bw > best) best = bw;
    }
  }
  return best;
}

// part_cap: workspace bytes available for stream-K partial tiles; a GEMM
// whose plan needs more runs whole tiles only (same results within
// rounding, without the last round's balancing).
TcShape make_shape(int64_t M, int64_t N, int64_t K, int64_t n_per_tile, int* err, bool pairs,
                   size_t part_cap) {
  TcShape s;
  s.M = (int)M;
  s.N = (int)N;
  s.K = (int)K;
  const int64_t bm = pairs ? TC2_BM : TC_BM;
  s.m_tiles = (int)((M + bm - 1) / bm);
  s.n_tiles = (int)((N + n_per_tile - 1) / n_per_tile);
  s.k_blocks = (int)((K + TC_BK - 1) / TC_BK);
  s.group_m = 16;
  s.wait_limit_ns = g_wait_limit_ns.load();
  s.err = err;
  s.inject_stall = take_inject() ? 1 : 0;
  // the workspace (whose first word is err) carries the stream-K scratch
  const TcPlan p = tc_plan((int64_t)s.m_tiles * s.n_tiles, s.k_blocks,
                           pairs ? tc2_units() : tc_nsm());
  s.sk_tiles = p.sk_tiles;
  s.seg_max = p.seg_max;
  if (tc_part_bytes(p, n_per_tile) * (pairs ? 2 : 1) > part_cap) {
    s.sk_tiles = 0;
    s.seg_max = 1;
  }
  s.counters = reinterpret_cast<int*>(reinterpret_cast<char*>(err) + WS_HEADER);
  s.part = reinterpret_cast<float*>(reinterpret_cast<char*>(err) + WS_HEADER + TC_SK_COUNTER_BYTES);
  return s;
}

// CTAs (or pairs) to launch: the stream-K plan's grid, or one per tile up to
// `units` when the GEMM runs whole tiles only.
int launch_units(const TcShape& s, int units) {
  const int64_t tiles = (int64_t)s.m_tiles * s.n_tiles;
  if (s.sk_tiles) return tc_plan(tiles, s.k_blocks, units).grid;
  return (int)(tiles < units ? tiles : units);
}

// The training kernels are launched in plain stream order: with a static
// round-robin tile split, a programmatic dependent whose CTAs start late on
// SMs still held by the predecessor's last wave also finishes late (measured
// slower than plain order).
template <int AM, int BMODE, bool BF16, class Epi>
cudaError_t launch_tc(int kid, const CUtensorMap& ta, const CUtensorMap& tb, const TcShape& s,
                      const typename Epi::Params& ep, cudaStream_t st) {
  auto kern = tc_gemm_kernel<TC_BN, TC_STAGES, AM, BMODE, BF16, Epi>;
  constexpr int smem = TcSmem<TC_BN, TC_STAGES>::DYN_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = launch_units(s, tc_nsm());
  ProfScope prof(kid, st);
  kern<<<grid, TC_THREADS, smem, st>>>(ta, tb, s, ep);
  g_last_launches.fetch_add(1);
  return cudaGetLastError();
}

// The pair kernel: clusters of two CTAs on the two SMs of a TPC.
// tg, tu: the TMA dG/dU epilogue's maps of G and U (other epilogues: unused)
template <int AM, int BMODE, bool BF16, class Epi, int BN = TC2_BN>
cudaError_t launch_tc2(int kid, const CUtensorMap& ta, const CUtensorMap& tb, const TcShape& s,
                       const typename Epi::Params& ep, cudaStream_t st,
                       const CUtensorMap* tg = nullptr, const CUtensorMap* tu = nullptr) {
  // the TMA dG/dU epilogue's slots (GU_SLOTS x 4 KB per epilogue warp) take
  // the room of GU_SLOTS - 1 ring stages; 512-column tiles (48 KB stages)
  // keep four
  constexpr bool gu = epi_tma_gu<Epi>::value;
  constexpr int stages = BN > 256 ? 4 : (gu ? TC2_STAGES + 1 - GU_SLOTS : TC2_STAGES);
  auto kern = tc2_gemm_kernel<stages, AM, BMODE, BF16, Epi, BN>;
  constexpr int smem = Tc2Smem<stages, gu, BN>::DYN_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int units = launch_units(s, tc2_units());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * units));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope prof(kid, st);
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, s, ep, tg != nullptr ? *tg : ta,
                         tu != nullptr ? *tu : tb);
  g_last_launches.fetch_add(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int AM, int BMODE, bool BF16, class Epi>
cudaError_t launch_gemm(bool pairs, int kid, const CUtensorMap& ta, const CUtensorMap& tb,
                        const TcShape& s, const typename Epi::Params& ep, cudaStream_t st) {
  return pairs ? launch_tc2<AM, BMODE, BF16, Epi>(kid, ta, tb, s, ep, st)
               : launch_tc<AM, BMODE, BF16, Epi>(kid, ta, tb, s, ep, st);
}

template <bool DUAL, class Epi>
cudaError_t launch_simt(int kid, SimtOperand A, SimtOperand B, SimtOperand B2, int64_t M,
                        int64_t N, int64_t K, const Epi& epi, const SimtCheck& chk,
                        cudaStream_t st) {
  dim3 grid((unsigned)((N + SG_BN - 1) / SG_BN), (unsigned)((M + SG_BM - 1) / SG_BM));
  ProfScope prof(kid, st);
  simt_gemm_kernel<DUAL, Epi>
      <<<grid, SG_THREADS, 0, st>>>(A, B, B2, (int)M, (int)N, (int)K, epi, chk);
  g_last_launches.fetch_add(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// packed weights for the few-token no-grad forward
// ---------------------------------------------------------------------------
// Layout: the gate/up boxes, then the down boxes, 16 KB each.  Gate/up box
// (t, kb), t < ceil(H/64), kb < ceil(D/64), sits at (t * ceil(D/64) + kb) * 16
// KB: rows 0..63 are Wg rows t*64.., rows 64..127 the Wu rows of the same
// units, 64 elements (128 bytes) of K from kb*64 each.  Down box (t, kb),
// t < ceil(D/128), kb < ceil(H/64): Wd rows t*128.., K from kb*64.  Within a
// box the 16-byte chunk c of row r is stored at r*128 + (c ^ (r & 7))*16 (the
// 128-byte swizzle of the tensor-map loads); elements past D or H are zero.
constexpr size_t PACK_BOX_BYTES = 16384;

size_t packed_gateup_bytes(int64_t D, int64_t H) {
  return (size_t)((H + 63) / 64) * (size_t)((D + 63) / 64) * PACK_BOX_BYTES;
}

size_t packed_down_bytes(int64_t D, int64_t H) {
  return (size_t)((D + 127) / 128) * (size_t)((H + 63) / 64) * PACK_BOX_BYTES;
}

// One thread per 16-byte chunk of the packed buffer.
__global__ void pack_weights_kernel(const uint8_t* __restrict__ Wgu, const uint8_t* __restrict__ Wd,
                                    uint4* __restrict__ out, int64_t D, int64_t H,
                                    int64_t gu_chunks, int64_t all_chunks) {
  const int64_t kb1 = (D + 63) / 64, kb2 = (H + 63) / 64;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < all_chunks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool gu = i < gu_chunks;
    const int64_t j = gu ? i : i - gu_chunks;
    const int64_t box = j / 1024;
    const int r = (int)((j % 1024) / 8);
    const int c = (int)(j % 8) ^ (r & 7);  // the chunk stored at this position
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (gu) {
      const int64_t t = box / kb1, kb = box % kb1;
      const int64_t unit = t * 64 + (r & 63);
      const int64_t k = kb * 64 + c * 8;
      if (unit < H && k < D)
        v = *reinterpret_cast<const uint4*>(Wgu + ((r < 64 ? unit : H + unit) * D + k) * 2);
    } else {
      const int64_t t = box / kb2, kb = box % kb2;
      const int64_t row = t * 128 + r;
      const int64_t k = kb * 64 + c * 8;
      if (row < D && k < H) v = *reinterpret_cast<const uint4*>(Wd + (row * H + k) * 2);
    }
    out[i] = v;
  }
}

// ---------------------------------------------------------------------------
// no-grad forward for M <= 64 tokens: split-contraction swap-AB kernels
// ---------------------------------------------------------------------------
constexpr int NG_MAX_M = 64;
constexpr int NG_MAX_CTAS = 256;  // stream-K CTAs per launch (one per SM, capped)

struct NgPlan {
  int NT;
  int t1, kb1;  // gate/up: tiles of 64 hidden units, k-blocks over D
  int t2, kb2;  // down: tiles of 128 output features, k-blocks over H
  size_t counter_bytes, part_bytes;
};

bool ng_eligible(int64_t M, int64_t D, int64_t H, swiglu_dtype dt) {
  return dt != SWIGLU_F32_IEEE && M >= 1 && M <= NG_MAX_M;
}

// A CTA's range of ceil(total / ctas) k-blocks meets at most
// ceil(range / kb) + 1 tiles, so ctas x seg_max <= tiles + 3 ctas partial
// slots for any grid up to NG_MAX_CTAS: the workspace bound below does not
// depend on the device.
// The token block: the smallest of 16, 32, 48, 64 that holds M (the two
// kernels' time tracks the token rows landed per weight box, padding rows
// included); the fused kernel takes 16, 32 or 64 (ng_fused_plan).
NgPlan ng_plan(int64_t M, int64_t D, int64_t H, int nt = 0) {
  NgPlan p;
  p.NT = nt > 0 ? nt : (M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 48 ? 48 : 64)));
  p.t1 = (int)((H + 63) / 64);
  p.kb1 = (int)((D + 63) / 64);
  p.t2 = (int)((D + 127) / 128);
  p.kb2 = (int)((H + 63) / 64);
  // arrival counters of both phases, then the fused kernel's ready mask
  p.counter_bytes = (((size_t)(p.t1 + p.t2 + (p.t1 + 31) / 32) * 4 + 255) / 256) * 256;
  const size_t slots = (size_t)(p.t1 > p.t2 ? p.t1 : p.t2) + 3 * NG_MAX_CTAS;
  p.part_bytes = slots * 128 * p.NT * 4;
  return p;
}

NgPlan ng_fused_plan(int64_t M, int64_t D, int64_t H) {
  return ng_plan(M, D, H, M <= 16 ? 16 : (M <= 32 ? 32 : 64));
}

// CTAs, stream-K tiles and partial slots per CTA of one GEMM over at most
// `grid` CTAs.  With tiles >= CTAs, all but (tiles mod CTAs) tiles are taken
// whole, the same number per CTA; with fewer k-blocks than CTAs to share, the
// count shrinks so that every sharing CTA owns at least one.
void ng_split(int tiles, int kb, int grid, int& ctas, int& sk_tiles, int& seg_max) {
  int64_t c = grid < 1 ? 1 : grid;
  sk_tiles = tiles >= c ? (int)(tiles % c) : tiles;
  const int64_t total = (int64_t)sk_tiles * kb;
  if (total > 0 && c > total && tiles < c) c = total;
  ctas = (int)c;
  const int64_t range = total > 0 ? (total + c - 1) / c : 0;
  seg_max = (int)((range + kb - 1) / kb) + 1;
}

int ng_max_grid() {
  const int nsm = sm_count();
  return nsm < 1 ? 1 : (nsm < NG_MAX_CTAS ? nsm : NG_MAX_CTAS);
}

void ng_grid(int tiles, int kb, int& ctas, int& sk_tiles, int& seg_max) {
  ng_split(tiles, kb, ng_max_grid(), ctas, sk_tiles, seg_max);
}

// The fused kernel's work units.  gate/up: runs of 64 k-blocks (the
// gate/up units all precede the down units, so their end overlaps the down
// units' start); down: runs of 32 k-blocks, then 16 and 8 over the last
// 2 x 32 k-blocks, so the last units handed out are short.  Per unit the
// epilogue writes a partial tile of 128 x NT fp32 (at most an eighth of the
// unit's weight bytes).  A GEMM whose k-blocks fit one run has whole tiles
// (no partials).  Measured on D = 4096, H = 11008: this pair beat 16 / 32-
// and 8 / 16-k-block units, with and without the taper, at 1 and 64 tokens.
struct NgDynPlan {
  int chunks0, chunks1, units0, units1, grid;
  int kb_at[2][NG_MAX_CHUNKS + 1];
  size_t part0_bytes, part1_bytes;
};

int ng_chunks(int kb, int q, bool taper, int* at) {
  int n = 0, k = 0;
  at[0] = 0;
  while (k < kb) {
    const int rem = kb - k;
    int len = q;
    if (taper && rem <= 2 * q) len = rem > q ? q / 2 : q / 4;
    if (len < 1) len = 1;
    if (len > rem) len = rem;
    // the table has NG_MAX_CHUNKS entries: the last one takes the rest
    if (n == NG_MAX_CHUNKS - 1) len = rem;
    k += len;
    at[++n] = k;
  }
  return n;
}

NgDynPlan ng_dyn_plan(const NgPlan& p) {
  NgDynPlan d;
  int q0 = 64, q1 = 32;
  // keep at most NG_MAX_CHUNKS runs per tile on very long contractions
  while ((p.kb1 + q0 - 1) / q0 > NG_MAX_CHUNKS / 2) q0 *= 2;
  while ((p.kb2 + q1 - 1) / q1 > NG_MAX_CHUNKS / 2) q1 *= 2;
  d.chunks0 = ng_chunks(p.kb1, q0, false, d.kb_at[0]);
  d.chunks1 = ng_chunks(p.kb2, q1, true, d.kb_at[1]);
  d.units0 = p.t1 * d.chunks0;
  d.units1 = p.t2 * d.chunks1;
  const int g = ng_max_grid();
  const int units = d.units0 + d.units1;
  d.grid = units < g ? units : g;
  d.part0_bytes = d.chunks0 > 1 ? (size_t)d.units0 * 128 * p.NT * 4 : 0;
  d.part1_bytes = d.chunks1 > 1 ? (size_t)d.units1 * 128 * p.NT * 4 : 0;
  return d;
}

// Workspace bytes of the fused kernel: one partial slot per unit.
size_t ng_fused_bytes(const NgPlan& p) {
  const NgDynPlan d = ng_dyn_plan(p);
  return WS_HEADER + p.counter_bytes + d.part0_bytes + d.part1_bytes;
}

// Workspace bytes of the two-kernel form with the current device's grids
// (the second kernel reuses the first one's partial slots).
size_t ng_two_bytes(const NgPlan& p) {
  int c1 = 1, s1 = 1, c2 = 1, s2 = 1, k1 = 0, k2 = 0;
  ng_grid(p.t1, p.kb1, c1, k1, s1);
  ng_grid(p.t2, p.kb2, c2, k2, s2);
  const size_t slots1 = (size_t)c1 * s1, slots2 = (size_t)c2 * s2;
  return WS_HEADER + p.counter_bytes + (slots1 > slots2 ? slots1 : slots2) * 128 * p.NT * 4;
}

template <int NT, bool GATE_UP, bool BF16, bool PACKED = false>
cudaError_t launch_ng(int kid, const CUtensorMap& tw, const CUtensorMap& tx, NgArgs a,
                      cudaStream_t st) {
  auto kern = ng_gemm_kernel<NT, GATE_UP, BF16, PACKED>;
  constexpr int smem = NgSmem<NT>::DYN_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = 1;
  ng_grid(a.tiles, a.kb_tile, grid, a.sk_tiles, a.seg_max);
  a.ctas = grid;
  ProfScope prof(kid, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NG_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // the down kernel overlaps its prologue and weight prefetch with gate/up's tail
  // (per-kernel event timing would serialise the two, so it is not used then)
  const bool pdl = a.dependent && !g_prof_on.load();
  if (!pdl) a.dependent = 0;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, tw, tx, a);
  g_last_launches.fetch_add(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ws layout: [0, 256) header (error word at 0); per-tile counters of the
// gate/up kernel then of the down kernel; fp32 partial tiles.  The counters
// must be zero when a call starts: each kernel zeroes the other's counters
// at its start and every tile's reducer zeroes its own, so a zero-filled
// workspace stays valid across calls.
// With `packed` (swiglu_mlp_pack_weights' layout) the weight boxes come from
// it by bulk copies and Wgu / Wd are not read.
template <int NT, bool BF16>
swiglu_status ng_forward_nt(const void* X, const void* Wgu, const void* Wd, void* Y, void* A,
                            int64_t M, int64_t D, int64_t H, const NgPlan& p, char* ws,
                            size_t ws_cap, const Opts& o, cudaStream_t st,
                            const uint8_t* packed = nullptr) {
  int* err = reinterpret_cast<int*>(ws);
  int* counters = reinterpret_cast<int*>(ws + WS_HEADER);
  float* part = reinterpret_cast<float*>(ws + WS_HEADER + p.counter_bytes);
  const uint64_t wl = g_wait_limit_ns.load();
  CUtensorMap tw = {}, tx;
  if ((packed == nullptr && !encode_gateup(&tw, BF16, Wgu, D, H, 64)) ||
      !map_kmajor(&tx, BF16, X, D, M, D, ng_x_rows(NT, (int)M)))
    return SWIGLU_ERR_CUDA;
  NgArgs a1{(int)M, (int)H, p.kb1, p.t1, 0, 0, part, counters, counters + p.t1, p.t2, 1, 0, 0,
            A, H, wl, err};
  a1.scale = o.gm;
  a1.wpack = packed;
  set_windows(a1, {{A, (size_t)(M * H * 2)}, {ws, ws_cap}});
  if ((packed ? launch_ng<NT, true, BF16, true>(K_NG_GATE_UP, tw, tx, a1, st)
              : launch_ng<NT, true, BF16>(K_NG_GATE_UP, tw, tx, a1, st)) != cudaSuccess)
    return SWIGLU_ERR_CUDA;
  if ((packed == nullptr && !map_kmajor(&tw, BF16, Wd, H, D, H, 128)) ||
      !map_kmajor(&tx, BF16, A, H, M, H, ng_x_rows(NT, (int)M)))
    return SWIGLU_ERR_CUDA;
  NgArgs a2{(int)M, (int)D, p.kb2, p.t2, 0, 0, part, counters + p.t1, counters, p.t1, 0, 1, 0,
            Y, D, wl, err};
  a2.scale = o.dm;
  a2.wpack = packed ? packed + packed_gateup_bytes(D, H) : nullptr;
  set_windows(a2, {{Y, (size_t)(M * D * 2)}, {ws, ws_cap}});
  return cuda_status(packed ? launch_ng<NT, false, BF16, true>(K_NG_DOWN, tw, tx, a2, st)
                            : launch_ng<NT, false, BF16>(K_NG_DOWN, tw, tx, a2, st));
}

constexpr size_t NG_DONE_OFFSET = 128;  // the fused kernel's finished-CTA count (header)
constexpr size_t NG_NEXT_OFFSET = 192;  // the fused kernel's work-queue counter (header)

// The fused form: one launch for both GEMMs with a dynamic work queue.  ws
// layout as for the two kernels (header, per-tile counters of both GEMMs),
// plus the ready mask after the counters, the queue counter and the
// finished-CTA count in the header, and one partial slot per unit.
template <int NT, bool BF16>
swiglu_status ng_forward_fused(const void* X, const void* Wgu, const void* Wd, void* Y, void* A,
                               int64_t M, int64_t D, int64_t H, const NgPlan& p, char* ws,
                               size_t ws_cap, const Opts& o, cudaStream_t st) {
  auto kern = ng_fused_kernel<NT, BF16>;
  constexpr int smem = NgDynSmem<NT>::DYN_BYTES;
  {
    static std::mutex mu;
    static bool set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SWIGLU_ERR_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (!set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return SWIGLU_ERR_CUDA;
      set[dev] = true;
    }
  }
  const NgDynPlan d = ng_dyn_plan(p);
  int* err = reinterpret_cast<int*>(ws);
  int* counters = reinterpret_cast<int*>(ws + WS_HEADER);
  NgDynArgs f;
  f.chunks[0] = d.chunks0;
  f.chunks[1] = d.chunks1;
  std::memcpy(f.kb_at, d.kb_at, sizeof(f.kb_at));
  f.units0 = d.units0;
  f.units = d.units0 + d.units1;
  f.ready = reinterpret_cast<uint32_t*>(counters + p.t1 + p.t2);
  f.next_unit = reinterpret_cast<uint32_t*>(ws + NG_NEXT_OFFSET);
  f.done = reinterpret_cast<uint32_t*>(ws + NG_DONE_OFFSET);
  f.inject_unready = take_inject() ? 1 : 0;
  float* part0 = reinterpret_cast<float*>(ws + WS_HEADER + p.counter_bytes);
  float* part1 = reinterpret_cast<float*>(ws + WS_HEADER + p.counter_bytes + d.part0_bytes);
  const uint64_t wl = g_wait_limit_ns.load();
  CUtensorMap twgu, tx, twd, ta;
  if (!encode_gateup(&twgu, BF16, Wgu, D, H, 64) || !map_kmajor(&tx, BF16, X, D, M, D, NT) ||
      !map_kmajor(&twd, BF16, Wd, H, D, H, 128) || !map_kmajor(&ta, BF16, A, H, M, H, NT))
    return SWIGLU_ERR_CUDA;
  f.ph[0] = NgArgs{(int)M, (int)H, p.kb1, p.t1, 0, 0, part0, counters, nullptr, 0, 1, 0, 0,
                   A, H, wl, err};
  f.ph[1] = NgArgs{(int)M, (int)D, p.kb2, p.t2, 0, 0, part1, counters + p.t1, nullptr, 0, 0, 0,
                   0, Y, D, wl, err};
  f.ph[0].scale = o.gm;
  f.ph[1].scale = o.dm;
  set_windows(f.ph[0], {{A, (size_t)(M * H * 2)}, {ws, ws_cap}});
  set_windows(f.ph[1], {{Y, (size_t)(M * D * 2)}, {ws, ws_cap}});
  ProfScope prof(K_NG_FUSED, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)d.grid);
  cfg.blockDim = dim3(NG_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, twgu, tx, twd, ta, f);
  g_last_launches.fetch_add(1);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

// The fused form when it is selected (swiglu_mlp_set_nograd_fused: never by
// default, for 33..64 tokens, or always) and its workspace fits `ws_cap` (a
// fixed scratch array may not hold it); else two kernels.
template <int NT, bool BF16>
swiglu_status ng_forward_t(const void* X, const void* Wgu, const void* Wd, void* Y, void* A,
                           int64_t M, int64_t D, int64_t H, const NgPlan& p, char* ws,
                           size_t ws_cap, const Opts& o, cudaStream_t st) {
  const int mode = g_ng_fused.load();
  if (mode == 2 || (mode == 1 && M > 32)) {
    const NgPlan pf = ng_fused_plan(M, D, H);
    if (ng_fused_bytes(pf) <= ws_cap) {
      switch (pf.NT) {
        case 16: return ng_forward_fused<16, BF16>(X, Wgu, Wd, Y, A, M, D, H, pf, ws, ws_cap, o, st);
        case 32: return ng_forward_fused<32, BF16>(X, Wgu, Wd, Y, A, M, D, H, pf, ws, ws_cap, o, st);
        default: return ng_forward_fused<64, BF16>(X, Wgu, Wd, Y, A, M, D, H, pf, ws, ws_cap, o, st);
      }
    }
  }
  if (ng_two_bytes(p) > ws_cap) return SWIGLU_ERR_UNSUPPORTED;
  return ng_forward_nt<NT, BF16>(X, Wgu, Wd, Y, A, M, D, H, p, ws, ws_cap, o, st);
}

template <bool BF16>
swiglu_status ng_forward(const void* X, const void* Wgu, const void* Wd, void* Y, void* A,
                         int64_t M, int64_t D, int64_t H, char* ws, size_t ws_cap,
                         const Opts& o, cudaStream_t st) {
  const NgPlan p = ng_plan(M, D, H);
  switch (p.NT) {
    case 16: return ng_forward_t<16, BF16>(X, Wgu, Wd, Y, A, M, D, H, p, ws, ws_cap, o, st);
    case 32: return ng_forward_t<32, BF16>(X, Wgu, Wd, Y, A, M, D, H, p, ws, ws_cap, o, st);
    case 48: return ng_forward_t<48, BF16>(X, Wgu, Wd, Y, A, M, D, H, p, ws, ws_cap, o, st);
    default: return ng_forward_t<64, BF16>(X, Wgu, Wd, Y, A, M, D, H, p, ws, ws_cap, o, st);
  }
}

// ---------------------------------------------------------------------------
// the same few-token no-grad forward with its scratch in a static device array
// ---------------------------------------------------------------------------
// Scratch (error word, tile counters, fp32 partial tiles) for callers that
// cannot allocate.  It is part of the module image: every GPU that loads this
// library holds these bytes until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES];  // device address of the array, per device

// Host code cannot use g_noalloc_scratch's name as a device address (it is a
// host-side shadow); the device address is looked up once per device, with
// that device current, and cached.
swiglu_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWIGLU_ERR_CUDA;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return SWIGLU_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SWIGLU_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SWIGLU_OK;
}

size_t elt_bytes(swiglu_dtype dt) {
  switch (dt) {
    case SWIGLU_BF16:
    case SWIGLU_F16: return 2;
    case SWIGLU_F32_IEEE: return 4;
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape/dtype/workspace checks shared by every entry point.  Pointers are
// checked by the callers (which know which ones they use).
swiglu_status check_common(int64_t M, int64_t D, int64_t H, swiglu_dtype dt, const void* ws,
                           size_t ws_bytes, int op) {
  if (elt_bytes(dt) == 0) return SWIGLU_ERR_INVALID_ARG;
  if (M < 0 || D <= 0 || H <= 0) return SWIGLU_ERR_INVALID_ARG;
  const int64_t mult = dt == SWIGLU_F32_IEEE ? 4 : 8;
  if (D % mult != 0 || H % mult != 0) return SWIGLU_ERR_ALIGNMENT;
  const int64_t lim = 0x7fffffffLL;
  if (M > lim || D > lim || 3 * H > lim) return SWIGLU_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < swiglu_mlp_workspace_min_bytes(M, D, H, dt, op))
    return SWIGLU_ERR_WORKSPACE;
  if (!aligned16(ws)) return SWIGLU_ERR_ALIGNMENT;
  return SWIGLU_OK;
}

swiglu_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr) return SWIGLU_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return SWIGLU_ERR_ALIGNMENT;
  return SWIGLU_OK;
}

swiglu_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

// Reads and checks the options of an _ex call (NULL: the defaults).
swiglu_status read_opts(const swiglu_mlp_options* in, bool backward, Opts* out) {
  Opts o;
  if (in != nullptr) {
    if (!std::isfinite(in->gate_multiplier) || !std::isfinite(in->down_multiplier))
      return SWIGLU_ERR_INVALID_ARG;
    if (in->accumulate != 0 && (in->accumulate != 1 || !backward)) return SWIGLU_ERR_INVALID_ARG;
    o.gm = in->gate_multiplier;
    o.dm = in->down_multiplier;
    o.acc = in->accumulate;
  }
  *out = o;
  return SWIGLU_OK;
}

// ---------------------------------------------------------------------------
// tensor-core (bf16 / fp16) paths
// ---------------------------------------------------------------------------
template <bool BF16>
swiglu_status tc_forward(const void* X, const void* Wgu, const void* Wd, void* Y, void* G,
                         void* U, int64_t ld_gu, void* A, int64_t ld_a, int64_t M, int64_t D,
                         int64_t H, int* err, size_t ws_bytes, const Opts& o, cudaStream_t st) {
  const size_t cap = part_capacity(ws_bytes);
  CUtensorMap tx, tw, ta, twd;
  // gate/up + SwiGLU: C[m, j | H + j], N counts hidden units, BN/2 per tile;
  // on a pair each CTA brings one of Wg, Wu
  const bool pairs1 = use_pairs(M, H, TC_BN / 2, D);
  if (!map_kmajor(&tx, BF16, X, D, M, D, TC_BM) ||
      !encode_gateup(&tw, BF16, Wgu, D, H, TC_BN / 2, pairs1 ? 1 : 2))
    return SWIGLU_ERR_CUDA;
  TcShape s1 = make_shape(M, H, D, TC_BN / 2, err, pairs1, cap);
  // training: G, U and A are column ranges of the saved rows; no-grad: A alone
  set_windows(s1, {{G != nullptr ? G : A, (size_t)(M * (G != nullptr ? ld_gu : ld_a) * 2)},
                   {err, ws_bytes}});
  EpiSwiGLU::Params p1{G, U, ld_gu, A, ld_a, o.gm};
  cudaError_t e = launch_gemm<LOAD_KMAJOR, LOAD_GATEUP, BF16, EpiSwiGLU>(
      pairs1, G != nullptr ? K_GATE_UP : K_GATE_UP_NOGRAD, tx, tw, s1, p1, st);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  // down projection: Y = A Wd^T (a K-major B tile is 256 rows on one SM,
  // 128 rows per CTA on a pair)
  const bool pairs2 = use_pairs(M, D, TC_BN, H);
  if (!map_kmajor(&ta, BF16, A, H, M, ld_a, TC_BM) ||
      !map_kmajor(&twd, BF16, Wd, H, D, H, pairs2 ? 128 : TC_BN))
    return SWIGLU_ERR_CUDA;
  const bool wide2 = use_wide(pairs2, M, D, H);
  TcShape s2 = make_shape(M, D, H, wide2 ? TC2_WIDE_BN : TC_BN, err, pairs2, cap);
  set_windows(s2, {{Y, (size_t)(M * D * 2)}, {err, ws_bytes}});
  EpiStore::Params p2{Y, D, o.dm, 0};
  const int kid2 = G != nullptr ? K_DOWN : K_DOWN_NOGRAD;
  return cuda_status(
      wide2 ? launch_tc2<LOAD_KMAJOR, LOAD_KMAJOR, BF16, EpiStore, TC2_WIDE_BN>(kid2, ta, twd, s2,
                                                                              p2, st)
            : launch_gemm<LOAD_KMAJOR, LOAD_KMAJOR, BF16, EpiStore>(pairs2, kid2, ta, twd, s2, p2,
                                                                   st));
}

template <bool BF16>
swiglu_status tc_backward(const void* dY, const void* X, const void* Wgu, const void* Wd,
                          void* saved, void* dX, void* dWgu, void* dWd, int64_t M, int64_t D,
                          int64_t H, int* err, size_t ws_bytes, const Opts& o,
                          cudaStream_t st) {
  const size_t cap = part_capacity(ws_bytes);
  const int64_t ld = 3 * H;
  char* sv = static_cast<char*>(saved);
  void* G = sv;
  void* U = sv + H * 2;
  void* A = sv + 2 * H * 2;
  CUtensorMap m1, m2;
  cudaError_t e;
  // dWd [D, H] = dY^T A: both operands MN-major over the token dimension
  if (!map_mnmajor(&m1, BF16, dY, D, M, D) || !map_mnmajor(&m2, BF16, A, H, M, ld))
    return SWIGLU_ERR_CUDA;
  {
    const bool pairs = use_pairs(D, H, TC_BN, M);
    const bool wide = use_wide(pairs, D, H, M);
    TcShape s = make_shape(D, H, M, wide ? TC2_WIDE_BN : TC_BN, err, pairs, cap);
    set_windows(s, {{dWd, (size_t)(D * H * 2)}, {err, ws_bytes}});
    EpiStore::Params p{dWd, H, o.dm, o.acc};
    e = wide ? launch_tc2<LOAD_MNMAJOR, LOAD_MNMAJOR, BF16, EpiStore, TC2_WIDE_BN>(K_DWD, m1, m2,
                                                                                 s, p, st)
             : launch_gemm<LOAD_MNMAJOR, LOAD_MNMAJOR, BF16, EpiStore>(pairs, K_DWD, m1, m2, s, p,
                                                                      st);
    if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  }
  // dA = dY Wd (Wd read MN-major as [K = D][N = H]); dG, dU written over G, U
  if (!map_kmajor(&m1, BF16, dY, D, M, D, TC_BM) || !map_mnmajor(&m2, BF16, Wd, H, D, H))
    return SWIGLU_ERR_CUDA;
  {
    const bool pairs = use_pairs(M, H, TC_BN, D);
    TcShape s = make_shape(M, H, D, TC_BN, err, pairs, cap);
    set_windows(s, {{saved, (size_t)(M * ld * 2)}, {err, ws_bytes}});
    EpiDSwiGLU::Params p{G, U, ld, o.gm, o.dm};
    if (pairs && D <= 2048) {
      // a short contraction leaves the epilogue the bound: G/U in and dG/dU
      // out by TMA, through per-warp slots loaded ahead
      CUtensorMap tg, tu;
      if (!encode_2d(&tg, BF16, G, H, M, ld * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
          !encode_2d(&tu, BF16, U, H, M, ld * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return SWIGLU_ERR_CUDA;
      e = launch_tc2<LOAD_KMAJOR, LOAD_MNMAJOR, BF16, EpiDSwiGLUTma>(
          K_DGU, m1, m2, s, EpiDSwiGLUTma::Params{o.gm, o.dm}, st, &tg, &tu);
    } else {
      // a short contraction on single SMs: direct G/U loads
      e = D <= 2048 ? launch_gemm<LOAD_KMAJOR, LOAD_MNMAJOR, BF16, EpiDSwiGLUT<true>>(
                          pairs, K_DGU, m1, m2, s, p, st)
                    : launch_gemm<LOAD_KMAJOR, LOAD_MNMAJOR, BF16, EpiDSwiGLUT<false>>(
                          pairs, K_DGU, m1, m2, s, p, st);
    }
    if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  }
  // [dWg; dWu] [2H, D] = [dG | dU]^T X: one GEMM over the 2H columns
  if (!map_mnmajor(&m1, BF16, G, 2 * H, M, ld) || !map_mnmajor(&m2, BF16, X, D, M, D))
    return SWIGLU_ERR_CUDA;
  {
    const bool pairs = use_pairs(2 * H, D, TC_BN, M);
    const bool wide = use_wide(pairs, 2 * H, D, M);
    TcShape s = make_shape(2 * H, D, M, wide ? TC2_WIDE_BN : TC_BN, err, pairs, cap);
    set_windows(s, {{dWgu, (size_t)(2 * H * D * 2)}, {err, ws_bytes}});
    EpiStore::Params p{dWgu, D, 1.0f, o.acc};
    e = wide ? launch_tc2<LOAD_MNMAJOR, LOAD_MNMAJOR, BF16, EpiStore, TC2_WIDE_BN>(K_DWGU, m1, m2,
                                                                                 s, p, st)
             : launch_gemm<LOAD_MNMAJOR, LOAD_MNMAJOR, BF16, EpiStore>(pairs, K_DWGU, m1, m2, s,
                                                                      p, st);
    if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  }
  // dX [M, D] = [dG | dU] [Wg; Wu]: K = 2H in one accumulator
  if (!map_kmajor(&m1, BF16, G, 2 * H, M, ld, TC_BM) || !map_mnmajor(&m2, BF16, Wgu, D, 2 * H, D))
    return SWIGLU_ERR_CUDA;
  {
    const bool pairs = use_pairs(M, D, TC_BN, 2 * H);
    const bool wide = use_wide(pairs, M, D, 2 * H);
    TcShape s = make_shape(M, D, 2 * H, wide ? TC2_WIDE_BN : TC_BN, err, pairs, cap);
    set_windows(s, {{dX, (size_t)(M * D * 2)}, {err, ws_bytes}});
    EpiStore::Params p{dX, D, 1.0f, 0};
    e = wide ? launch_tc2<LOAD_KMAJOR, LOAD_MNMAJOR, BF16, EpiStore, TC2_WIDE_BN>(K_DX, m1, m2, s,
                                                                                p, st)
             : launch_gemm<LOAD_KMAJOR, LOAD_MNMAJOR, BF16, EpiStore>(pairs, K_DX, m1, m2, s, p,
                                                                     st);
    if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  }
  return SWIGLU_OK;
}

// ---------------------------------------------------------------------------
// fp32 IEEE (CUDA-core FFMA) paths
// ---------------------------------------------------------------------------
swiglu_status simt_forward(const float* X, const float* Wgu, const float* Wd, float* Y, float* G,
                           float* U, int64_t ld_gu, float* A, int64_t ld_a, int64_t M, int64_t D,
                           int64_t H, int* err, const Opts& o, cudaStream_t st) {
  // training: G, U and A are column ranges of the saved rows; no-grad: A alone
  const Win out{G != nullptr ? (const void*)G : (const void*)A,
                (size_t)(M * (G != nullptr ? ld_gu : ld_a) * 4)};
  const Win x_w{X, (size_t)(M * D * 4)}, wgu_w{Wgu, (size_t)(2 * H * D * 4)},
      wd_w{Wd, (size_t)(D * H * 4)}, y_w{Y, (size_t)(M * D * 4)};
  SimtOperand x{X, D, 1}, wg{Wgu, D, 1}, wu{Wgu + H * D, D, 1};
  cudaError_t e = launch_simt<true>(K_SIMT_GATE_UP, x, wg, wu, M, H, D,
                                    SimtEpiSwiGLU{G, U, ld_gu, A, ld_a, o.gm},
                                    simt_check(err, {out, x_w, wgu_w}), st);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  SimtOperand a{A, ld_a, 1}, wd{Wd, H, 1};
  return cuda_status(launch_simt<false>(K_SIMT_DOWN, a, wd, wd, M, D, H,
                                        SimtEpiStore{Y, D, o.dm, 0},
                                        simt_check(err, {y_w, out, wd_w}), st));
}

swiglu_status simt_backward(const float* dY, const float* X, const float* Wgu, const float* Wd,
                            float* saved, float* dX, float* dWgu, float* dWd, int64_t M,
                            int64_t D, int64_t H, int* err, const Opts& o, cudaStream_t st) {
  const int64_t ld = 3 * H;
  float* G = saved;
  float* U = saved + H;
  float* A = saved + 2 * H;
  const Win dy_w{dY, (size_t)(M * D * 4)}, x_w{X, (size_t)(M * D * 4)},
      wgu_w{Wgu, (size_t)(2 * H * D * 4)}, wd_w{Wd, (size_t)(D * H * 4)},
      sv_w{saved, (size_t)(M * ld * 4)};
  cudaError_t e;
  // dA = dY Wd: A(m, d) = dY[m, d]; B(j, d) = Wd[d, j]
  e = launch_simt<false>(K_SIMT_DGU, SimtOperand{dY, D, 1}, SimtOperand{Wd, 1, H}, SimtOperand{Wd, 1, H}, M,
                         H, D, SimtEpiDSwiGLU{G, U, ld, o.gm, o.dm},
                         simt_check(err, {sv_w, dy_w, wd_w}), st);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  // dWd[d, j] = sum_m dY[m, d] A[m, j]
  e = launch_simt<false>(K_SIMT_DWD, SimtOperand{dY, 1, D}, SimtOperand{A, 1, ld}, SimtOperand{A, 1, ld}, D,
                         H, M, SimtEpiStore{dWd, H, o.dm, o.acc},
                         simt_check(err, {Win{dWd, (size_t)(D * H * 4)}, dy_w, sv_w}), st);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  // dWgu[j', d] = sum_m dGU[m, j'] X[m, d]
  e = launch_simt<false>(K_SIMT_DWGU, SimtOperand{G, 1, ld}, SimtOperand{X, 1, D}, SimtOperand{X, 1, D}, 2 * H,
                         D, M, SimtEpiStore{dWgu, D, 1.0f, o.acc},
                         simt_check(err, {Win{dWgu, (size_t)(2 * H * D * 4)}, sv_w, x_w}), st);
  if (e != cudaSuccess) return SWIGLU_ERR_CUDA;
  // dX[m, d] = sum_j' dGU[m, j'] Wgu[j', d]
  e = launch_simt<false>(K_SIMT_DX, SimtOperand{G, ld, 1}, SimtOperand{Wgu, 1, D}, SimtOperand{Wgu, 1, D}, M,
                         D, 2 * H, SimtEpiStore{dX, D, 1.0f, 0},
                         simt_check(err, {Win{dX, (size_t)(M * D * 4)}, sv_w, wgu_w}), st);
  return cuda_status(e);
}

// ---------------------------------------------------------------------------
// test hook: the epilogues' elementwise stage on chosen values
// ---------------------------------------------------------------------------
// One thread per 32 consecutive elements (the epilogue's chunk): the forward
// stage through swiglu_pair, the backward one through dswiglu_32, the device
// functions the tensor-core epilogues call.
template <bool BF16>
__global__ void elementwise_test_kernel(int64_t chunks, const float* acc_g, const float* acc_u,
                                        uint32_t* A, uint32_t* G, uint32_t* U, const float* dA,
                                        const uint4* gs, const uint4* us, uint4* dG, uint4* dU,
                                        float gate_mul, float down_mul) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= chunks) return;
  const int64_t e0 = c * 32;
  if (acc_g != nullptr) {
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      uint32_t a, g, u;
      // the branch the gate/up epilogue takes for this multiplier
      if (gate_mul == 1.0f)
        swiglu_pair<BF16, false>(gate_mul, acc_g[e0 + 2 * i], acc_g[e0 + 2 * i + 1],
                                 acc_u[e0 + 2 * i], acc_u[e0 + 2 * i + 1], a, g, u);
      else
        swiglu_pair<BF16>(gate_mul, acc_g[e0 + 2 * i], acc_g[e0 + 2 * i + 1], acc_u[e0 + 2 * i],
                          acc_u[e0 + 2 * i + 1], a, g, u);
      A[e0 / 2 + i] = a;
      G[e0 / 2 + i] = g;
      U[e0 / 2 + i] = u;
    }
  }
  if (dA != nullptr) {
    uint4 vg[4], vu[4];
    uint32_t r[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      vg[q] = gs[c * 4 + q];
      vu[q] = us[c * 4 + q];
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(dA[e0 + i]);
    uint32_t odg[16], odu[16];
    dswiglu_32<BF16>(vg, vu, r, gate_mul, down_mul, odg, odu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dG[c * 4 + q] = make_uint4(odg[4 * q], odg[4 * q + 1], odg[4 * q + 2], odg[4 * q + 3]);
      dU[c * 4 + q] = make_uint4(odu[4 * q], odu[4 * q + 1], odu[4 * q + 2], odu[4 * q + 3]);
    }
  }
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

size_t swiglu_mlp_element_bytes(swiglu_dtype dtype) { return elt_bytes(dtype); }

size_t swiglu_mlp_saved_bytes(int64_t M, int64_t H, swiglu_dtype dtype) {
  if (M < 0 || H < 0) return 0;
  return (size_t)M * (size_t)(3 * H) * elt_bytes(dtype);
}

size_t swiglu_mlp_workspace_bytes(int64_t M, int64_t D, int64_t H, swiglu_dtype dtype, int op) {
  if (op == SWIGLU_OP_FWD_NOGRAD && D > 0 && H > 0 && ng_eligible(M, D, H, dtype)) {
    const NgPlan p = ng_plan(M, D, H);
    const size_t two = WS_HEADER + p.counter_bytes + p.part_bytes;
    const size_t one = ng_fused_bytes(ng_fused_plan(M, D, H));
    return two > one ? two : one;
  }
  if (dtype == SWIGLU_BF16 || dtype == SWIGLU_F16)
    return WS_HEADER + TC_SK_COUNTER_BYTES + tc_ws_part_bytes(M, D, H, op);
  return WS_HEADER;
}

size_t swiglu_mlp_workspace_min_bytes(int64_t M, int64_t D, int64_t H, swiglu_dtype dtype,
                                      int op) {
  if (op == SWIGLU_OP_FWD_NOGRAD && D > 0 && H > 0 && ng_eligible(M, D, H, dtype))
    return ng_two_bytes(ng_plan(M, D, H));
  if (dtype == SWIGLU_BF16 || dtype == SWIGLU_F16) return WS_HEADER + TC_SK_COUNTER_BYTES;
  return WS_HEADER;
}

swiglu_status swiglu_mlp_fwd_ex(const void* X, const void* Wgu, const void* Wd, void* Y,
                                void* saved, int64_t M, int64_t D, int64_t H,
                                swiglu_dtype dtype, const swiglu_mlp_options* options,
                                void* ws, size_t ws_bytes, void* stream) {
  g_last_launches.store(0);
  Opts o;
  swiglu_status st = read_opts(options, false, &o);
  if (st != SWIGLU_OK) return st;
  st = check_common(M, D, H, dtype, ws, ws_bytes, SWIGLU_OP_FWD);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;
  if ((st = check_ptrs({X, Wgu, Wd, Y, saved})) != SWIGLU_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  if (cudaMemsetAsync(err, 0, ws_clear_bytes(dtype), s) != cudaSuccess) return SWIGLU_ERR_CUDA;
  const size_t e = elt_bytes(dtype);
  char* sv = static_cast<char*>(saved);
  void* G = sv;
  void* U = sv + H * e;
  void* A = sv + 2 * H * e;
  switch (dtype) {
    case SWIGLU_BF16:
      return tc_forward<true>(X, Wgu, Wd, Y, G, U, 3 * H, A, 3 * H, M, D, H, err, ws_bytes, o, s);
    case SWIGLU_F16:
      return tc_forward<false>(X, Wgu, Wd, Y, G, U, 3 * H, A, 3 * H, M, D, H, err, ws_bytes, o, s);
    default:
      return simt_forward((const float*)X, (const float*)Wgu, (const float*)Wd, (float*)Y,
                          (float*)G, (float*)U, 3 * H, (float*)A, 3 * H, M, D, H, err, o, s);
  }
}

swiglu_status swiglu_mlp_fwd(const void* X, const void* Wgu, const void* Wd, void* Y, void* saved,
                             int64_t M, int64_t D, int64_t H, swiglu_dtype dtype, void* ws,
                             size_t ws_bytes, void* stream) {
  return swiglu_mlp_fwd_ex(X, Wgu, Wd, Y, saved, M, D, H, dtype, nullptr, ws, ws_bytes, stream);
}

swiglu_status swiglu_mlp_fwd_nograd_ex(const void* X, const void* Wgu, const void* Wd, void* Y,
                                       void* A, int64_t M, int64_t D, int64_t H,
                                       swiglu_dtype dtype, const swiglu_mlp_options* options,
                                       void* ws, size_t ws_bytes, void* stream) {
  g_last_launches.store(0);
  Opts o;
  swiglu_status st = read_opts(options, false, &o);
  if (st != SWIGLU_OK) return st;
  st = check_common(M, D, H, dtype, ws, ws_bytes, SWIGLU_OP_FWD_NOGRAD);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;
  if ((st = check_ptrs({X, Wgu, Wd, Y, A})) != SWIGLU_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ng_eligible(M, D, H, dtype)) {
    char* w = static_cast<char*>(ws);
    return dtype == SWIGLU_BF16
               ? ng_forward<true>(X, Wgu, Wd, Y, A, M, D, H, w, ws_bytes, o, s)
               : ng_forward<false>(X, Wgu, Wd, Y, A, M, D, H, w, ws_bytes, o, s);
  }
  int* err = static_cast<int*>(ws);
  if (cudaMemsetAsync(err, 0, ws_clear_bytes(dtype), s) != cudaSuccess) return SWIGLU_ERR_CUDA;
  switch (dtype) {
    case SWIGLU_BF16:
      return tc_forward<true>(X, Wgu, Wd, Y, nullptr, nullptr, 0, A, H, M, D, H, err, ws_bytes, o, s);
    case SWIGLU_F16:
      return tc_forward<false>(X, Wgu, Wd, Y, nullptr, nullptr, 0, A, H, M, D, H, err, ws_bytes, o, s);
    default:
      return simt_forward((const float*)X, (const float*)Wgu, (const float*)Wd, (float*)Y,
                          nullptr, nullptr, 0, (float*)A, H, M, D, H, err, o, s);
  }
}

swiglu_status swiglu_mlp_fwd_nograd(const void* X, const void* Wgu, const void* Wd, void* Y,
                                    void* A, int64_t M, int64_t D, int64_t H, swiglu_dtype dtype,
                                    void* ws, size_t ws_bytes, void* stream) {
  return swiglu_mlp_fwd_nograd_ex(X, Wgu, Wd, Y, A, M, D, H, dtype, nullptr, ws, ws_bytes,
                                  stream);
}

size_t swiglu_mlp_packed_weights_bytes(int64_t D, int64_t H, swiglu_dtype dtype) {
  if (D <= 0 || H <= 0 || (dtype != SWIGLU_BF16 && dtype != SWIGLU_F16)) return 0;
  return packed_gateup_bytes(D, H) + packed_down_bytes(D, H);
}

swiglu_status swiglu_mlp_pack_weights(const void* Wgu, const void* Wd, void* packed, int64_t D,
                                      int64_t H, swiglu_dtype dtype, void* stream) {
  g_last_launches.store(0);
  if (dtype != SWIGLU_BF16 && dtype != SWIGLU_F16) return SWIGLU_ERR_UNSUPPORTED;
  if (D <= 0 || H <= 0) return SWIGLU_ERR_INVALID_ARG;
  if (D % 8 != 0 || H % 8 != 0) return SWIGLU_ERR_ALIGNMENT;
  if (D > 0x7fffffffLL || 3 * H > 0x7fffffffLL) return SWIGLU_ERR_UNSUPPORTED;
  swiglu_status st = check_ptrs({Wgu, Wd, packed});
  if (st != SWIGLU_OK) return st;
  const int64_t gu_chunks = (int64_t)(packed_gateup_bytes(D, H) / 16);
  const int64_t all = gu_chunks + (int64_t)(packed_down_bytes(D, H) / 16);
  const int nsm = sm_count();
  const int64_t want = (all + 255) / 256;
  const int grid = (int)(want < (int64_t)(nsm > 0 ? nsm : 1) * 8 ? want : (int64_t)(nsm > 0 ? nsm : 1) * 8);
  pack_weights_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(Wgu), static_cast<const uint8_t*>(Wd),
      static_cast<uint4*>(packed), D, H, gu_chunks, all);
  g_last_launches.fetch_add(1);
  return cuda_status(cudaGetLastError());
}

swiglu_status swiglu_mlp_fwd_nograd_packed(const void* X, const void* packed, void* Y, void* A,
                                           int64_t M, int64_t D, int64_t H, swiglu_dtype dtype,
                                           const swiglu_mlp_options* options, void* ws,
                                           size_t ws_bytes, void* stream) {
  g_last_launches.store(0);
  Opts o;
  swiglu_status st = read_opts(options, false, &o);
  if (st != SWIGLU_OK) return st;
  if (dtype != SWIGLU_BF16 && dtype != SWIGLU_F16) return SWIGLU_ERR_UNSUPPORTED;
  if (M > NG_MAX_M) return SWIGLU_ERR_UNSUPPORTED;
  st = check_common(M, D, H, dtype, ws, ws_bytes, SWIGLU_OP_FWD_NOGRAD);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;
  if ((st = check_ptrs({X, packed, Y, A})) != SWIGLU_OK) return st;
  const NgPlan p = ng_plan(M, D, H);
  if (ng_two_bytes(p) > ws_bytes) return SWIGLU_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  switch (p.NT) {
    case 16:
      return dtype == SWIGLU_BF16
                 ? ng_forward_nt<16, true>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk)
                 : ng_forward_nt<16, false>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk);
    case 32:
      return dtype == SWIGLU_BF16
                 ? ng_forward_nt<32, true>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk)
                 : ng_forward_nt<32, false>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk);
    case 48:
      return dtype == SWIGLU_BF16
                 ? ng_forward_nt<48, true>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk)
                 : ng_forward_nt<48, false>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk);
    default:
      return dtype == SWIGLU_BF16
                 ? ng_forward_nt<64, true>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk)
                 : ng_forward_nt<64, false>(X, nullptr, nullptr, Y, A, M, D, H, p, w, ws_bytes, o, s, pk);
  }
}

swiglu_status swiglu_mlp_fwd_nograd_noalloc(const void* X, const void* Wgu, const void* Wd,
                                            void* Y, void* A, int64_t M, int64_t D, int64_t H,
                                            swiglu_dtype dtype, void* stream) {
  g_last_launches.store(0);
  if (dtype != SWIGLU_BF16 && dtype != SWIGLU_F16) return SWIGLU_ERR_UNSUPPORTED;
  if (M < 0 || D <= 0 || H <= 0) return SWIGLU_ERR_INVALID_ARG;
  if (D % 8 != 0 || H % 8 != 0) return SWIGLU_ERR_ALIGNMENT;
  if (M > NG_MAX_M || D > 0x7fffffffLL || 3 * H > 0x7fffffffLL) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0) return SWIGLU_OK;
  swiglu_status st = check_ptrs({X, Wgu, Wd, Y, A});
  if (st != SWIGLU_OK) return st;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != SWIGLU_OK) return st;
  const NgPlan p = ng_plan(M, D, H);
  if (ng_two_bytes(p) > NOALLOC_SCRATCH_BYTES &&
      ng_fused_bytes(ng_fused_plan(M, D, H)) > NOALLOC_SCRATCH_BYTES)
    return SWIGLU_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: clear the error word, the
  // tile counters and the ready mask, which must start at zero
  if (cudaMemsetAsync(scratch, 0, WS_HEADER + p.counter_bytes, s) != cudaSuccess)
    return SWIGLU_ERR_CUDA;
  char* w = static_cast<char*>(scratch);
  return dtype == SWIGLU_BF16
             ? ng_forward<true>(X, Wgu, Wd, Y, A, M, D, H, w, NOALLOC_SCRATCH_BYTES, Opts{}, s)
             : ng_forward<false>(X, Wgu, Wd, Y, A, M, D, H, w, NOALLOC_SCRATCH_BYTES, Opts{}, s);
}

swiglu_status swiglu_mlp_bwd_ex(const void* dY, const void* X, const void* Wgu, const void* Wd,
                                void* saved, void* dX, void* dWgu, void* dWd, int64_t M,
                                int64_t D, int64_t H, swiglu_dtype dtype,
                                const swiglu_mlp_options* options, void* ws, size_t ws_bytes,
                                void* stream) {
  g_last_launches.store(0);
  Opts o;
  swiglu_status st = read_opts(options, true, &o);
  if (st != SWIGLU_OK) return st;
  st = check_common(M, D, H, dtype, ws, ws_bytes, SWIGLU_OP_BWD);
  if (st != SWIGLU_OK) return st;
  if (M == 0) return SWIGLU_OK;  // gradients of an empty batch: nothing is written
  if ((st = check_ptrs({dY, X, Wgu, Wd, saved, dX, dWgu, dWd})) != SWIGLU_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  if (cudaMemsetAsync(err, 0, ws_clear_bytes(dtype), s) != cudaSuccess) return SWIGLU_ERR_CUDA;
  switch (dtype) {
    case SWIGLU_BF16:
      return tc_backward<true>(dY, X, Wgu, Wd, saved, dX, dWgu, dWd, M, D, H, err, ws_bytes, o, s);
    case SWIGLU_F16:
      return tc_backward<false>(dY, X, Wgu, Wd, saved, dX, dWgu, dWd, M, D, H, err, ws_bytes, o, s);
    default:
      return simt_backward((const float*)dY, (const float*)X, (const float*)Wgu,
                           (const float*)Wd, (float*)saved, (float*)dX, (float*)dWgu,
                           (float*)dWd, M, D, H, err, o, s);
  }
}

swiglu_status swiglu_mlp_bwd(const void* dY, const void* X, const void* Wgu, const void* Wd,
                             void* saved, void* dX, void* dWgu, void* dWd, int64_t M, int64_t D,
                             int64_t H, swiglu_dtype dtype, void* ws, size_t ws_bytes,
                             void* stream) {
  return swiglu_mlp_bwd_ex(dY, X, Wgu, Wd, saved, dX, dWgu, dWd, M, D, H, dtype, nullptr, ws,
                           ws_bytes, stream);
}

struct swiglu_mlp_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
  int launches = 0;  // kernels one replay runs
};

swiglu_status swiglu_mlp_graph_create_fwd_nograd(const void* X, const void* Wgu, const void* Wd,
                                                 void* Y, void* A, int64_t M, int64_t D,
                                                 int64_t H, swiglu_dtype dtype, void* ws,
                                                 size_t ws_bytes, swiglu_mlp_graph** out) {
  if (out == nullptr) return SWIGLU_ERR_INVALID_ARG;
  *out = nullptr;
  swiglu_status st = check_common(M, D, H, dtype, ws, ws_bytes, SWIGLU_OP_FWD_NOGRAD);
  if (st != SWIGLU_OK) return st;
  if (M > 0 && (st = check_ptrs({X, Wgu, Wd, Y, A})) != SWIGLU_OK) return st;
  if (g_prof_on.load()) return SWIGLU_ERR_UNSUPPORTED;
  swiglu_mlp_graph* g = new swiglu_mlp_graph;
  if (cudaGetDevice(&g->device) != cudaSuccess) {
    delete g;
    return SWIGLU_ERR_CUDA;
  }
  if (M == 0) {  // nothing to record: launches of this graph do nothing
    *out = g;
    return SWIGLU_OK;
  }
  // device queries that are cached on first use run here, outside the capture
  sm_count();
  if (dtype != SWIGLU_F32_IEEE) tc2_units();
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    delete g;
    return SWIGLU_ERR_CUDA;
  }
  st = SWIGLU_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
    const swiglu_status inner =
        swiglu_mlp_fwd_nograd(X, Wgu, Wd, Y, A, M, D, H, dtype, ws, ws_bytes, cs);
    g->launches = g_last_launches.load();
    const cudaError_t ec = cudaStreamEndCapture(cs, &g->graph);
    if (inner != SWIGLU_OK)
      st = inner;
    else if (ec == cudaSuccess && g->graph != nullptr &&
             cudaGraphInstantiate(&g->exec, g->graph, 0) == cudaSuccess)
      st = SWIGLU_OK;
  }
  cudaGetLastError();  // clear the error a failed capture recorded
  cudaStreamDestroy(cs);
  if (st != SWIGLU_OK) {
    swiglu_mlp_graph_destroy(g);
    return st;
  }
  *out = g;
  return SWIGLU_OK;
}

swiglu_status swiglu_mlp_graph_launch(swiglu_mlp_graph* graph, void* stream) {
  if (graph == nullptr) return SWIGLU_ERR_INVALID_ARG;
  g_last_launches.store(0);
  if (graph->exec == nullptr) return SWIGLU_OK;  // M = 0
  const cudaError_t e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_last_launches.store(graph->launches);
  return cuda_status(e);
}

swiglu_status swiglu_mlp_graph_destroy(swiglu_mlp_graph* graph) {
  if (graph == nullptr) return SWIGLU_ERR_INVALID_ARG;
  cudaError_t e = cudaSuccess;
  if (graph->exec != nullptr) e = cudaGraphExecDestroy(graph->exec);
  if (graph->graph != nullptr) {
    const cudaError_t e2 = cudaGraphDestroy(graph->graph);
    if (e == cudaSuccess) e = e2;
  }
  delete graph;
  return cuda_status(e);
}

swiglu_status swiglu_mlp_query_error(const void* ws, void* stream) {
  if (ws == nullptr) return SWIGLU_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SWIGLU_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SWIGLU_ERR_CUDA;
  if (host == DEV_ERR_TIMEOUT) return SWIGLU_ERR_DEVICE_TIMEOUT;
  if (host == DEV_ERR_BOUNDS) return SWIGLU_ERR_DEVICE_BOUNDS;
  return host == 0 ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

void swiglu_mlp_debug_narrow_once(int on) { g_narrow_once.store(on ? 1 : 0); }

int swiglu_mlp_debug_build(void) {
#ifdef SWIGLU_DEBUG
  return 1;
#else
  return 0;
#endif
}

const char* swiglu_status_string(swiglu_status status) {
  switch (status) {
    case SWIGLU_OK: return "ok";
    case SWIGLU_ERR_INVALID_ARG: return "invalid argument (null pointer, bad size or dtype)";
    case SWIGLU_ERR_ALIGNMENT: return "misaligned pointer or D/H not a multiple of 8 (4 for fp32)";
    case SWIGLU_ERR_UNSUPPORTED: return "shape outside the supported range";
    case SWIGLU_ERR_WORKSPACE: return "workspace missing or too small";
    case SWIGLU_ERR_CUDA: return "CUDA error";
    case SWIGLU_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case SWIGLU_ERR_DEVICE_BOUNDS: return "device index check failed (debug build)";
    default: return "unknown status";
  }
}

uint64_t swiglu_mlp_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1000) ns = 1000;
  return g_wait_limit_ns.exchange(ns);
}

void swiglu_mlp_inject_stall_once(int on) { g_inject_stall.store(on > 0 ? on : 0); }

int swiglu_mlp_last_launch_count(void) { return g_last_launches.load(); }

int swiglu_mlp_set_nograd_fused(int mode) {
  return g_ng_fused.exchange(mode <= 0 ? 0 : (mode >= 2 ? 2 : 1));
}

int swiglu_mlp_set_cta_pairs(int mode) {
  return g_cta_pairs.exchange(mode <= 0 ? 0 : (mode >= 2 ? 2 : 1));
}

int swiglu_mlp_set_wide_tiles(int mode) {
  return g_wide_tiles.exchange(mode <= 0 ? 0 : (mode >= 2 ? 2 : 1));
}

void swiglu_mlp_profile_enable(int on) { g_prof_on.store(on ? 1 : 0); }

int swiglu_mlp_profile_read(int n, int64_t* launches, double* total_ms) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  int rc = K_COUNT;
  for (const ProfRec& r : g_prof_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      rc = -1;
    g_prof_ms[r.id] += ms;
    g_prof_n[r.id] += 1;
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_pending.clear();
  for (int i = 0; i < K_COUNT && i < n; ++i) {
    if (launches) launches[i] = g_prof_n[i];
    if (total_ms) total_ms[i] = g_prof_ms[i];
    g_prof_n[i] = 0;
    g_prof_ms[i] = 0.0;
  }
  return rc;
}

const char* swiglu_mlp_kernel_name(int id) {
  return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : nullptr;
}

swiglu_status swiglu_mlp_test_elementwise(swiglu_dtype dtype, int64_t n, const float* acc_g,
                                          const float* acc_u, void* A, void* G, void* U,
                                          const float* dA, const void* gs, const void* us,
                                          void* dG, void* dU, float gate_multiplier,
                                          float down_multiplier, void* stream) {
  g_last_launches.store(0);
  if (dtype != SWIGLU_BF16 && dtype != SWIGLU_F16) return SWIGLU_ERR_INVALID_ARG;
  if (n < 0 || n % 32 != 0 || n > 0x7fffffffLL) return SWIGLU_ERR_INVALID_ARG;
  const bool fwd = acc_g != nullptr, bwd = dA != nullptr;
  if (!fwd && !bwd) return SWIGLU_ERR_INVALID_ARG;
  swiglu_status st;
  if (fwd && (st = check_ptrs({acc_g, acc_u, A, G, U})) != SWIGLU_OK) return st;
  if (bwd && (st = check_ptrs({dA, gs, us, dG, dU})) != SWIGLU_OK) return st;
  if (n == 0) return SWIGLU_OK;
  const int64_t chunks = n / 32;
  const int threads = 128;
  const unsigned blocks = (unsigned)((chunks + threads - 1) / threads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto k = dtype == SWIGLU_BF16 ? elementwise_test_kernel<true> : elementwise_test_kernel<false>;
  k<<<blocks, threads, 0, s>>>(chunks, acc_g, acc_u, static_cast<uint32_t*>(A),
                               static_cast<uint32_t*>(G), static_cast<uint32_t*>(U), dA,
                               static_cast<const uint4*>(gs), static_cast<const uint4*>(us),
                               static_cast<uint4*>(dG), static_cast<uint4*>(dU), gate_multiplier,
                               down_multiplier);
  g_last_launches.fetch_add(1);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
