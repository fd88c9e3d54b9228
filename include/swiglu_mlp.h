/*
 * swiglu_mlp.h -- C ABI of the fused SwiGLU MLP library for GB300 (sm_103a).
 *
 * The operation ("[RFC] Full-pipeline SwiGLU MLP with forward/backward
 * co-optimization", Liger-Kernel issue #1347, section "Summary"):
 *
 *     G = X Wg^T,   U = X Wu^T,   A = SiLU(G) * U,   Y = A Wd^T
 *
 * and its gradients for Y's cotangent dY ("Correctness": dI = dX, dWg, dWu,
 * dWd).  SiLU(g) = g / (1 + e^-g).
 *
 * Layouts (all row-major, nn.Linear convention):
 *   X   [M, D]       M = B * S tokens
 *   Wgu [2H, D]      rows 0..H-1 are Wg, rows H..2H-1 are Wu (the two
 *                    projections concatenated, as one contiguous matrix)
 *   Wd  [D, H]
 *   Y   [M, D]
 *   saved [M, 3H]    one contiguous buffer holding, per token row, [G | U | A]
 *                    (Summary: the three saved activations share one buffer)
 *   dWgu [2H, D]     [dWg; dWu] in the layout of Wgu
 *   dWd [D, H],  dX [M, D],  dY [M, D]
 *
 * Element types (swiglu_dtype): bf16 or fp16 storage with fp32 accumulation
 * on the tensor cores, or SWIGLU_F32_IEEE: fp32 storage computed with IEEE
 * fp32 FMA on the CUDA cores -- never TF32 ("[RFC] Testing Methodology for
 * FP32 Convergence Tests on Fused SwiGLU/dSwiGLU Kernels", Liger-Kernel issue
 * #1383, section "Root Cause").
 *
 * Rounding: G and U are rounded once to the storage type from the fp32
 * accumulators; A = SiLU(G) * U is computed in fp32 from the unrounded
 * accumulators and rounded once ("Scope one-round FP32 SwiGLU to the exact
 * Qwen3.5 contract", xorl PR #51, review section); every other output is
 * rounded once from its fp32 accumulator, round-to-nearest-even.
 *
 * Pointers: every tensor pointer is a DEVICE pointer, owned by the caller,
 * 16-byte aligned.  Sizes: M >= 0, D >= 1, H >= 1; for bf16/fp16 D and H must
 * be multiples of 8 (row strides of D, H, 2H and 3H elements are then
 * multiples of 16 bytes, as the tensor-memory-access engine requires); for
 * fp32 D and H must be multiples of 4.  M = 0 returns SWIGLU_OK and launches
 * nothing.  ``stream`` is a cudaStream_t (0 = legacy default stream).
 *
 * Workspace: ``ws`` is a device buffer of swiglu_mlp_workspace_bytes() bytes
 * (a size for the current device; at least swiglu_mlp_workspace_min_bytes()
 * is accepted, see there), owned by the caller, ZERO-FILLED
 * before its first use.  It holds a device error word (cleared at the start
 * of every call), per-tile arrival counters (cleared by every training call,
 * left at zero by every completed few-token no-grad call) and fp32 partial
 * tiles: when a GEMM's last round of whole tiles would leave SMs idle, its
 * remaining tiles are split along K over all SMs (stream-K) and the partial
 * sums meet in the workspace.  After a SWIGLU_ERR_DEVICE_TIMEOUT, zero-fill
 * it again before reuse.  Calls that share one workspace must not overlap on
 * the GPU.  The library itself allocates no device buffers (the one
 * exception: an instantiated graph of swiglu_mlp_graph_create_fwd_nograd).
 *
 * Calls are asynchronous on ``stream`` and do not synchronise (except
 * swiglu_mlp_query_error).  Argument errors are detected on the host before
 * any launch and returned as a status; a device-side wait that runs past its
 * time limit (a stuck pipeline) is recorded in the workspace error word and
 * reported by swiglu_mlp_query_error as SWIGLU_ERR_DEVICE_TIMEOUT.
 *
 * Results are deterministic: no floating-point atomics; repeated calls on the
 * same inputs give the same bits.
 */
#ifndef SWIGLU_MLP_H
#define SWIGLU_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SWIGLU_BF16 = 0,
  SWIGLU_F16 = 1,
  SWIGLU_F32_IEEE = 2
} swiglu_dtype;

typedef enum {
  SWIGLU_OK = 0,
  SWIGLU_ERR_INVALID_ARG = 1,     /* null pointer, negative or zero size, bad enum */
  SWIGLU_ERR_ALIGNMENT = 2,       /* pointer not 16-byte aligned, or D/H not a multiple of 8 (4 for fp32) */
  SWIGLU_ERR_UNSUPPORTED = 3,     /* shape outside the supported range (e.g. > 2^31 - 1 rows) */
  SWIGLU_ERR_WORKSPACE = 4,       /* ws is NULL or smaller than swiglu_mlp_workspace_bytes() */
  SWIGLU_ERR_CUDA = 5,            /* a CUDA runtime/driver call or a launch failed */
  SWIGLU_ERR_DEVICE_TIMEOUT = 6,  /* a device pipeline wait ran past its limit */
  SWIGLU_ERR_DEVICE_BOUNDS = 7    /* debug builds only: a device index check failed */
} swiglu_status;

/* Operations, for sizing queries. */
enum { SWIGLU_OP_FWD = 0, SWIGLU_OP_FWD_NOGRAD = 1, SWIGLU_OP_BWD = 2 };

/* Bytes per element of a storage type (2, 2 or 4); 0 for an invalid value. */
size_t swiglu_mlp_element_bytes(swiglu_dtype dtype);

/* Bytes of the saved buffer: M * 3H elements ([G | U | A] per row). */
size_t swiglu_mlp_saved_bytes(int64_t M, int64_t H, swiglu_dtype dtype);

/* Bytes of workspace an operation needs (at least the 256-byte header that
 * holds the device error word), with room for every GEMM's stream-K partial
 * tiles and, for few tokens without gradients, for either kernel form. */
size_t swiglu_mlp_workspace_bytes(int64_t M, int64_t D, int64_t H, swiglu_dtype dtype, int op);

/* The smallest workspace an operation accepts: the header and tile counters
 * (1.25 KB) for the tensor-core paths, plus the two-kernel form's partial
 * tiles for few tokens without gradients.  With less than
 * swiglu_mlp_workspace_bytes(), each GEMM whose stream-K partial tiles do
 * not fit runs whole tiles only (results within the same tolerances; the
 * last round of tiles is no longer balanced over the SMs), and the few-token
 * no-grad call takes the fused kernel only if its partials fit.  This trades
 * a few percent of speed for up to ~40 MB at the largest shapes (training
 * intermediates at small S are then the [G|U|A] buffer alone). */
size_t swiglu_mlp_workspace_min_bytes(int64_t M, int64_t D, int64_t H, swiglu_dtype dtype,
                                      int op);

/* Training forward.  Writes Y [M,D] and saved [M,3H] = [G | U | A].
 * Reads X [M,D], Wgu [2H,D], Wd [D,H].  ("Summary": the gate and up
 * projections fused with SiLU and gating in one kernel; A, G, U stored in one
 * contiguous buffer.)  Kernels: gate/up + SwiGLU, then the down projection. */
swiglu_status swiglu_mlp_fwd(const void* X, const void* Wgu, const void* Wd, void* Y,
                             void* saved, int64_t M, int64_t D, int64_t H,
                             swiglu_dtype dtype, void* ws, size_t ws_bytes, void* stream);

/* Inference forward that saves neither G nor U ("Summary": a dedicated
 * no-grad path).  Writes A [M,H] (row stride H) and Y [M,D]. */
swiglu_status swiglu_mlp_fwd_nograd(const void* X, const void* Wgu, const void* Wd, void* Y,
                                    void* A, int64_t M, int64_t D, int64_t H,
                                    swiglu_dtype dtype, void* ws, size_t ws_bytes, void* stream);

/* The few-token no-grad forward (same kernels and results as
 * swiglu_mlp_fwd_nograd for M <= 64) for callers that cannot allocate device
 * memory: code that runs while a CUDA graph is being captured, a plug-in
 * whose host framework owns every device allocation and offers no workspace,
 * or a latency-critical decode loop that may not call cudaMalloc.  The pages
 * have no counterpart: it is an interface convenience of this library.
 *
 * The caller passes inputs and outputs as in swiglu_mlp_fwd_nograd; there is
 * no workspace argument.  Scratch (error word, per-tile counters, fp32
 * partial sums) lives in one file-scope static device array of 16 MiB, which
 * every GPU that loads this library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *
 * Limits: bf16/fp16 only, 0 <= M <= 64, D and H multiples of 8, and the
 * partial sums of the call must fit the array (on a 152-SM GB300 the fused
 * kernel's fit for M <= 32 and the two-kernel form's for every M <= 64, at
 * any D and H: each CTA holds at most two partial tiles per GEMM); anything
 * beyond returns SWIGLU_ERR_UNSUPPORTED without launching.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  Every call clears the error word
 * and counters in the array (an asynchronous memset, no allocation) and then
 * launches the kernels (one fused kernel or two).  All calls share the one array: calls that
 * overlap on the GPU (other streams, other threads) race and give undefined
 * results.  Device errors are not reported through a workspace; use
 * swiglu_mlp_fwd_nograd when they must be queried. */
swiglu_status swiglu_mlp_fwd_nograd_noalloc(const void* X, const void* Wgu, const void* Wd,
                                            void* Y, void* A, int64_t M, int64_t D, int64_t H,
                                            swiglu_dtype dtype, void* stream);

/* A no-grad forward captured once into a CUDA graph and replayed per call,
 * for decode loops ("Inference results": the fixed host cost of building
 * descriptors per call dominates at small shapes, and CUDA graphs are the
 * remedy the page names but did not validate).
 *
 * swiglu_mlp_graph_create_fwd_nograd validates its arguments exactly as
 * swiglu_mlp_fwd_nograd does, then records that call -- its workspace clear,
 * tensor maps and kernel launches, with every pointer and size fixed -- by
 * stream capture on a stream of its own, and instantiates the graph for the
 * current device.  Nothing runs on the GPU during create.  Each
 * swiglu_mlp_graph_launch(graph, stream) then performs the same computation
 * on the buffers given at create time: write the new tokens into X, launch,
 * read Y (and A) after the launch on ``stream`` completes.  Results are
 * bitwise equal to swiglu_mlp_fwd_nograd on the same inputs.
 *
 * Ownership: the caller keeps X, Wgu, Wd, Y, A and ws alive and unmoved for
 * the life of the graph; ``ws`` follows the workspace rules above (zero-filled
 * before first use; launches sharing it must not overlap on the GPU).  The
 * graph object (host memory plus what the CUDA runtime holds for an
 * instantiated graph) belongs to the library until
 * swiglu_mlp_graph_destroy(graph); launches still pending then complete, and
 * the runtime releases the graph after them (the caller's buffers must
 * outlive those launches).  Create must not itself be called during a stream capture, nor
 * while per-kernel profiling is enabled (SWIGLU_ERR_UNSUPPORTED).  M = 0
 * yields a graph whose launch does nothing.  Errors: the argument statuses of
 * swiglu_mlp_fwd_nograd; SWIGLU_ERR_INVALID_ARG for a NULL ``graph`` /
 * ``out``; SWIGLU_ERR_CUDA when capture, instantiation or launch fails. */
typedef struct swiglu_mlp_graph swiglu_mlp_graph;
swiglu_status swiglu_mlp_graph_create_fwd_nograd(const void* X, const void* Wgu, const void* Wd,
                                                 void* Y, void* A, int64_t M, int64_t D,
                                                 int64_t H, swiglu_dtype dtype, void* ws,
                                                 size_t ws_bytes, swiglu_mlp_graph** out);
swiglu_status swiglu_mlp_graph_launch(swiglu_mlp_graph* graph, void* stream);
swiglu_status swiglu_mlp_graph_destroy(swiglu_mlp_graph* graph);

/* Backward.  Consumes ``saved`` as written by swiglu_mlp_fwd on the same
 * X, Wgu, Wd: once G and U have been read they are no longer needed, and dG,
 * dU are written over them in place (Summary; Known limitations: for that
 * reason the graph cannot be retained and a second backward on the same
 * buffer is not possible -- a second call on the same ``saved`` gives
 * undefined values).
 *   dA = dY Wd is never stored: dU = dA * SiLU(G), dG = dA * U * SiLU'(G)
 *   with SiLU'(g) = s (1 + g (1 - s)), s = 1 / (1 + e^-g), G, U the stored
 *   values;
 *   dWd = dY^T A;  [dWg; dWu] = [dG | dU]^T X as one GEMM over the
 *   concatenated [dG | dU] (Summary: the two weight gradients are computed
 *   together);  dX = [dG | dU] [Wg; Wu], both halves summed in one fp32
 *   accumulator over K = 2H (Summary: the input gradient in one kernel).
 * Gradients are written, not accumulated (beta = 0).  Writes dX [M,D],
 * dWgu [2H,D], dWd [D,H]; rewrites columns [0, 2H) of ``saved``. */
swiglu_status swiglu_mlp_bwd(const void* dY, const void* X, const void* Wgu, const void* Wd,
                             void* saved, void* dX, void* dWgu, void* dWd, int64_t M, int64_t D,
                             int64_t H, swiglu_dtype dtype, void* ws, size_t ws_bytes,
                             void* stream);

/* Options of the _ex entry points.  NULL options (or the base entry points)
 * mean {1, 1, 0}: the standard MLP, gradients overwritten.
 *
 * gate_multiplier mg, down_multiplier md: the gate/down multiplier variant
 * that the maintainer thread of the RFC defers to a follow-up (Falcon-H1;
 * the pages do not define it -- this library takes the plain reading)
 *     A = SiLU(mg * X Wg^T) * (X Wu^T),   Y = md * (A Wd^T),
 * the stored G being the pre-activation mg * X Wg^T; backward follows the
 * chain rule: dA = md * (dY Wd), dU = dA * SiLU(G), dG = dA * U * SiLU'(G)
 * * mg, dWd = md * (dY^T A), dWg = dG^T X, dWu = dU^T X, dX = dG Wg + dU Wu.
 * Both multipliers must be finite.
 *
 * accumulate (backward only; must be 0 for the forward calls): 1 adds the
 * new weight gradients to the values already in dWgu and dWd (beta = 1,
 * gradient accumulation over micro-batches), with one rounding of the fp32
 * sum per element; dX is always overwritten. */
typedef struct {
  float gate_multiplier;
  float down_multiplier;
  int accumulate;
} swiglu_mlp_options;

swiglu_status swiglu_mlp_fwd_ex(const void* X, const void* Wgu, const void* Wd, void* Y,
                                void* saved, int64_t M, int64_t D, int64_t H,
                                swiglu_dtype dtype, const swiglu_mlp_options* options,
                                void* ws, size_t ws_bytes, void* stream);
swiglu_status swiglu_mlp_fwd_nograd_ex(const void* X, const void* Wgu, const void* Wd, void* Y,
                                       void* A, int64_t M, int64_t D, int64_t H,
                                       swiglu_dtype dtype, const swiglu_mlp_options* options,
                                       void* ws, size_t ws_bytes, void* stream);

/* Bytes of the packed copy of a layer's weights that
 * swiglu_mlp_pack_weights writes: ceil(H/64) * ceil(D/64) + ceil(D/128) *
 * ceil(H/64) blocks of 16 KB (about the size of Wgu and Wd together).  0 for
 * invalid sizes or a dtype other than bf16/fp16. */
size_t swiglu_mlp_packed_weights_bytes(int64_t D, int64_t H, swiglu_dtype dtype);

/* Writes a packed copy of Wgu [2H,D] and Wd [D,H] (bf16 or fp16) to
 * `packed` (device, 16-byte aligned, swiglu_mlp_packed_weights_bytes bytes)
 * for swiglu_mlp_fwd_nograd_packed.  The few-token no-grad kernels stream
 * each weight matrix as 16 KB blocks of 128 rows x 64 elements of K; the
 * packed copy stores each block contiguously, in the order the kernels
 * consume them and already in the 128-byte swizzled form they load into
 * shared memory, so each CTA reads one contiguous range (measured on GB300:
 * ~6.3 TB/s for contiguous 16 KB bulk copies against ~5.8 TB/s for the same
 * bytes as 128-byte rows of the row-major matrices).  The pages have no
 * counterpart: it is an inference-side layout option of this library.
 * Layout: the gate/up blocks, then the down blocks.  Gate/up block (t, kb)
 * at (t * ceil(D/64) + kb) * 16 KB: rows 0..63 are Wg rows t*64.., rows
 * 64..127 the Wu rows of the same hidden units, elements kb*64.. of K; down
 * block (t, kb) at gate/up bytes + (t * ceil(H/64) + kb) * 16 KB: Wd rows
 * t*128.., elements kb*64.. of K.  Within a block, the 16-byte chunk c of row
 * r is at r*128 + (c ^ (r mod 8))*16; elements past D or H are zero.  One
 * kernel on `stream`; D and H multiples of 8.  Rewrite the copy whenever the
 * weights change: the packed forward never reads Wgu or Wd. */
swiglu_status swiglu_mlp_pack_weights(const void* Wgu, const void* Wd, void* packed, int64_t D,
                                      int64_t H, swiglu_dtype dtype, void* stream);

/* swiglu_mlp_fwd_nograd (with options as swiglu_mlp_fwd_nograd_ex: the gate
 * and down multipliers) for 0 <= M <= 64 tokens, reading the weights from a
 * copy written by swiglu_mlp_pack_weights instead of Wgu / Wd.  Runs the
 * two-kernel few-token form; its outputs are bitwise equal to
 * swiglu_mlp_fwd_nograd's two-kernel form on the same weights (the kernels
 * see the same shared-memory contents).  M > 64 and fp32 return
 * SWIGLU_ERR_UNSUPPORTED (keep the row-major weights for larger batches);
 * the workspace is that of swiglu_mlp_fwd_nograd. */
swiglu_status swiglu_mlp_fwd_nograd_packed(const void* X, const void* packed, void* Y, void* A,
                                           int64_t M, int64_t D, int64_t H, swiglu_dtype dtype,
                                           const swiglu_mlp_options* options, void* ws,
                                           size_t ws_bytes, void* stream);

swiglu_status swiglu_mlp_bwd_ex(const void* dY, const void* X, const void* Wgu, const void* Wd,
                                void* saved, void* dX, void* dWgu, void* dWd, int64_t M,
                                int64_t D, int64_t H, swiglu_dtype dtype,
                                const swiglu_mlp_options* options, void* ws, size_t ws_bytes,
                                void* stream);

/* Synchronises ``stream`` and reads the device error word in ``ws``:
 * SWIGLU_OK, SWIGLU_ERR_DEVICE_TIMEOUT, SWIGLU_ERR_DEVICE_BOUNDS (debug
 * builds), or SWIGLU_ERR_CUDA if the stream reported an error. */
swiglu_status swiglu_mlp_query_error(const void* ws, void* stream);

/* 1 if this library was compiled as the debug build (-DSWIGLU_DEBUG, shipped
 * as libswiglu_mlp_debug.so), else 0.  In the debug build every plain
 * (non-TMA) global load and store of every kernel -- epilogue outputs, the
 * dG/dU epilogue's reads of G and U, stream-K partial tiles, tile counters,
 * the few-token queue and ready mask, the fp32 path's operands -- is checked
 * against the buffers that launch was given (the caller's tensors and the
 * workspace, with their sizes) and its table indices against their bounds.
 * A failed check skips the access and records SWIGLU_ERR_DEVICE_BOUNDS in the
 * workspace error word (read by swiglu_mlp_query_error); the kernel runs to
 * its end, nothing traps.  Same API, same results; slower. */
int swiglu_mlp_debug_build(void);

/* Test hook for the debug build's checks: when ``on`` is nonzero, the next
 * launch of this process gets its output buffer's window halved, so the
 * kernel's accesses to the buffer's second half fail their check, are
 * skipped, and SWIGLU_ERR_DEVICE_BOUNDS is recorded.  No access leaves the
 * caller's buffers.  The flag clears itself after one launch.  Outputs of
 * that call are undefined; the workspace stays valid.  In the release build
 * the flag has no effect. */
void swiglu_mlp_debug_narrow_once(int on);

/* Static description of a status code. */
const char* swiglu_status_string(swiglu_status status);

/* Limit, in nanoseconds, on every device-side pipeline wait of later calls
 * from this process (default 2e9 = 2 s; values below 1000 are raised to
 * 1000).  Returns the previous limit. */
uint64_t swiglu_mlp_set_wait_limit_ns(uint64_t ns);

/* Test hook for failure detection: when ``on`` = n > 0, the n-th
 * tensor-core launch of this process from now (1: the next) makes its load
 * producer skip the arrival of the first pipeline stage (or, in the fused
 * few-token no-grad kernel, leaves the first gate/up tile's ready bit clear),
 * so a consumer's wait runs out, the kernel records SWIGLU_ERR_DEVICE_TIMEOUT
 * and returns cleanly.  Training launches come in the order gate/up, down
 * (forward) and dWd, dG/dU, dWgu, dX (backward).  The hook clears itself at
 * that launch; on <= 0 clears it.  Outputs of that call are undefined. */
void swiglu_mlp_inject_stall_once(int on);

/* Selects how later calls of this process run their bf16/fp16 tensor-core
 * GEMMs: on pairs of SMs -- 2-CTA clusters issuing tcgen05.mma.cta_group::2
 * on 256 x 256 tiles, each SM loading half of each operand tile -- or on
 * single SMs (128 x 256 tiles).  mode 1 (the default): pairs for the GEMMs
 * with enough 256 x 256 tiles to give every pair one, K >= 1024 and rows
 * that 256-row tiles cover without more padding than 128-row ones, or with
 * K >= 16384; 2: pairs for every GEMM; 0: never.  All modes give
 * results within the same tolerances (accumulation order differs).  Returns
 * the previous mode.  A workspace sized by swiglu_mlp_workspace_bytes() fits
 * every mode. */
int swiglu_mlp_set_cta_pairs(int mode);

/* Selects the tile width of later training calls' weight-gradient and dX
 * GEMMs (dWd, dWgu, dX) and of the down projection when they run on SM
 * pairs.  256 x 256 tiles use two
 * TMEM accumulators, so that a tile's epilogue overlaps the next tile's
 * main loop; 256 x 512 tiles use one accumulator of all 512 TMEM columns,
 * each A k-block feeding twice the columns (half the B-panel reads per
 * FLOP).  mode 1 (the default): 512 columns where the contraction is at
 * least 16384 and every pair gets two whole tiles or more (measured 3.4%
 * faster per training step at B=8 S=8192 D=4096 H=11008), else 256; 0: 256
 * always; 2: 512 always.  All are deterministic and within the same
 * tolerances (their stream-K splits differ).  A workspace sized by
 * swiglu_mlp_workspace_bytes() fits every mode.  Returns the previous
 * mode. */
int swiglu_mlp_set_wide_tiles(int mode);

/* Selects how later few-token no-grad calls (M <= 64, bf16/fp16) of this
 * process run: as ONE persistent kernel that hands out fixed work units (a
 * gate/up or down tile x a run of k-blocks) from a queue in the workspace,
 * so faster SMs take more of the weight stream, and that starts each
 * down-projection k-block as soon as the A columns it reads are written (a
 * ready mask in the workspace); or as two kernels (gate/up, then the down
 * projection as a programmatic dependent launch).  mode 0 (the default):
 * always two kernels, measured faster at every size from 1 to 64 tokens
 * (62-63 vs 65-68 us at 1-16 tokens, 72-83 vs 87-89 us at 33-64, D = 4096,
 * H = 11008; the two kernels also take a 48-token block, the fused kernel
 * 16, 32 or 64); 1: the fused kernel for 33..64 tokens, two kernels below; 2:
 * always the fused kernel.  Both forms are
 * deterministic (partial sums are added in a fixed order); they split the
 * contractions at different points, so their results differ in rounding
 * only.  A workspace sized by swiglu_mlp_workspace_bytes() fits both.
 * Returns the previous mode. */
int swiglu_mlp_set_nograd_fused(int mode);

/* Number of kernels the last fwd / fwd_nograd / bwd call launched on the
 * device (for launch accounting in benchmarks). */
int swiglu_mlp_last_launch_count(void);

/* Per-kernel device timing for benchmarks.  While enabled, every kernel
 * launch is bracketed by two CUDA events recorded on its stream (do not
 * enable it during CUDA-graph stream capture).  swiglu_mlp_profile_read waits
 * for the recorded events, writes, for kernel ids 0 .. n-1, the number of
 * launches and their summed device time in milliseconds since the previous
 * read (either array may be NULL), resets the counters, and returns the
 * number of kernel ids (-1 if an event could not be read). */
void swiglu_mlp_profile_enable(int on);
int swiglu_mlp_profile_read(int n, int64_t* launches, double* total_ms);

/* Name of a kernel id (NULL outside 0 .. count-1). */
const char* swiglu_mlp_kernel_name(int id);

/* Test hook: the elementwise SwiGLU stage of the tensor-core epilogues,
 * applied by the same device functions to n caller-chosen values, so that
 * its fp32 arithmetic can be checked value by value ("Scope one-round FP32
 * SwiGLU to the exact Qwen3.5 contract", xorl PR #51, review section: SiLU
 * and the product in fp32, one rounding; "[RFC] Full-pipeline SwiGLU MLP
 * with forward/backward co-optimization", Liger-Kernel #1347, "Summary":
 * dG and dU from dA in registers).  dtype: SWIGLU_BF16 or SWIGLU_F16.
 *   Forward, when acc_g is not NULL: acc_g, acc_u are fp32 [n] (the gate
 *   and up accumulators); with g = gate_multiplier * acc_g it writes
 *   A = rnd(SiLU(g) acc_u), G = rnd(g), U = rnd(acc_u) ([n] each, dtype).
 *   Backward, when dA is not NULL: dA is fp32 [n] (the dY Wd accumulator),
 *   gs, us are the stored G, U ([n], dtype); it writes
 *   dU = rnd(down_multiplier dA SiLU(gs)) and
 *   dG = rnd(down_multiplier dA us SiLU'(gs) gate_multiplier) ([n], dtype).
 * All pointers are device pointers, 16-byte aligned; outputs of the unused
 * direction may be NULL.  n must be a multiple of 32 (the epilogue's
 * chunk), 0 <= n < 2^31.  Asynchronous on ``stream``.  Errors:
 * SWIGLU_ERR_INVALID_ARG (bad dtype, n, NULL input/output of a requested
 * direction, or neither direction), SWIGLU_ERR_ALIGNMENT, SWIGLU_ERR_CUDA. */
swiglu_status swiglu_mlp_test_elementwise(swiglu_dtype dtype, int64_t n, const float* acc_g,
                                          const float* acc_u, void* A, void* G, void* U,
                                          const float* dA, const void* gs, const void* us,
                                          void* dG, void* dU, float gate_multiplier,
                                          float down_multiplier, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_MLP_H */
