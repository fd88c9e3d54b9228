// ng_fused.cuh -- the few-token no-grad forward as ONE persistent kernel
// with a dynamic, deterministic work queue.
//
// Both GEMMs are cut into fixed work units:
//   gate/up: tile t (64 hidden units: Wg and Wu rows) x chunk c, a run of
//            k-blocks over D; unit u = t * chunks0 + c (tile-major);
//   down:    tile t (128 output features of Wd) x chunk c, a run of k-blocks
//            over H (shorter runs at the end); unit units0 + c * tiles1 + t
//            (chunk-major).
// Each CTA's producer takes the next unit id from a global counter shortly
// before it finishes issuing the current unit's loads, and hands it to the
// MMA warp and the epilogue through a small queue in shared memory.  Fast SMs therefore take
// more units, and the whole weight stream (gate/up, then the down
// projection) ends at nearly the same time on every SM -- a static split
// leaves the slowest SMs streaming for several microseconds after the rest.
//
// Results do not depend on which SM ran what: a unit's fp32 partial tile
// goes to the workspace slot of that unit, and the tile's last unit to finish
// (per-tile arrival counter) sums the tile's chunks in chunk order and writes
// the output (A = rnd(SiLU(g) * u), or Y = rnd(y)).  A tile of a single chunk
// writes its output straight from TMEM.
//
// The down projection's chunk c reads the A columns of gate/up tiles
// [c * q1, (c + 1) * q1) (one k-block of 64 hidden units per gate/up tile).
// Whoever writes a gate/up tile's A columns sets its bit in a ready mask
// (release OR after a proxy fence); a producer loads a down unit's Wd
// k-blocks at once and issues each activation load once its bit is set,
// keeping the last mask word it read so one L2 round trip clears up to 32
// k-blocks.  Gate/up units precede all down units in the queue and never
// wait for anything, and only running CTAs hold units, so every bit a
// producer waits for is eventually set -- no co-residency is needed.  Down
// units are chunk-major, so the first ones read the A columns written first.
// The last CTA to finish resets the queue counter and the mask for the next
// call.  Every wait is bounded (wait_limit_ns) and ends the kernel cleanly
// with DEV_ERR_TIMEOUT.
#pragma once

#include "ng_gemm.cuh"

namespace swiglu {

constexpr int NG_MAX_CHUNKS = 64;  // k-block runs per tile, per GEMM

struct NgDynArgs {
  NgArgs ph[2];        // gate/up (out = A) and down (out = Y): M, rows, kb_tile, tiles,
                       //   part (one slot per unit), counters, out, ld_out
  int chunks[2];       // units per tile
  // chunk c of GEMM g covers k-blocks [kb_at[g][c], kb_at[g][c + 1]); the down
  // projection's last chunks are shorter, so the last units to be handed
  // out finish at nearly the same time
  int kb_at[2][NG_MAX_CHUNKS + 1];
  int units0, units;   // gate/up units; all units
  uint32_t* ready;     // mask over gate/up tiles: bit t set once tile t's A columns are written
  uint32_t* next_unit; // the queue: next unit id to hand out
  uint32_t* done;      // CTAs finished; the last one resets next_unit, done and ready
  int inject_unready;  // test hook: tile 0's bit is never set, so the waits on it run out
};

// Weight ring of the fused kernel, per SM: 200 KB measured 2 us faster than
// 110 KB at 16-64 tokens (the two-kernel form does best with 110 KB).
constexpr int NG_FUSED_RING_KB = 200;

// The two-kernel form's ring layout (with the fused kernel's ring size) and
// staging, plus the unit queue and four TMEM accumulators (the MMA warp may
// run up to three units ahead of the epilogue, whose per-unit work includes
// a few L2 round trips).
template <int NT>
struct NgDynSmem {
  using B = NgSmem<NT, NG_FUSED_RING_KB>;
  static constexpr int UQ = 8;                    // unit queue entries
  static constexpr int NACC = 4;                  // TMEM accumulators
  static constexpr int UQ_BAR_OFFSET = B::TOTAL;  // uq_full[UQ], uq_empty[UQ]
  static constexpr int ACC_BAR_OFFSET = UQ_BAR_OFFSET + 2 * UQ * 8;  // accf[NACC], acce[NACC]
  static constexpr int UQ_ID_OFFSET = ACC_BAR_OFFSET + 2 * NACC * 8;
  static constexpr int TOTAL = UQ_ID_OFFSET + UQ * 4;
  static constexpr int DYN_BYTES = TOTAL + 1024;
  static constexpr int TMEM_COLS = NACC * NT < 32 ? 32 : NACC * NT;
};

// A unit's GEMM, tile and k-blocks.
struct NgUnit {
  int ph, tile, chunk, kb0, nkb;
};

__device__ __forceinline__ NgUnit ng_decode(const NgDynArgs& f, uint32_t u) {
  NgUnit w;
  if ((int)u < f.units0) {
    w.ph = 0;
    w.tile = (int)u / f.chunks[0];
    w.chunk = (int)u - w.tile * f.chunks[0];
  } else {
    const int v = (int)u - f.units0;
    w.ph = 1;
    w.chunk = v / f.ph[1].tiles;
    w.tile = v - w.chunk * f.ph[1].tiles;
  }
  if (!SWIGLU_CHECK(w.chunk < f.chunks[w.ph] && f.chunks[w.ph] <= NG_MAX_CHUNKS, f.ph[0].err))
    w.chunk = 0;
  w.kb0 = f.kb_at[w.ph][w.chunk];
  w.nkb = f.kb_at[w.ph][w.chunk + 1] - w.kb0;
  return w;
}

template <int NT, bool BF16>
__global__ void __launch_bounds__(NG_THREADS, 1)
    ng_fused_kernel(const __grid_constant__ CUtensorMap tmWgu,
                    const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmWd,
                    const __grid_constant__ CUtensorMap tmA, const NgDynArgs f) {
  using L = NgSmem<NT, NG_FUSED_RING_KB>;
  using Q = NgDynSmem<NT>;
  static_assert(NT == 16 || NT == 32 || NT == 64, "NT must be 16, 32 or 64");
  static_assert(Q::TOTAL + 1024 <= 232448, "shared memory plan exceeds 227 KB");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFFSET;
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (L::STAGES + i); };
  auto accf_bar = [&](int i) { return sbase + Q::ACC_BAR_OFFSET + 8u * i; };
  auto acce_bar = [&](int i) { return sbase + Q::ACC_BAR_OFFSET + 8u * (Q::NACC + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * L::STAGES + 4);
  auto uq_full = [&](int i) { return sbase + Q::UQ_BAR_OFFSET + 8u * i; };
  auto uq_empty = [&](int i) { return sbase + Q::UQ_BAR_OFFSET + 8u * (Q::UQ + i); };
  volatile uint32_t* uq_id = reinterpret_cast<volatile uint32_t*>(smem + Q::UQ_ID_OFFSET);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFFSET);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFFSET + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wl = f.ph[0].wait_limit_ns;
  int* const err = f.ph[0].err;
  const uint32_t units = (uint32_t)f.units;

  if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < Q::NACC; ++i) {
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), 128);
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < Q::UQ; ++i) {
      mbar_init(uq_full(i), 1);
      mbar_init(uq_empty(i), 5);  // the MMA warp and the four epilogue warps
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmWgu);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmWd);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Q::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int qs = 0;
      uint32_t qph = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      // activation loads of down units waiting for their ready bits (ring order)
      int q_stage[L::STAGES] = {}, q_kb[L::STAGES] = {};
      int q_head = 0, q_n = 0;
      uint32_t mask_word = 0;  // last ready-mask word read, and its index
      int mask_idx = -1;
      auto issue_front = [&]() {
        const int s = q_stage[q_head];
        tma_load_2d(sbase + s * L::STAGE_BYTES + L::W_BYTES, &tmA, full_bar(s),
                    q_kb[q_head] * TC_BK, 0);
        if (++q_head == L::STAGES) q_head = 0;
        --q_n;
      };
      // Issues the queued activation loads whose bits are set until barrier
      // `bar` completes phase `par` (with room in the queue if need_room), or,
      // for bar == 0, until the queue is empty; false on timeout or abort.
      // The ring slot a down unit reuses is the oldest: while the queue is not
      // full it is not queued, so the MMA warp can always free it.
      auto pump = [&](uint32_t bar, uint32_t par, bool need_room) -> bool {
        uint64_t t0 = global_timer_ns();
        for (uint32_t n = 1;; ++n) {
          if (q_n > 0) {
            const int kb = q_kb[q_head];
            const uint32_t bit = 1u << (kb & 31);
            bool ready = mask_idx == (kb >> 5) && (mask_word & bit) != 0u;
            if (!ready) {
              // a k-block outside the mask (debug check) counts as ready: no wait on it
              mask_word = SWIGLU_CHECK(kb >= 0 && kb < f.ph[0].tiles, err)
                              ? ld_acquire_gpu(f.ready + (kb >> 5))
                              : ~0u;
              mask_idx = kb >> 5;
              ready = (mask_word & bit) != 0u;
              // order the acquired A columns before this thread's TMA reads
              if (ready) fence_proxy_async_global();
            }
            if (ready) {
              issue_front();
              t0 = global_timer_ns();
              continue;
            }
          }
          if (bar == 0u ? q_n == 0
                        : ((!need_room || q_n < L::STAGES) && mbar_test_wait(bar, par)))
            return true;
          if ((n & 255u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > wl) {
              atomicCAS(err, DEV_ERR_NONE, DEV_ERR_TIMEOUT);
              *abort_flag = 1;
              return false;
            }
          }
        }
      };
      uint32_t next = atomicAdd(f.next_unit, 1u);
      for (;;) {
        const uint32_t u = next;
        // hand the unit (or the end mark, u >= units) to the MMA warp and the epilogue
        if (!pump(uq_empty(qs), qph ^ 1u, false)) {
          ok = false;
          break;
        }
        uq_id[qs] = u;
        mbar_arrive(uq_full(qs));
        if (++qs == Q::UQ) {
          qs = 0;
          qph ^= 1u;
        }
        if (u >= units) break;
        const NgUnit w = ng_decode(f, u);
        for (int i = 0; i < w.nkb; ++i) {
          // take the next unit two k-blocks before this one's last load: the
          // counter's round trip is hidden, and a CTA commits to new work
          // only when it is about to start it
          if (i == (w.nkb > 2 ? w.nkb - 2 : 0)) next = atomicAdd(f.next_unit, 1u);
          if (!pump(empty_bar(stage), phase ^ 1u, w.ph == 1)) {
            ok = false;
            break;
          }
          const uint32_t sw = sbase + stage * L::STAGE_BYTES;
          const int kb = w.kb0 + i;
          mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
          if (w.ph == 0) {
            tma_load_3d(sw, &tmWgu, full_bar(stage), kb * TC_BK, w.tile * 64, 0);
            tma_load_2d(sw + L::W_BYTES, &tmX, full_bar(stage), kb * TC_BK, 0);
          } else {
            tma_load_2d(sw, &tmWd, full_bar(stage), kb * TC_BK, w.tile * 128);
            int qt = q_head + q_n;
            if (qt >= L::STAGES) qt -= L::STAGES;
            q_stage[qt] = stage;
            q_kb[qt] = kb;
            ++q_n;
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == L::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (ok) ok = pump(0u, 0u, false);
      if (!ok) {
        // Complete every slot's transaction -- the activation loads still
        // queued read in-bounds A whatever its state -- then wait for all
        // copies in flight before the CTA may exit.
        while (q_n > 0) issue_front();
        for (int i = 0; i < L::STAGES; ++i)
          if (issued_mask & (1u << i))
            mbar_wait_bounded(full_bar(i), (issued_parity >> i) & 1u, wl, nullptr, err);
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
      int qs = 0;
      uint32_t qph = 0;
      bool ok = true;
      for (;;) {
        if (!mbar_wait_bounded(uq_full(qs), qph, wl, abort_flag, err)) break;
        const uint32_t u = uq_id[qs];
        mbar_arrive(uq_empty(qs));
        if (++qs == Q::UQ) {
          qs = 0;
          qph ^= 1u;
        }
        if (u >= units) break;
        const NgUnit w = ng_decode(f, u);
        if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, wl, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * NT;
        for (int i = 0; i < w.nkb; ++i) {
          if (!mbar_wait_bounded(full_bar(stage), phase, wl, abort_flag, err)) {
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
        if (++acc == Q::NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, wl, nullptr, err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = threadIdx.x - 64;  // 0..127 among the epilogue threads
    int acc = 0;
    uint32_t acc_phase = 0;
    int qs = 0;
    uint32_t qph = 0;
    float* ustage = reinterpret_cast<float*>(smem + L::USTAGE_OFFSET);
    for (;;) {
      int ok = 1;
      uint32_t u = 0;
      if (lane == 0) {
        ok = mbar_wait_bounded(uq_full(qs), qph, wl, abort_flag, err) ? 1 : 0;
        if (ok) {
          u = uq_id[qs];
          mbar_arrive(uq_empty(qs));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!epi_bar_and(ok)) break;  // all four epilogue warps leave together
      if (++qs == Q::UQ) {
        qs = 0;
        qph ^= 1u;
      }
      if (u >= units) break;
      const NgUnit w = ng_decode(f, u);
      if (lane == 0)
        ok = mbar_wait_bounded(accf_bar(acc), acc_phase, wl, abort_flag, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!epi_bar_and(ok)) break;
      const uint32_t tacc = tmem_base + acc * NT;
      const NgArgs& a = f.ph[w.ph];
      const int chunks = f.chunks[w.ph];
      bool wrote = true;
      if (chunks == 1) {
        if (w.ph == 0)
          ng_store_whole<NT, true, BF16>(a, w.tile, tacc, acce_bar(acc), ustage);
        else
          ng_store_whole<NT, false, BF16>(a, w.tile, tacc, acce_bar(acc), ustage);
      } else {
        // the slot of chunk c of this unit's tile
        const int tiles = a.tiles;
        const int ph = w.ph, tile = w.tile;
        auto slot = [&](int c) -> float* {
          const int s = ph == 0 ? tile * chunks + c : c * tiles + tile;
          return SWIGLU_CHECK(s >= 0 && s < tiles * chunks, err) ? a.part + (size_t)s * 128 * NT
                                                                  : nullptr;
        };
        float* const dst = slot(w.chunk);
        ng_store_partial<NT>(dst, tacc, acce_bar(acc),
                             SWIGLU_CHECK_PTR(a.dbg, dst, 128 * NT * 4, err));
        epi_bar_sync();
        if (e == 0) {
          int last = 0;
          __threadfence();  // the 128 threads' partial stores before the count
          if (!*abort_flag)
            last = SWIGLU_CHECK(tile < tiles, err) && atomicAdd(a.counters + tile, 1) == chunks - 1;
          *last_flag = last;
        }
        epi_bar_sync();
        wrote = *last_flag != 0;
        if (wrote) {
          __threadfence();
          auto part_of = [&](int c) -> const float* { return slot(c); };
          if (ph == 0)
            ng_reduce_store<NT, true, BF16>(a, tile, chunks, part_of);
          else
            ng_reduce_store<NT, false, BF16>(a, tile, chunks, part_of);
          if (e == 0 && SWIGLU_CHECK(tile < tiles, err)) a.counters[tile] = 0;  // next call
        }
      }
      if (w.ph == 0 && wrote) {
        // publish the tile's A columns to every CTA's down-unit TMA loads
        fence_proxy_async_global();
        epi_bar_sync();
        if (e == 0 && !(f.inject_unready && w.tile == 0) &&
            SWIGLU_CHECK(w.tile < f.ph[0].tiles, err)) {
          __threadfence();
          red_or_release_gpu(f.ready + (w.tile >> 5), 1u << (w.tile & 31));
        }
      }
      if (++acc == Q::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // every role of this CTA is done with the queue and the mask; the grid's
    // last CTA resets them for the next call
    uint32_t last = 0;
    if (lane == 0) {
      __threadfence();
      last = atomicAdd(f.done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      for (int j = lane; j < (f.ph[0].tiles + 31) / 32; j += 32) f.ready[j] = 0u;
      if (lane == 0) {
        *f.next_unit = 0u;
        *f.done = 0u;
      }
    }
  } else if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Q::TMEM_COLS);
  }
}

}  // namespace swiglu
