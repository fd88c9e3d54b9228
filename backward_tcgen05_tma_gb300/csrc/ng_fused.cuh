// ng_fused.cuh -- the few-token no-grad forward as ONE persistent kernel.
//
// The two-kernel form (ng_gemm.cuh) pays for two launches and two pipeline
// start-ups, and between them for the drain of the gate/up kernel, whose last
// reductions run while no weight bytes stream.  Here a single cooperative
// launch (every CTA resident at once, one per SM) runs both phases back to
// back on the same TMA ring, TMEM accumulators and epilogue warps:
//   phase 0: gate/up tiles of 64 hidden units -> A [M, H]
//   phase 1: down tiles of 128 output features -> Y [M, D]
// each split over the CTAs exactly as the two-kernel form splits it
// (stream-K hybrid, deterministic CTA-order reductions).
//
// Phase 1's k-block j (hidden units 64j .. 64j+63) reads exactly the A
// columns that phase 0's tile j writes.  The CTA that writes them (the
// tile's owner, or the last contributor of a shared tile) sets bit j of a
// ready mask in the workspace (one 32-bit word per 32 tiles, set with a
// release OR after a proxy fence).  A phase-1 producer loads its Wd k-blocks
// into the ring without waiting and issues a k-block's activation load only
// once its bit is set; it keeps the last mask word it read, so one L2 round
// trip clears up to 32 k-blocks (one acquire per k-block would cost about
// 0.6 us each, serialised in the producer).  Nothing in phase 0 waits for
// another CTA, so every bit is eventually set as long as all CTAs are
// resident, which the cooperative launch guarantees.  The last CTA to finish
// clears the mask for the next call.  Every wait is bounded (wait_limit_ns)
// and ends the kernel cleanly with DEV_ERR_TIMEOUT.
#pragma once

#include "ng_gemm.cuh"

namespace swiglu {

struct NgFusedArgs {
  NgArgs ph[2];     // phase 0: gate/up (out = A), phase 1: down (out = Y)
  uint32_t* ready;  // mask over phase 0's tiles: bit j set once tile j's A columns are written
  uint32_t* done;   // CTAs finished in this call; the last one resets it and ready
  int inject_unready;  // test hook: tile 0's flag is never raised, so the waits on it run out
};

template <int NT, bool BF16>
__global__ void __launch_bounds__(NG_THREADS, 1)
    ng_fused_kernel(const __grid_constant__ CUtensorMap tmWgu,
                    const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmWd,
                    const __grid_constant__ CUtensorMap tmA, const NgFusedArgs f) {
  using L = NgSmem<NT>;
  static_assert(NT == 16 || NT == 32 || NT == 64, "NT must be 16, 32 or 64");
  static_assert(L::TOTAL + 1024 <= 232448, "shared memory plan exceeds 227 KB");

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
  const NgArgs& a0 = f.ph[0];
  const NgArgs& a1 = f.ph[1];
  const uint64_t wl = a0.wait_limit_ns;
  int* const err = a0.err;

  if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0;
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
    tma_prefetch_desc(&tmWgu);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmWd);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Each phase's split: CTAs [0, ctas) share it; the rest sit the phase out.
  const int cta = blockIdx.x;
  const int64_t total0 = (int64_t)a0.sk_tiles * a0.kb_tile;
  const int64_t total1 = (int64_t)a1.sk_tiles * a1.kb_tile;
  auto segs0 = [&]() {
    const bool in = cta < a0.ctas;
    return NgSegIter{in ? ng_start(cta, total0, a0.ctas) : 0,
                     in ? ng_start(cta + 1, total0, a0.ctas) : 0, 0,
                     in ? (a0.tiles - a0.sk_tiles) / a0.ctas : 0, a0.kb_tile, a0.sk_tiles, cta,
                     a0.ctas};
  };
  auto segs1 = [&]() {
    const bool in = cta < a1.ctas;
    return NgSegIter{in ? ng_start(cta, total1, a1.ctas) : 0,
                     in ? ng_start(cta + 1, total1, a1.ctas) : 0, 0,
                     in ? (a1.tiles - a1.sk_tiles) / a1.ctas : 0, a1.kb_tile, a1.sk_tiles, cta,
                     a1.ctas};
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      auto advance = [&]() {
        if (++stage == L::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      };
      // phase 0: weights and tokens, nothing to wait for but ring slots
      {
        NgSegIter it = segs0();
        int tile, kb0, nkb;
        bool whole;
        while (ok && it.next(tile, kb0, nkb, whole)) {
          for (int i = 0; i < nkb; ++i) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, wl, abort_flag, err)) {
              ok = false;
              break;
            }
            const uint32_t sw = sbase + stage * L::STAGE_BYTES;
            const int k0 = (kb0 + i) * TC_BK;
            mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
            tma_load_3d(sw, &tmWgu, full_bar(stage), k0, tile * 64, 0);
            tma_load_2d(sw + L::W_BYTES, &tmX, full_bar(stage), k0, 0);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            advance();
          }
        }
      }
      // phase 1: the Wd half of a slot is loaded as soon as the slot is free;
      // the activation half waits in a FIFO (ring order) for its ready bit
      int q_stage[L::STAGES] = {}, q_kb[L::STAGES] = {};
      int q_head = 0, q_n = 0;
      uint32_t mask_word = 0;  // last ready-mask word read, and its index
      int mask_idx = -1;
      auto issue_front = [&]() {
        const int s = q_stage[q_head];
        tma_load_2d(sbase + s * L::STAGE_BYTES + L::W_BYTES, &tmA, full_bar(s), q_kb[q_head] * TC_BK,
                    0);
        if (++q_head == L::STAGES) q_head = 0;
        --q_n;
      };
      // Issues the activation loads whose flags are up until the ring slot
      // `stage` is free (need_slot) or the FIFO is empty; false on timeout or
      // abort.  The slot to reuse is the ring's oldest: while the FIFO is not
      // full it is not in the FIFO, so the MMA warp can always free it.
      auto pump = [&](bool need_slot) -> bool {
        uint64_t t0 = global_timer_ns();
        for (uint32_t n = 1;; ++n) {
          if (q_n > 0) {
            const int kb = q_kb[q_head];
            const uint32_t bit = 1u << (kb & 31);
            bool ready = mask_idx == (kb >> 5) && (mask_word & bit) != 0u;
            if (!ready) {
              mask_word = ld_acquire_gpu(f.ready + (kb >> 5));
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
          if (need_slot ? (q_n < L::STAGES && mbar_test_wait(empty_bar(stage), phase ^ 1u))
                        : q_n == 0)
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
      if (ok) {
        NgSegIter it = segs1();
        int tile, kb0, nkb;
        bool whole;
        while (ok && it.next(tile, kb0, nkb, whole)) {
          for (int i = 0; i < nkb; ++i) {
            if (!pump(true)) {
              ok = false;
              break;
            }
            const uint32_t sw = sbase + stage * L::STAGE_BYTES;
            mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
            tma_load_2d(sw, &tmWd, full_bar(stage), (kb0 + i) * TC_BK, tile * 128);
            int qt = q_head + q_n;
            if (qt >= L::STAGES) qt -= L::STAGES;
            q_stage[qt] = stage;
            q_kb[qt] = kb0 + i;
            ++q_n;
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            advance();
          }
        }
        if (ok) ok = pump(false);
      }
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
      bool ok = true;
      for (int p = 0; p < 2 && ok; ++p) {
        NgSegIter it = p == 0 ? segs0() : segs1();
        int tile, kb0, nkb;
        bool whole;
        while (ok && it.next(tile, kb0, nkb, whole)) {
          if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, wl, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * NT;
          for (int i = 0; i < nkb; ++i) {
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
                          make_sw128_desc(sx + kk * 32, 16, 1024), idesc,
                          (i | kk) != 0 ? 1u : 0u);
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
      }
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, wl, nullptr, err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = threadIdx.x - 64;  // 0..127 among the epilogue threads
    int acc = 0;
    uint32_t acc_phase = 0;
    float* ustage = reinterpret_cast<float*>(smem + L::USTAGE_OFFSET);
    bool ok = true;
    auto next_acc = [&]() {
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    };
    auto acc_ready = [&]() -> bool {
      int r = 1;
      if (lane == 0) r = mbar_wait_bounded(accf_bar(acc), acc_phase, wl, abort_flag, err) ? 1 : 0;
      r = __shfl_sync(0xffffffffu, r, 0);
      return epi_bar_and(r) != 0;  // all four epilogue warps decide together
    };
    {
      NgSegIter it = segs0();
      int tile, kb0, nkb, seg = 0;
      bool whole;
      for (; it.next(tile, kb0, nkb, whole); ++seg) {
        if (!acc_ready()) {
          ok = false;
          break;
        }
        if (ng_epilogue_segment<NT, true, BF16>(a0, tile, whole, seg, tmem_base + acc * NT,
                                                acce_bar(acc), total0, a0.ctas, ustage,
                                                abort_flag, last_flag)) {
          // this CTA wrote the tile's A columns: publish them to the TMA
          // loads of every CTA's phase 1
          fence_proxy_async_global();
          epi_bar_sync();
          if (e == 0 && !(f.inject_unready && tile == 0)) {
            __threadfence();
            red_or_release_gpu(f.ready + (tile >> 5), 1u << (tile & 31));
          }
        }
        next_acc();
      }
    }
    if (ok) {
      NgSegIter it = segs1();
      int tile, kb0, nkb, seg = 0;
      bool whole;
      for (; it.next(tile, kb0, nkb, whole); ++seg) {
        if (!acc_ready()) break;
        ng_epilogue_segment<NT, false, BF16>(a1, tile, whole, seg, tmem_base + acc * NT,
                                             acce_bar(acc), total1, a1.ctas, ustage, abort_flag,
                                             last_flag);
        next_acc();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // every role of this CTA is done with the flags; the grid's last CTA
    // lowers them (and the count) for the next call
    uint32_t last = 0;
    if (lane == 0) {
      __threadfence();
      last = atomicAdd(f.done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      for (int j = lane; j < (a0.tiles + 31) / 32; j += 32) f.ready[j] = 0u;
      if (lane == 0) *f.done = 0u;
    }
  } else if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace swiglu
