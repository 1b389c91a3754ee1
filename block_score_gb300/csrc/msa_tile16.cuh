// Persistent, warp-specialised block-score kernel for fp16 / bf16 keys on sm_103a.
//
// Per work unit (request b, kv head hk, query tile, KV chunk) the kernel takes
// the logical KV blocks of the chunk two at a time and computes
//     S = Q_tile (128 rows x 128) * [K_beta ; K_beta+1]^T (128 x 256 tokens)
// as one stream of M=128, N=256 tcgen05 MMAs (fp32 accumulator in TMEM), then
// reduces each row of S to one number per block: the max over the block's
// visible tokens (feature request "MsaIndexScore", "calculation": DOT -> MASK
// -> MAX).  Rows are (query position, head) pairs of one GQA group, so one K
// page read serves g heads.
//
// Why two blocks per MMA: the issuing thread stalls on every mbarrier wait
// until its queued MMAs have been dispatched, and a 64-cycle N=128 MMA cannot
// cover that pause, so the tensor pipe idles for a few hundred cycles per block.
// A 128-cycle N=256 MMA keeps the pipe busy across the wait.
//
// Roles (one CTA per SM, persistent over units fetched with an atomic counter):
//   warp 0       scheduler: claims the next unit from the global counter a few
//                blocks before the producer needs it and decodes it from the plan
//   warp 1       TMEM owner + single-thread tcgen05.mma issuer
//   warp 2       TMA producer (Q tiles, K pages through block_table)
//   warps 3..10  epilogue, two groups of four warps (one per TMEM lane
//                quarter); of every pair, group 0 takes the first block and
//                group 1 the second: TMEM -> registers, release of the
//                accumulator, then mask, 128-wide max, local-mask constants,
//                store
//
// Shared memory: Q double buffer (2 x 32 KiB) and a ring of five 32 KiB K
// slots.  A pair of blocks takes two consecutive slots: the first holds both
// pages' first 64-element halves (256 rows, so one descriptor spans both
// pages), the second both pages' second halves.  Each slot is released as soon
// as the four MMAs reading it are done.  TMEM: two 256-column accumulators.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

struct Tile16 {
  static constexpr int kThreads = 352;
  static constexpr int kQBufs = 2;
  static constexpr int kSlots = 5;                             // K slots of one K half of two pages
  static constexpr int kAcc = 2;                               // accumulators of 256 columns
  static constexpr int kGroups = 2;                            // epilogue groups
  static constexpr uint32_t kSlotBytes = 2 * kHalfBytes;       // 256 rows x 128 bytes
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQBufs * kTileBytes;
  static constexpr uint32_t ring_off = k_off + kSlots * kSlotBytes;
  static constexpr uint32_t bar_off = ring_off + kSched * sizeof(UnitDesc);
  static constexpr uint32_t n_bars = 2 * kSched + 2 * kQBufs + 2 * kSlots + 2 * kAcc + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;   // tmem base, abort flag
  static constexpr uint32_t end = misc_off + 16;
  static constexpr uint32_t bytes = end + 1024;                // + alignment slack
};

static_assert(Tile16::bytes <= 232448, "shared memory per CTA");

template <bool BF16>
__global__ void __launch_bounds__(Tile16::kThreads, 1)
    tile16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const Params p) {
  using C = Tile16;
  constexpr int PS = C::kSlots;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  UnitDesc* ring = reinterpret_cast<UnitDesc*>(smem + C::ring_off);
  const uint32_t bars = sbase + C::bar_off;
  const uint32_t b_sched_full = bars;
  const uint32_t b_sched_empty = b_sched_full + 8 * kSched;
  const uint32_t b_q_full = b_sched_empty + 8 * kSched;
  const uint32_t b_q_empty = b_q_full + 8 * C::kQBufs;
  const uint32_t b_k_full = b_q_empty + 8 * C::kQBufs;
  const uint32_t b_k_empty = b_k_full + 8 * PS;
  const uint32_t b_acc_full = b_k_empty + 8 * PS;
  const uint32_t b_acc_empty = b_acc_full + 8 * C::kAcc;
  const uint32_t b_drain = b_acc_empty + 8 * C::kAcc;
  const uint32_t b_sched_req = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // readers of each unit descriptor: producer, MMA, 8 epilogue warps
  constexpr int kConsumers = 2 + 4 * C::kGroups;

  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSched; ++i) {
      mbar_init(b_sched_full + 8 * i, 1);
      mbar_init(b_sched_empty + 8 * i, kConsumers);
    }
    for (int i = 0; i < C::kQBufs; ++i) {
      mbar_init(b_q_full + 8 * i, 1);
      mbar_init(b_q_empty + 8 * i, 1);
    }
    for (int i = 0; i < PS; ++i) {
      mbar_init(b_k_full + 8 * i, 1);
      mbar_init(b_k_empty + 8 * i, 1);
    }
    for (int i = 0; i < C::kAcc; ++i) {
      mbar_init(b_acc_full + 8 * i, 1);
      mbar_init(b_acc_empty + 8 * i, 4 * C::kGroups);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_sched_req, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // The plan written by the preceding kernel is visible after this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  const ReqInfo* req = reinterpret_cast<const ReqInfo*>(p.ws + sizeof(PlanHeader));
  const int32_t* prefix = plan_prefix(p.ws, p.B, 0);
  WaitCtl ctl{abort_flag, &hdr->err, p.wait_limit_ns};
  const int n_units0 = *reinterpret_cast<volatile int*>(&hdr->n_units[0]);

  if (n_units0 == 0) {
    // no tile-class requests in this call
  } else if (warp == 0) {
    // -------------------------------------------------------- scheduler --
    // Claims one unit ahead: the first at once, each later one when the
    // producer is kLead blocks from the end of its current unit.
    if (lane == 0) {
      const int n_units = *reinterpret_cast<volatile int*>(&hdr->n_units[0]);
      const int chunk = *reinterpret_cast<volatile int*>(&hdr->chunk[0]);
      const int n_req = *reinterpret_cast<volatile int*>(&hdr->n_req[0]);
      uint32_t ss = 0, sph = 0, rph = 0;
      for (bool first = true;; first = false) {
        if (!first) {
          if (!mbar_wait(b_sched_req, rph, ctl)) break;
          rph ^= 1;
        }
        UnitDesc d;
        make_unit(p, req, prefix, n_req, n_units, chunk, p.np, atomicAdd(&hdr->counter[0], 1), d);
        if (!mbar_wait(b_sched_empty + 8 * ss, sph ^ 1, ctl)) break;
        ring[ss] = d;
        mbar_arrive(b_sched_full + 8 * ss);
        if (++ss == kSched) { ss = 0; sph ^= 1; }
        if (!d.live) break;
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_k = l2_policy_evict_last();
      const uint32_t q_bytes = 2u * 128u * (uint32_t)(p.g * p.np);
      const bool paged = p.layout != 2;
      const int32_t page_oob = (int32_t)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);
      uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0;
      uint32_t n_q = 0, n_k = 0;   // loads issued (for the teardown drain)
      for (;;) {
        if (!mbar_wait(b_sched_full + 8 * ss, sph, ctl)) break;
        const UnitDesc d = ring[ss];
        mbar_arrive(b_sched_empty + 8 * ss);
        if (++ss == kSched) { ss = 0; sph ^= 1; }
        if (!d.live) break;
        if (d.b1 <= d.c0) {
          mbar_arrive(b_sched_req);
          continue;
        }
        const int req_at = max(d.c0, d.b1 - kLead);
        if (!mbar_wait(b_q_empty + 8 * qb, qph ^ 1, ctl)) break;
        const uint32_t qdst = sbase + C::q_off + qb * kTileBytes;
        mbar_arrive_expect_tx(b_q_full + 8 * qb, q_bytes);
        tma_load_3d(qdst, &tm_q, b_q_full + 8 * qb, 0, d.hk * p.g, d.t0);
        tma_load_3d(qdst + kHalfBytes, &tm_q, b_q_full + 8 * qb, 64, d.hk * p.g, d.t0);
        ++n_q;
        if (++qb == C::kQBufs) { qb = 0; qph ^= 1; }
        // page indices of the next pair are read one pair ahead
        const int32_t* trow = p.block_table + (int64_t)d.b * p.MB;
        int nx0 = 0, nx1 = 0;
        if (paged) {
          nx0 = __ldg(trow + d.c0);
          if (d.c0 + 1 < d.b1) nx1 = __ldg(trow + d.c0 + 1);
        }
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; beta += 2) {
          if (req_at >= beta && req_at < beta + 2) mbar_arrive(b_sched_req);
          const int nblk = beta + 1 < d.b1 ? 2 : 1;
          int pg[2] = {nx0, nx1};
          if (paged) {
            nx0 = beta + 2 < d.b1 ? __ldg(trow + beta + 2) : 0;
            nx1 = beta + 3 < d.b1 ? __ldg(trow + beta + 3) : 0;
          }
          int page[2] = {0, 0}, tok[2] = {0, 0};
          for (int j = 0; j < nblk; ++j) {
            if (paged) {
              page[j] = pg[j];
              if (page[j] < 0 || (int64_t)page[j] >= p.NP) {
                atomicOr(&hdr->err, kErrBlockTable);
                page[j] = page_oob;   // out of bounds: the copy fills zeros
              }
            } else {
              tok[j] = d.kbase + (beta + j) * kP;
            }
          }
          // K half x of both pages into one slot: page j's 128 rows at j * 16 KiB
          for (int x = 0; x < 2 && ok; ++x) {
            if (!mbar_wait(b_k_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
            const uint32_t kdst = sbase + C::k_off + ks * C::kSlotBytes;
            mbar_arrive_expect_tx(b_k_full + 8 * ks, (uint32_t)nblk * kHalfBytes);
            for (int j = 0; j < nblk; ++j)
              tma_k(kdst + (uint32_t)j * kHalfBytes, &tm_k, b_k_full + 8 * ks, 64 * x, tok[j], d.hk,
                    page[j], p.layout, pol_k);
            ++n_k;
            if (++ks == PS) { ks = 0; kph ^= 1; }
          }
          if (!ok) break;
        }
        if (!ok) break;
      }
      // Teardown: never leave the CTA with a TMA write in flight.  Only the
      // last (ring size) loads of each ring can still be pending.
      for (uint32_t j = n_k > (uint32_t)PS ? n_k - PS : 0; j < n_k; ++j) {
        const uint32_t st = j % PS, ph = (j / PS) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_k_full + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
      for (uint32_t j = n_q > (uint32_t)C::kQBufs ? n_q - C::kQBufs : 0; j < n_q; ++j) {
        const uint32_t st = j % C::kQBufs, ph = (j / C::kQBufs) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_q_full + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc2 = idesc_f16(BF16, 128, 256);   // two blocks
      constexpr uint32_t idesc1 = idesc_f16(BF16, 128, 128);   // odd last block of a unit
      uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0, ab = 0, aph = 0;
      bool issued = false;
      for (;;) {
        if (!mbar_wait(b_sched_full + 8 * ss, sph, ctl)) break;
        const UnitDesc d = ring[ss];
        mbar_arrive(b_sched_empty + 8 * ss);
        if (++ss == kSched) { ss = 0; sph ^= 1; }
        if (!d.live) break;
        if (d.b1 <= d.c0) continue;
        if (!mbar_wait(b_q_full + 8 * qb, qph, ctl)) break;
        const uint32_t qsrc = sbase + C::q_off + qb * kTileBytes;
        bool ok = true;
        for (int beta = d.c0; beta < d.b1 && ok; beta += 2) {
          if (!mbar_wait(b_acc_empty + 8 * ab, aph ^ 1, ctl)) { ok = false; break; }
          const uint32_t dt = tmem_base + ab * 256u;
          const uint32_t idesc = beta + 1 < d.b1 ? idesc2 : idesc1;
          for (int x = 0; x < 2; ++x) {
            if (!mbar_wait(b_k_full + 8 * ks, kph, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ksrc = sbase + C::k_off + ks * C::kSlotBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f16(dt, desc_at(qsrc, 4 * x + kk), smem_desc_sw128(ksrc + 32u * kk), idesc,
                         (x | kk) ? 1u : 0u);
            tc_commit(b_k_empty + 8 * ks);   // the slot is free once these four MMAs are done
            if (++ks == PS) { ks = 0; kph ^= 1; }
          }
          if (!ok) break;
          tc_commit(b_acc_full + 8 * ab);
          issued = true;
          if (++ab == C::kAcc) { ab = 0; aph ^= 1; }
        }
        if (!ok) break;
        tc_commit(b_q_empty + 8 * qb);
        if (++qb == C::kQBufs) { qb = 0; qph ^= 1; }
      }
      if (issued) {
        // every MMA of this CTA has landed before TMEM is released
        tc_commit(b_drain);
        uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_drain, 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp < kEpiWarp0 + 4 * C::kGroups) {
    // --------------------------------------------------------- epilogue --
    const int grp = (warp - kEpiWarp0) >> 2;       // block of each pair this group drains
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may read
    const int r = quarter * 32 + lane;             // MMA row = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)grp * 128u;
    const float ninf = __int_as_float(0xff800000);
    const int rows = p.g * p.np;
    const int pos = r / p.g;
    const int hl = r - pos * p.g;
    uint32_t ss = 0, sph = 0, ab = 0, aph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      const bool valid = r < rows && pos < d.npos;
      const bool warp_valid = __any_sync(0xffffffffu, valid);
      const int i = d.i0 + pos;
      const int lim = p.sparse_mode == 3 ? d.L - d.Lq + i : d.L - 1;   // last visible key
      const int h = d.hk * p.g + hl;
      float* orow = p.out + ((int64_t)h * p.T + (d.t0 + pos)) * (int64_t)p.MBp;
      const int lo = max(0, d.sl + 1 - p.local_blocks);
      // value of a column that has no computed score: the local-mask constant
      // if forced, else the fill value (padding columns >= MB always fill)
      const bool live_kv = d.L > 0;
      auto fill_value = [&](int beta) -> float {
        float f = ninf;
        if (live_kv && beta < p.init_blocks) f = 1e30f;
        if (live_kv && beta >= lo && beta <= d.sl) f = 1e29f;
        return beta < p.MB ? f : ninf;
      };
      auto forced = [&](int beta) -> bool {
        return live_kv && (beta < p.init_blocks || (beta >= lo && beta <= d.sl));
      };
      bool ok = true;
      int beta = d.c0;
      for (; beta < d.b1; beta += 2) {
        const uint32_t a = ab, a_ph = aph;
        if (++ab == C::kAcc) { ab = 0; aph ^= 1; }
        const int col = beta + grp;        // this group's block of the pair
        const bool has = col < d.b1;       // else a lone last block's partner (a fill column)
        const bool ld = warp_valid && has;
        if (!warp_wait(b_acc_full + 8 * a, a_ph, ctl)) { ok = false; break; }
        tc_fence_after();
        float x[128];
        if (ld) {
          tmem_ld128(t_lane + a * 256u, x);
          tmem_wait_ld();
        }
        // the accumulator is free once both groups hold their block in registers
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
        float m = ninf;
        if (ld && valid) m = masked_row_max(x, lim - col * kP);
        // local mask after the max: forced blocks take their constant
        if (!has || forced(col)) m = fill_value(col);
        if (valid) __stcs(orow + col, m);
      }
      if (!ok) break;
      // columns past the computed pairs (group 0): pairs up to a multiple of
      // 8, then whole groups of closed-form values
      if (grp != 0) continue;
      if (valid) {
        for (; (beta & 7) && beta < d.c1; beta += 2)
          __stcs(reinterpret_cast<float2*>(orow + beta), make_float2(fill_value(beta), fill_value(beta + 1)));
        for (; beta < d.c1; beta += 8) {
          float4* dst = reinterpret_cast<float4*>(orow + beta);
          __stcs(dst, make_float4(fill_value(beta), fill_value(beta + 1), fill_value(beta + 2),
                                  fill_value(beta + 3)));
          __stcs(dst + 1, make_float4(fill_value(beta + 4), fill_value(beta + 5),
                                      fill_value(beta + 6), fill_value(beta + 7)));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace msa
