// Persistent, warp-specialised block-score kernel for sm_103a.
//
// Per work unit (request b, kv head hk, query tile, KV chunk) the kernel
// computes, for each logical KV block beta of the chunk,
//     S = Q_tile (128 rows x 128) * K_beta^T (128 x 128 tokens)      (tcgen05, fp32 in TMEM)
// and reduces every row of S to one number: the max over the visible tokens
// of the block (feature request "MsaIndexScore", "calculation": DOT ->
// optional DEQUANT column multiply -> MASK -> MAX).  Rows are (query position,
// head) pairs of one GQA group, so one K page read serves g heads.
//
// Roles (one CTA per SM, persistent over units fetched with an atomic counter):
//   warp 0       scheduler: claims the next unit from the global counter a few
//                blocks before the producer needs it and decodes it from the plan
//   warp 1       TMEM owner + single-thread tcgen05.mma issuer
//   warp 2       TMA producer (Q tiles, K pages through block_table)
//   warps 3..6   epilogue: TMEM -> registers, (scale), mask, 128-wide max,
//                local-mask constants, 32-byte vector stores of the fp32 scores
//   warps 7..10  (int8 keys only) int8 -> fp16 conversion of K pages into the
//                swizzled operand layout, and the per-token scale for the epilogue
//
// Shared memory: Q double buffer (2 x 32 KiB), K ring of 32 KiB stages, for
// int8 also a ring of raw 16 KiB pages.  TMEM: 4 accumulators of 128 columns.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

template <bool KI8>
struct ScoreCfg;

template <>
struct ScoreCfg<false> {
  static constexpr int kStages = 5;      // 16-bit K pages in flight
  static constexpr int kRawStages = 0;
  static constexpr int kThreads = 224;
};

template <>
struct ScoreCfg<true> {
  static constexpr int kStages = 2;      // converted fp16 pages
  static constexpr int kRawStages = 5;   // int8 pages in flight
  static constexpr int kThreads = 352;
};


constexpr int kQBufs = 2;
constexpr int kAcc = 4;

template <bool KI8>
struct SmemLayout {
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQBufs * kTileBytes;
  static constexpr uint32_t raw_off = k_off + ScoreCfg<KI8>::kStages * kTileBytes;
  static constexpr uint32_t scale_off = raw_off + ScoreCfg<KI8>::kRawStages * kRawStride;
  static constexpr uint32_t scale_bytes = KI8 ? kAcc * 128 * 4 : 0;
  static constexpr uint32_t ring_off = scale_off + scale_bytes;        // UnitDesc x kSched
  static constexpr uint32_t bar_off = ring_off + kSched * sizeof(UnitDesc);
  static constexpr uint32_t n_bars = 2 * kSched + 2 * kQBufs + 2 * ScoreCfg<KI8>::kStages +
                                     2 * ScoreCfg<KI8>::kRawStages + 2 * kAcc +
                                     (KI8 ? 2 * kAcc : 0) + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;           // tmem base, abort, raw pages
  static constexpr uint32_t end = misc_off + 16 + 4 * (ScoreCfg<KI8>::kRawStages + 1);
  static constexpr uint32_t bytes = end + 1024;                        // + alignment slack
};


template <bool KI8, bool BF16>
__global__ void __launch_bounds__(ScoreCfg<KI8>::kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const Params p) {
  using Cfg = ScoreCfg<KI8>;
  using L = SmemLayout<KI8>;
  constexpr int S = Cfg::kStages;
  constexpr int R = Cfg::kRawStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  UnitDesc* ring = reinterpret_cast<UnitDesc*>(smem + L::ring_off);
  const uint32_t bars = sbase + L::bar_off;
  // barrier addresses
  const uint32_t b_sched_full = bars;
  const uint32_t b_sched_empty = b_sched_full + 8 * kSched;
  const uint32_t b_q_full = b_sched_empty + 8 * kSched;
  const uint32_t b_q_empty = b_q_full + 8 * kQBufs;
  const uint32_t b_k_full = b_q_empty + 8 * kQBufs;
  const uint32_t b_k_empty = b_k_full + 8 * S;
  const uint32_t b_raw_full = b_k_empty + 8 * S;
  const uint32_t b_raw_empty = b_raw_full + 8 * R;
  const uint32_t b_acc_full = b_raw_empty + 8 * R;
  const uint32_t b_acc_empty = b_acc_full + 8 * kAcc;
  const uint32_t b_sc_full = b_acc_empty + 8 * kAcc;
  const uint32_t b_sc_empty = b_sc_full + (KI8 ? 8 * kAcc : 0);
  const uint32_t b_drain = b_sc_empty + (KI8 ? 8 * kAcc : 0);
  const uint32_t b_sched_req = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  volatile int* raw_page = reinterpret_cast<volatile int*>(smem + L::misc_off + 16);
  float* scale_s = reinterpret_cast<float*>(smem + L::scale_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // readers of each unit descriptor: producer, MMA, 4 epilogue warps (+ 4 converter warps)
  constexpr int kConsumers = KI8 ? 10 : 6;

  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSched; ++i) {
      mbar_init(b_sched_full + 8 * i, 1);
      mbar_init(b_sched_empty + 8 * i, kConsumers);
    }
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(b_q_full + 8 * i, 1);
      mbar_init(b_q_empty + 8 * i, 1);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(b_k_full + 8 * i, KI8 ? 4 : 1);
      mbar_init(b_k_empty + 8 * i, 1);
    }
    for (int i = 0; i < R; ++i) {
      mbar_init(b_raw_full + 8 * i, 1);
      mbar_init(b_raw_empty + 8 * i, 4);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(b_acc_full + 8 * i, 1);
      mbar_init(b_acc_empty + 8 * i, 4);
      if (KI8) {
        mbar_init(b_sc_full + 8 * i, 4);
        mbar_init(b_sc_empty + 8 * i, 4);
      }
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
    // producer is kLead blocks from the end of its current unit, so a CTA
    // never sits on work another CTA could be doing.
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
        const uint32_t qdst = sbase + L::q_off + qb * kTileBytes;
        mbar_arrive_expect_tx(b_q_full + 8 * qb, q_bytes);
        tma_load_3d(qdst, &tm_q, b_q_full + 8 * qb, 0, d.hk * p.g, d.t0);
        tma_load_3d(qdst + kHalfBytes, &tm_q, b_q_full + 8 * qb, 64, d.hk * p.g, d.t0);
        ++n_q;
        if (++qb == kQBufs) { qb = 0; qph ^= 1; }
        // page indices run four blocks ahead of their use
        const int32_t* trow = p.block_table + (int64_t)d.b * p.MB;
        int pg0 = 0, pg1 = 0, pg2 = 0, pg3 = 0;
        if (paged) {
          pg0 = __ldg(trow + d.c0);
          if (d.c0 + 1 < d.b1) pg1 = __ldg(trow + d.c0 + 1);
          if (d.c0 + 2 < d.b1) pg2 = __ldg(trow + d.c0 + 2);
          if (d.c0 + 3 < d.b1) pg3 = __ldg(trow + d.c0 + 3);
        }
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; ++beta) {
          if (beta == req_at) mbar_arrive(b_sched_req);
          int page = 0, tok;
          if (paged) {
            page = pg0;
            pg0 = pg1;
            pg1 = pg2;
            pg2 = pg3;
            pg3 = beta + 4 < d.b1 ? __ldg(trow + beta + 4) : 0;
            tok = 0;
            if (page < 0 || (int64_t)page >= p.NP) {
              atomicOr(&hdr->err, kErrBlockTable);
              page = (int)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);   // out of bounds: zero fill
            }
          } else {
            tok = d.kbase + beta * kP;
          }
          if constexpr (KI8) {
            if (!mbar_wait(b_raw_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
            raw_page[ks] = paged ? page : tok;
            const uint32_t rdst = sbase + L::raw_off + ks * kRawStride;
            // the page's 128 scales ride along with the int8 tile (one bulk copy)
            const bool with_scale = paged && (int64_t)page < p.NP;
            mbar_arrive_expect_tx(b_raw_full + 8 * ks, kRawBytes + (with_scale ? kRawScaleBytes : 0u));
            tma_k(rdst, &tm_k, b_raw_full + 8 * ks, 0, tok, d.hk, page, p.layout, pol_k);
            if (with_scale)
              bulk_load(rdst + kRawBytes, p.scale + ((int64_t)page * p.H_kv + d.hk) * kP,
                        kRawScaleBytes, b_raw_full + 8 * ks);
            ++n_k;
            if (++ks == R) { ks = 0; kph ^= 1; }
          } else {
            if (!mbar_wait(b_k_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
            const uint32_t kdst = sbase + L::k_off + ks * kTileBytes;
            mbar_arrive_expect_tx(b_k_full + 8 * ks, kTileBytes);
            tma_k(kdst, &tm_k, b_k_full + 8 * ks, 0, tok, d.hk, page, p.layout, pol_k);
            tma_k(kdst + kHalfBytes, &tm_k, b_k_full + 8 * ks, 64, tok, d.hk, page, p.layout, pol_k);
            ++n_k;
            if (++ks == S) { ks = 0; kph ^= 1; }
          }
        }
        if (!ok) break;
      }
      // Teardown: never leave the CTA with a TMA write in flight.  Only the
      // last (ring size) loads of each ring can still be pending.
      const uint32_t nk_ring = KI8 ? (uint32_t)R : (uint32_t)S;
      const uint32_t kfull = KI8 ? b_raw_full : b_k_full;
      for (uint32_t j = n_k > nk_ring ? n_k - nk_ring : 0; j < n_k; ++j) {
        const uint32_t st = j % nk_ring, ph = (j / nk_ring) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(kfull + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
      for (uint32_t j = n_q > (uint32_t)kQBufs ? n_q - kQBufs : 0; j < n_q; ++j) {
        const uint32_t st = j % kQBufs, ph = (j / kQBufs) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_q_full + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BF16, 128, 128);
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
        const uint32_t qsrc = sbase + L::q_off + qb * kTileBytes;
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; ++beta) {
          if (!mbar_wait(b_k_full + 8 * ks, kph, ctl)) { ok = false; break; }
          if (!mbar_wait(b_acc_empty + 8 * ab, aph ^ 1, ctl)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ksrc = sbase + L::k_off + ks * kTileBytes;
          const uint32_t dt = tmem_base + ab * 128u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma_f16(dt, desc_at(qsrc, k), desc_at(ksrc, k), idesc, k > 0 ? 1u : 0u);
          tc_commit(b_k_empty + 8 * ks);
          tc_commit(b_acc_full + 8 * ab);
          issued = true;
          if (++ks == S) { ks = 0; kph ^= 1; }
          if (++ab == kAcc) { ab = 0; aph ^= 1; }
        }
        if (!ok) break;
        tc_commit(b_q_empty + 8 * qb);
        if (++qb == kQBufs) { qb = 0; qph ^= 1; }
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
  } else if (warp < kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may read
    const int r = quarter * 32 + lane;             // MMA row = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
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
      float v[8];
      bool ok = true;
      int beta = d.c0;
      for (; beta < d.b1; ++beta) {
        float m = ninf;
        if (!warp_wait(b_acc_full + 8 * ab, aph, ctl)) { ok = false; break; }
        tc_fence_after();
        float x[128];
        if (warp_valid) {
          const uint32_t ta = t_lane + ab * 128u;
          tmem_ld128(ta, x);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_acc_empty + 8 * ab);
        if constexpr (KI8) {
          // DEQUANT: column multiply by the per-token scale, before the mask
          if (!warp_wait(b_sc_full + 8 * ab, aph, ctl)) { ok = false; break; }
          if (warp_valid) {
            const float4* sc = reinterpret_cast<const float4*>(scale_s + ab * 128);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float4 s4 = sc[c];
              x[4 * c + 0] *= s4.x;
              x[4 * c + 1] *= s4.y;
              x[4 * c + 2] *= s4.z;
              x[4 * c + 3] *= s4.w;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_sc_empty + 8 * ab);
        }
        if (valid) m = masked_row_max(x, lim - beta * kP);
        if (++ab == kAcc) { ab = 0; aph ^= 1; }
        // local mask after the max: forced blocks take their constant
        if (live_kv && (beta < p.init_blocks || (beta >= lo && beta <= d.sl))) m = fill_value(beta);
        const int e = beta & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k == e) v[k] = m;
        if (e == 7 && valid) {
          float4* dst = reinterpret_cast<float4*>(orow + (beta - 7));
          __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
          __stcs(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
        }
      }
      if (!ok) break;
      // columns past the computed blocks: finish the open group of 8, then
      // write whole groups of closed-form values
      if (valid) {
        if (beta & 7) {
          for (; beta & 7; ++beta) {
            const float f = fill_value(beta);
            const int e = beta & 7;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (k == e) v[k] = f;
          }
          float4* dst = reinterpret_cast<float4*>(orow + (beta - 8));
          __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
          __stcs(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
        }
        for (; beta < d.c1; beta += 8) {
          float4* dst = reinterpret_cast<float4*>(orow + beta);
          __stcs(dst, make_float4(fill_value(beta), fill_value(beta + 1), fill_value(beta + 2),
                                  fill_value(beta + 3)));
          __stcs(dst + 1, make_float4(fill_value(beta + 4), fill_value(beta + 5),
                                      fill_value(beta + 6), fill_value(beta + 7)));
        }
      }
      if (!ok) break;
    }
  } else if (KI8) {
    // ------------------------------------------- int8 -> fp16 converters --
    const int ct = threadIdx.x - kCvtWarp0 * 32;   // 0..127
    uint32_t ss = 0, sph = 0, rs = 0, rph = 0, ks = 0, kph = 0, ab = 0, aph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; ++beta) {
        if (!warp_wait(b_raw_full + 8 * rs, rph, ctl)) { ok = false; break; }
        if (!warp_wait(b_k_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
        const uint8_t* src = smem + L::raw_off + rs * kRawStride;
        // this thread's token scale: from the stage (paged) or, for packed keys,
        // a global load issued now so that it overlaps the conversion
        const int page = raw_page[rs];
        float sv = 0.f;
        if (p.layout == 2) {
          const int64_t row = (int64_t)page + ct;      // page holds the first key row here
          if (row < (int64_t)d.kbase + d.L && row < p.NP) sv = __ldg(p.scale + row * p.H_kv + d.hk);
        } else if (page >= 0 && (int64_t)page < p.NP) {
          sv = reinterpret_cast<const float*>(src + kRawBytes)[ct];
        }
        uint8_t* dst = smem + L::k_off + ks * kTileBytes;
        // all eight 16-byte chunks of this thread are loaded before any store,
        // so the loads overlap (the compiler cannot reorder them past stores
        // into the same shared memory)
        int4 raw[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int id = ct + 128 * it;           // 16-byte chunk of the int8 page
          raw[it] = *reinterpret_cast<const int4*>(src + (id >> 3) * 128 + (id & 7) * 16);
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int id = ct + 128 * it;
          const int row = id >> 3, c16 = id & 7;
          const uint32_t w[4] = {(uint32_t)raw[it].x, (uint32_t)raw[it].y, (uint32_t)raw[it].z,
                                 (uint32_t)raw[it].w};
          uint32_t hv[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) int8x4_to_half4(w[q], hv[2 * q], hv[2 * q + 1]);
          // 16 fp16 values = two 16-byte chunks of the 128-byte swizzled row
          const int half = c16 >> 2;
          const int j0 = (c16 & 3) * 2;
          uint8_t* rowp = dst + half * kHalfBytes + row * 128;
          *reinterpret_cast<uint4*>(rowp + (((j0 + 0) ^ (row & 7)) << 4)) =
              make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(rowp + (((j0 + 1) ^ (row & 7)) << 4)) =
              make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(b_k_full + 8 * ks);
          mbar_arrive(b_raw_empty + 8 * rs);
        }
        if (++rs == R) { rs = 0; rph ^= 1; }
        if (++ks == S) { ks = 0; kph ^= 1; }
        // per-token scale of this block for the epilogue (slot follows the accumulator ring)
        if (!warp_wait(b_sc_empty + 8 * ab, aph ^ 1, ctl)) { ok = false; break; }
        scale_s[ab * 128 + ct] = sv;
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sc_full + 8 * ab);
        if (++ab == kAcc) { ab = 0; aph ^= 1; }
      }
      if (!ok) break;
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
