// Persistent, warp-specialised block-score kernel for query tiles, sm_103a.
//
// Per work unit (request b, kv head hk, query tile, KV chunk) the kernel takes
// the logical KV blocks of the chunk two at a time and computes
//     S = Q_tile (128 rows x 128) * [K_beta ; K_beta+1]^T (128 x 256 tokens)
// as one stream of M=128, N=256 tcgen05 MMAs (fp32 accumulator in TMEM), then
// reduces each row of S to one number per block: the max over the block's
// visible tokens (feature request "MsaIndexScore", "calculation": DOT ->
// optional DEQUANT -> MASK -> MAX).  Rows are (query position, head) pairs of
// one GQA group, so one K page read serves g heads.
//
// Why two blocks per MMA: the issuing thread stalls on every mbarrier wait
// until its queued MMAs have been dispatched, and a 64-cycle N=128 MMA cannot
// cover that pause, so the tensor pipe idles for a few hundred cycles per block.
// A 128-cycle N=256 MMA keeps the pipe busy across the wait.  The whole MMA
// warp runs the issue loop and its elected lane (elect.sync) issues: issued so,
// back-to-back N=256 MMAs complete every ~134 cycles, against ~168 when one
// lane issues them from a divergent branch.
//
// Roles (one CTA per SM, persistent over units fetched with an atomic counter):
//   warp 0       scheduler: claims the next unit from the global counter a few
//                blocks before the producer needs it and decodes it from the plan
//   warp 1       TMEM owner + tcgen05.mma issuer (converged warp, elected lane)
//   warp 2       TMA producer (Q tiles, K pages through block_table)
//   16-bit keys:
//   warps 3..10  epilogue, two groups of four warps (one per TMEM lane
//                quarter); of every pair, group 0 takes the first block and
//                group 1 the second: TMEM -> registers, release of the
//                accumulator, then mask, 128-wide max, local-mask constants,
//                store
//   int8 keys:
//   warps 3..10  epilogue as above, with the per-token scale multiply before
//                the mask
//   warps 11..18 converters, two groups of four: group j turns page j of every
//                pair from int8 into fp16 rows of the swizzled operand layout,
//                one K slot at a time, and hands over its per-token scales
//
// Shared memory: Q double buffer (2 x 32 KiB) and a ring of 32 KiB K slots.
// A pair of blocks takes two consecutive slots: the first holds both pages'
// first 64-element halves (256 rows, so one descriptor spans both pages), the
// second both pages' second halves.  Each slot is released as soon as the
// four MMAs reading it are done.  int8 keys add a ring of raw int8 pages (with
// their scales) and a ring of per-pair scale vectors for the epilogue.
// TMEM: two 256-column accumulators.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_fp16.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

// Key modes: 0 = fp16 / bf16 / fp8 keys, 1 = int8 (or FP4) keys converted by
// converter warps, 2 = int8 keys already converted into an fp16 copy of the
// pages (the mirror; TMA straight into the K slots, the scales loaded beside).
__host__ __device__ constexpr int tile_mode(bool ki8, bool km) { return ki8 ? 1 : (km ? 2 : 0); }

template <int MODE>
struct TileCfg;

template <>
struct TileCfg<0> {               // fp16 / bf16 / fp8 keys: TMA straight into the K slots
  static constexpr int kThreads = 384;         // the last warp feeds the MMA warp
  static constexpr int kSlots = 5;
  static constexpr int kRaw = 0;
  static constexpr int kScPairs = 0;
  static constexpr int kGroups = 2;            // epilogue groups
  static constexpr int kQBufs = 2;
  static constexpr int kCvtGroups = 0;
};

template <>
struct TileCfg<2> {               // int8 keys from the fp16 mirror: TMA into the K slots, scales by bulk copy
  static constexpr int kThreads = 384;         // the last warp feeds the MMA warp
  static constexpr int kSlots = 4;             // one slot fewer than mode 0: room for the scale ring
  static constexpr int kRaw = 0;
  static constexpr int kScPairs = 4;
  static constexpr int kGroups = 2;
  static constexpr int kQBufs = 2;
  static constexpr int kCvtGroups = 0;
};

template <>
struct TileCfg<1> {               // int8 keys: raw pages, converters, scales
  static constexpr int kThreads = 640;         // the last warp feeds the MMA warp
  static constexpr int kCvtGroups = 2;         // page j of every pair by group j
  static constexpr int kSlots = 3;
  static constexpr int kRaw = 5;               // int8 pages in flight (L2 latency)
  static constexpr int kScPairs = 4;
  static constexpr int kGroups = 2;
  static constexpr int kQBufs = 1;             // the shared memory goes to the raw ring
};

template <int MODE>
struct TileLayout {
  using Cfg = TileCfg<MODE>;
  static constexpr int kQBufs = Cfg::kQBufs;
  static constexpr int kAcc = 2;                               // accumulators of 256 columns
  static constexpr int kGroups = Cfg::kGroups;                 // epilogue groups
  static constexpr int kCvtW0 = kEpiWarp0 + 4 * kGroups;       // first converter warp (int8)
  static constexpr uint32_t kSlotBytes = 2 * kHalfBytes;       // 256 rows x 128 bytes
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQBufs * kTileBytes;
  static constexpr uint32_t raw_off = k_off + Cfg::kSlots * kSlotBytes;
  static constexpr uint32_t sc_off = raw_off + Cfg::kRaw * kRawStride;
  static constexpr uint32_t ring_off = sc_off + Cfg::kScPairs * 256 * 4;
  static constexpr uint32_t bar_off = ring_off + kSched * sizeof(UnitDesc);
  static constexpr uint32_t n_bars = 2 * kSched + 2 * kQBufs + 2 * Cfg::kSlots + 2 * Cfg::kRaw +
                                     2 * kAcc + 2 * Cfg::kScPairs + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;   // tmem base, abort flag, raw pages
  static constexpr uint32_t end = misc_off + 16 + 4 * (Cfg::kRaw + 1);
  static constexpr uint32_t bytes = end + 1024;                // + alignment slack
};

static_assert(TileLayout<0>::bytes <= 232448 && TileLayout<1>::bytes <= 232448 &&
                  TileLayout<2>::bytes <= 232448,
              "shared memory per CTA");

// Every writer of shared memory stays inside its own region, so nothing but
// mbarrier operations and tcgen05.commit ever touches the barrier words:
// regions in address order without overlap, 128-byte-swizzled operand tiles
// on 1 KiB boundaries, and each copy no larger than its destination.
template <int MODE>
constexpr bool tile_layout_ok() {
  using L = TileLayout<MODE>;
  using C = TileCfg<MODE>;
  return L::q_off % 1024 == 0 && L::k_off % 1024 == 0 && L::raw_off % 1024 == 0 &&
         kRawStride % 1024 == 0 && L::kSlotBytes % 1024 == 0 &&
         L::q_off + L::kQBufs * kTileBytes <= L::k_off &&                 // Q box: <= 128 rows x 256 B
         L::k_off + C::kSlots * L::kSlotBytes <= L::raw_off &&            // K slot: 2 pages x 16 KiB
         L::raw_off + C::kRaw * kRawStride <= L::sc_off &&                // raw page + scales
         kRawBytes + kRawScaleBytes <= kRawStride &&
         L::sc_off + C::kScPairs * 256 * 4 <= L::ring_off &&              // [pair][page][token] fp32
         L::ring_off + kSched * sizeof(UnitDesc) <= L::bar_off &&
         L::bar_off % 8 == 0 && L::bar_off + L::n_bars * 8 <= L::misc_off &&
         L::misc_off + 16 + 4 * C::kRaw <= L::end && L::end + 1024 <= L::bytes;
}
static_assert(tile_layout_ok<0>() && tile_layout_ok<1>() && tile_layout_ok<2>(),
              "tile kernel shared-memory layout");

// A claim costs an atomic and a chain of dependent L2 round trips (the search
// over the unit prefix sums, the request record, the first table entries):
// about 5,000 cycles while HBM is saturated, as long as a few FP8 block pairs
// of a decode unit.  The next unit is therefore claimed this many blocks
// before the end of the current one (at its start for short units).
constexpr int kTileLead = 16;

// MMA handoff of the 16-bit / FP8 kernel: helper warp -> MMA warp through
// named barrier kMmaBar; item codes (0 = stop)
// the helper is the last warp: after the two epilogue groups (16-bit / FP8
// keys) or after the converters (int8 keys)
constexpr uint32_t kMmaBar = 1;
constexpr uint32_t kCodeLive = 1, kCodeFirst = 2, kCodeLast = 4, kCodeLone = 8, kCodeUnitEnd = 16;

// F8: 0 = 16-bit operands (fp16 / bf16, or int8 keys converted to fp16);
// 1 = FP8 E4M3 query and keys; 2 = FP8 E5M2.  An FP8 row of 128 elements is
// one 128-byte swizzle row, so a query tile is one box and a pair of pages
// fills one K slot; four kind::f8f6f4 MMAs (K = 32) cover the head dimension.
// TOPK: the fused per-group selection (0 = off).  The epilogue keeps a
// running top-kTopkMax list of each query position's group score (the max over
// the position's g head rows, g dividing 32) over the blocks its group drains,
// and writes it as one partial list per unit; the scores are stored only if
// p.out is not null.  TOPK = 2: the list is spread over 8 lanes of the
// position (g >= 8), so the 128-column TMEM load of a block still fits the
// registers; TOPK = 16: every lane holds the whole list (g < 8) and a block is
// loaded in two 64-column pieces.
// KF4 (with KI8): FP4 key pages instead of int8, 1 = NVFP4 (E4M3 scale per 16
// elements, fp16 operands), 2 = MXFP4 (E8M0 scale per 32, bf16 operands): the
// converters dequantise each E2M1 element by its group scale exactly, so the
// epilogue has no per-token scale to apply.
// KM (without KI8): int8 keys read from their fp16 mirror (tm_k maps the
// mirror, BNBD order), the per-token scales bulk-copied by the producer into
// the scale ring, the int8 epilogue.
template <bool KI8, bool BF16, int F8 = 0, int TOPK = 0, int KF4 = 0, bool KM = false>
__global__ void __launch_bounds__(TileCfg<tile_mode(KI8, KM)>::kThreads, 1)
    tile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const Params p) {
  static_assert(F8 == 0 || !KI8, "FP8 operands come with FP8 keys");
  static_assert(KF4 == 0 || KI8, "FP4 pages go through the converter warps");
  static_assert(!KM || (!KI8 && F8 == 0 && !BF16), "the int8 mirror: fp16 query, no converters");
  constexpr bool kF8 = F8 != 0;
  constexpr int kHalves = kF8 ? 1 : 2;             // K slots (and Q boxes) per pair of blocks
  constexpr int kMode = tile_mode(KI8, KM);
  using Cfg = TileCfg<kMode>;
  using L = TileLayout<kMode>;
  constexpr int PS = Cfg::kSlots;
  constexpr int R = Cfg::kRaw;
  constexpr int SC = Cfg::kScPairs;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  UnitDesc* ring = reinterpret_cast<UnitDesc*>(smem + L::ring_off);
  float* scale_s = reinterpret_cast<float*>(smem + L::sc_off);   // [pair slot][page][token]
  const uint32_t bars = sbase + L::bar_off;
  const uint32_t b_sched_full = bars;
  const uint32_t b_sched_empty = b_sched_full + 8 * kSched;
  const uint32_t b_q_full = b_sched_empty + 8 * kSched;
  const uint32_t b_q_empty = b_q_full + 8 * L::kQBufs;
  const uint32_t b_k_full = b_q_empty + 8 * L::kQBufs;
  const uint32_t b_k_empty = b_k_full + 8 * PS;
  const uint32_t b_raw_full = b_k_empty + 8 * PS;
  const uint32_t b_raw_empty = b_raw_full + 8 * R;
  const uint32_t b_acc_full = b_raw_empty + 8 * R;
  const uint32_t b_acc_empty = b_acc_full + 8 * L::kAcc;
  const uint32_t b_sc_full = b_acc_empty + 8 * L::kAcc;
  const uint32_t b_sc_empty = b_sc_full + 8 * SC;
  const uint32_t b_drain = b_sc_empty + 8 * SC;
  const uint32_t b_sched_req = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  volatile int* raw_page = reinterpret_cast<volatile int*>(smem + L::misc_off + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // readers of each unit descriptor: producer, MMA, the epilogue and converter warps
  constexpr int kConsumers = 2 + 4 * L::kGroups + 4 * Cfg::kCvtGroups;

  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSched; ++i) {
      mbar_init(b_sched_full + 8 * i, 1);
      mbar_init(b_sched_empty + 8 * i, kConsumers);
    }
    for (int i = 0; i < L::kQBufs; ++i) {
      mbar_init(b_q_full + 8 * i, 1);
      mbar_init(b_q_empty + 8 * i, 1);
    }
    for (int i = 0; i < PS; ++i) {
      mbar_init(b_k_full + 8 * i, KI8 ? 4 * Cfg::kCvtGroups : 1);   // TMA, or the converter warps
      mbar_init(b_k_empty + 8 * i, 1);
    }
    for (int i = 0; i < R; ++i) {
      mbar_init(b_raw_full + 8 * i, 1);
      mbar_init(b_raw_empty + 8 * i, 4);
    }
    for (int i = 0; i < L::kAcc; ++i) {
      mbar_init(b_acc_full + 8 * i, 1);
      mbar_init(b_acc_empty + 8 * i, 4 * L::kGroups);
    }
    for (int i = 0; i < SC; ++i) {
      mbar_init(b_sc_full + 8 * i, KM ? 1 : 4 * Cfg::kCvtGroups);   // the producer, or the converter warps
      mbar_init(b_sc_empty + 8 * i, 4 * L::kGroups);
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
  // the header fields are read together: one round trip before the first claim
  // (plain loads: the header is constant during this grid)
  const int n_units0 = hdr->n_units[0];
  const int chunk0 = hdr->chunk[0];
  const int n_req0 = hdr->n_req[0];

  if (n_units0 == 0) {
    // no tile-class requests in this call
  } else if (warp == 0) {
    // -------------------------------------------------------- scheduler --
    // Claims one unit ahead: the first at once, each later one when the
    // producer is kTileLead blocks from the end of its current unit.  The
    // whole warp looks the unit up (make_unit_warp); lane 0 claims and
    // publishes it.
    uint32_t ss = 0, sph = 0, rph = 0;
    for (bool first = true;; first = false) {
      if (!first) {
        if (!warp_wait(b_sched_req, rph, ctl)) break;
        rph ^= 1;
      }
      // the first unit of CTA i is unit i; later claims count from the grid size
      int u = (int)blockIdx.x;
      if (!first) {
        if (lane == 0) u = (int)gridDim.x + atomicAdd(&hdr->counter[0], 1);
        u = __shfl_sync(0xffffffffu, u, 0);
      }
      UnitDesc d;
      make_unit_warp(p, req, prefix, n_req0, n_units0, chunk0, p.np, u, d);
      if (!warp_wait(b_sched_empty + 8 * ss, sph ^ 1, ctl)) break;
      if (lane == 0) {
        ring[ss] = d;
        mbar_arrive(b_sched_full + 8 * ss);
      }
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (u >= n_units0) break;
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_k = l2_policy_evict_last();
      const uint32_t q_bytes = (uint32_t)kHalves * 128u * (uint32_t)(p.g * p.np);
      const bool paged = p.layout != 2;
      const int32_t page_oob = (int32_t)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);
      uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0, scs = 0, scph = 0;
      uint32_t n_q = 0, n_k = 0, n_sc = 0;   // loads issued (for the teardown drain)
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
        const int req_at = max(d.c0, d.b1 - kTileLead);
        if (!mbar_wait(b_q_empty + 8 * qb, qph ^ 1, ctl)) break;
        const uint32_t qdst = sbase + L::q_off + qb * kTileBytes;
        mbar_arrive_expect_tx(b_q_full + 8 * qb, q_bytes);
        tma_load_3d(qdst, &tm_q, b_q_full + 8 * qb, 0, d.hk * p.g, d.t0);
        if constexpr (!kF8) tma_load_3d(qdst + kHalfBytes, &tm_q, b_q_full + 8 * qb, 64, d.hk * p.g, d.t0);
        ++n_q;
        if (++qb == L::kQBufs) { qb = 0; qph ^= 1; }
        const int32_t* trow = p.block_table + (int64_t)d.b * p.MB;
        // page indices two pairs ahead (an FP8 pair's MMAs take about one L2
        // round trip); the first pair's pages come with the unit
        int nx0 = d.pg0, nx1 = d.pg1, nn0 = 0, nn1 = 0;
        if (paged) {
          nn0 = d.c0 + 2 < d.b1 ? __ldg(trow + d.c0 + 2) : 0;
          nn1 = d.c0 + 3 < d.b1 ? __ldg(trow + d.c0 + 3) : 0;
        }
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; beta += 2) {
          if (req_at >= beta && req_at < beta + 2) mbar_arrive(b_sched_req);
          const int nblk = beta + 1 < d.b1 ? 2 : 1;
          int pg[2] = {nx0, nx1};
          nx0 = nn0;
          nx1 = nn1;
          if (paged) {
            nn0 = beta + 4 < d.b1 ? __ldg(trow + beta + 4) : 0;
            nn1 = beta + 5 < d.b1 ? __ldg(trow + beta + 5) : 0;
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
          if constexpr (KI8) {
            // one raw int8 page per ring stage, its scales riding along
            for (int j = 0; j < nblk; ++j) {
              if (!mbar_wait(b_raw_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
              raw_page[ks] = paged ? page[j] : tok[j];
              const uint32_t rdst = sbase + L::raw_off + ks * kRawStride;
              const bool with_scale = paged && (int64_t)page[j] < p.NP;
              // int8: a 16 KiB page and its 128 fp32 token scales; FP4: an 8 KiB
              // page and its tokens' group scale bytes
              const uint32_t data_bytes = KF4 ? kRawBytes / 2 : kRawBytes;
              const uint32_t sc_bytes = KF4 ? (uint32_t)(kP * p.fp4_ng) : kRawScaleBytes;
              mbar_arrive_expect_tx(b_raw_full + 8 * ks, data_bytes + (with_scale ? sc_bytes : 0u));
              tma_k(rdst, &tm_k, b_raw_full + 8 * ks, 0, tok[j], d.hk, page[j], p.layout, pol_k);
              if (with_scale) {
                if constexpr (KF4 != 0)
                  bulk_load(rdst + kRawBytes, p.k_scale8 + ((int64_t)page[j] * p.H_kv + d.hk) * kP * p.fp4_ng,
                            sc_bytes, b_raw_full + 8 * ks);
                else
                  bulk_load(rdst + kRawBytes, p.scale + ((int64_t)page[j] * p.H_kv + d.hk) * kP,
                            kRawScaleBytes, b_raw_full + 8 * ks);
              }
              ++n_k;
              if (++ks == R) { ks = 0; kph ^= 1; }
            }
          } else {
            // K half x of both pages into one slot: page j's 128 rows at j * 16 KiB
            // (the mirror is in BNBD order)
            for (int x = 0; x < kHalves && ok; ++x) {
              if (!mbar_wait(b_k_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
              const uint32_t kdst = sbase + L::k_off + ks * L::kSlotBytes;
              mbar_arrive_expect_tx(b_k_full + 8 * ks, (uint32_t)nblk * kHalfBytes);
              for (int j = 0; j < nblk; ++j)
                tma_k(kdst + (uint32_t)j * kHalfBytes, &tm_k, b_k_full + 8 * ks, 64 * x, tok[j], d.hk,
                      page[j], KM ? 1 : p.layout, pol_k);
              ++n_k;
              if (++ks == PS) { ks = 0; kph ^= 1; }
            }
            if constexpr (KM) {
              // the pair's per-token scales into the scale ring (pages outside
              // [0, NP) load as zeros above; their scales are written as zeros)
              if (ok && !mbar_wait(b_sc_empty + 8 * scs, scph ^ 1, ctl)) ok = false;
              if (ok) {
                uint32_t sb = 0;
                for (int j = 0; j < nblk; ++j) {
                  if ((int64_t)page[j] < p.NP) {
                    sb += kRawScaleBytes;
                  } else {
                    float* z = scale_s + scs * 256 + j * 128;
                    for (int c = 0; c < 128; ++c) z[c] = 0.f;
                  }
                }
                mbar_arrive_expect_tx(b_sc_full + 8 * scs, sb);
                for (int j = 0; j < nblk; ++j)
                  if ((int64_t)page[j] < p.NP)
                    bulk_load(sbase + L::sc_off + (uint32_t)(scs * 256 + j * 128) * 4u,
                              p.scale + ((int64_t)page[j] * p.H_kv + d.hk) * kP, kRawScaleBytes,
                              b_sc_full + 8 * scs);
                ++n_sc;
                if (++scs == SC) { scs = 0; scph ^= 1; }
              }
            }
          }
          if (!ok) break;
        }
        if (!ok) break;
      }
      // Teardown: never leave the CTA with a TMA write in flight.  Only the
      // last (ring size) loads of each ring can still be pending.
      constexpr uint32_t kRing = KI8 ? (uint32_t)R : (uint32_t)PS;
      const uint32_t kfull = KI8 ? b_raw_full : b_k_full;
      for (uint32_t j = n_k > kRing ? n_k - kRing : 0; j < n_k; ++j) {
        const uint32_t st = j % kRing, ph = (j / kRing) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(kfull + 8 * st, ph) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
      for (uint32_t j = n_q > (uint32_t)L::kQBufs ? n_q - L::kQBufs : 0; j < n_q; ++j) {
        const uint32_t st = j % L::kQBufs, ph = (j / L::kQBufs) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_q_full + 8 * st, ph) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
      if constexpr (KM) {
        for (uint32_t j = n_sc > (uint32_t)SC ? n_sc - SC : 0; j < n_sc; ++j) {
          const uint32_t st = j % SC, ph = (j / SC) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(b_sc_full + 8 * st, ph) && global_timer_ns() - t0 < kDrainLimitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    // The warp waits on nothing but a named barrier
    // shared with the helper warp, which waits on the mbarriers and passes each
    // K slot on as the popcount of its lanes' predicates (kCode* bits; 0 =
    // stop): an mbarrier wait by this warp would first let its queued MMAs
    // drain, idling the tensor pipe for a few hundred cycles per wait.
    constexpr uint32_t idesc2 = kF8 ? idesc_f8(F8 == 2, 128, 256) : idesc_f16(BF16, 128, 256);
    constexpr uint32_t idesc1 = kF8 ? idesc_f8(F8 == 2, 128, 128) : idesc_f16(BF16, 128, 128);
    uint32_t qb = 0, ks = 0, ab = 0, x = 0;
    bool issued = false;
    for (;;) {
      __syncwarp();   // the barrier counts whole warps: reconverge first
      const uint32_t code = named_bar_popc(kMmaBar, 64, false);
      if (code == 0) break;
      tc_fence_after();
      if (code & kCodeFirst) x = 0;
      {
        // the whole (converged) warp runs the issue, its elected lane issues
        const uint32_t qsrc = sbase + L::q_off + qb * kTileBytes;
        const uint32_t dt = tmem_base + ab * 256u;
        const uint32_t idesc = (code & kCodeLone) ? idesc1 : idesc2;
        const uint32_t ksrc = sbase + L::k_off + ks * L::kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if constexpr (kF8)
            tc_mma_f8_w(dt, desc_at(qsrc, kk), smem_desc_sw128(ksrc + 32u * kk), idesc, kk ? 1u : 0u);
          else
            tc_mma_f16_w(dt, desc_at(qsrc, 4 * (int)x + kk), smem_desc_sw128(ksrc + 32u * kk), idesc,
                         (x | (uint32_t)kk) ? 1u : 0u);
        }
        tc_commit_w(b_k_empty + 8 * ks);   // the slot is free once these four MMAs are done
        if (code & kCodeLast) tc_commit_w(b_acc_full + 8 * ab);
        if (code & kCodeUnitEnd) tc_commit_w(b_q_empty + 8 * qb);
      }
      ++x;
      if (++ks == (uint32_t)PS) ks = 0;
      if ((code & kCodeLast) && ++ab == (uint32_t)L::kAcc) ab = 0;
      if ((code & kCodeUnitEnd) && ++qb == (uint32_t)L::kQBufs) qb = 0;
      issued = true;
    }
    __syncwarp();
    if (issued) {
      // every MMA of this CTA has landed before TMEM is released
      tc_commit_w(b_drain);
      if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_drain, 0) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == Cfg::kThreads / 32 - 1) {
    // ------------------------------------------------------ MMA helper --
    // Waits for what each K slot's MMAs need (the unit's query tile, a free
    // accumulator at a pair's first slot, the slot's pages) and passes the
    // slot on.  Every path out of the loop ends with exactly one stop code,
    // so the MMA warp's barrier waits always pair up.
    uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0, ab = 0, aph = 0;
    // watchdog test: the drain barrier's first phase completes only after the
    // MMA warp's last commit, which waits for this warp, so the wait runs out
    const bool go = !p.stall || warp_wait(b_drain, 0, ctl);
    for (; go;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      if (d.b1 <= d.c0) continue;
      if (!warp_wait(b_q_full + 8 * qb, qph, ctl)) break;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1 && ok; beta += 2) {
        if (!warp_wait(b_acc_empty + 8 * ab, aph ^ 1, ctl)) { ok = false; break; }
        for (int xx = 0; xx < kHalves; ++xx) {
          if (!warp_wait(b_k_full + 8 * ks, kph, ctl)) { ok = false; break; }
          const uint32_t code = kCodeLive | (xx == 0 ? kCodeFirst : 0u) |
                                (xx == kHalves - 1 ? kCodeLast : 0u) |
                                (beta + 1 < d.b1 ? 0u : kCodeLone) |
                                (xx == kHalves - 1 && beta + 2 >= d.b1 ? kCodeUnitEnd : 0u);
          __syncwarp();
          (void)named_bar_popc(kMmaBar, 64, (uint32_t)lane < code);
          if (++ks == PS) { ks = 0; kph ^= 1; }
        }
        if (!ok) break;
        if (++ab == L::kAcc) { ab = 0; aph ^= 1; }
      }
      if (!ok) break;
      if (++qb == L::kQBufs) { qb = 0; qph ^= 1; }
    }
    __syncwarp();
    (void)named_bar_popc(kMmaBar, 64, false);
  } else if (warp < kEpiWarp0 + 4 * L::kGroups) {
    // --------------------------------------------------------- epilogue --
    const int grp = (warp - kEpiWarp0) >> 2;       // block of each pair this group drains
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may read
    const int r = quarter * 32 + lane;             // MMA row = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const float ninf = __int_as_float(0xff800000);
    const int rows = p.g * p.np;
    const int pos = r / p.g;
    const int hl = r - pos * p.g;
    const bool write_out = p.out != nullptr;
    uint32_t ss = 0, sph = 0, ab = 0, aph = 0, sc = 0, scph = 0;
    using Sel = std::conditional_t<TOPK == 2, TopList2, TopList>;
    Sel sel;
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
      // fused selection: the group score of this position for block col
      auto select = [&](float m, int col) {
        if constexpr (TOPK != 0) select_block(sel, m, valid, col, p.MB, hl, p.g);
      };
      if constexpr (TOPK != 0) sel.clear();
      bool ok = true;
      int beta = d.c0;
      for (; beta < d.b1; beta += 2) {
        const uint32_t a = ab, a_ph = aph;
        if (++ab == L::kAcc) { ab = 0; aph ^= 1; }
        if (!warp_wait(b_acc_full + 8 * a, a_ph, ctl)) { ok = false; break; }
        tc_fence_after();
        if constexpr (KM) {
          // this group's block of the pair from the fp16 mirror: the 16-bit
          // path's TMEM loads, then DEQUANT (column multiply by the per-token
          // scale) before the mask
          const uint32_t s = sc, s_ph = scph;
          if (++sc == SC) { sc = 0; scph ^= 1; }
          if (!warp_wait(b_sc_full + 8 * s, s_ph, ctl)) { ok = false; break; }
          const int col = beta + grp;
          const bool has = col < d.b1;
          const bool ld = warp_valid && has;
          const float4* sv = reinterpret_cast<const float4*>(scale_s + s * 256 + grp * 128);
          float m = ninf;
          if constexpr (TOPK != 0) {          // the running selection holds registers
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              float x[64];
              if (ld) {
                tmem_ld64(t_lane + a * 256u + (uint32_t)grp * 128u + 64u * hf, x);
                tmem_wait_ld();
              }
              if (hf == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
              }
              if (ld && valid) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const float4 s4 = sv[16 * hf + c];
                  x[4 * c + 0] *= s4.x;
                  x[4 * c + 1] *= s4.y;
                  x[4 * c + 2] *= s4.z;
                  x[4 * c + 3] *= s4.w;
                }
                m = fmaxf(m, masked_max<64>(x, lim - col * kP - 64 * hf));
              }
            }
          } else {
            float x[128];
            if (ld) {
              tmem_ld128(t_lane + a * 256u + (uint32_t)grp * 128u, x);
              tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
            if (ld && valid) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const float4 s4 = sv[c];
                x[4 * c + 0] *= s4.x;
                x[4 * c + 1] *= s4.y;
                x[4 * c + 2] *= s4.z;
                x[4 * c + 3] *= s4.w;
              }
              m = masked_max<128>(x, lim - col * kP);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_sc_empty + 8 * s);
          if (!has || forced(col)) m = fill_value(col);
          if (valid && write_out) __stcs(orow + col, m);
          select(m, col);
          continue;
        }
        if constexpr (KI8) {
          // this group's block of the pair.  DEQUANT: column multiply by the
          // per-token scale, before the mask; 64-column pieces keep the
          // register footprint down; the accumulator is handed back after the
          // last TMEM load
          const uint32_t s = sc, s_ph = scph;
          if (++sc == SC) { sc = 0; scph ^= 1; }
          if (!warp_wait(b_sc_full + 8 * s, s_ph, ctl)) { ok = false; break; }
          float mb = ninf;
          const int b = grp;
          const bool ld = warp_valid && beta + b < d.b1;
#pragma unroll
          for (int hq = 0; hq < 4; ++hq) {          // 32-column quarters of the block
            float x[32];
            if (ld) {
              tmem_ld32(t_lane + a * 256u + (uint32_t)(128 * b + 32 * hq), x);
              tmem_wait_ld();
            }
            if (hq == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
            }
            if (ld && valid) {
              if constexpr (KF4 == 0) {               // FP4: the scales are in the operands
                const float4* sv = reinterpret_cast<const float4*>(scale_s + s * 256 + b * 128 + hq * 32);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const float4 s4 = sv[c];
                  x[4 * c + 0] *= s4.x;
                  x[4 * c + 1] *= s4.y;
                  x[4 * c + 2] *= s4.z;
                  x[4 * c + 3] *= s4.w;
                }
              }
              mb = fmaxf(mb, masked_max<32>(x, lim - (beta + b) * kP - 32 * hq));
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_sc_empty + 8 * s);
          // local mask after the max: forced blocks take their constant; a
          // lone last block's partner column is a fill column
          const int col = beta + b;
          if (col >= d.b1 || forced(col)) mb = fill_value(col);
          if (valid && write_out) __stcs(orow + col, mb);
          select(mb, col);
          continue;
        }
        const int col = beta + grp;        // this group's block of the pair
        const bool has = col < d.b1;       // else a lone last block's partner (a fill column)
        const bool ld = warp_valid && has;
        float m = ninf;
        if constexpr (TOPK == 16) {
          // two 64-column pieces: the running selection holds the registers
          // that the other half of a 128-column load would take
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float x[64];
            if (ld) {
              tmem_ld64(t_lane + a * 256u + (uint32_t)grp * 128u + 64u * hf, x);
              tmem_wait_ld();
            }
            if (hf == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
            }
            if (ld && valid) m = fmaxf(m, masked_max<64>(x, lim - col * kP - 64 * hf));
          }
        } else {
          float x[128];
          if (ld) {
            tmem_ld128(t_lane + a * 256u + (uint32_t)grp * 128u, x);
            tmem_wait_ld();
          }
          // the accumulator is free once both groups hold their block in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_acc_empty + 8 * a);
          if (ld && valid) m = masked_max<128>(x, lim - col * kP);
        }
        // local mask after the max: forced blocks take their constant
        if (!has || forced(col)) m = fill_value(col);
        if (valid && write_out) __stcs(orow + col, m);
        select(m, col);
      }
      if (!ok) break;
      // one partial selection per (unit, epilogue group): part 2 * chunk + group
      const bool store_sel = valid && 2 * d.ch + 1 < p.cand_parts;
      if constexpr (TOPK != 0) {
        if (grp != 0 && store_sel) sel.store(cand_row(p, d.t0 + pos, d.hk, 2 * d.ch + 1), p.topk_k, hl);
      }
      // columns past the computed pairs (group 0): pairs up to a multiple of
      // 8, then whole groups of closed-form values
      if (grp != 0) continue;
      if constexpr (TOPK != 0) {
        if (live_kv) insert_forced(sel, beta, min(d.c1, p.MB), p.init_blocks, lo, d.sl, hl, p.g);
        if (store_sel) sel.store(cand_row(p, d.t0 + pos, d.hk, 2 * d.ch), p.topk_k, hl);
      }
      if (valid && write_out) {
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
  } else if (warp >= L::kCvtW0 && warp < L::kCvtW0 + 4 * Cfg::kCvtGroups) {
    if constexpr (KI8) {
    // ------------------------------------------- int8 -> fp16 converters --
    // Group cgp converts the pages j of every pair with j % kCvtGroups == cgp,
    // one K slot at a time (elements 0..63 of each row into the pair's first
    // slot, 64..127 into the second), so the MMA can start on the first slot
    // while the second is converted.  Lane
    // mapping: in each 8-lane shared-memory phase, lanes 0..3 take four
    // 16-byte chunks of row a and lanes 4..7 of row a + 4, and the latter
    // write their two output chunks in the opposite order: reads of the
    // swizzled int8 page and writes of the swizzled fp16 rows are then
    // conflict-free.
    const int cgp = (warp - L::kCvtW0) >> 2;
    const int wq = (warp - L::kCvtW0) & 3;                 // warp within the group
    const int ct = wq * 32 + lane;                         // token whose scale this thread moves
    const int ph = lane >> 3, pl = lane & 7;
    const int ci = pl & 3;                                 // 16-byte int8 chunk within the half
    const int rsub = ph + 4 * (pl >> 2);                   // row within an 8-row step
    const bool odd_first = (pl >> 2) != 0;
    uint32_t ss = 0, sph = 0, rc = 0, ks = 0, kph = 0, sc = 0, scph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1 && ok; beta += 2) {
        const int nblk = beta + 1 < d.b1 ? 2 : 1;
        uint32_t rs[2];
        float sv[2] = {0.f, 0.f};
        uint2 gsc[2] = {make_uint2(0u, 0u), make_uint2(0u, 0u)};   // FP4: this token's group scale bytes
        for (int j = cgp; j < nblk && ok; j += Cfg::kCvtGroups) {
          const uint32_t rpage = rc + (uint32_t)j;   // the page's place in the raw ring
          rs[j] = rpage % R;
          if (!warp_wait(b_raw_full + 8 * rs[j], (rpage / R) & 1u, ctl)) { ok = false; break; }
          // this thread's token scale: from the stage (paged) or, for packed
          // keys, a global load issued now so that it overlaps the conversion
          const uint8_t* src = smem + L::raw_off + rs[j] * kRawStride;
          const int page = raw_page[rs[j]];
          if constexpr (KF4 != 0) {
            // FP4: the group scales of token ct (4 bytes MXFP4, 8 bytes NVFP4);
            // the epilogue's token scale is 1
            sv[j] = 1.f;
            const uint8_t* g = nullptr;
            if (p.layout == 2) {
              const int64_t row = (int64_t)page + ct;
              if (row < (int64_t)d.kbase + d.L && row < p.NP)
                g = p.k_scale8 + (row * p.H_kv + d.hk) * (int64_t)p.fp4_ng;
            } else if (page >= 0 && (int64_t)page < p.NP) {
              g = src + kRawBytes + ct * p.fp4_ng;
            }
            if (g) {
              if constexpr (KF4 == 1) gsc[j] = *reinterpret_cast<const uint2*>(g);
              else gsc[j].x = *reinterpret_cast<const uint32_t*>(g);
            }
          } else if (p.layout == 2) {
            const int64_t row = (int64_t)page + ct;      // page holds the first key row here
            if (row < (int64_t)d.kbase + d.L && row < p.NP) sv[j] = __ldg(p.scale + row * p.H_kv + d.hk);
          } else if (page >= 0 && (int64_t)page < p.NP) {
            sv[j] = reinterpret_cast<const float*>(src + kRawBytes)[ct];
          }
        }
        if (!ok) break;
        rc += (uint32_t)nblk;
        for (int x = 0; x < 2; ++x) {
          const uint32_t k = ks, k_ph = kph;
          if (++ks == PS) { ks = 0; kph ^= 1; }
          if (!warp_wait(b_k_empty + 8 * k, k_ph ^ 1, ctl)) { ok = false; break; }
          for (int j = cgp; j < nblk; j += Cfg::kCvtGroups) {
            const uint8_t* src = smem + L::raw_off + rs[j] * kRawStride;
            uint8_t* dst = smem + L::k_off + k * L::kSlotBytes + j * kHalfBytes;
            if constexpr (KF4 != 0) {
              // FP4: thread = token row ct; half x = elements 64x .. 64x+63 =
              // bytes 32x .. 32x+31 of the 64-byte row (64-byte swizzled: chunk
              // c at (c ^ ((row >> 1) & 3)) * 16), written as 8 chunks of 8
              // 16-bit values into the 128-byte swizzled operand row
              const int row = ct;
              const int sw = (row >> 1) & 3;
              const uint4 in0 = *reinterpret_cast<const uint4*>(src + row * 64 + (((2 * x) ^ sw) << 4));
              const uint4 in1 = *reinterpret_cast<const uint4*>(src + row * 64 + (((2 * x + 1) ^ sw) << 4));
              const uint32_t wv[8] = {in0.x, in0.y, in0.z, in0.w, in1.x, in1.y, in1.z, in1.w};
              uint8_t* rowp = dst + row * 128;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                uint4 o;
                if constexpr (KF4 == 1) {
                  // NVFP4: group (64x + 8i) / 16 = 4x + i / 2 of 8 scale bytes
                  const int gi = 4 * x + (i >> 1);
                  const uint32_t sb = ((gi < 4 ? gsc[j].x : gsc[j].y) >> (8 * (gi & 3))) & 0xffu;
                  o = fp4x8_to_f16(wv[i], e4m3_scale2(sb));
                } else {
                  // MXFP4: group (64x + 8i) / 32 = 2x + i / 4 of 4 scale bytes
                  const uint32_t sb = (gsc[j].x >> (8 * (2 * x + (i >> 2)))) & 0xffu;
                  o = fp4x8_to_bf16(wv[i], e8m0_scale(sb));
                }
                *reinterpret_cast<uint4*>(rowp + ((i ^ (row & 7)) << 4)) = o;
              }
            } else {
              int4 raw[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int row = wq * 32 + t * 8 + rsub;
                const int c = 4 * x + ci;
                raw[t] = *reinterpret_cast<const int4*>(src + row * 128 + ((c ^ (row & 7)) << 4));
              }
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int row = wq * 32 + t * 8 + rsub;
                uint32_t hv[8];
                int8x4_to_half4((uint32_t)raw[t].x, hv[0], hv[1]);
                int8x4_to_half4((uint32_t)raw[t].y, hv[2], hv[3]);
                int8x4_to_half4((uint32_t)raw[t].z, hv[4], hv[5]);
                int8x4_to_half4((uint32_t)raw[t].w, hv[6], hv[7]);
                // 16 fp16 values = output chunks 2ci, 2ci + 1 of the 128-byte row
                uint8_t* rowp = dst + row * 128;
                const int ca = (2 * ci + (odd_first ? 1 : 0)) ^ (row & 7);
                const int cb = (2 * ci + (odd_first ? 0 : 1)) ^ (row & 7);
                const uint4 lo = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                const uint4 hi = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                *reinterpret_cast<uint4*>(rowp + (ca << 4)) = odd_first ? hi : lo;
                *reinterpret_cast<uint4*>(rowp + (cb << 4)) = odd_first ? lo : hi;
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_k_full + 8 * k);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0)
          for (int j = cgp; j < nblk; j += Cfg::kCvtGroups) mbar_arrive(b_raw_empty + 8 * rs[j]);
        // the pages' token scales for the epilogue
        const uint32_t s = sc, s_ph = scph;
        if (++sc == SC) { sc = 0; scph ^= 1; }
        if (!warp_wait(b_sc_empty + 8 * s, s_ph ^ 1, ctl)) { ok = false; break; }
        for (int j = cgp; j < nblk; j += Cfg::kCvtGroups) scale_s[s * 256 + j * 128 + ct] = sv[j];
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sc_full + 8 * s);
      }
      if (!ok) break;
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

// Launch one instantiation: persistent grid of one CTA per SM, programmatic
// dependent launch after the plan kernel.
template <bool KI8, bool BF16, int F8, int TOPK, int KF4 = 0, bool KM = false>
inline cudaError_t launch_tile_variant(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  using L = TileLayout<tile_mode(KI8, KM)>;
  auto kern = tile_kernel<KI8, BF16, F8, TOPK, KF4, KM>;
  static std::atomic<uint64_t> configured[64];   // per device: context the limit was raised in
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(kern, (int)L::bytes, configured, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_sms);
  cfg.blockDim = dim3(TileCfg<tile_mode(KI8, KM)>::kThreads);
  cfg.dynamicSmemBytes = L::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tq),
                            *static_cast<const CUtensorMap*>(tk), p);
}

// The plain scores, or the fused per-group selection when p.topk_k > 0.
template <bool KI8, bool BF16, int F8, bool KM = false>
inline cudaError_t launch_tile(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  if (p.topk_k <= 0) return launch_tile_variant<KI8, BF16, F8, 0, 0, KM>(tq, tk, p, s);
  return p.g >= 8 ? launch_tile_variant<KI8, BF16, F8, 2, 0, KM>(tq, tk, p, s)
                  : launch_tile_variant<KI8, BF16, F8, 16, 0, KM>(tq, tk, p, s);
}

}  // namespace msa
