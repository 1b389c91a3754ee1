// Persistent block-score kernel for short-query requests with int8 or FP4
// keys (Lq * g <= 32 query rows: decode and speculative decode), sm_103a.
//
// The MMA is turned around with respect to the tile kernel: the 128 tokens of
// one key page are the M side and the request's query rows are the N side,
//     D[token, row] = K_page (128 x 128) * Q_rows^T (128 x N), N = 16 or 32
// so a page costs eight small MMAs instead of a 128 x 128 x 128 product.  The
// block max is then a max over TMEM lanes: each epilogue warp reduces its 32
// tokens for all rows with a butterfly of shuffles, and a separate warp
// combines the four partial maxima of each block (feature request
// "MsaIndexScore", "calculation": DOT -> DEQUANT -> MASK -> MAX, with the
// per-token scale applied per lane before the mask).
//
// int8 keys never touch shared memory as fp16: converter warps read the int8
// page (TMA, 128-byte swizzle), convert one token row per thread and store it
// straight into tensor memory, where the MMA reads its A operand; the token's
// scale goes into a TMEM column that the epilogue reads with the accumulator.
// FP4 pages (E2M1 codes, 64-byte rows, 64-byte swizzle, with their group
// scale bytes) take the same route: a converter dequantises its token row
// exactly into the 16-bit operand type (fp16 for NVFP4, bf16 for MXFP4; the
// MiniMax Sparse Attention notes, sec. 8.2, "FP4 Indexer") and there is no
// per-token scale.
//
// Pipeline granularity.  Per page there is little arithmetic, and an mbarrier
// wait costs a warp ~100-150 cycles even when the phase is already complete.
// So every stage works on items of two consecutive pages of a unit: one TMA
// stage, one converted-A slot, one accumulator pair, one partial-maximum slot
// and one set of waits per item.
//
// The MMA warp never waits on an mbarrier: any shared-memory access by the
// warp that issues tcgen05.mma first lets its queued MMAs drain, which with
// these small MMAs idles the tensor pipe for a few hundred cycles per wait.  A
// helper warp waits instead and passes each item on through a named barrier
// (bar.red.popc: the count of the helper's set predicates is the item's code),
// which keeps the queue flowing.
//
// Roles (one CTA per SM, units fetched from the short class's counter):
//   warp 0        scheduler         warp 1  TMEM owner + MMA issuer
//   warp 2        TMA producer      warp 3  combine: the four partial maxima of
//                                           each block, local mask, stores
//   warps 4..7    epilogue (partial maxima per token quarter)
//   warps 8..11   converters (one token quarter of both pages of an item)
//   warp 12       MMA helper: waits for each item's operands
#pragma once
#include <atomic>
#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_fp16.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

struct Short8 {
  static constexpr int kCombineWarp = 3;
  static constexpr int kEpiW0 = 4;
  static constexpr int kCvtW0 = 8;
  // converter warp sets (set s converts pages s, s + kCvtSets, ... of an item);
  // more sets put more than four warps on a sub-partition, which caps the
  // registers of every warp at 96
  static constexpr int kCvtSets = 1;
  static constexpr int kCvtWarps = 4 * kCvtSets;
  static constexpr int kHelperWarp = kCvtW0 + kCvtWarps;
  static constexpr int kThreads = 32 * (kHelperWarp + 1);
  static constexpr uint32_t kMmaBar = 1;                 // named barrier: helper -> MMA warp
  // item codes passed through that barrier (0 = no more items)
  static constexpr uint32_t kCodeLive = 1, kCodeTwo = 2, kCodeNarrow = 4, kCodeLast = 8;
  static constexpr uint32_t kPageBytes = 16384 + 1024;   // int8 page + its 128 scales
  static constexpr int kStages = 5;                      // items (two pages) in flight
  static constexpr uint32_t kStageBytes = 2 * kPageBytes;
  static constexpr int kN = kShortRows;                  // MMA N: the request's query rows, padded
  static constexpr int kA = 2;                           // converted items (2 x 64 columns each)
  static constexpr int kD = 3;                           // accumulator items (2 x kN columns each)
  static constexpr uint32_t kDCol0 = kA * 128;
  static constexpr uint32_t kScCol0 = kDCol0 + kD * 2 * kN;   // per-token scale ring, one column a page
  static constexpr uint32_t kScCols = kTmemCols - kScCol0;
  static constexpr int kRed = 8;                         // partial-maximum ring (items)
  static constexpr uint32_t kQHalf = kN * 128;           // one 64-element half of the query rows
  static constexpr uint32_t kQBytes = 2 * kQHalf;
  static constexpr int kQBufs = 4;                      // query rows of the next units (8 KiB each)
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kQBufs * kQBytes;
  static constexpr uint32_t red_off = k_off + kStages * kStageBytes;
  static constexpr uint32_t red_bytes = kRed * 4 * 2 * kN * 4;   // [item][quarter][page][row]
  static constexpr uint32_t ring_off = red_off + red_bytes;
  // the first kReqCache request records and the short class's unit prefix
  // sums, copied once so that a claim costs one atomic and no dependent
  // global loads
  static constexpr int kReqCache = 128;
  static constexpr uint32_t req_off = ring_off + kSched * sizeof(UnitDesc);
  static constexpr uint32_t pfx_off = req_off + kReqCache * sizeof(ReqInfo);
  static constexpr uint32_t bar_off = pfx_off + kReqCache * 4;
  static constexpr uint32_t n_bars =
      2 * kSched + 2 * kQBufs + 2 * kStages + 2 * kA + 2 * kD + 2 * kRed + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t end = misc_off + 16 + 8 * kStages;
  static constexpr uint32_t bytes = end + 1024;
};

static_assert(Short8::bytes <= 232448, "shared memory per CTA");
// Regions in address order without overlap (nothing but mbarrier operations
// and tcgen05.commit touches the barrier words); swizzled tiles 1 KiB aligned.
static_assert(Short8::q_off % 1024 == 0 && Short8::k_off % 1024 == 0 &&
                  Short8::kQBytes % 1024 == 0 && Short8::kPageBytes % 1024 == 0 &&
                  Short8::q_off + Short8::kQBufs * Short8::kQBytes <= Short8::k_off &&
                  kRawBytes + kRawScaleBytes <= Short8::kPageBytes &&
                  Short8::k_off + Short8::kStages * Short8::kStageBytes <= Short8::red_off &&
                  Short8::red_off + Short8::red_bytes <= Short8::ring_off &&
                  Short8::ring_off + kSched * sizeof(UnitDesc) <= Short8::req_off &&
                  Short8::req_off + Short8::kReqCache * sizeof(ReqInfo) <= Short8::pfx_off &&
                  Short8::pfx_off + Short8::kReqCache * 4 <= Short8::bar_off &&
                  Short8::bar_off % 8 == 0 &&
                  Short8::bar_off + Short8::n_bars * 8 <= Short8::misc_off &&
                  Short8::misc_off + 16 + 8 * Short8::kStages <= Short8::end,
              "short-query kernel shared-memory layout");
// A converter writes page p's scale into column p % kScCols once the MMAs of
// the item kA back are done; by then the epilogue has read every page up to
// (kA + kD) items back, so the ring never overwrites an unread scale.
static_assert(Short8::kScCols >= 2 * (Short8::kA + Short8::kD + 1), "scale ring too short");

// Butterfly transpose-reduction: lane l holds 32 values (one per column);
// returns, on lane c, the max over all 32 lanes of column c.  31 shuffles.
__device__ __forceinline__ float warp_transpose_max32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = upper ? v[w + i] : v[i];
      const float send = upper ? v[i] : v[w + i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
  return v[0];
}

// TOPK: the fused per-group selection (0 = off).  The combine warp keeps,
// per query position, a running top-kTopkMax list of the group score (the max
// over the position's g head lanes, g dividing 32) over every block of a unit
// and writes it as the unit's partial list (part 2 * chunk; part 2 * chunk + 1
// is written empty); the scores are stored only if p.out is not null.
// TOPK = 2: the list is spread over 8 lanes of the position (g >= 8);
// TOPK = 16: every lane of the position holds the whole list.
// KF4: FP4 key pages instead of int8, 1 = NVFP4 (E4M3 scale per 16 elements,
// fp16 operands), 2 = MXFP4 (E8M0 scale per 32, bf16 operands).
template <bool BF16, int TOPK = 0, int KF4 = 0>
__global__ void __launch_bounds__(Short8::kThreads, 1)
    short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const Params p) {
  using C = Short8;
  constexpr int S = C::kStages;
  static_assert(KF4 == 0 || BF16 == (KF4 == 2), "FP4 operand type: fp16 for NVFP4, bf16 for MXFP4");
  constexpr bool kTokScale = KF4 == 0;                   // int8: DEQUANT by the per-token scale
  // bytes of one page in a stage: int8 16 KiB, FP4 8 KiB of codes
  constexpr uint32_t kData = KF4 ? kRawBytes / 2 : kRawBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  UnitDesc* ring = reinterpret_cast<UnitDesc*>(smem + C::ring_off);
  float* red = reinterpret_cast<float*>(smem + C::red_off);
  const uint32_t b_sched_full = sbase + C::bar_off;
  const uint32_t b_sched_empty = b_sched_full + 8 * kSched;
  const uint32_t b_q_full = b_sched_empty + 8 * kSched;
  const uint32_t b_q_empty = b_q_full + 8 * C::kQBufs;
  const uint32_t b_st_full = b_q_empty + 8 * C::kQBufs;      // item's int8 pages landed
  const uint32_t b_st_empty = b_st_full + 8 * S;             // item's pages read by the converters
  const uint32_t b_a_full = b_st_empty + 8 * S;              // item converted into TMEM
  const uint32_t b_a_free = b_a_full + 8 * C::kA;            // its MMAs are done
  const uint32_t b_d_full = b_a_free + 8 * C::kA;            // item's accumulators ready
  const uint32_t b_d_free = b_d_full + 8 * C::kD;            // accumulators read by the epilogue
  const uint32_t b_red_full = b_d_free + 8 * C::kD;          // four partial maxima written
  const uint32_t b_red_empty = b_red_full + 8 * C::kRed;     // partial maxima combined
  const uint32_t b_drain = b_red_empty + 8 * C::kRed;
  const uint32_t b_sched_req = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::misc_off + 4);
  volatile int* raw_page = reinterpret_cast<volatile int*>(smem + C::misc_off + 16);   // [stage][2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // readers of each unit descriptor: producer, MMA helper, combine, 4 epilogue, the converter warps
  constexpr int kConsumers = 7 + C::kCvtWarps;

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
    for (int i = 0; i < S; ++i) {
      mbar_init(b_st_full + 8 * i, 1);
      mbar_init(b_st_empty + 8 * i, C::kCvtWarps);
    }
    for (int i = 0; i < C::kA; ++i) {
      mbar_init(b_a_full + 8 * i, C::kCvtWarps);
      mbar_init(b_a_free + 8 * i, 1);
    }
    for (int i = 0; i < C::kD; ++i) {
      mbar_init(b_d_full + 8 * i, 1);
      mbar_init(b_d_free + 8 * i, 4);
    }
    for (int i = 0; i < C::kRed; ++i) {
      mbar_init(b_red_full + 8 * i, 4);
      mbar_init(b_red_empty + 8 * i, 1);
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

  // The plan written by the plan kernel is visible after this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  // The header fields (constant during this grid) and, in warp 0, the first
  // request records and the class's prefix sums are fetched together: their
  // addresses depend only on B, so the first claim waits one round trip.
  const int n_units = hdr->n_units[1];
  const int n_req0 = hdr->n_req[0];
  const int n_req = hdr->n_req[1];
  const int chunk = hdr->chunk[1];
  const int n_cache = p.B < C::kReqCache ? (int)p.B : C::kReqCache;
  if (warp == 0) {
    constexpr int kV = C::kReqCache * (int)(sizeof(ReqInfo) / 16) / 32;   // int4 per lane
    constexpr int kP = C::kReqCache / 32;
    const int4* grec = reinterpret_cast<const int4*>(p.ws + sizeof(PlanHeader));
    const int32_t* gpfx = plan_prefix(p.ws, p.B, 1);
    const int n4 = n_cache * (int)(sizeof(ReqInfo) / 16);
    int4 v[kV];
    int32_t pf[kP];
#pragma unroll
    for (int k = 0; k < kV; ++k)
      if (lane + 32 * k < n4) v[k] = grec[lane + 32 * k];
#pragma unroll
    for (int k = 0; k < kP; ++k)
      if (lane + 32 * k < n_cache) pf[k] = gpfx[lane + 32 * k];
    int4* crec = reinterpret_cast<int4*>(smem + C::req_off);
    int32_t* cpfx = reinterpret_cast<int32_t*>(smem + C::pfx_off);
#pragma unroll
    for (int k = 0; k < kV; ++k)
      if (lane + 32 * k < n4) crec[lane + 32 * k] = v[k];
#pragma unroll
    for (int k = 0; k < kP; ++k)
      if (lane + 32 * k < n_cache) cpfx[lane + 32 * k] = pf[k];
    __syncwarp();
  }
  WaitCtl ctl{abort_flag, &hdr->err, p.wait_limit_ns};

  if (n_units == 0) {
    // no short requests in this call
  } else if (warp == 0) {
    // -------------------------------------------------------- scheduler --
    const bool cached = n_req0 + n_req <= n_cache;
    const ReqInfo* req = (cached ? reinterpret_cast<const ReqInfo*>(smem + C::req_off)
                                 : reinterpret_cast<const ReqInfo*>(p.ws + sizeof(PlanHeader))) + n_req0;
    const int32_t* prefix = cached ? reinterpret_cast<const int32_t*>(smem + C::pfx_off) : plan_prefix(p.ws, p.B, 1);
    if (lane == 0) {
      uint32_t ss = 0, sph = 0, rph = 0;
      for (bool first = true;; first = false) {
        if (!first) {
          if (!mbar_wait(b_sched_req, rph, ctl)) break;
          rph ^= 1;
        }
        UnitDesc d;
        // the first unit of CTA i is unit i; later claims count from the grid size
        make_unit(p, req, prefix, n_req, n_units, chunk, p.np_short,
                  first ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&hdr->counter[1], 1), d);
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
      const uint64_t pol_k = l2_policy_evict_first();
      const uint32_t q_bytes = 2u * 128u * (uint32_t)(p.g * p.np_short);
      const bool paged = p.layout != 2;
      const int page_oob = (int)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);
      // a page's scales: 128 fp32 token scales (int8) or 128 rows of FP4
      // group scale bytes (4 MXFP4, 8 NVFP4)
      const uint32_t sc_bytes = KF4 ? (uint32_t)(kP * p.fp4_ng) : kRawScaleBytes;
      uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0;
      uint32_t n_q = 0, n_k = 0;
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
        const uint32_t qdst = sbase + C::q_off + qb * C::kQBytes;
        mbar_arrive_expect_tx(b_q_full + 8 * qb, q_bytes);
        tma_load_3d(qdst, &tm_q, b_q_full + 8 * qb, 0, d.hk * p.g, d.t0);
        tma_load_3d(qdst + C::kQHalf, &tm_q, b_q_full + 8 * qb, 64, d.hk * p.g, d.t0);
        ++n_q;
        if (++qb == C::kQBufs) { qb = 0; qph ^= 1; }
        const int32_t* trow = p.block_table + (int64_t)d.b * p.MB;
        int nx0 = d.pg0, nx1 = d.pg1;   // the first pair's pages come with the unit
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; beta += 2) {
          if (req_at >= beta && req_at < beta + 2) mbar_arrive(b_sched_req);
          const int npg = beta + 1 < d.b1 ? 2 : 1;
          int pg[2] = {nx0, nx1};
          if (paged) {
            nx0 = beta + 2 < d.b1 ? __ldg(trow + beta + 2) : 0;
            nx1 = beta + 3 < d.b1 ? __ldg(trow + beta + 3) : 0;
          }
          if (!mbar_wait(b_st_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
          const uint32_t dst = sbase + C::k_off + ks * C::kStageBytes;
          uint32_t bytes = 0;
          bool with_scale[2] = {false, false};
          for (int j = 0; j < npg; ++j) {
            int page = 0, tok = 0;
            if (paged) {
              page = pg[j];
              if (page < 0 || (int64_t)page >= p.NP) {
                atomicOr(&hdr->err, kErrBlockTable);
                page = page_oob;   // out of bounds: zero fill
              }
              pg[j] = page;
              with_scale[j] = (int64_t)page < p.NP;
            } else {
              tok = d.kbase + (beta + j) * kP;
              pg[j] = tok;
            }
            raw_page[2 * ks + j] = pg[j];
            bytes += kData + (with_scale[j] ? sc_bytes : 0u);
          }
          mbar_arrive_expect_tx(b_st_full + 8 * ks, bytes);
          for (int j = 0; j < npg; ++j) {
            const uint32_t pdst = dst + (uint32_t)j * C::kPageBytes;
            tma_k(pdst, &tm_k, b_st_full + 8 * ks, 0, paged ? 0 : pg[j], d.hk, paged ? pg[j] : 0,
                  p.layout, pol_k);
            if (with_scale[j]) {
              if constexpr (KF4 != 0)
                bulk_load(pdst + kRawBytes, p.k_scale8 + ((int64_t)pg[j] * p.H_kv + d.hk) * kP * p.fp4_ng,
                          sc_bytes, b_st_full + 8 * ks);
              else
                bulk_load(pdst + kRawBytes, p.scale + ((int64_t)pg[j] * p.H_kv + d.hk) * kP,
                          kRawScaleBytes, b_st_full + 8 * ks);
            }
          }
          ++n_k;
          if (++ks == S) { ks = 0; kph ^= 1; }
        }
        if (!ok) break;
      }
      // never leave the CTA with a TMA write in flight
      for (uint32_t j = n_k > (uint32_t)S ? n_k - S : 0; j < n_k; ++j) {
        const uint32_t st = j % S, ph = (j / S) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_st_full + 8 * st, ph) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
      for (uint32_t j = n_q > (uint32_t)C::kQBufs ? n_q - C::kQBufs : 0; j < n_q; ++j) {
        const uint32_t st = j % C::kQBufs, ph = (j / C::kQBufs) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_q_full + 8 * st, ph) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    // Items are numbered in stream order (it); item it uses A slot it % kA and
    // accumulator pair it % kD.  The warp touches no shared memory: the helper
    // warp does the waiting and hands over each item through a named barrier
    // whose thread count carries the item's code (kCode* bits; 0 = stop), so
    // the MMAs of one item are still running while the next is issued.
    constexpr uint32_t idesc32 = idesc_f16(BF16, 128, 32);
    constexpr uint32_t idesc16 = idesc_f16(BF16, 128, 16);
    uint32_t qb = 0, it = 0;
    bool issued = false;
    for (;; ++it) {
      __syncwarp();   // the barrier counts whole warps: reconverge first
      const uint32_t code = named_bar_popc(C::kMmaBar, 64, false);
      if (code == 0) break;
      tc_fence_after();
      {
        // the whole (converged) warp runs the issue, its elected lane issues
        const uint32_t as = it % C::kA, ds = it % C::kD;
        const uint32_t qsrc = sbase + C::q_off + qb * C::kQBytes;
        const uint32_t idesc = (code & C::kCodeNarrow) ? idesc16 : idesc32;   // N = 16 or 32 query rows
        const int npg = (code & C::kCodeTwo) ? 2 : 1;
        for (int j = 0; j < npg; ++j) {
          const uint32_t at = tmem_base + as * 128u + 64u * j;
          const uint32_t dt = tmem_base + C::kDCol0 + ds * (2u * C::kN) + (uint32_t)C::kN * j;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma_f16_ta_w(dt, at + 8u * k,
                            smem_desc_sw128(qsrc + (uint32_t)(k >> 2) * C::kQHalf + (k & 3) * 32u),
                            idesc, k > 0 ? 1u : 0u);
        }
        tc_commit_w(b_a_free + 8 * as);
        tc_commit_w(b_d_full + 8 * ds);
        if (code & C::kCodeLast) tc_commit_w(b_q_empty + 8 * qb);
      }
      if (code & C::kCodeLast) qb = qb + 1 == (uint32_t)C::kQBufs ? 0u : qb + 1;
      issued = true;
    }
    __syncwarp();
    if (issued) {
      tc_commit_w(b_drain);
      if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_drain, 0) && global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == C::kHelperWarp) {
    // ------------------------------------------------------ MMA helper --
    // Waits for what each item's MMAs read (the unit's query rows, the
    // converted page pair, which also implies a free accumulator pair) and
    // passes the item to the MMA warp.  Every path out of the loop ends with
    // exactly one stop code, so the MMA warp's barrier waits always pair up.
    uint32_t ss = 0, sph = 0, qb = 0, qph = 0, it = 0;
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
      const uint32_t narrow = d.Lq * p.g <= 16 ? C::kCodeNarrow : 0u;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; beta += 2, ++it) {
        // the first converter warp saw the accumulator pair free before it
        // arrived, so one wait covers both operands' readiness
        if (!warp_wait(b_a_full + 8 * (it % C::kA), (it / C::kA) & 1u, ctl)) {
          ok = false;
          break;
        }
        const uint32_t code = C::kCodeLive | narrow | (beta + 1 < d.b1 ? C::kCodeTwo : 0u) |
                              (beta + 2 >= d.b1 ? C::kCodeLast : 0u);
        __syncwarp();
        (void)named_bar_popc(C::kMmaBar, 64, (uint32_t)lane < code);
      }
      if (!ok) break;
      if (++qb == C::kQBufs) { qb = 0; qph ^= 1; }
    }
    __syncwarp();
    (void)named_bar_popc(C::kMmaBar, 64, false);
  } else if (warp >= C::kEpiW0 && warp < C::kEpiW0 + 4) {
    // --------------------------------------------------------- epilogue --
    // Every warp reduces its 32 tokens of each page of an item for all rows
    // and posts the partial maxima to a ring that the combine warp drains.
    const int quarter = warp & 3;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const float ninf = __int_as_float(0xff800000);
    uint32_t ss = 0, sph = 0, rr = 0, rph = 0, it = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      const bool narrow = d.Lq * p.g <= 16;               // the MMA used N = 16
      // first visible row for a token t: rows r with floor(r / g) >= t - (L - Lq)
      // (sparse_mode 3), all rows if t < L (mode 0); no row if t >= L
      const int qbase = p.sparse_mode == 3 ? d.L - d.Lq : 0x3fffffff;
      auto first_row = [&](int beta) -> int {
        const int t = beta * kP + quarter * 32 + lane;    // this lane's token of block beta
        if (t >= d.L) return C::kN;
        if (t <= qbase) return 0;
        const int64_t m = (int64_t)(t - qbase) * p.g;
        return m > C::kN ? C::kN : (int)m;
      };
      // both pages of the item below the kv length and at or before the
      // first row's position: nothing to mask (warp-uniform)
      auto all_visible = [&](int beta, bool two) -> bool {
        const int t_end = (beta + 2) * kP;                // one past the item's last token
        return two && t_end <= d.L && t_end - 1 <= qbase;
      };
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; beta += 2, ++it) {
        const uint32_t ds = it % C::kD;
        const bool two = beta + 1 < d.b1;
        if (!warp_wait(b_d_full + 8 * ds, (it / C::kD) & 1u, ctl)) { ok = false; break; }
        tc_fence_after();
        // page p's scale sits in column p % kScCols; items hold pages 2it, 2it + 1
        const uint32_t dcol = t_lane + C::kDCol0 + ds * (2u * C::kN);
        const uint32_t scol = t_lane + C::kScCol0;
        const float sc0 = kTokScale ? tmem_ld1(scol + (2u * it) % C::kScCols) : 1.f;
        const float sc1 = kTokScale ? tmem_ld1(scol + (2u * it + 1u) % C::kScCols) : 1.f;
        float* rslot = red + rr * (4 * 2 * C::kN) + quarter * (2 * C::kN);
        if (narrow) {
          // both pages' 16 columns in one 32-wide transpose: lane c < 16 gets
          // row c of the first page, lane c >= 16 row c - 16 of the second
          float x[32];
          tmem_ld16(dcol, *reinterpret_cast<float(*)[16]>(&x[0]));
          tmem_ld16(dcol + C::kN, *reinterpret_cast<float(*)[16]>(&x[16]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_d_free + 8 * ds);
          if (all_visible(beta, two)) {
            if constexpr (kTokScale) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                x[c] *= sc0;                                     // DEQUANT
                x[16 + c] *= sc1;
              }
            }
          } else {
            const int n0 = first_row(beta), n1 = two ? first_row(beta + 1) : C::kN;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              x[c] = c >= n0 ? x[c] * sc0 : ninf;               // DEQUANT, MASK
              x[16 + c] = c >= n1 ? x[16 + c] * sc1 : ninf;
            }
          }
          const float mine = warp_transpose_max32(x, lane);
          if (!warp_wait(b_red_empty + 8 * rr, rph ^ 1, ctl)) { ok = false; break; }
          rslot[(lane >> 4) * C::kN + (lane & 15)] = mine;
        } else {
          float x0[32], x1[32];
          tmem_ld32(dcol, x0);
          tmem_ld32(dcol + C::kN, x1);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_d_free + 8 * ds);
          if (all_visible(beta, two)) {
            if constexpr (kTokScale) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                x0[c] *= sc0;
                x1[c] *= sc1;
              }
            }
          } else {
            const int n0 = first_row(beta), n1 = two ? first_row(beta + 1) : C::kN;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              x0[c] = c >= n0 ? x0[c] * sc0 : ninf;
              x1[c] = c >= n1 ? x1[c] * sc1 : ninf;
            }
          }
          const float m0 = warp_transpose_max32(x0, lane);
          const float m1 = warp_transpose_max32(x1, lane);
          if (!warp_wait(b_red_empty + 8 * rr, rph ^ 1, ctl)) { ok = false; break; }
          rslot[lane] = m0;
          rslot[C::kN + lane] = m1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(b_red_full + 8 * rr);
        if (++rr == C::kRed) { rr = 0; rph ^= 1; }
      }
      if (!ok) break;
    }
  } else if (warp == C::kCombineWarp) {
    // ---------------------------------------------------------- combine --
    // Lane r owns output row r = (position r / g, head r % g): the max of the
    // four partial maxima of each computed block, the local-mask constants, the
    // fill of the other columns, and 16-byte stores of 4 blocks at a time.
    const float ninf = __int_as_float(0xff800000);
    const bool write_out = p.out != nullptr;
    uint32_t ss = 0, sph = 0, rr = 0, rph = 0;
    using Sel = std::conditional_t<TOPK == 2, TopList2, TopList>;
    Sel sel;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      const int rows = d.Lq * p.g;                        // valid query rows (<= 32)
      const bool row_valid = lane < rows;
      if constexpr (TOPK != 0) sel.clear();
      const int hl = lane - (lane / p.g) * p.g;
      auto select = [&](float m, int col) {
        if constexpr (TOPK != 0) select_block(sel, m, row_valid, col, p.MB, hl, p.g);
      };
      const int pos = lane / p.g;
      const int h = d.hk * p.g + (lane - pos * p.g);
      float* orow = p.out + ((int64_t)h * p.T + (d.t0 + pos)) * (int64_t)p.MBp;
      const int lo = max(0, d.sl + 1 - p.local_blocks);
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
      float v[4];
      bool ok = true;
      int beta = d.c0;
      for (; beta < d.b1; beta += 2) {
        if (!warp_wait(b_red_full + 8 * rr, rph, ctl)) { ok = false; break; }
        const float* r4 = red + rr * (4 * 2 * C::kN) + lane;
        float m0 = fmax3(r4[0], r4[2 * C::kN], fmaxf(r4[4 * C::kN], r4[6 * C::kN]));
        float m1 = fmax3(r4[C::kN], r4[3 * C::kN], fmaxf(r4[5 * C::kN], r4[7 * C::kN]));
        __syncwarp();
        if (lane == 0) mbar_arrive(b_red_empty + 8 * rr);
        if (++rr == C::kRed) { rr = 0; rph ^= 1; }
        // local mask after the max; a lone last block's partner is a fill column
        if (forced(beta)) m0 = fill_value(beta);
        if (beta + 1 >= d.b1 || forced(beta + 1)) m1 = fill_value(beta + 1);
        select(m0, beta);
        select(m1, beta + 1);
        // 16-byte stores of 4 columns (units start on multiples of 4)
        if ((beta & 3) == 0) {
          v[0] = m0;
          v[1] = m1;
        } else {
          v[2] = m0;
          v[3] = m1;
          if (row_valid && write_out)
            __stcs(reinterpret_cast<float4*>(orow + (beta - 2)), make_float4(v[0], v[1], v[2], v[3]));
        }
      }
      if (!ok) break;
      if constexpr (TOPK != 0) {
        // the forced columns past the computed pairs, then this unit's partial
        // list (and an empty second list: every unit owns two parts)
        if (live_kv) insert_forced(sel, beta, min(d.c1, p.MB), p.init_blocks, lo, d.sl, hl, p.g);
        if (row_valid && 2 * d.ch + 1 < p.cand_parts) {
          sel.store(cand_row(p, d.t0 + pos, d.hk, 2 * d.ch), p.topk_k, hl);
          Sel none;
          none.clear();
          none.store(cand_row(p, d.t0 + pos, d.hk, 2 * d.ch + 1), p.topk_k, hl);
        }
      }
      if (row_valid && write_out) {
        if (beta & 3) {   // an open group of 4 (beta is even): close it with fill columns
          v[2] = fill_value(beta);
          v[3] = fill_value(beta + 1);
          __stcs(reinterpret_cast<float4*>(orow + (beta - 2)), make_float4(v[0], v[1], v[2], v[3]));
          beta += 2;
        }
        for (; beta < d.c1; beta += 4)
          __stcs(reinterpret_cast<float4*>(orow + beta), make_float4(fill_value(beta), fill_value(beta + 1),
                                                                     fill_value(beta + 2), fill_value(beta + 3)));
      }
    }
  } else if (warp >= C::kCvtW0 && warp < C::kCvtW0 + C::kCvtWarps) {
    // ------------------------------ int8 or FP4 -> 16 bits into TMEM --
    // Warp q of set s converts token rows 32q..32q+31 of pages s, s + kCvtSets,
    // ... of every item (its TMEM lane quarter is q = warp % 4).
    const int quarter = warp & 3;
    const int set = (warp - C::kCvtW0) >> 2;
    const int row = quarter * 32 + lane;                  // token row of the page
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t ss = 0, sph = 0, it = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; beta += 2, ++it) {
        const uint32_t rs = it % S, as = it % C::kA;
        const int npg = beta + 1 < d.b1 ? 2 : 1;
        if (!warp_wait(b_st_full + 8 * rs, (it / S) & 1u, ctl)) { ok = false; break; }
        if (set >= npg) {                                 // no page of this item: the stage is read
          __syncwarp();
          if (lane == 0) mbar_arrive(b_st_empty + 8 * rs);
        }
        for (int jp = set; jp < npg; jp += C::kCvtSets) {
          const bool last_read = jp + C::kCvtSets >= npg;
          const uint8_t* src = smem + C::k_off + rs * C::kStageBytes + (uint32_t)jp * C::kPageBytes;
          const int page = raw_page[2 * rs + jp];
          uint32_t hv[64];
          float sv = 0.f;
          if constexpr (KF4 != 0) {
            // this token's group scale bytes (8 NVFP4, 4 MXFP4): from the stage
            // (paged) or from global memory (packed keys)
            uint2 gs = make_uint2(0u, 0u);
            const uint8_t* g = nullptr;
            if (p.layout == 2) {
              const int64_t trow = (int64_t)page + row;   // page holds the first key row here
              if (trow < (int64_t)d.kbase + d.L && trow < p.NP)
                g = p.k_scale8 + (trow * p.H_kv + d.hk) * (int64_t)p.fp4_ng;
            } else if (page >= 0 && (int64_t)page < p.NP) {
              g = src + kRawBytes + row * p.fp4_ng;
            }
            if (g) {
              if constexpr (KF4 == 1) gs = *reinterpret_cast<const uint2*>(g);
              else gs.x = *reinterpret_cast<const uint32_t*>(g);
            }
            // the 64-byte row of codes, 64-byte swizzled: chunk c at (c ^ ((row >> 1) & 3)) * 16
            const int sw = (row >> 1) & 3;
            uint4 in[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              in[c] = *reinterpret_cast<const uint4*>(src + row * 64 + ((c ^ sw) << 4));
            if (last_read) {
              __syncwarp();
              if (lane == 0) mbar_arrive(b_st_empty + 8 * rs);
            }
            // word w = elements 8w .. 8w+7 (element 2i in the low nibble of byte i)
#pragma unroll
            for (int w = 0; w < 16; ++w) {
              const uint4 v4 = in[w >> 2];
              const uint32_t word = (w & 3) == 0 ? v4.x : (w & 3) == 1 ? v4.y : (w & 3) == 2 ? v4.z : v4.w;
              uint4 o;
              if constexpr (KF4 == 1) {
                const int gi = w >> 1;                    // group of 16 elements
                const uint32_t sb = ((gi < 4 ? gs.x : gs.y) >> (8 * (gi & 3))) & 0xffu;
                o = fp4x8_to_f16(word, e4m3_scale2(sb));
              } else {
                const uint32_t sb = (gs.x >> (8 * (w >> 2))) & 0xffu;   // group of 32 elements
                o = fp4x8_to_bf16(word, e8m0_scale(sb));
              }
              hv[4 * w + 0] = o.x;
              hv[4 * w + 1] = o.y;
              hv[4 * w + 2] = o.z;
              hv[4 * w + 3] = o.w;
            }
          } else {
            if (p.layout == 2) {
              const int64_t trow = (int64_t)page + row;   // page holds the first key row here
              if (trow < (int64_t)d.kbase + d.L && trow < p.NP) sv = __ldg(p.scale + trow * p.H_kv + d.hk);
            } else if (page >= 0 && (int64_t)page < p.NP) {
              sv = reinterpret_cast<const float*>(src + kRawBytes)[row];
            }
            // row of the page: 8 chunks of 16 bytes, stored 128-byte swizzled
            int4 raw[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              raw[c] = *reinterpret_cast<const int4*>(src + row * 128 + ((c ^ (row & 7)) << 4));
            if (last_read) {
              __syncwarp();
              if (lane == 0) mbar_arrive(b_st_empty + 8 * rs);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              int8x4_to_half4((uint32_t)raw[c].x, hv[8 * c + 0], hv[8 * c + 1]);
              int8x4_to_half4((uint32_t)raw[c].y, hv[8 * c + 2], hv[8 * c + 3]);
              int8x4_to_half4((uint32_t)raw[c].z, hv[8 * c + 4], hv[8 * c + 5]);
              int8x4_to_half4((uint32_t)raw[c].w, hv[8 * c + 6], hv[8 * c + 7]);
            }
          }
          if (jp == set) {
            if (!warp_wait(b_a_free + 8 * as, ((it / C::kA) & 1u) ^ 1u, ctl)) { ok = false; break; }
            tc_fence_after();
          }
          tmem_st64(t_lane + as * 128u + 64u * jp, hv);
          if constexpr (kTokScale) tmem_st1(t_lane + C::kScCol0 + (2u * it + jp) % C::kScCols, __float_as_uint(sv));
        }
        if (!ok) break;
        tmem_wait_st();
        // one warp also waits until the epilogue has read the accumulator pair
        // this item will use: the item is ready only after all four arrived
        if (quarter == 0 && set == 0 &&
            !warp_wait(b_d_free + 8 * (it % C::kD), ((it / C::kD) & 1u) ^ 1u, ctl)) {
          ok = false;
          break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_a_full + 8 * as);
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

// One persistent CTA per SM, launched as a programmatic dependent of the plan.
template <bool BF16, int TOPK, int KF4>
cudaError_t launch_short_kernel(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  auto kern = short_kernel<BF16, TOPK, KF4>;
  static std::atomic<uint64_t> configured[64];   // per device: context the limit was raised in
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(kern, (int)Short8::bytes, configured, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_sms);
  cfg.blockDim = dim3(Short8::kThreads);
  cfg.dynamicSmemBytes = Short8::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tq),
                            *static_cast<const CUtensorMap*>(tk), p);
}

}  // namespace msa
