// Persistent block-score kernel for short-query requests (Lq * g <= 32 query
// rows: decode and speculative decode), sm_103a.
//
// The MMA is turned around with respect to the tile kernel: the 128 tokens of
// one key page are the M side and the request's query rows are the N side,
//     D[token, row] = K_page (128 x 128) * Q_rows^T (128 x 32)        (fp32 in TMEM)
// so a page costs a 128 x 32 x 128 MMA instead of a 128 x 128 x 128 one, and
// the shared-memory traffic per page is the page itself plus a 4 KiB read of
// the query rows.  The block max is then a max over TMEM lanes: each epilogue
// warp reduces its 32 tokens for all rows with a butterfly of shuffles, and a
// separate warp combines the four partial maxima of each block (feature request "MsaIndexScore", "calculation": DOT ->
// optional DEQUANT -> MASK -> MAX, with the per-token scale applied per lane).
//
// int8 keys never touch shared memory as fp16: converter warps read the int8
// page (TMA, 128-byte swizzle), convert one token row per thread and store it
// straight into tensor memory, where the MMA reads its A operand; the page's
// per-token scale goes into the next TMEM column.
//
// Roles (one CTA per SM, units fetched from the short class's counter):
//   warp 0       scheduler      warp 1  TMEM owner + MMA issuer
//   warp 2       TMA producer   warps 3..6  epilogue (partial maxima per token quarter)
//   warps 7..10  (int8 only) converters
//   last warp    combine: the four partial maxima of each block, local mask, stores
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

template <bool KI8>
struct ShortCfg;

template <>
struct ShortCfg<false> {
  static constexpr int kStages = 6;                 // 32 KiB key pages in flight
  static constexpr int kSlots = 8;                  // accumulators of 32 columns
  static constexpr uint32_t kSlotCols = 32;
  static constexpr uint32_t kDCol = 0;              // accumulator column inside a slot
  static constexpr uint32_t kStageBytes = 32768;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr int kThreads = 256;
};

template <>
struct ShortCfg<true> {
  static constexpr int kStages = 12;                // int8 pages (+ their scales) in flight
  static constexpr int kSlots = 4;                  // [A: 64 cols | scale: 1 col | D: 32 cols]
  static constexpr uint32_t kSlotCols = 128;
  static constexpr uint32_t kDCol = 96;
  static constexpr uint32_t kStageBytes = 16384 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 384;
};

constexpr int kShortN = kShortRows;                 // MMA N: the request's query rows, padded
constexpr uint32_t kShortQHalf = kShortN * 128;     // one 64-element half of the query rows
constexpr uint32_t kShortQBytes = 2 * kShortQHalf;
constexpr int kShortQBufs = 2;
constexpr uint32_t kSlotScaleCol = 64;
constexpr int kRed = 8;                             // partial-maximum ring (blocks)
template <bool KI8>
__host__ __device__ constexpr int short_combine_warp() { return KI8 ? 11 : 7; }

template <bool KI8>
struct ShortSmem {
  using C = ShortCfg<KI8>;
  static constexpr uint32_t q_off = 0;
  static constexpr uint32_t k_off = q_off + kShortQBufs * kShortQBytes;
  static constexpr uint32_t red_off = k_off + C::kStages * C::kStageBytes;
  static constexpr uint32_t red_bytes = kRed * 4 * kShortN * 4;
  static constexpr uint32_t ring_off = red_off + red_bytes;
  static constexpr uint32_t bar_off = ring_off + kSched * sizeof(UnitDesc);
  static constexpr uint32_t n_bars =
      2 * kSched + 2 * kShortQBufs + 2 * C::kStages + 3 * C::kSlots + 2 * kRed + 2;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t end = misc_off + 16 + 4 * C::kStages;
  static constexpr uint32_t bytes = end + 1024;
};

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

// Same for 16 columns: four halving steps inside each 16-lane group, then one
// exchange between the two groups; lanes c and c + 16 return column c.
__device__ __forceinline__ float warp_transpose_max16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = upper ? v[w + i] : v[i];
      const float send = upper ? v[i] : v[w + i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
    }
  }
  return fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 16));
}

// Masked, scaled partial max over this warp's 32 tokens for N query rows:
// lane c (c < N) returns row c's maximum.
template <int N, bool KI8>
__device__ __forceinline__ float short_partial_max(uint32_t taddr, float sc, int n_min, int lane) {
  const float ninf = __int_as_float(0xff800000);
  float x[N];
  if constexpr (N == 32) {
    tmem_ld32(taddr, x);
  } else {
    tmem_ld16(taddr, x);
  }
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < N; ++c) x[c] = c >= n_min ? (KI8 ? x[c] * sc : x[c]) : ninf;   // DEQUANT, MASK
  if constexpr (N == 32) {
    return warp_transpose_max32(x, lane);
  } else {
    return warp_transpose_max16(x, lane);
  }
}

template <bool KI8, bool BF16>
__global__ void __launch_bounds__(ShortCfg<KI8>::kThreads, 1)
    short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const Params p) {
  using C = ShortCfg<KI8>;
  using L = ShortSmem<KI8>;
  constexpr int S = C::kStages;
  constexpr int A = C::kSlots;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  UnitDesc* ring = reinterpret_cast<UnitDesc*>(smem + L::ring_off);
  float* red = reinterpret_cast<float*>(smem + L::red_off);   // [slot][warp quarter][row]
  const uint32_t b_sched_full = sbase + L::bar_off;
  const uint32_t b_sched_empty = b_sched_full + 8 * kSched;
  const uint32_t b_q_full = b_sched_empty + 8 * kSched;
  const uint32_t b_q_empty = b_q_full + 8 * kShortQBufs;
  const uint32_t b_st_full = b_q_empty + 8 * kShortQBufs;
  const uint32_t b_st_empty = b_st_full + 8 * S;
  const uint32_t b_a_full = b_st_empty + 8 * S;      // int8: converted page in TMEM
  const uint32_t b_slot_free = b_a_full + 8 * A;     // epilogue done with a slot
  const uint32_t b_d_full = b_slot_free + 8 * A;     // accumulator ready
  const uint32_t b_red_full = b_d_full + 8 * A;      // four partial maxima written
  const uint32_t b_red_empty = b_red_full + 8 * kRed;  // partial maxima combined
  const uint32_t b_drain = b_red_empty + 8 * kRed;
  const uint32_t b_sched_req = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);
  volatile int* raw_page = reinterpret_cast<volatile int*>(smem + L::misc_off + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // readers of each unit descriptor: producer, MMA, 4 epilogue, combine (+ 4 converter) warps
  constexpr int kConsumers = KI8 ? 11 : 7;
  constexpr int kCombineWarp = short_combine_warp<KI8>();

  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSched; ++i) {
      mbar_init(b_sched_full + 8 * i, 1);
      mbar_init(b_sched_empty + 8 * i, kConsumers);
    }
    for (int i = 0; i < kShortQBufs; ++i) {
      mbar_init(b_q_full + 8 * i, 1);
      mbar_init(b_q_empty + 8 * i, 1);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(b_st_full + 8 * i, 1);
      mbar_init(b_st_empty + 8 * i, KI8 ? 4 : 1);
    }
    for (int i = 0; i < A; ++i) {
      mbar_init(b_a_full + 8 * i, 4);
      mbar_init(b_slot_free + 8 * i, 4);
      mbar_init(b_d_full + 8 * i, 1);
    }
    for (int i = 0; i < kRed; ++i) {
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
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // The plan written by the plan kernel is visible after this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  const int n_units = *reinterpret_cast<volatile int*>(&hdr->n_units[1]);
  WaitCtl ctl{abort_flag, &hdr->err, p.wait_limit_ns};

  if (n_units == 0) {
    // no short requests in this call
  } else if (warp == 0) {
    // -------------------------------------------------------- scheduler --
    if (lane == 0) {
      const int n_req0 = *reinterpret_cast<volatile int*>(&hdr->n_req[0]);
      const int n_req = *reinterpret_cast<volatile int*>(&hdr->n_req[1]);
      const int chunk = *reinterpret_cast<volatile int*>(&hdr->chunk[1]);
      const ReqInfo* req = reinterpret_cast<const ReqInfo*>(p.ws + sizeof(PlanHeader)) + n_req0;
      const int32_t* prefix = plan_prefix(p.ws, p.B, 1);
      uint32_t ss = 0, sph = 0, rph = 0;
      for (bool first = true;; first = false) {
        if (!first) {
          if (!mbar_wait(b_sched_req, rph, ctl)) break;
          rph ^= 1;
        }
        UnitDesc d;
        make_unit(p, req, prefix, n_req, n_units, chunk, p.np_short,
                  atomicAdd(&hdr->counter[1], 1), d);
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
        const uint32_t qdst = sbase + L::q_off + qb * kShortQBytes;
        mbar_arrive_expect_tx(b_q_full + 8 * qb, q_bytes);
        tma_load_3d(qdst, &tm_q, b_q_full + 8 * qb, 0, d.hk * p.g, d.t0);
        tma_load_3d(qdst + kShortQHalf, &tm_q, b_q_full + 8 * qb, 64, d.hk * p.g, d.t0);
        ++n_q;
        if (++qb == kShortQBufs) { qb = 0; qph ^= 1; }
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
          if (!mbar_wait(b_st_empty + 8 * ks, kph ^ 1, ctl)) { ok = false; break; }
          const uint32_t dst = sbase + L::k_off + ks * C::kStageBytes;
          if constexpr (KI8) {
            raw_page[ks] = paged ? page : tok;
            const bool with_scale = paged && (int64_t)page < p.NP;
            mbar_arrive_expect_tx(b_st_full + 8 * ks, kRawBytes + (with_scale ? kRawScaleBytes : 0u));
            tma_k(dst, &tm_k, b_st_full + 8 * ks, 0, tok, d.hk, page, p.layout, pol_k);
            if (with_scale)
              bulk_load(dst + kRawBytes, p.scale + ((int64_t)page * p.H_kv + d.hk) * kP,
                        kRawScaleBytes, b_st_full + 8 * ks);
          } else {
            mbar_arrive_expect_tx(b_st_full + 8 * ks, 32768u);
            tma_k(dst, &tm_k, b_st_full + 8 * ks, 0, tok, d.hk, page, p.layout, pol_k);
            tma_k(dst + 16384u, &tm_k, b_st_full + 8 * ks, 64, tok, d.hk, page, p.layout, pol_k);
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
        while (!mbar_try_wait(b_st_full + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
      for (uint32_t j = n_q > (uint32_t)kShortQBufs ? n_q - kShortQBufs : 0; j < n_q; ++j) {
        const uint32_t st = j % kShortQBufs, ph = (j / kShortQBufs) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_q_full + 8 * st, ph) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc32 = idesc_f16(BF16, 128, 32);
      constexpr uint32_t idesc16 = idesc_f16(BF16, 128, 16);
      uint32_t ss = 0, sph = 0, qb = 0, qph = 0, ks = 0, kph = 0, sl = 0, slph = 0;
      bool issued = false;
      for (;;) {
        if (!mbar_wait(b_sched_full + 8 * ss, sph, ctl)) break;
        const UnitDesc d = ring[ss];
        mbar_arrive(b_sched_empty + 8 * ss);
        if (++ss == kSched) { ss = 0; sph ^= 1; }
        if (!d.live) break;
        if (d.b1 <= d.c0) continue;
        if (!mbar_wait(b_q_full + 8 * qb, qph, ctl)) break;
        const uint32_t qsrc = sbase + L::q_off + qb * kShortQBytes;
        const uint32_t idesc = d.Lq * p.g <= 16 ? idesc16 : idesc32;   // N = 16 or 32 query rows
        bool ok = true;
        for (int beta = d.c0; beta < d.b1; ++beta) {
          const uint32_t dt = tmem_base + sl * C::kSlotCols + C::kDCol;
          if constexpr (KI8) {
            // converters filled the slot's A columns (they waited for it to be free)
            if (!mbar_wait(b_a_full + 8 * sl, slph, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t at = tmem_base + sl * C::kSlotCols;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc_mma_f16_ta(dt, at + 8u * k,
                            smem_desc_sw128(qsrc + (uint32_t)(k >> 2) * kShortQHalf + (k & 3) * 32u),
                            idesc, k > 0 ? 1u : 0u);
          } else {
            if (!mbar_wait(b_st_full + 8 * ks, kph, ctl)) { ok = false; break; }
            if (!mbar_wait(b_slot_free + 8 * sl, slph ^ 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ksrc = sbase + L::k_off + ks * C::kStageBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc_mma_f16(dt, desc_at(ksrc, k),
                         smem_desc_sw128(qsrc + (uint32_t)(k >> 2) * kShortQHalf + (k & 3) * 32u),
                         idesc, k > 0 ? 1u : 0u);
            tc_commit(b_st_empty + 8 * ks);
            if (++ks == S) { ks = 0; kph ^= 1; }
          }
          tc_commit(b_d_full + 8 * sl);
          issued = true;
          if (++sl == A) { sl = 0; slph ^= 1; }
        }
        if (!ok) break;
        tc_commit(b_q_empty + 8 * qb);
        if (++qb == kShortQBufs) { qb = 0; qph ^= 1; }
      }
      if (issued) {
        tc_commit(b_drain);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(b_drain, 0) && global_timer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp < kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue --
    // Every warp reduces its 32 tokens of each block for all rows and posts
    // the partial maxima to a ring that the combine warp drains; the epilogue
    // warps never wait for one another.
    const int quarter = warp & 3;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t ss = 0, sph = 0, sl = 0, slph = 0, rr = 0, rph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      const bool narrow = d.Lq * p.g <= 16;               // the MMA used N = 16
      // first visible row for a token t: rows n with floor(n / g) >= t - (L - Lq)
      // (sparse_mode 3), all rows if t < L (mode 0); no row if t >= L
      const int qbase = p.sparse_mode == 3 ? d.L - d.Lq : 0x3fffffff;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; ++beta) {
        if (!warp_wait(b_d_full + 8 * sl, slph, ctl)) { ok = false; break; }
        tc_fence_after();
        float sc = 1.f;
        if constexpr (KI8) sc = tmem_ld1(t_lane + sl * C::kSlotCols + kSlotScaleCol);
        const int t = beta * kP + quarter * 32 + lane;    // this lane's token
        int n_min = 0;
        if (t >= d.L) {
          n_min = kShortN;
        } else if (t > qbase) {
          const int64_t m = (int64_t)(t - qbase) * p.g;
          n_min = m > kShortN ? kShortN : (int)m;
        }
        // MAX over the warp's 32 tokens for every row at once (butterfly of
        // shuffles: each step a lane keeps half of its columns and takes the max
        // with its partner's copy of them)
        const uint32_t dcol = t_lane + sl * C::kSlotCols + C::kDCol;
        const float mine = narrow ? short_partial_max<16, KI8>(dcol, sc, n_min, lane)
                                  : short_partial_max<32, KI8>(dcol, sc, n_min, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_slot_free + 8 * sl);
        if (++sl == A) { sl = 0; slph ^= 1; }
        if (!warp_wait(b_red_empty + 8 * rr, rph ^ 1, ctl)) { ok = false; break; }
        red[(rr * 4 + quarter) * kShortN + lane] = mine;
        __syncwarp();
        if (lane == 0) mbar_arrive(b_red_full + 8 * rr);
        if (++rr == kRed) { rr = 0; rph ^= 1; }
      }
      if (!ok) break;
    }
  } else if (warp == kCombineWarp) {
    // ---------------------------------------------------------- combine --
    // Lane n owns output row n = (position n / g, head n % g): the max of the
    // four partial maxima of each computed block, the local-mask constants, the
    // fill of the other columns, and 32-byte stores of 8 blocks at a time.
    const float ninf = __int_as_float(0xff800000);
    uint32_t ss = 0, sph = 0, rr = 0, rph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      const int rows = d.Lq * p.g;                        // valid query rows (<= 32)
      const int n = lane;
      const bool row_valid = n < rows;
      const int pos = n / p.g;
      const int h = d.hk * p.g + (n - pos * p.g);
      float* orow = p.out + ((int64_t)h * p.T + (d.t0 + pos)) * (int64_t)p.MBp;
      const int lo = max(0, d.sl + 1 - p.local_blocks);
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
        if (!warp_wait(b_red_full + 8 * rr, rph, ctl)) { ok = false; break; }
        const float* r4 = red + rr * 4 * kShortN + lane;
        float m = fmax3(r4[0], r4[kShortN], fmaxf(r4[2 * kShortN], r4[3 * kShortN]));
        __syncwarp();
        if (lane == 0) mbar_arrive(b_red_empty + 8 * rr);
        if (++rr == kRed) { rr = 0; rph ^= 1; }
        if (live_kv && (beta < p.init_blocks || (beta >= lo && beta <= d.sl))) m = fill_value(beta);
        const int e = beta & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k == e) v[k] = m;
        if (e == 7 && row_valid) {
          float4* dst = reinterpret_cast<float4*>(orow + (beta - 7));
          __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
          __stcs(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
        }
      }
      if (!ok) break;
      if (row_valid) {
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
    }
  } else if (KI8 && warp >= kCvtWarp0 && warp < kCvtWarp0 + 4) {
    // ----------------------------------------- int8 -> fp16 into TMEM --
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;                    // token row of the page
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t ss = 0, sph = 0, rs = 0, rph = 0, sl = 0, slph = 0;
    for (;;) {
      if (!warp_wait(b_sched_full + 8 * ss, sph, ctl)) break;
      const UnitDesc d = ring[ss];
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sched_empty + 8 * ss);
      if (++ss == kSched) { ss = 0; sph ^= 1; }
      if (!d.live) break;
      bool ok = true;
      for (int beta = d.c0; beta < d.b1; ++beta) {
        if (!warp_wait(b_st_full + 8 * rs, rph, ctl)) { ok = false; break; }
        const uint8_t* src = smem + L::k_off + rs * C::kStageBytes;
        const int page = raw_page[rs];
        float sv = 0.f;
        if (p.layout == 2) {
          const int64_t row = (int64_t)page + j;          // page holds the first key row here
          if (row < (int64_t)d.kbase + d.L && row < p.NP) sv = __ldg(p.scale + row * p.H_kv + d.hk);
        } else if (page >= 0 && (int64_t)page < p.NP) {
          sv = reinterpret_cast<const float*>(src + kRawBytes)[j];
        }
        // row j of the page: 8 chunks of 16 bytes, stored 128-byte swizzled
        int4 raw[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          raw[c] = *reinterpret_cast<const int4*>(src + j * 128 + ((c ^ (j & 7)) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(b_st_empty + 8 * rs);
        if (++rs == S) { rs = 0; rph ^= 1; }
        uint32_t hv[64];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          int8x4_to_half4((uint32_t)raw[c].x, hv[8 * c + 0], hv[8 * c + 1]);
          int8x4_to_half4((uint32_t)raw[c].y, hv[8 * c + 2], hv[8 * c + 3]);
          int8x4_to_half4((uint32_t)raw[c].z, hv[8 * c + 4], hv[8 * c + 5]);
          int8x4_to_half4((uint32_t)raw[c].w, hv[8 * c + 6], hv[8 * c + 7]);
        }
        if (!warp_wait(b_slot_free + 8 * sl, slph ^ 1, ctl)) { ok = false; break; }
        tc_fence_after();
        tmem_st64(t_lane + sl * C::kSlotCols, hv);
        tmem_st1(t_lane + sl * C::kSlotCols + kSlotScaleCol, __float_as_uint(sv));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_a_full + 8 * sl);
        if (++sl == A) { sl = 0; slph ^= 1; }
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace msa
