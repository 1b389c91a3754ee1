// Sparse main branch of MiniMax Sparse Attention on sm_103a: softmax attention
// restricted to the KV blocks each query's GQA group selected (MiniMax Sparse
// Attention notes, sec. 4.8 Equation (8); group-shared selection, sec. 4.3
// Equation (3)), computed KV-outer in two phases (sec. 4.11 Equations
// (13)-(16), sec. 5.5-5.10):
//
//   CSR build   the selection [T, H_kv, k] (query -> blocks) is turned into
//               block -> query lists (count, prefix sum, scatter), one list per
//               (kv head, request, logical block), and the lists are cut into
//               units of at most floor(128 / g) queries (sec. 5.6, 5.7);
//   K1          one unit at a time: the block's K and V pages are loaded once,
//               the unit's queries x the g heads of the group are gathered into
//               the 128 MMA rows (sec. 5.9), S = Q K^T on the tensor cores, a
//               masked softmax of each row over the block's visible keys, O = P V
//               with P read from tensor memory; each (query, head, selected
//               block) gets a partial (O normalised by its own sum, LSE);
//   K2          per (query, head) the partials are merged by the exact
//               log-sum-exp identity (sec. 5.10).
//
// The value cache shares the key cache's layout, dtype (fp16 or bf16), page
// stride and block table.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "msa_common.cuh"
#include "msa_ptx.cuh"
#include "msa_units.cuh"

namespace msa {

namespace {

// Workspace header of a sparse-attention call (the error word at the same
// offset as the block-score plan's, so msa_get_device_error reads it).
struct SparseHeader {
  int32_t n_units;
  int32_t pad0[7];
  int32_t err;
  int32_t pad1[7];
};
static_assert(sizeof(SparseHeader) == 64, "header");
static_assert(offsetof(SparseHeader, err) == offsetof(PlanHeader, err), "error word offset");

__device__ __forceinline__ int request_search(const int32_t* cu_q, int B, int64_t t) {
  int lo = 0, hi = B - 1;                       // last b with cu_q[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int64_t kv_length(const SparseParams& sp, int b) {
  const Params& p = sp.p;
  int64_t L;
  if (p.layout == 2) {
    L = (int64_t)__ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
  } else {
    L = __ldg(p.kv_len + b);
  }
  return L < 0 ? 0 : L;
}

// A selection entry names a block with keys: 0 <= beta < min(MB, ceil(L / P)).
__device__ __forceinline__ bool entry_valid(int beta, int MB, int64_t L) {
  return beta >= 0 && beta < MB && (int64_t)beta * kP < L;
}

// ------------------------------------------------------------ CSR build ----
// Thread per (token, kv head): validates the selection row and counts its
// entries into the rows of the block -> query lists.
__global__ void count_kernel(const SparseParams sp) {
  const Params& p = sp.p;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.T * (int64_t)p.H_kv) return;
  const int64_t t = idx / p.H_kv;
  const int r = (int)(idx - t * p.H_kv);
  const int b = request_search(p.cu_q, p.B, t);
  const int64_t L = kv_length(sp, b);
  const int32_t* row = sp.sel + idx * sp.k;
  SparseHeader* hdr = reinterpret_cast<SparseHeader*>(p.ws);
  int prev = -1, err = 0;
  for (int s = 0; s < sp.k; ++s) {
    const int beta = __ldg(row + s);
    if (beta < 0) { prev = 0x7fffffff; continue; }      // -1 tail: nothing may follow
    if (beta <= prev || beta >= p.MB) err = 1;           // not ascending, repeated, or beyond MB
    prev = beta;
    if (entry_valid(beta, p.MB, L)) atomicAdd(sp.cnt + ((int64_t)r * p.B + b) * p.MB + beta, 1);
  }
  if (err) atomicOr(&hdr->err, kErrSelection);
}

// One CTA: exclusive prefix sums of the list lengths (row_ptr) and of the
// units per list (unit_ptr); the scatter cursors start at row_ptr.
__global__ void __launch_bounds__(1024) scan_kernel(const SparseParams sp) {
  __shared__ int64_t s_sum[2][1024];
  const int tid = threadIdx.x;
  const int64_t rows = sp.rows;
  const int64_t per = (rows + 1023) / 1024;
  const int64_t r0 = min(rows, tid * per), r1 = min(rows, r0 + per);
  int64_t a = 0, u = 0;
  for (int64_t i = r0; i < r1; ++i) {
    const int c = sp.cnt[i];
    a += c;
    u += (c + sp.qpu - 1) / sp.qpu;
  }
  s_sum[0][tid] = a;
  s_sum[1][tid] = u;
  __syncthreads();
  // Hillis-Steele inclusive scan of the per-thread totals
  for (int off = 1; off < 1024; off <<= 1) {
    int64_t xa = 0, xu = 0;
    if (tid >= off) { xa = s_sum[0][tid - off]; xu = s_sum[1][tid - off]; }
    __syncthreads();
    s_sum[0][tid] += xa;
    s_sum[1][tid] += xu;
    __syncthreads();
  }
  a = tid ? s_sum[0][tid - 1] : 0;
  u = tid ? s_sum[1][tid - 1] : 0;
  for (int64_t i = r0; i < r1; ++i) {
    const int c = sp.cnt[i];
    sp.row_ptr[i] = (int32_t)a;
    sp.cursor[i] = (int32_t)a;
    sp.unit_ptr[i] = (int32_t)u;
    a += c;
    u += (c + sp.qpu - 1) / sp.qpu;
  }
  if (tid == 1023) {
    sp.row_ptr[rows] = (int32_t)s_sum[0][1023];
    sp.unit_ptr[rows] = (int32_t)s_sum[1][1023];
    reinterpret_cast<SparseHeader*>(sp.p.ws)->n_units = (int32_t)s_sum[1][1023];
  }
}

// Thread per (token, kv head): writes token * k + slot into its blocks' lists.
__global__ void scatter_kernel(const SparseParams sp) {
  const Params& p = sp.p;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.T * (int64_t)p.H_kv) return;
  const int64_t t = idx / p.H_kv;
  const int r = (int)(idx - t * p.H_kv);
  const int b = request_search(p.cu_q, p.B, t);
  const int64_t L = kv_length(sp, b);
  const int32_t* row = sp.sel + idx * sp.k;
  for (int s = 0; s < sp.k; ++s) {
    const int beta = __ldg(row + s);
    if (!entry_valid(beta, p.MB, L)) continue;
    const int64_t list = ((int64_t)r * p.B + b) * p.MB + beta;
    const int pos = atomicAdd(sp.cursor + list, 1);
    sp.qidx[pos] = (int32_t)(t * sp.k + s);
  }
}

// Thread per list: its units {list, first entry, entries}.
__global__ void units_kernel(const SparseParams sp) {
  const int64_t list = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (list >= sp.rows) return;
  const int c = sp.cnt[list];
  const int base = sp.row_ptr[list];
  int4* dst = sp.units + sp.unit_ptr[list];
  for (int u = 0; u * sp.qpu < c; ++u)
    dst[u] = make_int4((int)list, base + u * sp.qpu, min(sp.qpu, c - u * sp.qpu), 0);
}

// ------------------------------------------------------------------- K1 ----
struct K1Layout {
  static constexpr uint32_t kTile = 32768;             // 128 x 128 16-bit operand (two 16 KiB halves)
  static constexpr uint32_t kStage = 3 * kTile;        // Q, K, V (rows = tokens)
  static constexpr uint32_t stage_off = 0;
  static constexpr uint32_t vt_off = 2 * kStage;       // V transposed: rows = dims, K-major over tokens
  static constexpr uint32_t bar_off = vt_off + kTile;
  static constexpr uint32_t n_bars = 4 * 2 + 9;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t end = misc_off + 16;
  static constexpr uint32_t bytes = end + 1024;
};
static_assert(K1Layout::bytes <= 232448, "shared memory per CTA");

constexpr int kK1Threads = 320;       // 10 warps
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Roles: warp 0 TMA producer (K and V pages), warp 1 TMEM owner + MMA issuer,
// warps 2..5 softmax and partial stores (thread = MMA row = TMEM lane), warps
// 6..9 loaders (gather the unit's query rows, transpose V into a K-major tile).
// Units are taken round-robin (unit i of CTA c is c + i * gridDim.x); every
// role walks the same sequence, two stages of Q/K/V in flight.
template <bool BF16>
__global__ void __launch_bounds__(kK1Threads, 1)
    sparse_k1_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const SparseParams sp) {
  using Lo = K1Layout;
  const Params& p = sp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + Lo::bar_off;
  const uint32_t b_k_full = bars;                 // [2] K page landed
  const uint32_t b_v_full = b_k_full + 16;        // [2] V page landed
  const uint32_t b_q_full = b_v_full + 16;        // [2] query rows written (4 loader warps)
  const uint32_t b_stage_empty = b_q_full + 16;   // [2] the stage's last MMA done
  const uint32_t b_s_full = b_stage_empty + 16;
  const uint32_t b_s_empty = b_s_full + 8;        // 4 softmax warps read S
  const uint32_t b_p_full = b_s_empty + 8;        // 4 softmax warps wrote P
  const uint32_t b_o_full = b_p_full + 8;
  const uint32_t b_o_empty = b_o_full + 8;        // 4 softmax warps read O
  const uint32_t b_vt_full = b_o_empty + 8;       // 4 loader warps wrote V^T
  const uint32_t b_vt_empty = b_vt_full + 8;      // the MMA reading V^T done
  const uint32_t b_drain = b_vt_empty + 8;
  const uint32_t b_spare = b_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lo::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lo::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_k_full + 8 * i, 1);
      mbar_init(b_v_full + 8 * i, 1);
      mbar_init(b_q_full + 8 * i, 4);
      mbar_init(b_stage_empty + 8 * i, 1);
    }
    mbar_init(b_s_full, 1);
    mbar_init(b_s_empty, 4);
    mbar_init(b_p_full, 4);
    mbar_init(b_o_full, 1);
    mbar_init(b_o_empty, 4);
    mbar_init(b_vt_full, 4);
    mbar_init(b_vt_empty, 1);
    mbar_init(b_drain, 1);
    mbar_init(b_spare, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  SparseHeader* hdr = reinterpret_cast<SparseHeader*>(p.ws);
  const int n_units = hdr->n_units;
  WaitCtl ctl{abort_flag, &hdr->err, p.wait_limit_ns};
  const int g = p.g;

  // unit -> (kv head, request, block, first list entry, entries)
  auto unit_at = [&](int u, int& r, int& b, int& beta, int& e0, int& ne) {
    const int4 d = __ldg(sp.units + u);
    const int64_t list = d.x;
    beta = (int)(list % p.MB);
    const int64_t rb = list / p.MB;
    b = (int)(rb % p.B);
    r = (int)(rb / p.B);
    e0 = d.y;
    ne = d.z;
  };

  if (warp == 0) {
    // -------------------------------------------------------- producer --
    if (lane == 0) {
      const bool paged = p.layout != 2;
      const uint64_t pol = l2_policy_evict_last();      // a block's pages serve all its units
      uint32_t n_issued[2] = {0, 0};
      int i = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++i) {
        const int st = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;
        if (!mbar_wait(b_stage_empty + 8 * st, ph ^ 1, ctl)) break;
        int r, b, beta, e0, ne;
        unit_at(u, r, b, beta, e0, ne);
        int page = 0, tok = 0;
        if (paged) {
          page = __ldg(p.block_table + (int64_t)b * p.MB + beta);
          if (page < 0 || (int64_t)page >= p.NP) {
            atomicOr(&hdr->err, kErrBlockTable);
            page = (int32_t)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);   // out of bounds: zero fill
          }
        } else {
          tok = __ldg(p.cu_k + b) + beta * kP;
        }
        const uint32_t st_base = sbase + Lo::stage_off + st * Lo::kStage;
        mbar_arrive_expect_tx(b_k_full + 8 * st, Lo::kTile);
        for (int x = 0; x < 2; ++x)
          tma_k(st_base + Lo::kTile + x * kHalfBytes, &tm_k, b_k_full + 8 * st, 64 * x, tok, r, page,
                p.layout, pol);
        mbar_arrive_expect_tx(b_v_full + 8 * st, Lo::kTile);
        for (int x = 0; x < 2; ++x)
          tma_k(st_base + 2 * Lo::kTile + x * kHalfBytes, &tm_v, b_v_full + 8 * st, 64 * x, tok, r, page,
                p.layout, pol);
        ++n_issued[st];
      }
      // teardown: the last load of each stage may still be in flight
      for (int st = 0; st < 2; ++st) {
        if (!n_issued[st]) continue;
        const uint32_t ph = (n_issued[st] - 1) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!(mbar_try_wait(b_k_full + 8 * st, ph) && mbar_try_wait(b_v_full + 8 * st, ph)) &&
               global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer --
    constexpr uint32_t idesc = idesc_f16(BF16, 128, 128);
    bool issued = false;
    int i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++i) {
      const int st = i & 1;
      const uint32_t ph2 = (uint32_t)(i >> 1) & 1u, ph1 = (uint32_t)i & 1u;
      if (!warp_wait(b_k_full + 8 * st, ph2, ctl)) break;
      if (!warp_wait(b_q_full + 8 * st, ph2, ctl)) break;
      if (!warp_wait(b_s_empty, ph1 ^ 1, ctl)) break;
      tc_fence_after();
      const uint32_t st_base = sbase + Lo::stage_off + st * Lo::kStage;
      if (lane == 0) {
        // S = Q K^T: rows = (query, head), columns = the block's 128 tokens
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem_base + kColS, desc_at(st_base, kk), desc_at(st_base + Lo::kTile, kk), idesc,
                     kk ? 1u : 0u);
        tc_commit(b_s_full);
      }
      __syncwarp();
      if (!warp_wait(b_p_full, ph1, ctl)) break;
      if (!warp_wait(b_vt_full, ph1, ctl)) break;
      if (!warp_wait(b_o_empty, ph1 ^ 1, ctl)) break;
      tc_fence_after();
      if (lane == 0) {
        // O = P V: P (bf16 / fp16 pairs) from tensor memory, V^T K-major in shared memory
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_ta(tmem_base + kColO, tmem_base + kColP + 8u * kk,
                        desc_at(sbase + Lo::vt_off, kk), idesc, kk ? 1u : 0u);
        tc_commit(b_o_full);
        tc_commit(b_vt_empty);
        tc_commit(b_stage_empty + 8 * st);
      }
      __syncwarp();
      issued = true;
    }
    if (lane == 0 && issued) {
      tc_commit(b_drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(b_drain, 0) && global_timer_ns() - t0 < kDrainLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 6) {
    // --------------------------------------------------------- softmax --
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;              // MMA row = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const float ninf = __int_as_float(0xff800000);
    const float kscale = sp.sm_scale * 1.4426950408889634f;   // base-2 softmax
    int i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++i) {
      const uint32_t ph1 = (uint32_t)i & 1u;
      int r, b, beta, e0, ne;
      unit_at(u, r, b, beta, e0, ne);
      const bool valid = row < ne * g;
      int64_t t = 0;
      int s = 0, h = 0;
      int lim = -1;                                    // last visible column of the block (-1: none)
      if (valid) {
        const int entry = __ldg(sp.qidx + e0 + row / g);
        t = entry / sp.k;
        s = entry - (int)(t * sp.k);
        h = r * g + row % g;
        const int64_t L = kv_length(sp, b);
        const int64_t t0 = __ldg(p.cu_q + b);
        const int64_t Lq = (int64_t)__ldg(p.cu_q + b + 1) - t0;
        int64_t last = L - 1;
        if (p.sparse_mode == 3) last = min(last, L - Lq + (t - t0));
        const int64_t c = last - (int64_t)beta * kP;
        lim = c < 0 ? -1 : (c > kP - 1 ? kP - 1 : (int)c);
      }
      if (!warp_wait(b_s_full, ph1, ctl)) break;
      tc_fence_after();
      float x[128];
      tmem_ld128(t_lane + kColS, x);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_s_empty);
      float m = ninf;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        x[c] = c <= lim ? x[c] * kscale : ninf;
        m = fmaxf(m, x[c]);
      }
      const bool any = lim >= 0;
      float l = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float a0 = any ? ex2(x[2 * c] - m) : 0.f;
        const float a1 = any ? ex2(x[2 * c + 1] - m) : 0.f;
        l += a0 + a1;
        pk[c] = pack2(a0, a1, BF16);
      }
      tmem_st64(t_lane + kColP, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p_full);
      if (!warp_wait(b_o_full, ph1, ctl)) break;
      tc_fence_after();
      tmem_ld128(t_lane + kColO, x);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_o_empty);
      if (valid) {
        const int64_t slot = (t * p.H_q + h) * (int64_t)sp.k + s;
        float4* o = reinterpret_cast<float4*>(sp.o_part + slot * kD);
        const float inv = any ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          o[c] = make_float4(x[4 * c] * inv, x[4 * c + 1] * inv, x[4 * c + 2] * inv, x[4 * c + 3] * inv);
        // natural-log LSE of the block's visible keys
        sp.lse_part[slot] = any ? (m + __log2f(l)) * 0.6931471805599453f : ninf;
      }
    }
  } else {
    // --------------------------------------------------------- loaders --
    const int wq = warp - 6;                           // 0..3
    const int row = wq * 32 + lane;
    int i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++i) {
      const int st = i & 1;
      const uint32_t ph2 = (uint32_t)(i >> 1) & 1u, ph1 = (uint32_t)i & 1u;
      int r, b, beta, e0, ne;
      unit_at(u, r, b, beta, e0, ne);
      if (!warp_wait(b_stage_empty + 8 * st, ph2 ^ 1, ctl)) break;
      const uint32_t st_base = sbase + Lo::stage_off + st * Lo::kStage;
      uint8_t* qtile = smem + Lo::stage_off + st * Lo::kStage;
      // the unit's query rows (query entry row / g, head r * g + row % g)
      if (row < ne * g) {
        const int entry = __ldg(sp.qidx + e0 + row / g);
        const int64_t t = entry / sp.k;
        const int h = r * g + row % g;
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(sp.query) + (t * p.H_q + h) * (int64_t)kD);
        uint4 v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = __ldg(src + c);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int half = c >> 3, ch = c & 7;
          *reinterpret_cast<uint4*>(qtile + half * kHalfBytes + row * 128 + ((ch ^ (row & 7)) << 4)) = v[c];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_q_full + 8 * st);
      // V^T: 8x8 transposes, rows = tokens (V page) -> rows = dims (K-major over tokens)
      if (!warp_wait(b_v_full + 8 * st, ph2, ctl)) break;
      if (!warp_wait(b_vt_empty, ph1 ^ 1, ctl)) break;
      const uint32_t vraw = st_base + 2 * Lo::kTile;
      const uint32_t vt = sbase + Lo::vt_off;
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll 4
      for (int combo = wq; combo < 64; combo += 4) {
        const int a = combo & 15;                       // token group 8a .. 8a+7
        const int hd = (combo >> 4) & 1;                // dims 0..63 / 64..127
        const int c0 = (combo >> 5) * 4;                // dim chunks c0 .. c0+3 of the half
        const uint32_t src = vraw + hd * kHalfBytes + (8 * a + ri) * 128 + (((c0 + mi) ^ ri) << 4);
        const int dim = 64 * hd + 8 * (c0 + mi) + ri;
        const uint32_t dst = vt + (a >> 3) * kHalfBytes + dim * 128 + (((a & 7) ^ ri) << 4);
        uint32_t frag[4];
        ldsm_x4_trans(src, frag);
        stsm_x4(dst, frag);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_vt_full);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------- K2 ----
// Warp per (token, head): merges the partials of the token's selected blocks
// with the log-sum-exp identity; lane l holds dims 4l .. 4l+3.
__global__ void combine_kernel(const SparseParams sp, float* __restrict__ out,
                               float* __restrict__ lse) {
  const Params& p = sp.p;
  const int lane = threadIdx.x & 31;
  const int64_t rowid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (rowid >= p.T * (int64_t)p.H_q) return;
  const int64_t t = rowid / p.H_q;
  const int h = (int)(rowid - t * p.H_q);
  const int r = h / p.g;
  const int b = request_search(p.cu_q, p.B, t);
  const int64_t L = kv_length(sp, b);
  const int32_t* selrow = sp.sel + (t * p.H_kv + r) * sp.k;
  const float ninf = __int_as_float(0xff800000);
  float mx = ninf;
  for (int s = 0; s < sp.k; ++s)
    if (entry_valid(__ldg(selrow + s), p.MB, L)) mx = fmaxf(mx, sp.lse_part[rowid * sp.k + s]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx > ninf) {
    for (int s = 0; s < sp.k; ++s) {
      if (!entry_valid(__ldg(selrow + s), p.MB, L)) continue;
      const float w = __expf(sp.lse_part[rowid * sp.k + s] - mx);
      const float4 o = reinterpret_cast<const float4*>(sp.o_part + (rowid * sp.k + s) * kD)[lane];
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  reinterpret_cast<float4*>(out + rowid * kD)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && lane == 0) lse[rowid] = wsum > 0.f ? mx + __logf(wsum) : ninf;
}

}  // namespace

cudaError_t launch_sparse_attention(const void* tm_k, const void* tm_v, const SparseParams& sp,
                                    bool bf16, float* out, float* lse, cudaStream_t s) {
  const Params& p = sp.p;
  const int64_t th = p.T * (int64_t)p.H_kv;
  cudaError_t e = cudaMemsetAsync(sp.p.ws, 0, sizeof(SparseHeader), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(sp.cnt, 0, sizeof(int32_t) * (size_t)sp.rows, s);
  if (e != cudaSuccess) return e;
  const int threads = 256;
  if (th > 0) count_kernel<<<(unsigned)((th + threads - 1) / threads), threads, 0, s>>>(sp);
  scan_kernel<<<1, 1024, 0, s>>>(sp);
  if (th > 0) scatter_kernel<<<(unsigned)((th + threads - 1) / threads), threads, 0, s>>>(sp);
  units_kernel<<<(unsigned)((sp.rows + threads - 1) / threads), threads, 0, s>>>(sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  auto k1 = bf16 ? sparse_k1_kernel<true> : sparse_k1_kernel<false>;
  static std::atomic<uint64_t> configured[2][64];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit(k1, (int)K1Layout::bytes, configured[bf16 ? 1 : 0], dev)) != cudaSuccess)
    return e;
  k1<<<(unsigned)p.num_sms, kK1Threads, K1Layout::bytes, s>>>(*static_cast<const CUtensorMap*>(tm_k),
                                                               *static_cast<const CUtensorMap*>(tm_v), sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = p.T * (int64_t)p.H_q;
  if (rows > 0) combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(sp, out, lse);
  return cudaGetLastError();
}

}  // namespace msa
