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
//               block) gets a partial (O normalised by its own sum, in the
//               input's 16-bit type; LSE in fp32);
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
// Thread per (kv head, token), tokens fastest: validates the selection row
// and counts its entries into the rows of the block -> query lists.  Lanes of
// a warp that name the same list (neighbouring tokens share most of their
// blocks) add to it with one atomic.
__global__ void count_kernel(const SparseParams sp) {
  const Params& p = sp.p;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = idx < p.T * (int64_t)p.H_kv;
  const int r = live ? (int)(idx / p.T) : 0;
  const int64_t t = live ? idx - (int64_t)r * p.T : 0;
  const int b = request_search(p.cu_q, p.B, t);
  const int64_t L = kv_length(sp, b);
  const int32_t* row = sp.sel + (t * p.H_kv + r) * sp.k;
  SparseHeader* hdr = reinterpret_cast<SparseHeader*>(p.ws);
  const int lane = threadIdx.x & 31;
  int prev = -1, err = 0;
  for (int s = 0; s < sp.k; ++s) {
    const int beta = live ? __ldg(row + s) : -1;
    if (beta < 0) {
      prev = 0x7fffffff;                                 // -1 tail: nothing may follow
    } else {
      if (beta <= prev || beta >= p.MB) err = 1;         // not ascending, repeated, or beyond MB
      prev = beta;
    }
    const bool valid = live && entry_valid(beta, p.MB, L);
    const long long list = valid ? ((long long)r * p.B + b) * p.MB + beta : -1ll - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, list);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(sp.cnt + list, __popc(peers));
  }
  if (err) atomicOr(&hdr->err, kErrSelection);
}

// One CTA: exclusive prefix sums of the list lengths (row_ptr) and of the
// units per list (unit_ptr); the scatter cursors start at row_ptr.  Tiles of
// 1024 lists: one coalesced count per thread (the next tile's already in
// flight), a shuffle scan in each warp, one pass over the 32 warp totals, and a
// running carry from tile to tile.  (Every partial sum is at most the entry
// count, below 2^31.)
__global__ void __launch_bounds__(1024) scan_kernel(const SparseParams sp) {
  __shared__ int s_w[2][32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t rows = sp.rows;
  int carry_a = 0, carry_u = 0;                     // lists and units before the tile
  int c_next = tid < rows ? sp.cnt[tid] : 0;
  for (int64_t base = 0; base < rows; base += 1024) {
    const int64_t i = base + tid;
    const int c = c_next;
    c_next = i + 1024 < rows ? sp.cnt[i + 1024] : 0;
    const int cu = (c + sp.qpu - 1) / sp.qpu;
    int a = c, u = cu;                               // inclusive scans within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int na = __shfl_up_sync(0xffffffffu, a, o), nu = __shfl_up_sync(0xffffffffu, u, o);
      if (lane >= o) {
        a += na;
        u += nu;
      }
    }
    if (lane == 31) {
      s_w[0][wid] = a;
      s_w[1][wid] = u;
    }
    __syncthreads();
    if (wid == 0) {                                  // inclusive scan of the warp totals
      int wa = s_w[0][lane], wu = s_w[1][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int na = __shfl_up_sync(0xffffffffu, wa, o), nu = __shfl_up_sync(0xffffffffu, wu, o);
        if (lane >= o) {
          wa += na;
          wu += nu;
        }
      }
      s_w[0][lane] = wa;
      s_w[1][lane] = wu;
    }
    __syncthreads();
    const int pa = carry_a + (wid ? s_w[0][wid - 1] : 0) + a - c;   // exclusive
    const int pu = carry_u + (wid ? s_w[1][wid - 1] : 0) + u - cu;
    if (i < rows) {
      sp.row_ptr[i] = pa;
      sp.cursor[i] = pa;
      sp.unit_ptr[i] = pu;
    }
    carry_a += s_w[0][31];
    carry_u += s_w[1][31];
    __syncthreads();                                 // the totals are read before the next tile writes them
  }
  if (tid == 0) {
    sp.row_ptr[rows] = carry_a;
    sp.unit_ptr[rows] = carry_u;
    reinterpret_cast<SparseHeader*>(sp.p.ws)->n_units = carry_u;
  }
}

// Thread per (kv head, token), tokens fastest: writes token * k + slot into
// its blocks' lists; lanes that name the same list take consecutive positions
// from one atomic.
__global__ void scatter_kernel(const SparseParams sp) {
  const Params& p = sp.p;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = idx < p.T * (int64_t)p.H_kv;
  const int r = live ? (int)(idx / p.T) : 0;
  const int64_t t = live ? idx - (int64_t)r * p.T : 0;
  const int b = request_search(p.cu_q, p.B, t);
  const int64_t L = kv_length(sp, b);
  const int32_t* row = sp.sel + (t * p.H_kv + r) * sp.k;
  const int lane = threadIdx.x & 31;
  // the last key the token sees (rightDownCausal and kv_len), or -1: what K1
  // masks by, decided once per entry here rather than per unit and row there
  int64_t lastk = L - 1;
  if (live && p.sparse_mode == 3) lastk = min(lastk, L - ((int64_t)p.cu_q[b + 1] - p.cu_q[b]) + (t - p.cu_q[b]));
  const int last = (int)max(lastk, (int64_t)-1);
  for (int s = 0; s < sp.k; ++s) {
    const int beta = live ? __ldg(row + s) : -1;
    const bool valid = live && entry_valid(beta, p.MB, L);
    const long long list = valid ? ((long long)r * p.B + b) * p.MB + beta : -1ll - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, list);
    if (valid) {
      const int leader = __ffs(peers) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(sp.cursor + list, __popc(peers));
      base = __shfl_sync(peers, base, leader);
      sp.qrec[base + __popc(peers & ((1u << lane) - 1u))] = make_int2((int)(t * 32 + s), last);
    }
  }
}

// Thread per list: its units {list, first entry, entries}.
__global__ void units_kernel(const SparseParams sp) {
  const int64_t list = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (list >= sp.rows) return;
  const int c = sp.cnt[list];
  const int base = sp.row_ptr[list];
  int4* dst = sp.units + sp.unit_ptr[list];
  // the list's (kv head, request, block), decoded once here: K1 reads a unit
  // descriptor on its softmax warps' critical path, where 64-bit divisions by
  // runtime values cost ~1 us per unit
  const int beta = (int)(list % sp.p.MB);
  const int64_t rb = list / sp.p.MB;
  const int b = (int)(rb % sp.p.B), r = (int)(rb / sp.p.B);
  for (int u = 0; u * sp.qpu < c; ++u)
    dst[u] = make_int4(beta, base + u * sp.qpu, min(sp.qpu, c - u * sp.qpu) | (r << 16), b);
}

// ------------------------------------------------------------------- K1 ----
// Shared memory: two stages of {Q, K, V}, each a 128 x 128 16-bit tile stored
// as two 16 KiB halves of 64 columns, 128-byte swizzled as TMA writes them
// (Q: rows = query entry x head; K and V: rows = the block's tokens), then
// one staging area per softmax warp for the O rows it writes out.
struct K1Layout {
  static constexpr uint32_t kTile = 32768;
  static constexpr uint32_t kStage = 3 * kTile;          // Q, K, V
  static constexpr uint32_t stage_off = 0;
  static constexpr uint32_t kORow = 64 + 16;             // 32 16-bit columns + a 16-byte pad
  static constexpr uint32_t kOWarp = 32 * kORow;
  static constexpr uint32_t ostage_off = 2 * kStage;
  static constexpr uint32_t bar_off = ostage_off + 8 * kOWarp;
  static constexpr uint32_t n_bars = 9 * 2 + 1;
  static constexpr uint32_t misc_off = bar_off + n_bars * 8;
  static constexpr uint32_t end = misc_off + 16;
  static constexpr uint32_t bytes = end + 1024;
};
static_assert(K1Layout::bytes <= 232448, "shared memory per CTA");
static_assert(K1Layout::kStage % 1024 == 0 && K1Layout::ostage_off % 1024 == 0, "1 KiB aligned tiles");

constexpr int kK1Threads = 352;       // 11 warps
constexpr int kVWarp = 10;            // the V-page producer
// tensor memory: two buffers of [S (128 columns, P over its first 64) | O (128 columns)]
constexpr uint32_t kBufCols = 256, kColO = 128;

// Shared-memory descriptor of the V page as the B operand of O = P V in
// MN-major form (N = the 128 head dims contiguous, K = tokens): 128-byte
// swizzle atoms of 64 dims x 8 tokens; the next 64 dims are the tile's other
// half (leading byte offset 16 KiB), the next 8 tokens 1 KiB further (stride
// byte offset).  Slice kk covers tokens 16 kk .. 16 kk + 15.
__device__ __forceinline__ uint64_t v_desc_mn(uint32_t tile_base, int kk) {
  const uint32_t a = tile_base + (uint32_t)kk * 2048u;
  uint64_t d = 0;
  d |= static_cast<uint64_t>((a & 0x3FFFFu) >> 4);            // start address
  d |= static_cast<uint64_t>(kHalfBytes >> 4) << 16;           // leading byte offset
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
  return d;
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

// A unit: (kv head r, request b, block beta) and its query entries [e0, e0 + ne).
struct UnitInfo {
  int r, b, beta, e0, ne;
};

// Read-only global loads issued where they stand in the program: the
// compiler may not sink an asm volatile load down to the first use of its
// value (it may sink an __ldg), so a prefetch issued early stays early and
// only its consumer waits for it.
__device__ __forceinline__ int2 ldg_now2(const int2* ptr) {
  int2 v;
  asm volatile("ld.global.nc.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ptr));
  return v;
}
__device__ __forceinline__ int4 ldg_now4(const int4* ptr) {
  int4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// A unit descriptor: {block, first entry, entries | kv head << 16, request}
// (entries <= 128).
__device__ __forceinline__ UnitInfo unit_of(const SparseParams& sp, int4 d) {
  (void)sp;
  UnitInfo ui;
  ui.beta = d.x;
  ui.e0 = d.y;
  ui.ne = d.z & 0xffff;
  ui.r = d.z >> 16;
  ui.b = d.w;
  return ui;
}

__device__ __forceinline__ UnitInfo unit_info(const SparseParams& sp, int u) {
  return unit_of(sp, __ldg(sp.units + u));
}

// What one MMA row (query entry row / g, head r * g + row % g) needs of a unit.
struct RowInfo {
  bool valid;
  int t;            // token (< 2^27)
  int s, h;
  int lim;          // last visible column of the block (-1: none)
};

// The loads behind a RowInfo, issued early (row_pre) and turned into the
// RowInfo later (row_fin), so their latency hides under other work.
struct RowPre {
  bool valid;
  int2 rec;                      // the query entry's {token * 32 + slot, last visible key}
  int r, beta;
};

// The load is unconditional, from an index clamped into range, so that no
// instruction depends on the loaded value before row_fin.
__device__ __forceinline__ RowPre row_pre(const SparseParams& sp, const UnitInfo& ui, int row) {
  const Params& p = sp.p;
  RowPre q;
  q.valid = row < ui.ne * p.g;
  q.r = ui.r;
  q.beta = ui.beta;
  const int e = ui.e0 + max(0, min(row / p.g, ui.ne - 1));
  q.rec = ldg_now2(sp.qrec + e);
  return q;
}

__device__ __forceinline__ RowInfo row_fin(const SparseParams& sp, const RowPre& q, int row) {
  const Params& p = sp.p;
  RowInfo ri;
  ri.valid = q.valid;
  ri.t = 0;
  ri.s = ri.h = 0;
  ri.lim = -1;
  if (ri.valid) {
    ri.t = (int)((uint32_t)q.rec.x >> 5);
    ri.s = q.rec.x & 31;
    ri.h = q.r * p.g + row % p.g;
    const int c = q.rec.y - q.beta * kP;       // last visible column of the block
    ri.lim = c < 0 ? -1 : (c > kP - 1 ? kP - 1 : c);
  }
  return ri;
}

// Roles: warp 0 producer of the K page and the query rows (the rows by TMA
// when g is a multiple of 8, one g-row box per query entry and half, else
// gathered by the warp's lanes), warp 10 producer of the V page, warp 1 TMEM
// owner + MMA issuer, warps 2..9 two groups of four softmax warps (group =
// unit index % 2) that also store the partials.
// Units are taken round-robin (unit i of CTA c is c + i * gridDim.x); every
// role walks the same sequence.  Unit i uses stage i % 2 and tensor-memory
// buffer i % 2, which belong to softmax group i % 2.  Q and K of a stage are
// released when S = Q K^T is done, V when O = P V is; the MMA warp issues S(i)
// before O(i-1), and each softmax group turns S(i) into P(i) before it stores
// O(i-2), so one group's softmax runs while the other stores and the tensor
// core works on both.  (10 warps and more cap a thread at 168 registers, so a
// softmax warp reads S in 64- and 32-column pieces and O in two halves.)
template <bool BF16, bool QTMA>
__global__ void __launch_bounds__(kK1Threads, 1)
    sparse_k1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_qr,
                     const SparseParams sp) {
  using Lo = K1Layout;
  const Params& p = sp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + Lo::bar_off;
  const uint32_t b_k_full = bars;                 // [2] K page (and, by TMA, the query rows) landed
  const uint32_t b_v_full = b_k_full + 16;        // [2] V page landed
  const uint32_t b_q_full = b_v_full + 16;        // [2] query rows written (gathered by the producer warp)
  const uint32_t b_kq_empty = b_q_full + 16;      // [2] the stage's Q K^T product done (Q, K free)
  const uint32_t b_v_empty = b_kq_empty + 16;     // [2] the stage's P V product done (V free)
  const uint32_t b_s_full = b_v_empty + 16;       // [2] S in the buffer
  const uint32_t b_p_full = b_s_full + 16;        // [2] P written (4 softmax warps)
  const uint32_t b_o_full = b_p_full + 16;        // [2] O in the buffer
  const uint32_t b_o_empty = b_o_full + 16;       // [2] O read (4 softmax warps)
  const uint32_t b_drain = b_o_empty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lo::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lo::misc_off + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_k_full + 8 * i, 1);
      mbar_init(b_v_full + 8 * i, 1);
      mbar_init(b_q_full + 8 * i, 1);
      mbar_init(b_kq_empty + 8 * i, 1);
      mbar_init(b_v_empty + 8 * i, 1);
      mbar_init(b_s_full + 8 * i, 1);
      mbar_init(b_p_full + 8 * i, 4);
      mbar_init(b_o_full + 8 * i, 1);
      mbar_init(b_o_empty + 8 * i, 4);
    }
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (QTMA) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_qr);
    }
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
  const int first = blockIdx.x, step = gridDim.x;

  if (warp == 0) {
    // -------------------------------------------------------- producer --
    const bool paged = p.layout != 2;
    const uint64_t pol = l2_policy_evict_last();      // a block's pages serve all its units
    uint32_t n_k[2] = {0, 0};
    int i = 0;
    for (int u = first; u < n_units; u += step, ++i) {
      const int st = i & 1;
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      const UnitInfo ui = unit_info(sp, u);
      int page = 0, tok = 0;
      if (paged) {
        page = __ldg(p.block_table + (int64_t)ui.b * p.MB + ui.beta);
        if (page < 0 || (int64_t)page >= p.NP) {
          if (lane == 0) atomicOr(&hdr->err, kErrBlockTable);
          page = (int32_t)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);   // out of bounds: zero fill
        }
      } else {
        tok = __ldg(p.cu_k + ui.b) + ui.beta * kP;
      }
      // the unit's query tokens (entry / k), lane e holding entry e
      int qt = 0;
      if (QTMA && lane < ui.ne) qt = __ldg(&sp.qrec[ui.e0 + lane].x) >> 5;
      // entries of consecutive tokens t0, t0 + 1, ... (the blocks every token
      // of a range selects): one box of 128 / g positions per half brings
      // the whole tile (positions past the entries are rows the softmax skips)
      const int t0 = __shfl_sync(0xffffffffu, qt, 0);
      const bool run = QTMA && __all_sync(0xffffffffu, lane >= ui.ne || qt == t0 + lane);
      const uint32_t q_bytes = !QTMA ? 0u : run ? 2u * (uint32_t)(sp.qpu * g) * 128u : (uint32_t)(ui.ne * g) * 2u * 128u;
      const uint32_t st_base = sbase + Lo::stage_off + st * Lo::kStage;
      if (!warp_wait(b_kq_empty + 8 * st, ph ^ 1u, ctl)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(b_k_full + 8 * st, Lo::kTile + q_bytes);
        for (int x = 0; x < 2; ++x)
          tma_k(st_base + Lo::kTile + x * kHalfBytes, &tm_k, b_k_full + 8 * st, 64 * x, tok, ui.r, page,
                p.layout, pol);
      }
      if (QTMA) {
        // entry e's g heads land in rows e*g .. e*g+g-1 of each half (1 KiB
        // aligned: g % 8 == 0).  Lane e issues entry e's two boxes (ne <= 128 / g
        // <= 16): one lane issuing all of them took ~2 us a unit and held back
        // the next QK (one box per lane instead gains nothing more: the copy
        // engine's ~45 ns a box is then the limit).
        __syncwarp();   // lane 0's expect_tx above first
        if (run) {
          if (lane == 0)
            for (int x = 0; x < 2; ++x)
              tma_load_3d(st_base + x * kHalfBytes, &tm_qr, b_k_full + 8 * st, 64 * x, ui.r * g, t0);
        } else if (lane < ui.ne) {
          for (int x = 0; x < 2; ++x)
            tma_load_3d(st_base + x * kHalfBytes + (uint32_t)(lane * g) * 128u, &tm_q, b_k_full + 8 * st,
                        64 * x, ui.r * g, qt);
        }
      }
      if (!QTMA) {
        // the unit's query rows (query entry row / g, head r * g + row % g):
        // lane l takes rows l + 32 q, two rows' loads in flight at a time
        uint8_t* qtile = smem + Lo::stage_off + st * Lo::kStage;
#pragma unroll
        for (int q0 = 0; q0 < 4; q0 += 2) {
          uint4 v[2][16];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int row = (q0 + q) * 32 + lane;
            const bool have = row < ui.ne * g;
            const int64_t t = have ? __ldg(&sp.qrec[ui.e0 + row / g].x) >> 5 : 0;
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(sp.query) +
                                                              (t * p.H_q + ui.r * g + row % g) * (int64_t)kD);
#pragma unroll
            for (int c = 0; c < 16; ++c) v[q][c] = have ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int row = (q0 + q) * 32 + lane;
            if (row < ui.ne * g) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int half = c >> 3, ch = c & 7;
                *reinterpret_cast<uint4*>(qtile + half * kHalfBytes + row * 128 + ((ch ^ (row & 7)) << 4)) = v[q][c];
              }
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_q_full + 8 * st);
      }
      ++n_k[st];
    }
    // teardown: the last loads of each stage may still be in flight
    if (lane == 0) {
      for (int st = 0; st < 2; ++st) {
        const uint64_t t0 = global_timer_ns();
        if (n_k[st])
          while (!mbar_try_wait(b_k_full + 8 * st, (n_k[st] - 1) & 1u) && global_timer_ns() - t0 < kDrainLimitNs) {
          }

      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer --
    constexpr uint32_t idesc_s = idesc_f16(BF16, 128, 128);
    constexpr uint32_t idesc_o = idesc_f16(BF16, 128, 128) | (1u << 16);   // B (V) MN-major
    bool issued = false, ok = true;
    // O(j) = P(j) V(j): P from tensor memory, V as loaded
    auto pv = [&](int j) -> bool {
      const int bj = j & 1;
      const uint32_t phj = (uint32_t)(j >> 1) & 1u;
      if (!warp_wait(b_p_full + 8 * bj, phj, ctl)) return false;
      if (!warp_wait(b_v_full + 8 * bj, phj, ctl)) return false;
      if (!warp_wait(b_o_empty + 8 * bj, phj ^ 1u, ctl)) return false;   // O(j-2) read
      tc_fence_after();
      {
        // the whole (converged) warp runs the issue, its elected lane issues
        const uint32_t buf = tmem_base + bj * kBufCols;
        const uint32_t vt = sbase + Lo::stage_off + bj * Lo::kStage + 2 * Lo::kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_ta_w(buf + kColO, buf + 8u * kk, v_desc_mn(vt, kk), idesc_o, kk ? 1u : 0u);
        tc_commit_w(b_o_full + 8 * bj);
        tc_commit_w(b_v_empty + 8 * bj);
      }
      __syncwarp();
      return true;
    };
    int i = 0;
    for (int u = first; u < n_units; u += step, ++i) {
      const int st = i & 1;
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      // S(i) overwrites P(i-2) in this buffer: P(i-2) V(i-2) must be done
      if (!warp_wait(b_k_full + 8 * st, ph, ctl) || (!QTMA && !warp_wait(b_q_full + 8 * st, ph, ctl)) ||
          !warp_wait(b_v_empty + 8 * st, ph ^ 1u, ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        // S = Q K^T: rows = (query, head), columns = the block's 128 tokens
        const uint32_t st_base = sbase + Lo::stage_off + st * Lo::kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_w(tmem_base + st * kBufCols, desc_at(st_base, kk), desc_at(st_base + Lo::kTile, kk),
                       idesc_s, kk ? 1u : 0u);
        tc_commit_w(b_s_full + 8 * st);
        tc_commit_w(b_kq_empty + 8 * st);
      }
      __syncwarp();
      issued = true;
      if (i > 0 && !pv(i - 1)) { ok = false; break; }
    }
    if (ok && i > 0) pv(i - 1);
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
  } else if (warp == kVWarp) {
    // ------------------------------------------------------ V producer --
    // The V page of unit i goes into stage i % 2 once O = P V of unit i - 2
    // is done; a warp of its own, so that the K and query loads of the next
    // units never wait behind it.
    if (lane == 0) {
      const bool paged = p.layout != 2;
      const uint64_t pol = l2_policy_evict_last();
      uint32_t n_v[2] = {0, 0};
      int i = 0;
      for (int u = first; u < n_units; u += step, ++i) {
        const int st = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;
        const UnitInfo ui = unit_info(sp, u);
        int page = 0, tok = 0;
        if (paged) {
          page = __ldg(p.block_table + (int64_t)ui.b * p.MB + ui.beta);
          if (page < 0 || (int64_t)page >= p.NP) page = (int32_t)(p.NP < 0x7fffffffLL ? p.NP : 0x7fffffffLL);
        } else {
          tok = __ldg(p.cu_k + ui.b) + ui.beta * kP;
        }
        if (!mbar_wait(b_v_empty + 8 * st, ph ^ 1u, ctl)) break;
        mbar_arrive_expect_tx(b_v_full + 8 * st, Lo::kTile);
        const uint32_t vdst = sbase + Lo::stage_off + st * Lo::kStage + 2 * Lo::kTile;
        for (int x = 0; x < 2; ++x)
          tma_k(vdst + x * kHalfBytes, &tm_v, b_v_full + 8 * st, 64 * x, tok, ui.r, page, p.layout, pol);
        ++n_v[st];
      }
      // teardown: the last V load of each stage may still be in flight
      for (int st = 0; st < 2; ++st) {
        const uint64_t t0 = global_timer_ns();
        if (n_v[st])
          while (!mbar_try_wait(b_v_full + 8 * st, (n_v[st] - 1) & 1u) && global_timer_ns() - t0 < kDrainLimitNs) {
          }
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- softmax --
    // Two groups of four warps take alternate units: group grp handles units
    // i = grp, grp + 2, ... of this CTA, whose tensor-memory buffer is grp.
    // Thread = MMA row = TMEM lane of the warp's quarter.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_s = tmem_base + ((uint32_t)(quarter * 32) << 16) + grp * kBufCols;   // S / P; O at + kColO
    uint8_t* ostage = smem + Lo::ostage_off + (warp - 2) * Lo::kOWarp;
    const float ninf = __int_as_float(0xff800000);
    const float kscale = sp.sm_scale * 1.4426950408889634f;   // base-2 softmax
    bool ok = true;
    RowInfo prev{};                                    // the unit whose O is stored next
    float prev_l = 0.f, prev_m = 0.f;
    // store O(j) (j = the group's previous unit), normalised, and its LSE.  O
    // comes out of tensor memory in two 64-column halves; each 32-column
    // quarter of the warp's rows goes through the warp's staging area (each
    // thread writes its row's 64 bytes), then every store instruction writes
    // eight 64-byte row segments.
    // the stored unit's row state comes by value: a by-reference capture of
    // it kept it in local memory (a 40-byte stack frame), whose reloads from
    // L2 showed as ~1 us per 64-column half of the store
    auto store_o = [&](int j, const RowInfo prev, const float prev_l, const float prev_m) -> bool {
      if (!warp_wait(b_o_full + 8 * grp, (uint32_t)(j >> 1) & 1u, ctl)) return false;
      tc_fence_after();
      int64_t slot = -1;
      float inv = 0.f;
      if (prev.valid) {
        const bool any = prev.lim >= 0;
        slot = ((int64_t)prev.t * p.H_q + prev.h) * sp.k + prev.s;
        inv = any ? 1.f / prev_l : 0.f;
        // natural-log LSE of the block's visible keys
        sp.lse_part[slot] = any ? (prev_m + __log2f(prev_l)) * 0.6931471805599453f : ninf;
      }
      // the partial in the input's 16-bit type (fp16: clamped to the finite
      // range; the exact value is at most max |V|, its rounding may step past it)
      const float lim16 = BF16 ? 3.0e38f : 65504.f;
      const int rsub = lane >> 2, chunk = lane & 3;  // read-back: row rsub + 8 it, 16-byte chunk
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x[64];
        tmem_ld64(t_s + kColO + 64 * hh, x);
        tmem_wait_ld();
        if (hh == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_o_empty + 8 * grp);
        }
#pragma unroll
        for (int qh = 0; qh < 2; ++qh) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = 32 * qh + 8 * c + 2 * e;
              if constexpr (BF16)   // bfloat16 has fp32's range: nothing to clamp
                w[e] = pack2(x[col] * inv, x[col + 1] * inv, true);
              else
                w[e] = pack2(fminf(fmaxf(x[col] * inv, -lim16), lim16),
                             fminf(fmaxf(x[col + 1] * inv, -lim16), lim16), false);
            }
            *reinterpret_cast<uint4*>(ostage + lane * Lo::kORow + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int rr = 8 * it + rsub;
            const int64_t sl = __shfl_sync(0xffffffffu, slot, rr);
            const uint4 v = *reinterpret_cast<const uint4*>(ostage + rr * Lo::kORow + 16 * chunk);
            if (sl >= 0) __stcs(reinterpret_cast<uint4*>(sp.o_part + sl * kD + 64 * hh + 32 * qh) + chunk, v);
          }
          __syncwarp();
        }
      }
      return true;
    };
    const int u0 = first + grp * step, ustep = 2 * step;
    int i = grp;
    RowInfo cur = u0 < n_units ? row_fin(sp, row_pre(sp, unit_info(sp, u0), row), row) : RowInfo{};
    // unit descriptors are read at clamped indices (never past the last
    // unit); whether a unit exists is decided from u alone
    int4 d_next = n_units > 0 ? __ldg(sp.units + min(u0 + ustep, n_units - 1)) : make_int4(0, 0, 0, 0);
    for (int u = u0; u < n_units; u += ustep, i += 2) {
      // the group's next unit's row loads and the descriptor of the one after,
      // issued now and used after this unit's softmax and the previous store
      RowPre pre = row_pre(sp, unit_of(sp, d_next), row);
      pre.valid = pre.valid && u + ustep < n_units;
      const int4 d_after = ldg_now4(sp.units + min(u + 2 * ustep, n_units - 1));
      if (!warp_wait(b_s_full + 8 * grp, (uint32_t)(i >> 1) & 1u, ctl)) { ok = false; break; }
      tc_fence_after();
      // every row of the warp sees the whole block (or has no entry): no
      // per-element mask (blocks off the causal diagonal, most of them)
      const bool full = __all_sync(0xffffffffu, cur.lim >= kP - 1 || !cur.valid);
      // pass 1: row max over the visible columns (eight independent chains)
      float mp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mp[a] = ninf;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x[64];
        tmem_ld64(t_s + 64 * hh, x);
        tmem_wait_ld();
        if (full) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) mp[(c >> 1) & 7] = fmax3(mp[(c >> 1) & 7], x[c], x[c + 1]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (64 * hh + c <= cur.lim) mp[c & 7] = fmaxf(mp[c & 7], x[c]);
        }
      }
      const float m = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                            fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * kscale;
      const bool any = cur.lim >= 0;
      // the unmasked exponentials' offset: +inf for a row with no visible key,
      // so that each of its p is exactly 0
      const float m_off = any ? m : __int_as_float(0x7f800000);
      // pass 2: p = 2^(s * scale - m) over each 32-column quarter; the 16
      // packed pairs of quarter hq go to P columns 16 hq .. 16 hq + 15 (S
      // columns this thread has already read)
      float lp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) lp[a] = 0.f;
#pragma unroll
      for (int hq = 0; hq < 4; ++hq) {
        float x[32];
        tmem_ld32(t_s + 32 * hq, x);
        tmem_wait_ld();
        uint32_t pk[16];
        if (full) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float a0 = ex2(fmaf(x[2 * c], kscale, -m_off));
            const float a1 = ex2(fmaf(x[2 * c + 1], kscale, -m_off));
            lp[c & 7] += a0 + a1;
            pk[c] = pack2(a0, a1, BF16);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int c0 = 32 * hq + 2 * c;
            const float a0 = any && c0 <= cur.lim ? ex2(fmaf(x[2 * c], kscale, -m)) : 0.f;
            const float a1 = any && c0 + 1 <= cur.lim ? ex2(fmaf(x[2 * c + 1], kscale, -m)) : 0.f;
            lp[c & 7] += a0 + a1;
            pk[c] = pack2(a0, a1, BF16);
          }
        }
        tmem_st16(t_s + 16 * hq, pk);
      }
      const float l = ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p_full + 8 * grp);
      if (i >= 2 && !store_o(i - 2, prev, prev_l, prev_m)) { ok = false; break; }
      prev = cur;
      prev_l = l;
      prev_m = m;
      cur = row_fin(sp, pre, row);
      d_next = d_after;
    }
    if (ok && i > grp) store_o(i - 2, prev, prev_l, prev_m);
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
__device__ __forceinline__ float4 load_partial(const uint16_t* src, bool bf16) {
  const uint2 w = __ldcs(reinterpret_cast<const uint2*>(src));
  if (bf16) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <bool BF16>
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
  // lane s (< k) reads slot s's selection entry and log-sum-exp; the row's
  // maximum and every slot's weight come from one round of loads
  const bool valid = lane < sp.k && entry_valid(__ldg(selrow + lane), p.MB, L);
  const float ls = valid ? sp.lse_part[rowid * sp.k + lane] : ninf;
  float mx = ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float wl = valid && mx > ninf ? __expf(ls - mx) : 0.f;
  float wsum = wl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const uint32_t vmask = __ballot_sync(0xffffffffu, valid && mx > ninf);
  // the valid slots' partial rows, four loads in flight at a time (lane l
  // holds dims 4l .. 4l+3)
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint16_t* base = sp.o_part + rowid * sp.k * (int64_t)kD + 4 * lane;
  uint32_t m = vmask;
  while (m) {
    int sl[4];
    int n = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sl[j] = m ? __ffs(m) - 1 : 0;
      if (m) { m &= m - 1; ++n; }
    }
    float4 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = j < n ? load_partial(base + (int64_t)sl[j] * kD, BF16) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float w = __shfl_sync(0xffffffffu, wl, sl[j]);
      if (j < n) {
        acc.x += w * o[j].x;
        acc.y += w * o[j].y;
        acc.z += w * o[j].z;
        acc.w += w * o[j].w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  reinterpret_cast<float4*>(out + rowid * kD)[lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && lane == 0) lse[rowid] = wsum > 0.f ? mx + __logf(wsum) : ninf;
}

}  // namespace

cudaError_t launch_sparse_attention(const void* tm_q, const void* tm_k, const void* tm_v, const void* tm_qr,
                                    const SparseParams& sp, bool bf16, float* out, float* lse, cudaStream_t s) {
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

  // query rows by TMA when a query entry's g rows start on a 1 KiB boundary
  const bool qtma = p.g % 8 == 0;
  auto k1 = bf16 ? (qtma ? sparse_k1_kernel<true, true> : sparse_k1_kernel<true, false>)
                 : (qtma ? sparse_k1_kernel<false, true> : sparse_k1_kernel<false, false>);
  static std::atomic<uint64_t> configured[4][64];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit(k1, (int)K1Layout::bytes, configured[(bf16 ? 2 : 0) + (qtma ? 1 : 0)], dev)) !=
      cudaSuccess)
    return e;
  k1<<<(unsigned)p.num_sms, kK1Threads, K1Layout::bytes, s>>>(*static_cast<const CUtensorMap*>(tm_q),
                                                               *static_cast<const CUtensorMap*>(tm_k),
                                                               *static_cast<const CUtensorMap*>(tm_v),
                                                               *static_cast<const CUtensorMap*>(tm_qr), sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = p.T * (int64_t)p.H_q;
  if (rows > 0) {
    if (bf16) combine_kernel<true><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(sp, out, lse);
    else combine_kernel<false><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(sp, out, lse);
  }
  return cudaGetLastError();
}

}  // namespace msa
