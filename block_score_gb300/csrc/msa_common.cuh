// Internal definitions shared by the host launcher and the kernels of the
// block-score library: workspace (plan) layout, kernel parameters, unit
// descriptors.  Nothing here is part of the public ABI.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace msa {

constexpr int kD = 128;          // head dim handled by this library
constexpr int kP = 128;          // tokens per page (block_size)
constexpr int kTileRows = 128;   // MMA rows per work unit: floor(128/g) positions x g heads

constexpr int kErrCuQ = 0x01;
constexpr int kErrKvLen = 0x02;
constexpr int kErrCuK = 0x04;
constexpr int kErrBlockTable = 0x08;
constexpr int kErrTimeout = 0x10;
constexpr int kErrSelection = 0x20;   // a selection row out of range, repeated or not ascending

// Requests are split into two classes, each consumed by its own kernel:
//   class 0 ("tile" class): query tiles of floor(128/g) positions x g heads,
//           QK^T with the query tile as the MMA's M side;
//   class 1 ("short" class, int8 or FP4 keys): Lq * g <= kShortRows, all query
//           rows of the request as the MMA's N side against 128-token key
//           pages (M side).
constexpr int kShortRows = 32;

// Workspace layout:
//   [PlanHeader | ReqInfo x B | int32 prefix0 x (B+1) | int32 prefix1 x (B+1)]
// Class-0 request records come first (schedule order), then class 1.
struct PlanHeader {
  int32_t counter[2];   // next unit of each class (atomic)
  int32_t n_units[2];   // units of each class
  int32_t n_req[2];     // request records of each class
  int32_t chunk[2];     // blocks per KV chunk of each class (multiple of 8)
  int32_t err;          // device error bits
  int32_t pad[7];
};
static_assert(sizeof(PlanHeader) == 64, "header is 64 bytes");

// One request in schedule order.  Its units are H_kv x ntiles x nchunks,
// numbered kv-head-major, then query tiles from the last (most blocks) to the
// first, then KV chunks.  Short-class requests have ntiles == 1.
struct ReqInfo {
  int32_t b;         // original request index
  int32_t t0;        // first global query token (cu_seqlens_q[b])
  int32_t Lq;        // query tokens
  int32_t L;         // visible KV length
  int32_t ntiles;    // ceil(Lq / positions per tile)
  int32_t nchunks;   // KV chunks per tile
  int32_t kbase;     // TND: first key row of the request; else 0
  int32_t sl;        // start_loc[b]
};
static_assert(sizeof(ReqInfo) == 32, "ReqInfo is 32 bytes");

__host__ __device__ constexpr size_t workspace_bytes_for(int64_t B) {
  return (sizeof(PlanHeader) + sizeof(ReqInfo) * (size_t)B +
          2 * sizeof(int32_t) * (size_t)(B + 1) + 255) / 256 * 256;
}

__host__ __device__ inline const int32_t* plan_prefix(const uint8_t* ws, int B, int cls) {
  return reinterpret_cast<const int32_t*>(ws + sizeof(PlanHeader) + sizeof(ReqInfo) * B) +
         (cls ? (B + 1) : 0);
}

struct Params {
  int64_t T;
  int64_t NP;              // pages (paged) or T2 (TND)
  int32_t H_q, H_kv, g, np;   // np: positions per class-0 tile = floor(128 / g)
  int32_t np_short;            // positions the class-1 query box covers = floor(32 / g)
  int32_t B, MB, MBp;
  int32_t layout;          // 0 BBND, 1 BNBD, 2 TND
  int32_t short_cls;       // int8 or FP4 keys: the short-query class is enabled
  int32_t sparse_mode, init_blocks, local_blocks;
  int32_t max_q;            // host bound on every request's query length (0: none)
  int32_t num_sms;
  const int32_t* block_table;
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* cu_k;
  const int32_t* start_loc;
  const float* scale;
  float* out;
  uint8_t* ws;
  uint64_t wait_limit_ns;  // bound of every on-chip wait
  int32_t stall;           // nonzero: the MMA helper first waits on a barrier nothing completes
  // fused per-group selection (msa_index_score_topk); zero / null otherwise
  int32_t topk_k;          // blocks per selection (1..kTopkMax)
  uint64_t* cand;          // partial selections: [T][H_kv][cand_parts][topk_k] candidate keys
  int32_t cand_parts;      // partial lists per (token, group) row: 2 per KV chunk
  int32_t chunk_min[2];    // lower bound of each class's KV chunk (caps the chunks per tile)
  // FP4 keys (msa_index_score_fp4): group scale bytes of the key cache, in
  // logical page order (paged [NP, H_kv, P, D/G]; TND [T2, H_kv, D/G])
  const uint8_t* k_scale8;
  int32_t fp4_ng;          // scale bytes per row: D/32 (MXFP4) or D/16 (NVFP4)
  int32_t pad_;
};

// Blocks per selection that the fused per-group selection supports (the
// pages' selector fixes 16).
constexpr int kTopkMax = 16;

// One work unit as handed from the scheduler thread to the other roles.
struct alignas(16) UnitDesc {
  int32_t live;      // 1 = unit, 0 = no more work
  int32_t b, hk;     // request, kv head
  int32_t t0;        // global token of the tile's first position
  int32_t npos;      // valid positions in the tile
  int32_t i0;        // position of the tile's first token inside its request
  int32_t Lq, L;     // request query / KV lengths
  int32_t c0, c1;    // output columns [c0, c1) this unit writes (multiples of 8)
  int32_t b1;        // blocks [c0, b1) are computed; [b1, c1) are fill / forced
  int32_t kbase;     // TND key row base
  int32_t sl;        // start_loc of the request
  int32_t pg0, pg1;  // paged layouts: block_table entries of blocks c0 and c0 + 1 (if computed)
  int32_t ch;        // KV chunk index of the unit within its query tile
};
static_assert(sizeof(UnitDesc) == 64, "UnitDesc is 64 bytes");

__host__ __device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// One request as the plan sees it, read and validated from the per-request
// arrays (the plan kernel and the per-group selection merge both use it, so
// they agree on every request's class and KV chunk count).
struct ReqScratch {
  int Lq, L, t0, kbase, ntiles, nbc_max, cls;
};

__device__ inline ReqScratch read_request(const Params& p, int b, int& err) {
  ReqScratch r;
  const int64_t q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
  if ((b == 0 && q0 != 0) || q1 < q0 || q0 < 0 || q1 > p.T || (b == p.B - 1 && q1 != p.T))
    err |= kErrCuQ;
  int64_t lo = q0 < 0 ? 0 : (q0 > p.T ? p.T : q0);
  int64_t hi = q1 < lo ? lo : (q1 > p.T ? p.T : q1);
  r.t0 = (int)lo;
  r.Lq = (int)(hi - lo);
  // a host length bound that this request breaks: the launch may have left
  // out the kernel that would have scored it
  if (p.max_q > 0 && r.Lq > p.max_q) err |= kErrCuQ;
  int64_t L;
  if (p.layout == 2) {
    const int64_t k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    if ((b == 0 && k0 != 0) || k1 < k0 || k0 < 0 || k1 > p.NP) err |= kErrCuK;
    int64_t a = k0 < 0 ? 0 : (k0 > p.NP ? p.NP : k0);
    int64_t e = k1 < a ? a : (k1 > p.NP ? p.NP : k1);
    r.kbase = (int)a;
    L = e - a;
  } else {
    L = p.kv_len[b];
    r.kbase = 0;
    if (L < 0) {
      err |= kErrKvLen;
      L = 0;
    }
  }
  const int64_t nb = (L + kP - 1) / kP;
  if (nb > p.MB) err |= kErrKvLen;
  r.L = (int)(L > 0x7fffffff ? 0x7fffffff : L);
  // short class (int8 or FP4 keys, converted per page): every query row of
  // the request fits the N side of one MMA; 16-bit and FP8 keys stream
  // through the tile kernel at HBM speed
  r.cls = (p.short_cls && r.Lq > 0 && (int64_t)r.Lq * p.g <= kShortRows) ? 1 : 0;
  r.ntiles = r.cls ? 1 : cdiv(r.Lq, p.np);
  // the last query row sees the most blocks: q_pos = L - 1 in both modes
  r.nbc_max = L > 0 ? (int)(nb < p.MB ? nb : p.MB) : 0;
  return r;
}

// Record the message returned by msa_last_error_message() on this host thread.
void set_last_error_message(const char* msg);

// Sparse main-branch attention (msa_sparse_attention): the block-score call's
// parameters for the query, the key / value layout and the request arrays, plus
// the selection and the workspace arrays of the CSR build and the partials.
struct SparseParams {
  Params p;                // p.ws: the workspace header
  const void* query;       // [T, H_q, D] fp16 / bf16
  const int32_t* sel;      // [T, H_kv, k] logical blocks, ascending, -1 tail
  int32_t k;
  int32_t qpu;             // queries per unit: floor(128 / g)
  float sm_scale;
  int32_t pad_;
  int64_t rows;            // block -> query lists: H_kv * B * MB
  int32_t* cnt;            // [rows] list lengths
  int32_t* row_ptr;        // [rows + 1]
  int32_t* cursor;         // [rows] scatter positions
  int32_t* unit_ptr;       // [rows + 1] first unit of each list
  int2* qrec;              // [T * H_kv * k] {token * 32 + slot, last visible key of the token}, grouped by list
  int4* units;             // [T * H_kv * k] {list, first entry, entries, 0}
  uint16_t* o_part;        // [T, H_q, k, D] per-block outputs, normalised, fp16 / bf16 as the input
  float* lse_part;         // [T, H_q, k] per-block natural log-sum-exp
};

// tm_q: the query map with a box of (64 columns, g heads, 1 position), read
// when g is a multiple of 8; tm_k / tm_v: one 128-token page of one kv head.
// tm_q: query boxes of one position (one query entry's g heads); tm_qr: of
// 128 / g positions (a run of consecutive query tokens)
cudaError_t launch_sparse_attention(const void* tm_q, const void* tm_k, const void* tm_v, const void* tm_qr,
                                    const SparseParams& sp, bool bf16, float* out, float* lse,
                                    cudaStream_t s);

// Unique id (+1) of the CUDA context current on this host thread, 0 if there
// is none or the driver cannot say.  Per-device host caches are keyed by it:
// a device reset or another context on the same device invalidates them.
uint64_t current_context_id();

// Raise a kernel's dynamic shared-memory limit, once per device context.
// `done[dev]` holds the context id it was last raised for; host threads that
// race both set it, which is harmless.
template <class Kern>
inline cudaError_t ensure_smem_limit(Kern kern, int bytes, std::atomic<uint64_t> (&done)[64], int dev) {
  const uint64_t ctx = current_context_id();
  const bool cached = ctx != 0 && dev >= 0 && dev < 64;
  if (cached && done[dev].load(std::memory_order_relaxed) == ctx) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(ctx, std::memory_order_relaxed);
  return e;
}

// Host-side launchers (defined in the .cu files).
cudaError_t launch_plan(const Params& p, cudaStream_t s);
cudaError_t launch_topk(const float* score, int H, long long T, int MBp, int MB, int k, int32_t* out,
                        int num_sms, cudaStream_t s);
// The score launchers run the fused-selection variant of their kernel when
// p.topk_k > 0.
cudaError_t launch_score_16(const void* tmap_q, const void* tmap_k, const Params& p, bool bf16,
                            cudaStream_t s);
cudaError_t launch_score_f8(const void* tmap_q, const void* tmap_k, const Params& p, bool e5m2,
                            cudaStream_t s);
cudaError_t launch_score_i8(const void* tmap_q, const void* tmap_k, const Params& p,
                            cudaStream_t s);
// int8 keys read from their fp16 mirror (tmap_k maps the mirror, BNBD order)
cudaError_t launch_score_i8_mirror(const void* tmap_q, const void* tmap_k, const Params& p,
                                   cudaStream_t s);
// The int8 key pages of the query-tile requests into the fp16 mirror [NP, H_kv, P, D]
// (paged layouts; page_stride in elements of the int8 cache).
cudaError_t launch_i8_mirror(const Params& p, const void* key, int64_t page_stride, void* mirror,
                             cudaStream_t s);
// The FP4 key pages of every request into the 16-bit mirror [NP, H_kv, P, D]
// (fp16 for NVFP4, bf16 for MXFP4; paged layouts; page stride in bytes).
cudaError_t launch_fp4_mirror(const Params& p, const void* key, int64_t page_stride_bytes, bool nv,
                              void* mirror, cudaStream_t s);
cudaError_t launch_short_i8(const void* tmap_q, const void* tmap_k, const Params& p,
                            cudaStream_t s);
// FP4 keys, short-query requests: the short-query kernel with E2M1 pages
// dequantised into TMEM (nv: fp16 operands, else bf16).
cudaError_t launch_short_fp4(const void* tmap_q, const void* tmap_k, const Params& p, bool nv,
                             cudaStream_t s);
// FP4 keys: the tile kernel with E2M1 pages dequantised into 16-bit operands
// (nv: E4M3 scales per 16 elements, fp16 operands; else E8M0 per 32, bf16).
cudaError_t launch_score_fp4(const void* tmap_q, const void* tmap_k, const Params& p, bool nv,
                             cudaStream_t s);
// FP4 queries [T, H_q, D/2] with scales [T, H_q, D/G] -> 16-bit [T, H_q, D] (exact).
cudaError_t launch_fp4_dequant_query(const uint8_t* q, const uint8_t* q_scale, int64_t rows, bool nv,
                                     void* out, cudaStream_t s);
// Merge of the partial selections into [T, H_kv, k] indices (after the score kernels).
cudaError_t launch_group_select(const Params& p, int local_slot, int32_t* out, cudaStream_t s);

}  // namespace msa
