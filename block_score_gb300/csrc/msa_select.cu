// Per-GQA-group block selection, final step (sm_103a).
//
// The score kernels of msa_index_score_topk leave, for every (query token,
// group) row, one partial list per KV chunk and epilogue group: the
// kTopkMax largest candidate keys (group score, block) of the blocks that
// part covered.  Every block of the row belongs to exactly one part, so the
// row's k best blocks are among the parts' first k entries.  This kernel takes
// them, gives the query's own block a slot when asked, and writes the indices
// in ascending order with a -1 tail (MiniMax Sparse Attention notes, section
// 4.3 Equation (3): one index set per GQA group; section 4.7 Equation (7) and
// the selector contract; section 10, checklist items 7-9).
//
// One warp per row.  The row's candidates are read 32 at a time (one per
// lane); only keys above the current k-th best survive, and ballots compact
// them into a staging batch of one key per lane.  A full batch is sorted
// descending across the lanes (bitonic sort) and its best 16 are merged into
// the running best 16 held in lanes 0..15 (the two halves form a bitonic
// sequence, so one bitonic merge suffices).  Rows with many sparse partial
// lists (short KV chunks) thus sort only the few keys that can still enter.
// Keys embed the block index, so they are distinct and no block is picked twice.
#include <cstdint>
#include <cuda_runtime.h>

#include "msa_common.cuh"
#include "msa_units.cuh"

namespace msa {
namespace {

constexpr int kSelectWarps = 8;     // warps per CTA
constexpr int kWarpRowKeys = 128;   // candidate keys a row may have for one warp to take it

// Compare-exchange of one bitonic stage across lanes (partner lane ^ stride):
// the lane keeps the larger key when keep_max.
__device__ __forceinline__ uint64_t cx(uint64_t v, int stride, bool keep_max) {
  const uint64_t w = __shfl_xor_sync(0xffffffffu, v, stride);
  return keep_max ? (w > v ? w : v) : (w < v ? w : v);
}

// Sort one key per lane descending across the warp (lane 0 = largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const bool desc = (lane & size) == 0 || size == 32;
      v = cx(v, stride, ((lane & stride) == 0) == desc);
    }
  }
  return v;
}

// Lanes 0..15 hold a descending list, lanes 16..31 an ascending one (a
// bitonic sequence); afterwards lanes 0..15 hold the best 16 keys, descending.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t v, int lane) {
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) v = cx(v, stride, (lane & stride) == 0);
  return v;
}

// Request of query token t: the last b with cu_q[b] <= t (skips requests
// without query tokens).  Whole warp; every lane gets the answer.
__device__ __forceinline__ int request_of(const Params& p, int64_t t) {
  const int lane = (int)(threadIdx.x & 31);
  int base = 0, span = p.B;
  while (span > 1) {
    const int step = (span + 31) >> 5;
    const int off = lane * step;
    const int v = off < span ? __ldg(p.cu_q + base + off) : 0x7fffffff;
    const uint32_t m = __ballot_sync(0xffffffffu, (int64_t)v <= t);
    const int l = m ? 31 - __clz((int)m) : 0;
    base += l * step;
    span = min(step, span - l * step);
  }
  return base;
}

// Running selection of one warp over the keys src[i], i = first, first +
// step, ... < n: keys above the current want-th best are compacted into a
// staging batch (one key per lane) with ballots; a full batch is sorted and its
// best 16 merged into `best` (lanes 0..15, descending).
struct WarpSelect {
  uint64_t best = 0ull, thr = 0ull, stage = 0ull;
  int ns = 0;
  __device__ __forceinline__ void flush(int lane, int want) {
    const uint64_t c = warp_sort_desc(lane < ns ? stage : 0ull, lane);
    // lanes 16..31 take the batch's best 16 in ascending order
    const uint64_t rev = __shfl_sync(0xffffffffu, c, 31 - lane);
    best = warp_merge_desc(lane < 16 ? best : rev, lane);
    thr = __shfl_sync(0xffffffffu, best, want - 1);
    ns = 0;
  }
  // c: this lane's key of a batch (0 = none)
  __device__ __forceinline__ void add(uint64_t c, int own, int lane, int want) {
    const bool keep = c > thr && cand_block(c) != own;   // the own block takes its slot separately
    const uint32_t m = __ballot_sync(0xffffffffu, keep);
    if (m == 0u) return;
    const int cnt = __popc(m);
    if (ns + cnt > 32) flush(lane, want);
    // staging lane ns + r takes the r-th kept key
    const int r = lane - ns;
    const bool mine = r >= 0 && r < cnt;
    const uint64_t v = __shfl_sync(0xffffffffu, c, mine ? (int)__fns(m, 0, r + 1) : lane);
    if (mine) stage = v;
    ns += cnt;
  }
  __device__ __forceinline__ void finish(int lane, int want) {
    if (ns > 0) flush(lane, want);
  }
};

// The row's request and selection parameters (every lane computes the same).
struct RowInfo {
  int own, want, n;      // own block (-1: none), blocks to select, candidate keys
};

__device__ __forceinline__ RowInfo row_info(const Params& p, int64_t t, int local_slot) {
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(p.ws);
  const int b = request_of(p, t);
  int err = 0;
  const ReqScratch r = read_request(p, b, err);
  const int chunk = hdr->chunk[r.cls];
  const int nchunks = r.nbc_max > 0 && chunk > 0 ? cdiv(r.nbc_max, chunk) : 1;
  const int nparts = min(2 * nchunks, p.cand_parts);
  const int64_t i = t - r.t0;                       // position inside the request
  const int64_t qpos = (int64_t)r.L - r.Lq + i;     // rightDownCausal position
  RowInfo ri;
  ri.own = -1;
  if (local_slot && i >= 0 && i < r.Lq && qpos >= 0 && qpos < r.L && qpos / kP < p.MB)
    ri.own = (int)(qpos / kP);
  ri.want = ri.own >= 0 ? p.topk_k - 1 : p.topk_k;
  ri.n = ri.want > 0 ? nparts * p.topk_k : 0;
  return ri;
}

// The selected blocks of one row (best: lanes 0..15 descending) plus the own
// block, in ascending order with a -1 tail.
__device__ __forceinline__ void write_row(uint64_t best, const RowInfo& ri, int k, int lane,
                                          int32_t* dst) {
  int mine = 0x7fffffff;                            // block index this lane outputs
  const bool chosen = lane < ri.want && best != 0ull;
  if (chosen) mine = cand_block(best);
  int count = __popc(__ballot_sync(0xffffffffu, chosen));
  if (ri.own >= 0) {
    if (lane == count) mine = ri.own;
    ++count;
  }
  // ascending order: rank of each lane's block among the chosen ones
  int rank = 0;
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const int o = __shfl_sync(0xffffffffu, mine, l);
    rank += (l < count) && (o < mine);
  }
  if (lane < count) dst[rank] = mine;
  else if (lane < k) dst[lane] = -1;
}

// One warp per row: rows whose partial lists are few (up to kWarpRowKeys keys).
__global__ void __launch_bounds__(kSelectWarps * 32)
    group_select_kernel(const Params p, int local_slot, int32_t* __restrict__ out) {
  // launched as a programmatic dependent of the score kernel: the partial
  // lists (and, transitively, the plan) are complete after this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = (int)(threadIdx.x & 31);
  const int64_t row = (int64_t)blockIdx.x * kSelectWarps + (threadIdx.x >> 5);
  if (row >= p.T * (int64_t)p.H_kv) return;
  const RowInfo ri = row_info(p, row / p.H_kv, local_slot);
  const uint64_t* cand = p.cand + (row * p.cand_parts) * (int64_t)p.topk_k;
  WarpSelect ws;
  for (int base = 0; base < ri.n; base += 32)
    ws.add(base + lane < ri.n ? __ldg(reinterpret_cast<const unsigned long long*>(cand + base + lane)) : 0ull,
           ri.own, lane, ri.want);
  ws.finish(lane, ri.want);
  write_row(ws.best, ri, p.topk_k, lane, out + row * p.topk_k);
}

// One CTA per row: rows with many partial lists (short KV chunks: decode).
// Each warp selects over every 8th batch of 32 keys; warp 0 then selects over
// the warps' best 16.
__global__ void __launch_bounds__(kSelectWarps * 32)
    group_select_row_kernel(const Params p, int local_slot, int32_t* __restrict__ out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ uint64_t s_best[kSelectWarps][16];
  const int lane = (int)(threadIdx.x & 31), warp = (int)(threadIdx.x >> 5);
  const int64_t row = blockIdx.x;
  const RowInfo ri = row_info(p, row / p.H_kv, local_slot);
  const uint64_t* cand = p.cand + (row * p.cand_parts) * (int64_t)p.topk_k;
  WarpSelect ws;
  for (int base = warp * 32; base < ri.n; base += kSelectWarps * 32)
    ws.add(base + lane < ri.n ? __ldg(reinterpret_cast<const unsigned long long*>(cand + base + lane)) : 0ull,
           ri.own, lane, ri.want);
  ws.finish(lane, ri.want);
  if (lane < 16) s_best[warp][lane] = ws.best;
  __syncthreads();
  if (warp != 0) return;
  WarpSelect all;
  const uint64_t* sb = &s_best[0][0];
  for (int base = 0; base < kSelectWarps * 16; base += 32) all.add(sb[base + lane], ri.own, lane, ri.want);
  all.finish(lane, ri.want);
  write_row(all.best, ri, p.topk_k, lane, out + row * p.topk_k);
}

}  // namespace

cudaError_t launch_group_select(const Params& p, int local_slot, int32_t* out, cudaStream_t s) {
  const int64_t rows = p.T * (int64_t)p.H_kv;
  if (rows == 0) return cudaSuccess;
  // rows with few partial lists: a warp each; many (short KV chunks): a CTA each
  const bool per_cta = (int64_t)p.cand_parts * p.topk_k > kWarpRowKeys;
  const int64_t blocks = per_cta ? rows : (rows + kSelectWarps - 1) / kSelectWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kSelectWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return per_cta ? cudaLaunchKernelEx(&cfg, group_select_row_kernel, p, local_slot, out)
                 : cudaLaunchKernelEx(&cfg, group_select_kernel, p, local_slot, out);
}

}  // namespace msa
