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
// One warp per row.  Selection by rounds: each round every lane takes the
// largest of its candidates below the previous pick and a warp max gives the
// next key; keys embed the block index, so they are distinct and a round
// never picks a block twice.
#include <cstdint>
#include <cuda_runtime.h>

#include "msa_common.cuh"
#include "msa_units.cuh"

namespace msa {
namespace {

constexpr int kSelectWarps = 8;   // rows per CTA

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
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

__global__ void __launch_bounds__(kSelectWarps * 32)
    group_select_kernel(const Params p, int local_slot, int32_t* __restrict__ out) {
  const int lane = (int)(threadIdx.x & 31);
  const int64_t row = (int64_t)blockIdx.x * kSelectWarps + (threadIdx.x >> 5);
  if (row >= p.T * (int64_t)p.H_kv) return;
  const int64_t t = row / p.H_kv;
  const int k = p.topk_k;
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(p.ws);

  // the request of this token and its KV chunks, as the plan counted them
  const int b = request_of(p, t);
  int err = 0;
  const ReqScratch r = read_request(p, b, err);
  const int chunk = hdr->chunk[r.cls];
  const int nchunks = r.nbc_max > 0 && chunk > 0 ? cdiv(r.nbc_max, chunk) : 1;
  const int nparts = min(2 * nchunks, p.cand_parts);
  const int64_t i = t - r.t0;                       // position inside the request
  const int64_t qpos = (int64_t)r.L - r.Lq + i;     // rightDownCausal position
  int own = -1;
  if (local_slot && i >= 0 && i < r.Lq && qpos >= 0 && qpos < r.L && qpos / kP < p.MB)
    own = (int)(qpos / kP);
  const int want = own >= 0 ? k - 1 : k;

  const uint64_t* cand = p.cand + (row * p.cand_parts) * (int64_t)k;
  const int n = nparts * k;
  uint64_t prev = ~0ull;
  int mine = 0x7fffffff;                            // block index this lane outputs
  int count = 0;
  for (int s = 0; s < want; ++s) {
    uint64_t best = 0ull;
    for (int j = lane; j < n; j += 32) {
      const uint64_t c = __ldg(reinterpret_cast<const unsigned long long*>(cand + j));
      if (c < prev && c > best && cand_block(c) != own) best = c;
    }
    best = warp_max_u64(best);
    if (best == 0ull) break;                        // no valid candidate left
    if (lane == s) mine = cand_block(best);
    prev = best;
    ++count;
  }
  if (own >= 0) {
    if (lane == count) mine = own;
    ++count;
  }
  // ascending order: rank of each lane's block among the chosen ones
  int rank = 0;
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const int o = __shfl_sync(0xffffffffu, mine, l);
    rank += (l < count) && (o < mine);
  }
  int32_t* dst = out + row * k;
  if (lane < count) dst[rank] = mine;
  else if (lane < k) dst[lane] = -1;
}

}  // namespace

cudaError_t launch_group_select(const Params& p, int local_slot, int32_t* out, cudaStream_t s) {
  const int64_t rows = p.T * (int64_t)p.H_kv;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + kSelectWarps - 1) / kSelectWarps;
  group_select_kernel<<<(unsigned)blocks, kSelectWarps * 32, 0, s>>>(p, local_slot, out);
  return cudaGetLastError();
}

}  // namespace msa
