// Plan kernel: one CTA turns the per-request arrays (cu_seqlens_q, kv_len or
// cu_seqlens_k, start_loc) into the work plan the score kernel consumes.
//
// A work unit is (request, kv head, query tile, KV chunk).  A query tile packs
// floor(128/g) consecutive query positions x the g heads of one GQA group into
// the 128 MMA rows (the "query concatenation" of the MSA kernel notes, sec.
// 5.9).  Blocks are independent maxima, so splitting the KV range of a tile
// into chunks needs no combine step; chunks keep every SM busy on short-query
// (decode) batches, in the spirit of the reference tiling's KV split for
// "short M, long S" decode (torch API guide, sec. 8.3).
//
// The plan also validates the device arrays (guide sec. 4 rules) and records
// violations in the error word instead of faulting.
#include "msa_common.cuh"

namespace msa {

namespace {

constexpr int kPlanThreads = 1024;

// Inclusive block scan of one value per thread (blockDim.x threads, a
// multiple of 32 and at most 1024).
__device__ int block_incl_scan(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += s_warp[warp - 1];
  __syncthreads();
  return v;
}

__device__ int chunk_for(unsigned long long work, int num_sms, int MBp, int gran) {
  // about 16 units per SM on average, never below `gran` blocks (the tail of
  // a call is then a fraction of one short unit); a multiple of `gran` (the
  // store width of the kernel's epilogue: 8 for the tile kernel, 4 for the
  // short-query kernel)
  const unsigned long long target = (unsigned long long)num_sms * 16ull;
  const unsigned long long g = (unsigned long long)gran;
  unsigned long long c = (work + target - 1) / target;
  if (c < g) c = g;
  c = (c + g - 1) / g * g;
  if (c > (unsigned long long)MBp) c = (unsigned long long)MBp;
  return (int)c;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const Params p) {
  // Let the score kernels start their prologue (barrier init, TMEM
  // allocation); they wait for this grid's completion before reading the plan.
  asm volatile("griddepcontrol.launch_dependents;");
  // This grid is launched as a programmatic dependent of whatever precedes it
  // on the stream, so its launch overlaps that kernel's last units; it reads
  // nothing until the preceding kernel has completed (its request arrays may
  // be that kernel's output, and a previous call's score kernel still reads
  // the workspace).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  __shared__ int s_warp[32];
  __shared__ unsigned long long s_work[2];
  __shared__ int s_err;
  __shared__ __align__(16) int s_key[kPlanThreads];
  __shared__ int s_units[kPlanThreads];
  __shared__ int s_tot[2];
  __shared__ int s_nreq[2];

  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  ReqInfo* req = reinterpret_cast<ReqInfo*>(p.ws + sizeof(PlanHeader));
  int32_t* prefix0 = const_cast<int32_t*>(plan_prefix(p.ws, p.B, 0));
  int32_t* prefix1 = const_cast<int32_t*>(plan_prefix(p.ws, p.B, 1));
  const int tid = threadIdx.x;

  if (tid == 0) {
    s_work[0] = s_work[1] = 0ull;
    s_err = 0;
    s_nreq[0] = s_nreq[1] = 0;
  }
  __syncthreads();

  // pass 1: read every request once, validate, sum the work of each class
  // (blocks x kv heads x tiles, an upper bound that only sets the chunk sizes)
  const bool small = p.B <= (int)blockDim.x;
  int err = 0;
  unsigned long long work[2] = {0ull, 0ull};
  int nreq[2] = {0, 0};
  ReqScratch mine{};
  int my_sl = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int sl = __ldg(p.start_loc + b);       // issued together with the length loads
    ReqScratch r = read_request(p, b, err);
    work[r.cls] += (unsigned long long)p.H_kv * r.ntiles * r.nbc_max;
    nreq[r.cls] += 1;
    if (small) {
      mine = r;
      my_sl = sl;
    }
  }
  // warp-level reductions first: one shared atomic per warp, not per request
  err = __reduce_or_sync(0xffffffffu, (unsigned)err);
  nreq[0] = __reduce_add_sync(0xffffffffu, (unsigned)nreq[0]);
  nreq[1] = __reduce_add_sync(0xffffffffu, (unsigned)nreq[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    work[0] += __shfl_xor_sync(0xffffffffu, work[0], o);
    work[1] += __shfl_xor_sync(0xffffffffu, work[1], o);
  }
  if ((tid & 31) == 0) {
    if (err) atomicOr(&s_err, err);
    if (work[0]) atomicAdd(&s_work[0], work[0]);
    if (work[1]) atomicAdd(&s_work[1], work[1]);
    if (nreq[0]) atomicAdd(&s_nreq[0], nreq[0]);
    if (nreq[1]) atomicAdd(&s_nreq[1], nreq[1]);
  }
  __syncthreads();
  // a caller-side floor (the fused selection bounds the KV chunks of a tile)
  const int chunk0 = max(chunk_for(s_work[0], p.num_sms, p.MBp, 8), min(p.chunk_min[0], p.MBp));
  const int chunk1 = max(chunk_for(s_work[1], p.num_sms, p.MBp, 4), min(p.chunk_min[1], p.MBp));
  const int n0 = s_nreq[0];

  if (small) {
    // schedule order: class 0 first, then class 1; inside a class longest
    // first by the cost of the request's largest unit; the rank of a
    // request is the number of requests that go before it
    int cls = 0, units = 0, nchunks = 1;
    // one sort key per request: class 0 before class 1, then larger unit cost
    // first (requests without query rows last in their class), then index
    int key = 0x7fffffff;
    if (tid < p.B) {
      cls = mine.cls;
      const int chunk = cls ? chunk1 : chunk0;
      nchunks = mine.nbc_max > 0 ? cdiv(mine.nbc_max, chunk) : 1;
      units = mine.Lq > 0 ? p.H_kv * mine.ntiles * nchunks : 0;
      const int cost = mine.Lq > 0 ? (mine.nbc_max < chunk ? mine.nbc_max : chunk) + 1 : 0;
      key = (cls << 30) | (0x3fffffff - cost);
    }
    s_key[tid] = key;
    __syncthreads();
    if (tid < p.B) {
      // rank = requests that sort before this one; keys are read four at a time
      int rank = 0;
      const int4* k4 = reinterpret_cast<const int4*>(s_key);
      const int nq = (p.B + 3) >> 2;
#pragma unroll 4
      for (int q = 0; q < nq; ++q) {
        const int4 v = k4[q];
        const int j = q * 4;
        rank += (v.x < key) || (v.x == key && j + 0 < tid);
        rank += (j + 1 < p.B) && ((v.y < key) || (v.y == key && j + 1 < tid));
        rank += (j + 2 < p.B) && ((v.z < key) || (v.z == key && j + 2 < tid));
        rank += (j + 3 < p.B) && ((v.w < key) || (v.w == key && j + 3 < tid));
      }
      ReqInfo ri;
      ri.b = tid;
      ri.t0 = mine.t0;
      ri.Lq = mine.Lq;
      ri.L = mine.L;
      ri.ntiles = mine.ntiles;
      ri.nchunks = nchunks;
      ri.kbase = mine.kbase;
      ri.sl = my_sl;
      req[rank] = ri;
      s_units[rank] = units;
    }
    __syncthreads();
    // per-class inclusive scans over the ranked slots
    const int v0 = tid < n0 ? s_units[tid] : 0;
    const int incl0 = block_incl_scan(v0, s_warp);
    if (tid < n0) prefix0[tid + 1] = incl0;
    if (tid == (int)blockDim.x - 1) s_tot[0] = incl0;
    const int n1 = p.B - n0;
    const int v1 = tid < n1 ? s_units[n0 + tid] : 0;
    const int incl1 = block_incl_scan(v1, s_warp);
    if (tid < n1) prefix1[tid + 1] = incl1;
    if (tid == (int)blockDim.x - 1) s_tot[1] = incl1;
    __syncthreads();
  } else {
    // large batches: natural order inside each class; compaction by a scan of
    // the class flags, then per-class unit prefix sums
    int carry_slot[2] = {0, 0}, carry_units[2] = {0, 0};
    for (int base = 0; base < p.B; base += (int)blockDim.x) {
      const int b = base + tid;
      ReqScratch r{};
      int units = 0, nchunks = 1;
      const bool live = b < p.B;
      if (live) {
        int e2 = 0;
        r = read_request(p, b, e2);
        const int chunk = r.cls ? chunk1 : chunk0;
        nchunks = r.nbc_max > 0 ? cdiv(r.nbc_max, chunk) : 1;
        units = r.Lq > 0 ? p.H_kv * r.ntiles * nchunks : 0;
      }
      for (int c = 0; c < 2; ++c) {
        const int mine_c = live && r.cls == c;
        const int slot_incl = block_incl_scan(mine_c, s_warp);
        const int units_incl = block_incl_scan(mine_c ? units : 0, s_warp);
        if (mine_c) {
          const int slot = carry_slot[c] + slot_incl - 1;
          ReqInfo ri;
          ri.b = b;
          ri.t0 = r.t0;
          ri.Lq = r.Lq;
          ri.L = r.L;
          ri.ntiles = r.ntiles;
          ri.nchunks = nchunks;
          ri.kbase = r.kbase;
          ri.sl = p.start_loc[b];
          req[(c ? n0 : 0) + slot] = ri;
          (c ? prefix1 : prefix0)[slot + 1] = carry_units[c] + units_incl;
        }
        if (tid == (int)blockDim.x - 1) {
          s_tot[0] = slot_incl;
          s_tot[1] = units_incl;
        }
        __syncthreads();
        carry_slot[c] += s_tot[0];
        carry_units[c] += s_tot[1];
        __syncthreads();
      }
    }
    if (tid == 0) {
      s_tot[0] = carry_units[0];
      s_tot[1] = carry_units[1];
    }
    __syncthreads();
  }
  if (tid == 0) {
    prefix0[0] = 0;
    prefix1[0] = 0;
    hdr->counter[0] = hdr->counter[1] = 0;
    hdr->n_units[0] = s_tot[0];
    hdr->n_units[1] = s_tot[1];
    hdr->n_req[0] = n0;
    hdr->n_req[1] = p.B - n0;
    hdr->chunk[0] = chunk0;
    hdr->chunk[1] = chunk1;
    hdr->err = s_err;
  }
}

}  // namespace

cudaError_t launch_plan(const Params& p, cudaStream_t s) {
  // small batches need few threads: fewer warps make every barrier cheaper
  const int threads = p.B <= 128 ? 128 : kPlanThreads;
  // programmatic dependent of whatever precedes it on the stream: behind a
  // previous call's score kernel, which triggers at its start, the plan is
  // launched and resident before that kernel ends (see griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace msa
