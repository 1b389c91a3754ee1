// Short-query kernel instantiations for FP4 keys and queries: E2M1 codes with
// E4M3 group scales per 16 elements (NVFP4, fp16 operands) or E8M0 group
// scales per 32 (MXFP4, bf16 operands) (MiniMax Sparse Attention notes, sec.
// 8.2, "FP4 Indexer"); the query is the 16-bit copy the FP4 query
// dequantisation kernel writes.
#include "msa_short.cuh"

namespace msa {

cudaError_t launch_short_fp4(const void* tq, const void* tk, const Params& p, bool nv, cudaStream_t s) {
  return nv ? launch_short_kernel<false, 0, 1>(tq, tk, p, s) : launch_short_kernel<true, 0, 2>(tq, tk, p, s);
}

}  // namespace msa
