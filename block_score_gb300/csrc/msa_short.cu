// Short-query kernel instantiations: int8 keys with an fp16 query.
#include "msa_short.cuh"

namespace msa {

// The plain scores, or the fused per-group selection when p.topk_k > 0.
cudaError_t launch_short_i8(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  if (p.topk_k <= 0) return launch_short_kernel<false, 0, 0>(tq, tk, p, s);
  return p.g >= 8 ? launch_short_kernel<false, 2, 0>(tq, tk, p, s)
                  : launch_short_kernel<false, 16, 0>(tq, tk, p, s);
}

}  // namespace msa
