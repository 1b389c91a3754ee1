// Tile kernel instantiations for fp16 / bf16 keys (same type as the query).
#include "msa_tile.cuh"

namespace msa {

cudaError_t launch_score_16(const void* tq, const void* tk, const Params& p, bool bf16,
                            cudaStream_t s) {
  return bf16 ? launch_tile<false, true, 0>(tq, tk, p, s) : launch_tile<false, false, 0>(tq, tk, p, s);
}

}  // namespace msa
