// Tile kernel instantiations for int8 keys with an fp16 query (pre-quantised
// K cache with per-token scale): converted per tile by converter warps, or
// read from the fp16 mirror of the pages.
#include "msa_tile.cuh"

namespace msa {

cudaError_t launch_score_i8(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  return launch_tile<true, false, 0>(tq, tk, p, s);
}

cudaError_t launch_score_i8_mirror(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  return launch_tile<false, false, 0, true>(tq, tk, p, s);
}

}  // namespace msa
