// Tile kernel instantiations for FP8 query and keys of one type (E4M3 or
// E5M2, no scale: torch API guide "CANN ops-transformer ... msa_index_score",
// sec. 7.2), on tcgen05.mma kind::f8f6f4.
#include "msa_tile.cuh"

namespace msa {

cudaError_t launch_score_f8(const void* tq, const void* tk, const Params& p, bool e5m2,
                            cudaStream_t s) {
  return e5m2 ? launch_tile<false, false, 2>(tq, tk, p, s) : launch_tile<false, false, 1>(tq, tk, p, s);
}

}  // namespace msa
