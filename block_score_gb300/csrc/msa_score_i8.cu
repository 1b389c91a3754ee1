// Tile kernel instantiation for int8 keys with an fp16 query (pre-quantised
// K cache with per-token scale).
#include "msa_tile.cuh"

namespace msa {

cudaError_t launch_score_i8(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  using L = TileLayout<true>;
  auto kern = tile_kernel<true, false>;
  static bool configured[64] = {};   // per device; setting it twice is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_sms);
  cfg.blockDim = dim3(TileCfg<true>::kThreads);
  cfg.dynamicSmemBytes = L::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tq),
                            *static_cast<const CUtensorMap*>(tk), p);
}

}  // namespace msa
