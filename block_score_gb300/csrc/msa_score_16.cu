// Tile kernel instantiations for fp16 / bf16 keys (same type as the query).
#include "msa_tile.cuh"

namespace msa {

template <bool KI8, bool BF16>
static cudaError_t launch_tile(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  using L = TileLayout<KI8>;
  auto kern = tile_kernel<KI8, BF16>;
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
  cfg.blockDim = dim3(TileCfg<KI8>::kThreads);
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

cudaError_t launch_score_16(const void* tq, const void* tk, const Params& p, bool bf16,
                            cudaStream_t s) {
  return bf16 ? launch_tile<false, true>(tq, tk, p, s) : launch_tile<false, false>(tq, tk, p, s);
}

}  // namespace msa
