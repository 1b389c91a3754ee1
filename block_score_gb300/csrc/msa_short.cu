// Short-query kernel instantiation: int8 keys with an fp16 query.
#include "msa_short.cuh"

namespace msa {

template <int TOPK>
cudaError_t launch_short_variant(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  auto kern = short_kernel<false, TOPK>;
  static std::atomic<uint64_t> configured[64];   // per device: context the limit was raised in
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = ensure_smem_limit(kern, (int)Short8::bytes, configured, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_sms);
  cfg.blockDim = dim3(Short8::kThreads);
  cfg.dynamicSmemBytes = Short8::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tq),
                            *static_cast<const CUtensorMap*>(tk), p);
}

// The plain scores, or the fused per-group selection when p.topk_k > 0.
cudaError_t launch_short_i8(const void* tq, const void* tk, const Params& p, cudaStream_t s) {
  if (p.topk_k <= 0) return launch_short_variant<0>(tq, tk, p, s);
  return p.g >= 8 ? launch_short_variant<2>(tq, tk, p, s) : launch_short_variant<16>(tq, tk, p, s);
}

}  // namespace msa
