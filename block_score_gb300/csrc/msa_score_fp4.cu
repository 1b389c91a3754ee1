// Tile kernel instantiations for FP4 keys and queries: E2M1 codes with E4M3
// group scales per 16 elements (NVFP4) or E8M0 group scales per 32 (MXFP4)
// (MiniMax Sparse Attention notes, sec. 8.2, "FP4 Indexer"), plus the kernel
// that dequantises the query into the 16-bit operand the tile kernel loads.
#include "msa_tile.cuh"

namespace msa {

cudaError_t launch_score_fp4(const void* tq, const void* tk, const Params& p, bool nv,
                             cudaStream_t s) {
  return nv ? launch_tile_variant<true, false, 0, 0, 1>(tq, tk, p, s)
            : launch_tile_variant<true, true, 0, 0, 2>(tq, tk, p, s);
}

namespace {

// One thread per 8 elements (a 32-bit word of codes) of a query row of D = 128:
// the row's 64 bytes of codes and 4 (MXFP4) or 8 (NVFP4) scale bytes.
template <bool NV>
__global__ void fp4_dequant_query_kernel(const uint8_t* __restrict__ q,
                                         const uint8_t* __restrict__ q_scale, int64_t rows,
                                         uint4* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // word index
  if (i >= rows * 16) return;
  const int64_t row = i >> 4;
  const int w = (int)(i & 15);                        // elements 8w .. 8w+7
  const uint32_t codes = __ldg(reinterpret_cast<const uint32_t*>(q) + i);
  if constexpr (NV) {
    const uint32_t sb = __ldg(q_scale + row * 8 + (w >> 1));
    out[i] = fp4x8_to_f16(codes, e4m3_scale2(sb));
  } else {
    const uint32_t sb = __ldg(q_scale + row * 4 + (w >> 2));
    out[i] = fp4x8_to_bf16(codes, e8m0_scale(sb));
  }
}

}  // namespace

cudaError_t launch_fp4_dequant_query(const uint8_t* q, const uint8_t* q_scale, int64_t rows, bool nv,
                                     void* out, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (rows * 16 + threads - 1) / threads;
  if (nv)
    fp4_dequant_query_kernel<true><<<(unsigned)blocks, threads, 0, s>>>(q, q_scale, rows,
                                                                        static_cast<uint4*>(out));
  else
    fp4_dequant_query_kernel<false><<<(unsigned)blocks, threads, 0, s>>>(q, q_scale, rows,
                                                                         static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace msa
