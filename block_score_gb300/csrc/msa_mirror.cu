// Key pages converted once per call into a 16-bit copy (the mirror) in the
// workspace, sm_103a: the int8 pages of a call's query-tile requests, and the
// FP4 pages of prefill-heavy FP4 calls.
//
// The tile kernel applies every key page to each of the request's query
// tiles; with int8 keys it would otherwise convert the page once per tile.
// Here each (request, block) page is converted exactly (every int8 value is an
// fp16 integer) for all kv heads, and the tile kernel then streams the fp16
// pages by TMA like 16-bit keys, with the per-token scale applied to the dot
// products before the mask as before (feature request "MsaIndexScore",
// "calculation": DOT -> DEQUANT -> MASK -> MAX; the guide's int8 path, which
// also converts the keys into a scratch buffer before the matrix unit reads
// them, sec. 7.1).
//
// The mirror keeps the cache's page indices, in BNBD order [NP, H_kv, P, D]
// 16-bit with compact pages.  Requests of the short-query class (Lq * g <= 32)
// are scored from the int8 or FP4 pages by the short-query kernel and are
// skipped.
#include <cstdint>
#include <cuda_runtime.h>

#include "msa_common.cuh"
#include "msa_units.cuh"

namespace msa {
namespace {

// CTA per (request, logical block): the page of that block, all kv heads.
__global__ void __launch_bounds__(256)
    i8_mirror_kernel(const Params p, const int8_t* __restrict__ key, int64_t page_stride,
                     uint16_t* __restrict__ mirror) {
  const int b = (int)(blockIdx.x / (unsigned)p.MB);
  const int beta = (int)(blockIdx.x - (unsigned)b * (unsigned)p.MB);
  const int64_t Lq = (int64_t)__ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b);
  if (Lq <= 0 || Lq * p.g <= kShortRows) return;       // no query rows, or a short-query request
  const int64_t L = __ldg(p.kv_len + b);
  if (L <= 0) return;
  const int64_t nb = (L + kP - 1) / kP;
  if (beta >= nb || beta >= p.MB) return;
  const int page = __ldg(p.block_table + (int64_t)b * p.MB + beta);
  if (page < 0 || (int64_t)page >= p.NP) return;       // the tile kernel flags and zero-fills it
  const int8_t* src = key + (int64_t)page * page_stride;
  uint16_t* dst = mirror + (int64_t)page * p.H_kv * kP * kD;
  const int chunks = p.H_kv * kP * (kD / 16);          // 16-element chunks of the page
  for (int e = threadIdx.x; e < chunks; e += blockDim.x) {
    const int row = e >> 3, c = e & 7;                 // row = r * P + t (the mirror's order)
    const int r = row / kP, t = row - r * kP;
    const int64_t so = (p.layout == 0 ? (int64_t)t * p.H_kv + r : (int64_t)r * kP + t) * kD + 16 * c;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src + so));
    uint32_t h[8];
    int8x4_to_half4(w.x, h[0], h[1]);
    int8x4_to_half4(w.y, h[2], h[3]);
    int8x4_to_half4(w.z, h[4], h[5]);
    int8x4_to_half4(w.w, h[6], h[7]);
    uint4* d = reinterpret_cast<uint4*>(dst + (int64_t)row * kD + 16 * c);
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// CTA per (request, logical block): the page of that block dequantised from
// FP4 (E2M1 codes with their group scales) into 16-bit values, all kv heads.
// Every E2M1 value times its group scale is exact in the operand type (NVFP4
// in fp16, MXFP4 in bf16), so the mirror holds exactly what the converter
// warps would write for each query tile.
template <bool NV>
__global__ void __launch_bounds__(256)
    fp4_mirror_kernel(const Params p, const uint8_t* __restrict__ key, int64_t page_stride_bytes,
                      uint4* __restrict__ mirror) {
  const int b = (int)(blockIdx.x / (unsigned)p.MB);
  const int beta = (int)(blockIdx.x - (unsigned)b * (unsigned)p.MB);
  const int64_t Lq = (int64_t)__ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b);
  if (Lq <= 0 || Lq * p.g <= kShortRows) return;       // no query rows, or a short-query request
  const int64_t L = __ldg(p.kv_len + b);
  if (L <= 0) return;
  const int64_t nb = (L + kP - 1) / kP;
  if (beta >= nb || beta >= p.MB) return;
  const int page = __ldg(p.block_table + (int64_t)b * p.MB + beta);
  if (page < 0 || (int64_t)page >= p.NP) return;       // the tile kernel flags and zero-fills it
  const uint8_t* src = key + (int64_t)page * page_stride_bytes;
  const int words = p.H_kv * kP * (kD / 8);            // 8 codes (4 bytes) per word
  for (int e = threadIdx.x; e < words; e += blockDim.x) {
    const int row = e >> 4, w = e & 15;                // row = r * P + t (the mirror's order)
    const int r = row / kP, t = row - r * kP;
    const int64_t so = (p.layout == 0 ? (int64_t)t * p.H_kv + r : (int64_t)r * kP + t) * (kD / 2) + 4 * w;
    const uint32_t codes = __ldg(reinterpret_cast<const uint32_t*>(src + so));
    const int64_t srow = ((int64_t)page * p.H_kv + r) * kP + t;   // the scale bytes' row
    const int64_t di = ((int64_t)page * p.H_kv * kP + row) * (kD / 8) + w;
    if constexpr (NV) {
      const uint32_t sb = __ldg(p.k_scale8 + srow * (kD / 16) + (w >> 1));
      mirror[di] = fp4x8_to_f16(codes, e4m3_scale2(sb));
    } else {
      const uint32_t sb = __ldg(p.k_scale8 + srow * (kD / 32) + (w >> 2));
      mirror[di] = fp4x8_to_bf16(codes, e8m0_scale(sb));
    }
  }
}

}  // namespace

cudaError_t launch_fp4_mirror(const Params& p, const void* key, int64_t page_stride_bytes, bool nv,
                              void* mirror, cudaStream_t s) {
  const int64_t ctas = (int64_t)p.B * p.MB;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (nv)
    fp4_mirror_kernel<true><<<(unsigned)ctas, 256, 0, s>>>(p, static_cast<const uint8_t*>(key), page_stride_bytes,
                                                            static_cast<uint4*>(mirror));
  else
    fp4_mirror_kernel<false><<<(unsigned)ctas, 256, 0, s>>>(p, static_cast<const uint8_t*>(key), page_stride_bytes,
                                                             static_cast<uint4*>(mirror));
  return cudaGetLastError();
}

cudaError_t launch_i8_mirror(const Params& p, const void* key, int64_t page_stride, void* mirror,
                             cudaStream_t s) {
  const int64_t ctas = (int64_t)p.B * p.MB;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  i8_mirror_kernel<<<(unsigned)ctas, 256, 0, s>>>(
      p, static_cast<const int8_t*>(key), page_stride, static_cast<uint16_t*>(mirror));
  return cudaGetLastError();
}

}  // namespace msa
