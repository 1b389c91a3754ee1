// Block top-k selection over msa_index_score's output (sm_103a).
//
// For every row (index head h, query token t) of score[H, T, MBp], the k
// blocks with the highest score, listed by block index in ascending order,
// with a -1 tail when fewer than k blocks are valid (MiniMax Sparse Attention
// notes, section 4.7: Equation (7) TopK_b over a query's block scores and the
// selector contract quoted there; section 5.3).  A block is valid when
// beta < MB and its score is above -inf (no NaN); equal scores rank the
// smaller block index first.
//
// One warp per row, two passes over the row (the second hits L1):
//  1. each lane keeps the maximum of its strided elements; the k-th largest
//     of the 32 lane maxima is a lower bound T0 for the row's k-th largest
//     value (k lanes hold an element >= T0), so no element below T0 can be
//     selected;
//  2. the row is scanned in index order, 32 elements at a time; an element
//     at or above T0 that beats the current k-th best is inserted into a
//     sorted list held one entry per lane (key descending; an equal key that
//     is already listed has the smaller index, so it stays ahead).
// The list's indices are then sorted ascending with a warp bitonic network.
// The row is HBM-bound (one read of MBp floats, k int32 written); the
// candidate bound keeps insertions to about k..2k per row on score rows.
#include <cstdint>
#include <cuda_runtime.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kTopkWarps = 8;   // rows per CTA

// Order-preserving map of fp32 onto uint32 (larger float -> larger key);
// -inf and NaN map to 0, below every valid score.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (!(x > __int_as_float(0xff800000))) return 0u;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Bitonic sort of one value per lane across the warp.
template <bool kDescending, typename V>
__device__ __forceinline__ V warp_sort(V s, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const V other = __shfl_xor_sync(0xffffffffu, s, stride);
      const bool same = ((lane & size) == 0) == ((lane & stride) == 0);
      const V hi = s > other ? s : other, lo = s > other ? other : s;
      s = (same == kDescending) ? hi : lo;
    }
  }
  return s;
}

__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ score, int H, long long T, int MBp, int MB, int k,
                int32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)H * T;
  for (long long r = (long long)blockIdx.x * kTopkWarps + (threadIdx.x >> 5); r < nrows;
       r += (long long)gridDim.x * kTopkWarps) {
    const float* row = score + r * (long long)MBp;   // rows are (h, t) in h-major order
    // pass 1: lane maxima and the bound T0
    uint32_t lmax = 0;
    for (int c = lane; c < MB; c += 32) lmax = max(lmax, order_key(__ldg(row + c)));
    const uint32_t t0 = __shfl_sync(0xffffffffu, warp_sort<true>(lmax, lane), k - 1);
    const uint32_t lo = t0 > 0 ? t0 : 1u;
    // pass 2: ordered insertion of the candidates
    uint32_t lk = 0;            // this lane's list entry (lanes < cnt)
    int li = 0x7fffffff;
    int cnt = 0;
    uint32_t kth = 0;           // key of the k-th entry once the list is full
    for (int base = 0; base < MB; base += 32) {
      const int c = base + lane;
      const uint32_t key = c < MB ? order_key(__ldg(row + c)) : 0u;
      uint32_t m = __ballot_sync(0xffffffffu, key >= lo && (cnt < k || key > kth));
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const uint32_t nk = __shfl_sync(0xffffffffu, key, src);
        if (cnt == k && nk <= kth) continue;   // beaten by an earlier insertion of this chunk
        const int pos = __popc(__ballot_sync(0xffffffffu, lane < cnt && lk >= nk));
        const uint32_t uk = __shfl_up_sync(0xffffffffu, lk, 1);
        const int ui = __shfl_up_sync(0xffffffffu, li, 1);
        if (lane > pos) {
          lk = uk;
          li = ui;
        } else if (lane == pos) {
          lk = nk;
          li = base + src;
        }
        if (cnt < k) ++cnt;
        kth = __shfl_sync(0xffffffffu, lk, k - 1);
      }
    }
    // ascending block indices, -1 tail
    const int s = warp_sort<false>(lane < cnt ? li : 0x7fffffff, lane);
    if (lane < k) {
      const long long h = r / T, t = r - h * T;
      out[(t * H + h) * k + lane] = s == 0x7fffffff ? -1 : s;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const float* score, int H, long long T, int MBp, int MB, int k, int32_t* out,
                        int num_sms, cudaStream_t s) {
  const long long rows = (long long)H * T;
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + kTopkWarps - 1) / kTopkWarps;
  const long long cap = (long long)num_sms * 8;   // 8 CTAs of 8 warps fill an SM
  if (blocks > cap) blocks = cap;
  topk_kernel<<<(unsigned)blocks, kTopkWarps * 32, 0, s>>>(score, H, T, MBp, MB, k, out);
  return cudaGetLastError();
}

}  // namespace msa
