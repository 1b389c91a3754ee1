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
// One warp per row; the row is read once.  Scores become order-preserving
// 32-bit keys (invalid = 0).
//  1. Bound: each lane keeps the maximum of its strided elements; the k-th
//     largest of the 32 lane maxima, T0, is a lower bound for the row's k-th
//     largest key (k lanes hold an element >= T0), so only elements >= T0 can
//     be selected.
//  2. Candidates (>= T0) are counted with ballots.  Up to 32 of them are
//     compacted in index order into one slot per lane (shared memory); a
//     bitonic sort of their keys gives the k-th largest key K; the keys above
//     K are kept, and the keys equal to K in index order until k are kept.
//     Because the slots are in index order, a ballot writes the kept indices
//     ascending with no second sort.
//  3. Rows with more candidates (long runs of equal scores at the
//     threshold) take an ordered insertion into a sorted list held one entry
//     per lane instead, and a final sort of the kept indices.
// Rows of up to 32 * R elements stay in registers (R is picked per call from
// MB); longer rows are streamed in tiles of 32 * R, the second pass hitting L1.
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

// Per-lane directions of the 15 compare-exchange stages of a 32-wide bitonic
// sort (stage j of the (size, stride) sequence 2/1, 4/2, 4/1, ...): bit j is
// set when this lane keeps the larger value in a descending sort.  Depends
// only on the lane, so it is computed once per thread.
__device__ __forceinline__ uint32_t bitonic_dirs(int lane) {
  uint32_t d = 0;
  int j = 0;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1, ++j)
      if (((lane & size) == 0) == ((lane & stride) == 0)) d |= 1u << j;
  }
  return d;
}

// Bitonic sort of one value per lane across the warp; `dirs` from
// bitonic_dirs(lane).  Each stage is one shuffle, a min, a max and a select.
template <bool kDescending, typename V>
__device__ __forceinline__ V warp_sort(V s, uint32_t dirs) {
  int j = 0;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1, ++j) {
      const V other = __shfl_xor_sync(0xffffffffu, s, stride);
      const V hi = max(s, other), lo = min(s, other);
      s = (((dirs >> j) & 1u) != 0) == kDescending ? hi : lo;
    }
  }
  return s;
}

// Keys of tile `tile` (elements tile * 32R + 32 i + lane, i < R).
template <int R>
__device__ __forceinline__ void load_tile(const float* row, int MB, int tile, int lane, uint32_t (&key)[R]) {
  float v[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int c = tile * 32 * R + 32 * i + lane;
    v[i] = c < MB ? __ldg(row + c) : __int_as_float(0xff800000);
  }
#pragma unroll
  for (int i = 0; i < R; ++i) key[i] = order_key(v[i]);
}

template <int R>
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ score, int H, long long T, int MBp, int MB, int k,
                int32_t* __restrict__ out) {
  __shared__ unsigned long long s_cand[kTopkWarps][32];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const uint32_t dirs = bitonic_dirs(lane);
  const int ntiles = (MB + 32 * R - 1) / (32 * R);
  // grid: x strides over the tokens, y over the heads (no division per row)
  for (int h = blockIdx.y; h < H; h += gridDim.y)
  for (long long t = (long long)blockIdx.x * kTopkWarps + w; t < T; t += (long long)gridDim.x * kTopkWarps) {
    const float* row = score + ((long long)h * T + t) * (long long)MBp;   // rows are (h, t) in h-major order
    uint32_t key[R];
    // ---- 1. lane maxima over all tiles; the first tile stays in registers
    uint32_t lmax = 0;
    for (int tile = ntiles - 1; tile >= 0; --tile) {
      load_tile<R>(row, MB, tile, lane, key);
#pragma unroll
      for (int i = 0; i < R; ++i) lmax = max(lmax, key[i]);
    }
    const uint32_t t0 = __shfl_sync(0xffffffffu, warp_sort<true>(lmax, dirs), k - 1);
    const uint32_t lo = t0 > 0 ? t0 : 1u;
    int cur = 0;   // the tile whose keys are in registers
    // ---- 2. candidates, compacted in index order (lane j's slot: the j-th);
    // counting goes on past 32 to detect an overflow
    int ncand = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
      if (tile != cur) {
        load_tile<R>(row, MB, tile, lane, key);
        cur = tile;
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const bool c = key[i] >= lo;
        const unsigned b = __ballot_sync(0xffffffffu, c);
        const int slot = ncand + __popc(b & lt);
        if (c && slot < 32)
          s_cand[w][slot] = ((unsigned long long)key[i] << 32) | (uint32_t)(tile * 32 * R + 32 * i + lane);
        ncand += __popc(b);
      }
    }
    int32_t* orow = out + (t * H + h) * (long long)k;
    if (ncand <= 32) {
      __syncwarp();
      const unsigned long long word = lane < ncand ? s_cand[w][lane] : 0ull;
      __syncwarp();
      const uint32_t ck = (uint32_t)(word >> 32);   // 0 on lanes past the candidates
      // the k-th largest key; keys above it are kept, equal ones in index order
      const uint32_t kk = __shfl_sync(0xffffffffu, warp_sort<true>(ck, dirs), k - 1);
      const bool gt = ck > kk;
      const bool eq = ck == kk && ck != 0u;
      const int ngt = __popc(__ballot_sync(0xffffffffu, gt));
      const unsigned eqb = __ballot_sync(0xffffffffu, eq);   // all lanes vote: not under `||`
      const bool keep = gt || (eq && __popc(eqb & lt) < k - ngt);
      const unsigned kb = __ballot_sync(0xffffffffu, keep);
      if (keep) orow[__popc(kb & lt)] = (int32_t)(uint32_t)word;   // ascending: slots are in index order
      if (lane >= __popc(kb) && lane < k) orow[lane] = -1;
    } else {
      // ordered insertion of the candidates into a sorted list, one entry per lane
      uint32_t lk = 0;
      int li = 0x7fffffff;
      int cnt = 0;
      uint32_t kth = 0;
      for (int tile = 0; tile < ntiles; ++tile) {
        load_tile<R>(row, MB, tile, lane, key);
#pragma unroll 1
        for (int i = 0; i < R; ++i) {
          uint32_t kk = key[0];
#pragma unroll
          for (int j = 1; j < R; ++j)
            if (j == i) kk = key[j];
          unsigned m = __ballot_sync(0xffffffffu, kk >= lo && (cnt < k || kk > kth));
          while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const uint32_t nk = __shfl_sync(0xffffffffu, kk, src);
            if (cnt == k && nk <= kth) continue;   // beaten by an earlier insertion
            const int pos = __popc(__ballot_sync(0xffffffffu, lane < cnt && lk >= nk));
            const uint32_t uk = __shfl_up_sync(0xffffffffu, lk, 1);
            const int ui = __shfl_up_sync(0xffffffffu, li, 1);
            if (lane > pos) {
              lk = uk;
              li = ui;
            } else if (lane == pos) {
              lk = nk;
              li = tile * 32 * R + 32 * i + src;
            }
            if (cnt < k) ++cnt;
            kth = __shfl_sync(0xffffffffu, lk, k - 1);
          }
        }
      }
      // ascending block indices, -1 tail
      const int sidx = warp_sort<false>(lane < cnt ? li : 0x7fffffff, dirs);
      if (lane < k) orow[lane] = sidx == 0x7fffffff ? -1 : sidx;
    }
  }
}

template <int R>
cudaError_t launch_r(const float* score, int H, long long T, int MBp, int MB, int k, int32_t* out,
                     int num_sms, cudaStream_t s) {
  // 8 CTAs of 8 warps fill an SM; the heads share that budget
  long long bx = (T + kTopkWarps - 1) / kTopkWarps;
  long long cap = (long long)num_sms * 8 / H;
  if (cap < 1) cap = 1;
  if (bx > cap) bx = cap;
  const unsigned by = H < 65535 ? (unsigned)H : 65535u;
  topk_kernel<R><<<dim3((unsigned)bx, by), kTopkWarps * 32, 0, s>>>(score, H, T, MBp, MB, k, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const float* score, int H, long long T, int MBp, int MB, int k, int32_t* out,
                        int num_sms, cudaStream_t s) {
  if ((long long)H * T == 0) return cudaSuccess;
  const int per_lane = (MB + 31) / 32;
  if (per_lane <= 4) return launch_r<4>(score, H, T, MBp, MB, k, out, num_sms, s);
  if (per_lane <= 8) return launch_r<8>(score, H, T, MBp, MB, k, out, num_sms, s);
  if (per_lane <= 16) return launch_r<16>(score, H, T, MBp, MB, k, out, num_sms, s);
  return launch_r<36>(score, H, T, MBp, MB, k, out, num_sms, s);
}

}  // namespace msa
