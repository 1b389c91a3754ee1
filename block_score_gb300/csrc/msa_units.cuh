// Device helpers shared by the score kernels: int8 -> fp16 conversion, K page
// TMA loads, decoding a work unit from the plan, and the masked row max.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "msa_common.cuh"
#include "msa_ptx.cuh"

namespace msa {

// warp roles and pipeline constants shared by the score kernels
constexpr int kEpiWarp0 = 3;             // first epilogue warp
constexpr int kCvtWarp0 = 7;             // first int8 converter warp
constexpr int kLead = 4;                 // blocks before the end of a unit at which the next is claimed
constexpr int kSched = 4;
constexpr uint32_t kTmemCols = 512;         // TMEM columns a score kernel allocates
constexpr uint32_t kTileBytes = 128 * 128 * 2;   // one 16-bit 128x128 operand tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // 64-element (128-byte) K half
constexpr uint32_t kRawBytes = 128 * 128;        // one int8 page tile
constexpr uint32_t kRawScaleBytes = 128 * 4;     // the page's per-token scales (paged layouts)
constexpr uint32_t kRawStride = kRawBytes + 1024;  // int8 tile + scales, 1 KiB aligned

__device__ __forceinline__ uint64_t desc_at(uint32_t tile_base, int k) {
  // k-th 16-element slice of a 128-deep K-major tile: halves of 64 elements
  // are separate 16 KiB swizzled tiles; inside a half, slices are 32 bytes apart.
  return smem_desc_sw128(tile_base + (uint32_t)(k >> 2) * kHalfBytes + (uint32_t)(k & 3) * 32u);
}

// Four signed int8 values (one 32-bit word, little-endian) to four fp16
// values, exactly: x + 128 is placed in the low mantissa byte of 1024.0
// (bit pattern 0x64xx, whose unit in the last place is 1), and 1152 = 1024 + 128
// is subtracted; every step is exact for |x| <= 128.
__device__ __forceinline__ void int8x4_to_half4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                      // bytes x + 128 in [0, 255]
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // (1024 + u0, 1024 + u1)
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // (1024 + u2, 1024 + u3)
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152.0
  const __half2 ra = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 rb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ra);
  hi = *reinterpret_cast<const uint32_t*>(&rb);
}

// ------------------------------------------------------------- FP4 (E2M1) --
// Codes c0..c7 of a 32-bit word sit in its nibbles 0..7 (element 2i in the
// low nibble of byte i); one byte is a pair of codes, which the hardware
// conversion (cvt.rn.f16x2.e2m1x2, through cuda_fp4.h) turns into a binary16
// pair with the low nibble in the low half.

// 8 E2M1 codes times an NVFP4 group scale (E4M3, as binary16) -> 8 binary16
// values: the hardware converts each byte (a pair of codes, the low nibble
// first) to a binary16 pair, one multiplication applies the scale.  Exact:
// every product of an E2M1 value and an E4M3 value is a binary16 number.
__device__ __forceinline__ uint4 fp4x8_to_f16(uint32_t w, __half2 scale2) {
  uint32_t r[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(w >> (8 * q)), __NV_E2M1);
    const __half2 v = __hmul2(__half2(hr), scale2);
    r[q] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// 8 E2M1 codes times an MXFP4 group scale 2^(e-127) (E8M0 code e, as an fp32
// power of two) -> 8 bfloat16 values: the hardware converts each byte (a pair
// of codes, the low nibble first) to a binary16 pair, which widens exactly to
// fp32; the scale multiplies in fp32 and the pair is rounded to bfloat16.
// Exact for every code 0 .. 252: an E2M1 value has at most two significant
// bits, and every product lies in fp32's (and bfloat16's) normal or
// subnormal range at a multiple of 2^-128 (codes 253 and 254 put the largest
// magnitudes beyond both types' range).  Everything but the conversion runs
// on the FMA pipe, where the permute-table decode this replaces kept the
// half-rate ALU pipe busy.
__device__ __forceinline__ uint4 fp4x8_to_bf16(uint32_t w, float scale) {
  uint32_t r[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(w >> (8 * q)), __NV_E2M1);
    const float2 f = __half22float2(__half2(hr));
    const __nv_bfloat162 v = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    r[q] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// Group scale bytes as the converters' multipliers.
__device__ __forceinline__ __half2 e4m3_scale2(uint32_t byte) {
  const __half h = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3));
  return __half2half2(h);
}
__device__ __forceinline__ float e8m0_scale(uint32_t byte) {
  // 2^(e-127): the code is an fp32 exponent field; 0 is 2^-127 (subnormal), 255 NaN
  return __uint_as_float(byte == 0xffu ? 0x7fc00000u : (byte ? (byte << 23) : 0x00400000u));
}

// K page tile load.  The tensor map's dimensions are ordered by increasing
// stride: BNBD (D, P, H_kv, NP); BBND (D, H_kv, P, NP); TND (D, H_kv, T2, 1).
__device__ __forceinline__ void tma_k(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x,
                                      int tok, int hk, int page, int layout, uint64_t pol) {
  if (layout == 1)
    tma_load_4d(dst, m, bar, x, tok, hk, page, pol);
  else
    tma_load_4d(dst, m, bar, x, hk, tok, page, pol);
}

// Build the descriptor of unit u of one request class from the plan
// (scheduler thread only).  `req` / `prefix` point at that class's records and
// unit prefix sums; `np` is the number of query positions per tile.
// Unit `ul` of request record `ri` (its units counted from 0).
__device__ __forceinline__ void unit_of_request(const Params& p, const ReqInfo& ri, int ul,
                                                int chunk, int np, UnitDesc& d) {
  const int per_hk = ri.ntiles * ri.nchunks;
  const int hk = ul / per_hk;
  const int rem = ul - hk * per_hk;
  const int tile_rank = rem / ri.nchunks;
  const int ch = rem - tile_rank * ri.nchunks;
  const int tile = ri.ntiles - 1 - tile_rank;
  const int i0 = tile * np;
  const int npos = min(np, ri.Lq - i0);
  const int i_last = i0 + npos - 1;
  const int lim_last = p.sparse_mode == 3 ? ri.L - ri.Lq + i_last : ri.L - 1;
  const int nbc = (ri.L > 0 && lim_last >= 0) ? min(p.MB, lim_last / kP + 1) : 0;
  d.live = 1;
  d.b = ri.b;
  d.hk = hk;
  d.t0 = ri.t0 + i0;
  d.npos = npos;
  d.i0 = i0;
  d.Lq = ri.Lq;
  d.L = ri.L;
  d.c0 = ch * chunk;
  d.c1 = (ch == ri.nchunks - 1) ? p.MBp : d.c0 + chunk;
  d.b1 = max(d.c0, min(d.c1, nbc));
  d.kbase = ri.kbase;
  d.sl = ri.sl;
  d.ch = ch;
  // the first pair's pages, so the producer can start the unit's loads at once
  d.pg0 = d.pg1 = 0;
  if (p.layout != 2 && d.b1 > d.c0) {
    const int32_t* trow = p.block_table + (int64_t)ri.b * p.MB;
    d.pg0 = __ldg(trow + d.c0);
    if (d.c0 + 1 < d.b1) d.pg1 = __ldg(trow + d.c0 + 1);
  }
}

__device__ __forceinline__ void make_unit(const Params& p, const ReqInfo* req,
                                          const int32_t* prefix, int n_req, int n_units,
                                          int chunk, int np, int u, UnitDesc& d) {
  d.live = 0;
  if (u >= n_units) return;
  // request r: last r with prefix[r] <= u
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  unit_of_request(p, req[lo], u - prefix[lo], chunk, np, d);
}

// The same lookup by a whole warp over records in global memory: each round
// reads 32 prefix sums at once and narrows the range 32-fold, so the chain
// of dependent loads is ceil(log32(n_req)) + 2 long instead of
// log2(n_req) + 2.  Every lane passes the same u; the descriptor is valid in
// lane 0 only.
__device__ __forceinline__ void make_unit_warp(const Params& p, const ReqInfo* req,
                                               const int32_t* prefix, int n_req, int n_units,
                                               int chunk, int np, int u, UnitDesc& d) {
  const int lane = (int)(threadIdx.x & 31);
  d.live = 0;
  if (u >= n_units) return;
  // invariant: prefix[base] == at <= u (prefix[0] == 0); the answer is in [base, base + span)
  int base = 0, span = n_req, at = 0;
  while (span > 1) {
    const int step = (span + 31) >> 5;
    const int off = lane * step;
    const int v = off < span ? __ldg(prefix + base + off) : 0x7fffffff;
    const uint32_t m = __ballot_sync(0xffffffffu, v <= u);
    const int l = 31 - __clz((int)m);
    at = __shfl_sync(0xffffffffu, v, l);
    base += l * step;
    span = min(step, span - l * step);
  }
  if (lane == 0) unit_of_request(p, req[base], u - at, chunk, np, d);
}

// Max of the first (climit + 1) of N values (all if climit >= N - 1).
template <int N>
__device__ __forceinline__ float masked_max(const float (&x)[N], int climit) {
  static_assert(N % 16 == 0, "groups of 16");
  const float ninf = __int_as_float(0xff800000);
  if (climit < 0) return ninf;
  float a0 = ninf, a1 = ninf, a2 = ninf, a3 = ninf;
  if (climit >= N - 1) {
    // eight independent chains (depth N / 16), folded at the end
    float b0 = ninf, b1 = ninf, b2 = ninf, b3 = ninf;
#pragma unroll
    for (int c = 0; c < N; c += 16) {
      a0 = fmax3(a0, x[c + 0], x[c + 1]);
      a1 = fmax3(a1, x[c + 2], x[c + 3]);
      a2 = fmax3(a2, x[c + 4], x[c + 5]);
      a3 = fmax3(a3, x[c + 6], x[c + 7]);
      b0 = fmax3(b0, x[c + 8], x[c + 9]);
      b1 = fmax3(b1, x[c + 10], x[c + 11]);
      b2 = fmax3(b2, x[c + 12], x[c + 13]);
      b3 = fmax3(b3, x[c + 14], x[c + 15]);
    }
    a0 = fmax3(a0, b0, b1);
    a1 = fmax3(a1, b2, b3);
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 8) {
      a0 = fmax3(a0, c + 0 <= climit ? x[c + 0] : ninf, c + 1 <= climit ? x[c + 1] : ninf);
      a1 = fmax3(a1, c + 2 <= climit ? x[c + 2] : ninf, c + 3 <= climit ? x[c + 3] : ninf);
      a2 = fmax3(a2, c + 4 <= climit ? x[c + 4] : ninf, c + 5 <= climit ? x[c + 5] : ninf);
      a3 = fmax3(a3, c + 6 <= climit ? x[c + 6] : ninf, c + 7 <= climit ? x[c + 7] : ninf);
    }
  }
  return fmax3(a0, a1, fmaxf(a2, a3));
}

// ------------------------------------------------ fused per-group selection --
// A candidate is one (score, block) pair packed into 64 bits so that one
// unsigned comparison ranks it: the score's order-preserving bits above, the
// complement of the block index below (a larger score first, then the
// smaller block).  0 is "no candidate" (-inf, NaN): below every real key.
__device__ __forceinline__ uint64_t cand_key(float x, int beta) {
  if (!(x > __int_as_float(0xff800000))) return 0ull;
  const uint32_t u = __float_as_uint(x);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)o << 32) | (uint64_t)(0xffffffffu - (uint32_t)beta);
}

__device__ __forceinline__ int cand_block(uint64_t key) {
  return (int)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
}

// Running selection of one query position's group score: the kTopkMax
// largest keys seen, in descending order (unused entries 0).
//
// TopList keeps the whole list in every lane of the position (32 registers;
// any g).  Insertion into a sorted list, branch-free per entry:
// new[i] = max(v[i], min(v[i-1], x)).
struct TopList {
  uint64_t v[kTopkMax];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < kTopkMax; ++i) v[i] = 0ull;
  }
  // the list's smallest entry: a key at or below it changes nothing
  __device__ __forceinline__ uint64_t threshold() const { return v[kTopkMax - 1]; }
  // x: the position's key (the same in all its lanes); whole warp
  __device__ __forceinline__ void insert(uint64_t x, int /*hl*/, int /*g*/) {
    if (x > v[kTopkMax - 1]) {
#pragma unroll
      for (int i = kTopkMax - 1; i > 0; --i) v[i] = max(v[i], min(v[i - 1], x));
      v[0] = max(v[0], x);
    }
  }
  __device__ __forceinline__ void store(uint64_t* dst, int k, int hl) const {
    if (hl != 0) return;
#pragma unroll
    for (int i = 0; i < kTopkMax; ++i)
      if (i < k) dst[i] = v[i];
  }
};

// TopList2 spreads the list over the first 8 lanes of a position with g >= 8
// head lanes: lane j (0 <= j < 8) holds entries 2j and 2j+1, so a thread
// spends 6 registers on it.  The same per-entry rule; entry 2j-1 comes from
// the lane before.  Lanes j >= 8 (g = 16, 32) carry values nobody reads.
struct TopList2 {
  uint64_t a, b;      // entries 2j, 2j+1
  uint64_t thr;       // entry 15, the same in every lane of the position
  __device__ __forceinline__ void clear() { a = b = thr = 0ull; }
  __device__ __forceinline__ uint64_t threshold() const { return thr; }
  __device__ __forceinline__ void insert(uint64_t x, int hl, int g) {
    uint64_t up = __shfl_up_sync(0xffffffffu, b, 1, g);
    if (hl == 0) up = ~0ull;
    const uint64_t nb = max(b, min(a, x));
    a = max(a, min(up, x));
    b = nb;
    thr = __shfl_sync(0xffffffffu, b, 7, g);
  }
  __device__ __forceinline__ void store(uint64_t* dst, int k, int hl) const {
    if (hl >= kTopkMax / 2) return;
    if (2 * hl < k) dst[2 * hl] = a;
    if (2 * hl + 1 < k) dst[2 * hl + 1] = b;
  }
};

// Max over the g consecutive lanes that hold the g heads of one query
// position (g divides 32, so the lanes of a position form an aligned group).
__device__ __forceinline__ float group_max(float m, int g) {
  for (int o = 1; o < g; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// One block of a position: `m` is this lane's row score of block col.  A
// warp vote first: when no lane's own score beats its list's threshold, no
// group score can, and the shuffles and the insertion are skipped.  Whole warp.
template <class Sel>
__device__ __forceinline__ void select_block(Sel& sel, float m, bool row_valid, int col, int MB,
                                             int hl, int g) {
  const uint64_t own = (row_valid && col < MB) ? cand_key(m, col) : 0ull;
  if (__any_sync(0xffffffffu, own > sel.threshold())) {
    const float gm = group_max(row_valid ? m : __int_as_float(0xff800000), g);
    sel.insert(col < MB ? cand_key(gm, col) : 0ull, hl, g);
  }
}

// The forced columns of the local mask within [c_lo, c_hi) (a request with
// kv_len > 0): init blocks take 1e30, the window [lo, sl] 1e29 (it wins).
// Whole warp (the ranges are the same in every lane).
template <class Sel>
__device__ __forceinline__ void insert_forced(Sel& sel, int c_lo, int c_hi, int init_blocks,
                                              int lo, int sl, int hl, int g) {
  for (int c = c_lo; c < min(c_hi, init_blocks); ++c)
    if (!(c >= lo && c <= sl)) sel.insert(cand_key(1e30f, c), hl, g);
  for (int c = max(c_lo, lo); c < min(c_hi, sl + 1); ++c) sel.insert(cand_key(1e29f, c), hl, g);
}

// Partial list `part` of row (token t, group hk).
__device__ __forceinline__ uint64_t* cand_row(const Params& p, int64_t t, int hk, int part) {
  return p.cand + ((t * p.H_kv + hk) * (int64_t)p.cand_parts + part) * (int64_t)p.topk_k;
}

}  // namespace msa
