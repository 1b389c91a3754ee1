// C ABI of the block-score library: argument validation (the op's rules from
// the torch API guide "CANN ops-transformer ... msa_index_score", sec. 3, 4,
// 8.1 and 10), output shape (sec. 5 / 8.5), workspace sizing, TMA tensor maps
// and the launches (plan, tile-class score kernel, short-query score kernel).
// No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "msa_index_score.h"
#include "msa_common.cuh"

namespace {

thread_local char g_msg[512] = "";

msa_status_t fail(msa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

msa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round16(int64_t x) { return (x + 15) / 16 * 16; }

bool is_f8(msa_dtype_t t) { return t == MSA_E4M3 || t == MSA_E5M2; }

int elem_size(msa_dtype_t t) { return (t == MSA_I8 || is_f8(t) || t == MSA_E2M1) ? 1 : 2; }

// Storage elements of one key row of D values (FP4: two values per byte).
int64_t row_elems(const msa_index_score_args* a) {
  return a->k_dtype == MSA_E2M1 ? a->D / 2 : a->D;
}

// Host-side checks; everything that can be decided without reading device memory.
// `fp4`: the call is msa_index_score_fp4 (E2M1 query and key, scales given apart).
msa_status_t validate(const msa_index_score_args* a, bool fp4 = false) {
  if (!a) return fail(MSA_ERR_INVALID_ARG, "args is NULL");
  if (fp4 != (a->q_dtype == MSA_E2M1 || a->k_dtype == MSA_E2M1)) {
    if (fp4) return fail(MSA_ERR_INVALID_ARG, "msa_index_score_fp4 takes E2M1 query and key");
    return fail(MSA_ERR_INVALID_ARG, "E2M1 (FP4) inputs go through msa_index_score_fp4");
  }
  if (a->layout != MSA_LAYOUT_BBND && a->layout != MSA_LAYOUT_BNBD && a->layout != MSA_LAYOUT_TND)
    return fail(MSA_ERR_INVALID_ARG, "layout must be BBND, BNBD or TND");
  if (a->sparse_mode != 0 && a->sparse_mode != 3)
    return fail(MSA_ERR_INVALID_ARG, "sparse_mode must be 0 or 3");
  if (a->q_dtype != MSA_F16 && a->q_dtype != MSA_BF16 && !is_f8(a->q_dtype) && !fp4)
    return fail(MSA_ERR_INVALID_ARG, "query dtype must be fp16, bf16, fp8 e4m3 or fp8 e5m2");
  if (fp4) {
    if (a->q_dtype != MSA_E2M1 || a->k_dtype != MSA_E2M1)
      return fail(MSA_ERR_INVALID_ARG, "FP4 query and key must both be E2M1");
    if (a->scale) return fail(MSA_ERR_INVALID_ARG, "FP4 inputs take their group scales, not scale");
  } else if (is_f8(a->q_dtype) || is_f8(a->k_dtype)) {
    if (a->k_dtype != a->q_dtype)
      return fail(MSA_ERR_INVALID_ARG, "fp8 query and key must be of the same fp8 type");
    if (a->scale) return fail(MSA_ERR_INVALID_ARG, "fp8 inputs take no scale");
  } else if (a->k_dtype == MSA_I8) {
    if (a->q_dtype != MSA_F16) return fail(MSA_ERR_INVALID_ARG, "int8 key requires an fp16 query");
    if (!a->scale) return fail(MSA_ERR_INVALID_ARG, "int8 key requires scale");
  } else if (a->k_dtype == MSA_F16 || a->k_dtype == MSA_BF16) {
    if (a->k_dtype != a->q_dtype) return fail(MSA_ERR_INVALID_ARG, "key dtype must match query");
    if (a->scale) return fail(MSA_ERR_INVALID_ARG, "scale is only allowed with int8 keys");
  } else {
    return fail(MSA_ERR_INVALID_ARG, "key dtype must be fp16, bf16 or int8");
  }
  if (a->T < 0 || a->B < 0) return fail(MSA_ERR_INVALID_ARG, "T and B must be >= 0");
  if (a->B == 0 && a->T > 0) return fail(MSA_ERR_INVALID_ARG, "T > 0 needs at least one request");
  if (a->H_q <= 0 || a->H_kv <= 0) return fail(MSA_ERR_INVALID_ARG, "head counts must be > 0");
  if (a->H_q % a->H_kv != 0) return fail(MSA_ERR_INVALID_ARG, "H_q must be a multiple of H_kv");
  if (a->D != msa::kD) return fail(MSA_ERR_UNSUPPORTED, "only D = 128 is built (got %d)", a->D);
  if (a->P != msa::kP) return fail(MSA_ERR_UNSUPPORTED, "only block_size P = 128 is built (got %d)", a->P);
  if (a->H_q / a->H_kv > 128)
    return fail(MSA_ERR_UNSUPPORTED, "GQA group size H_q/H_kv > 128 is not built");
  if (a->MB < 1) return fail(MSA_ERR_INVALID_ARG, "MB must be >= 1");
  const int64_t mbp = round16(a->MB);
  const int64_t cap = a->layout == MSA_LAYOUT_TND ? mbp : a->MB;
  if (a->init_blocks < 0 || a->local_blocks < 0 || a->init_blocks > cap || a->local_blocks > cap)
    return fail(MSA_ERR_INVALID_ARG, "init_blocks/local_blocks must be in [0, %lld]", (long long)cap);
  if (a->max_seqlen_q < 0) return fail(MSA_ERR_INVALID_ARG, "max_seqlen_q must be >= 0 (0: not given)");
  if (a->T > 0x7fffffffLL - 1) return fail(MSA_ERR_UNSUPPORTED, "T too large");
  if (a->NP < 1 || a->NP > 0x7fffffffLL - 1)
    return fail(MSA_ERR_INVALID_ARG, "NP (pages or TND rows) must be in [1, 2^31-2]");
  const int es = elem_size(a->k_dtype);
  if (a->layout == MSA_LAYOUT_TND) {
    if (a->block_table) return fail(MSA_ERR_INVALID_ARG, "TND takes no block_table");
    if (!a->cu_seqlens_k || a->kv_len)
      return fail(MSA_ERR_INVALID_ARG, "TND takes cu_seqlens_k [B+1] and no kv_len");
    if (a->page_stride != (int64_t)a->H_kv * row_elems(a))
      return fail(MSA_ERR_INVALID_ARG, "TND key must be contiguous");
  } else {
    if (a->B > 0 && !a->block_table) return fail(MSA_ERR_INVALID_ARG, "paged layout needs block_table");
    if (a->B > 0 && !a->kv_len) return fail(MSA_ERR_INVALID_ARG, "paged layout needs kv_len [B]");
    if (a->cu_seqlens_k) return fail(MSA_ERR_INVALID_ARG, "cu_seqlens_k is for TND only");
    if (a->page_stride < (int64_t)a->P * a->H_kv * row_elems(a))
      return fail(MSA_ERR_INVALID_ARG, "page_stride smaller than a compact page");
    if ((a->page_stride * es) % 16 != 0)
      return fail(MSA_ERR_UNSUPPORTED, "page stride must be a multiple of 16 bytes");
  }
  if (a->T > 0 && a->B > 0) {
    if (!a->query || !a->key_cache || !a->cu_seqlens_q || !a->start_loc)
      return fail(MSA_ERR_INVALID_ARG, "query, key_cache, cu_seqlens_q and start_loc are required");
    if (!aligned(a->query, 16) || !aligned(a->key_cache, 16))
      return fail(MSA_ERR_INVALID_ARG, "query and key_cache must be 16-byte aligned");
    if (a->scale && !aligned(a->scale, 4)) return fail(MSA_ERR_INVALID_ARG, "scale must be 4-byte aligned");
    if (a->scale && a->layout != MSA_LAYOUT_TND && !aligned(a->scale, 16))
      return fail(MSA_ERR_UNSUPPORTED, "paged int8 scale must be 16-byte aligned");
  }
  return MSA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Watchdog controls (msa_set_watchdog): limit of one on-chip pipeline wait
// (0 = default) and the test stall.
constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;   // 4 s: far above any legitimate wait
std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int32_t> g_wait_stall{0};

int sm_count(int dev) {
  static std::atomic<int> cache[64];   // per device; threads that race store the same value
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

msa_status_t fill_params(const msa_index_score_args* a, float* out, void* ws, msa::Params& p) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int g = a->H_q / a->H_kv;
  p.T = a->T;
  p.NP = a->NP;
  p.H_q = a->H_q;
  p.H_kv = a->H_kv;
  p.g = g;
  p.np = msa::kTileRows / g;
  p.np_short = g <= msa::kShortRows ? msa::kShortRows / g : 1;
  p.B = a->B;
  p.MB = a->MB;
  p.MBp = (int32_t)round16(a->MB);
  p.layout = (int32_t)a->layout;
  p.short_cls = (a->k_dtype == MSA_I8 || a->k_dtype == MSA_E2M1) ? 1 : 0;
  p.sparse_mode = a->sparse_mode;
  p.init_blocks = a->init_blocks;
  p.local_blocks = a->local_blocks;
  p.max_q = a->max_seqlen_q;
  p.num_sms = sm_count(dev);
  p.block_table = a->block_table;
  p.cu_q = a->cu_seqlens_q;
  p.kv_len = a->kv_len;
  p.cu_k = a->cu_seqlens_k;
  p.start_loc = a->start_loc;
  p.scale = a->scale;
  p.out = out;
  p.ws = static_cast<uint8_t*>(ws);
  const uint64_t lim = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.wait_limit_ns = lim ? lim : kDefaultWaitLimitNs;
  p.stall = g_wait_stall.load(std::memory_order_relaxed) ? 1 : 0;
  p.topk_k = 0;
  p.cand = nullptr;
  p.cand_parts = 0;
  p.chunk_min[0] = p.chunk_min[1] = 0;
  p.k_scale8 = nullptr;
  p.fp4_ng = 0;
  p.pad_ = 0;
  return MSA_OK;
}

// Fused per-group selection: the partial lists of all rows (T x H_kv rows,
// 2 per KV chunk of a tile, k keys of 8 bytes each) are kept within
// kCandBudget bytes by capping the KV chunks of a tile (the plan's chunk floor).
constexpr int64_t kCandBudget = 64ll << 20;

struct SelectPlan {
  int32_t chunks;         // KV chunks per tile at most
  int32_t parts;          // partial lists per row
  int32_t chunk_min[2];   // plan chunk floors (tile class: multiple of 8, short class: of 4)
  size_t plan_bytes;      // the score plan's workspace
  size_t cand_bytes;      // the partial lists
};

SelectPlan select_plan(const msa_index_score_args* a, int k) {
  SelectPlan sp;
  const int64_t mbp = round16(a->MB);
  const int64_t most = (mbp + 3) / 4;               // chunks of the smallest chunk size (4 blocks)
  const int64_t per_chunk = a->T * (int64_t)a->H_kv * 2 * k * 8;
  int64_t c = per_chunk > 0 ? kCandBudget / per_chunk : most;
  c = c < 1 ? 1 : (c > most ? most : c);
  const int64_t floor_blocks = (mbp + c - 1) / c;
  sp.chunks = (int32_t)c;
  sp.parts = (int32_t)(2 * c);
  sp.chunk_min[0] = (int32_t)((floor_blocks + 7) / 8 * 8);
  sp.chunk_min[1] = (int32_t)((floor_blocks + 3) / 4 * 4);
  sp.plan_bytes = msa::workspace_bytes_for(a->B);
  sp.cand_bytes = (size_t)(a->T * (int64_t)a->H_kv * sp.parts * k) * 8;
  return sp;
}

msa_status_t validate_select(const msa_index_score_args* a, int k) {
  if (k < 1 || k > msa::kTopkMax)
    return fail(MSA_ERR_INVALID_ARG, "k must be in [1, %d]", msa::kTopkMax);
  const int g = a->H_q / a->H_kv;
  if (32 % g != 0)
    return fail(MSA_ERR_UNSUPPORTED,
                "the fused per-group selection needs H_q / H_kv in {1, 2, 4, 8, 16, 32} (got %d)", g);
  return MSA_OK;
}

msa_status_t check_ws(const msa_index_score_args* a, void* ws, size_t bytes) {
  if (!ws) return fail(MSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(MSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const size_t need = msa::workspace_bytes_for(a->B);
  if (bytes < need)
    return fail(MSA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, bytes);
  return MSA_OK;
}

// Encoded tensor maps of recent calls, per host thread: re-encoding costs
// microseconds of host time per launch, and repeated calls on the same
// buffers (a decode loop) reuse the same maps.
struct MapKey {
  const void* base;
  int32_t dtype, rank, swizzle;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5];
};

CUresult encode_cached(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank,
                       void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                       const cuuint32_t* box, const cuuint32_t* es, CUtensorMapSwizzle sw) {
  constexpr int kEntries = 16;
  struct Entry {
    MapKey key;
    CUtensorMap map;
    uint64_t stamp;
  };
  thread_local Entry cache[kEntries];
  thread_local uint64_t clock = 0;
  MapKey k;
  std::memset(&k, 0, sizeof k);
  k.base = base;
  k.dtype = (int32_t)dt;
  k.rank = (int32_t)rank;
  k.swizzle = (int32_t)sw;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  int victim = 0;
  for (int i = 0; i < kEntries; ++i) {
    if (cache[i].stamp && std::memcmp(&cache[i].key, &k, sizeof k) == 0) {
      cache[i].stamp = ++clock;
      *m = cache[i].map;
      return CUDA_SUCCESS;
    }
    if (cache[i].stamp < cache[victim].stamp) victim = i;
  }
  CUresult r = enc(m, dt, rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    cache[victim].key = k;
    cache[victim].map = *m;
    cache[victim].stamp = ++clock;
  }
  return r;
}

// fp4_q16: FP4 call, the dequantised query (fp16 for NVFP4, bf16 for MXFP4)
// that the tile kernel reads, else NULL.
msa_status_t make_maps(const msa_index_score_args* a, const msa::Params& p, CUtensorMap* tq,
                       CUtensorMap* tk, CUtensorMap* tq_short, CUtensorMap* tk_short,
                       const void* fp4_q16 = nullptr, bool fp4_nv = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const bool fp4 = fp4_q16 != nullptr;
  const bool f8 = is_f8(a->q_dtype);
  const CUtensorMapDataType qdt = fp4 ? (fp4_nv ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
                                  : f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : a->q_dtype == MSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const void* qbase = fp4 ? fp4_q16 : a->query;
  const cuuint64_t qsz = f8 ? 1 : 2;
  // query [T, H_q, D]: dims (D, H_q, T); a box is (128 bytes of D, g, positions):
  // one GQA group x a run of positions, 128-byte swizzled
  auto qmap = [&](CUtensorMap* m, int positions, const char* what) -> msa_status_t {
    cuuint64_t dims[3] = {(cuuint64_t)a->D, (cuuint64_t)a->H_q, (cuuint64_t)a->T};
    cuuint64_t strides[2] = {(cuuint64_t)a->D * qsz, (cuuint64_t)a->H_q * a->D * qsz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / qsz), (cuuint32_t)p.g, (cuuint32_t)positions};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode_cached(enc, m, qdt, 3, const_cast<void*>(qbase), dims, strides, box, es,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "%s tensor map: CUresult %d", what, (int)r);
    return MSA_OK;
  };
  // one 128-token key page of one kv head; dims ordered by increasing stride
  auto kmap = [&](CUtensorMap* m, bool swizzle_int8, const char* what) -> msa_status_t {
    const bool i8 = a->k_dtype == MSA_I8;
    const bool byte = i8 || f8 || fp4;           // one-byte elements: a 128-element row is 128 bytes
    const cuuint64_t esz = byte ? 1 : 2;
    const CUtensorMapDataType kdt = byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : qdt;
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    cuuint32_t box[4];
    // FP4: a row is 64 bytes of packed codes (the whole row in one box)
    const cuuint32_t bx = fp4 ? 64 : (byte ? 128 : 64);
    const cuuint64_t dx = fp4 ? (cuuint64_t)a->D / 2 : (cuuint64_t)a->D;   // row elements in storage
    if (a->layout == MSA_LAYOUT_BNBD) {         // [NP, H_kv, P, D]
      dims[0] = dx; dims[1] = a->P; dims[2] = a->H_kv; dims[3] = a->NP;
      strides[0] = dx * esz; strides[1] = (cuuint64_t)a->P * dx * esz;
      strides[2] = (cuuint64_t)a->page_stride * esz;
      box[0] = bx; box[1] = 128; box[2] = 1; box[3] = 1;
    } else if (a->layout == MSA_LAYOUT_BBND) {  // [NP, P, H_kv, D]
      dims[0] = dx; dims[1] = a->H_kv; dims[2] = a->P; dims[3] = a->NP;
      strides[0] = dx * esz; strides[1] = (cuuint64_t)a->H_kv * dx * esz;
      strides[2] = (cuuint64_t)a->page_stride * esz;
      box[0] = bx; box[1] = 1; box[2] = 128; box[3] = 1;
    } else {                                    // TND [T2, H_kv, D]
      dims[0] = dx; dims[1] = a->H_kv; dims[2] = a->NP; dims[3] = 1;
      strides[0] = dx * esz; strides[1] = (cuuint64_t)a->H_kv * dx * esz;
      strides[2] = (cuuint64_t)a->NP * a->H_kv * dx * esz;
      box[0] = bx; box[1] = 1; box[2] = 128; box[3] = 1;
    }
    cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw = fp4 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : (!i8 || swizzle_int8) ? CU_TENSOR_MAP_SWIZZLE_128B
                                                          : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = encode_cached(enc, m, kdt, 4, const_cast<void*>(a->key_cache), dims, strides,
                               box, es, sw);
    if (r != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "%s tensor map: CUresult %d", what, (int)r);
    return MSA_OK;
  };
  msa_status_t st;
  if ((st = qmap(tq, p.np, "query")) != MSA_OK) return st;
  if ((st = kmap(tk, true, "key")) != MSA_OK) return st;
  if (tq_short) {
    if ((st = qmap(tq_short, p.np_short, "short query")) != MSA_OK) return st;
    if ((st = kmap(tk_short, true, "short key")) != MSA_OK) return st;
  }
  return MSA_OK;
}

// The fp16 mirror of an int8 paged key cache (query-tile requests read their
// pages from it): [NP, H_kv, P, D] fp16, compact pages; 0 when not used.
size_t mirror_bytes(const msa_index_score_args* a) {
  if (!a || a->k_dtype != MSA_I8 || a->layout == MSA_LAYOUT_TND) return 0;
  return (size_t)a->NP * (size_t)a->H_kv * (size_t)a->P * (size_t)a->D * 2;
}

// FP4 paged keys: the same 16-bit mirror, used when the call has at least one
// full query tile per request on average (T * g >= 128 * B); a decode-heavy
// call reads each page about once, and the conversion would only add traffic.
size_t fp4_mirror_bytes(const msa_index_score_args* a) {
  if (!a || a->layout == MSA_LAYOUT_TND) return 0;
  return (size_t)a->NP * (size_t)a->H_kv * (size_t)a->P * (size_t)a->D * 2;
}

bool fp4_mirror_pays(const msa_index_score_args* a) {
  const int64_t g = a->H_kv > 0 ? a->H_q / a->H_kv : 1;
  return a->T * g >= (int64_t)msa::kTileRows * a->B;
}

// One 128-token page of one kv head of the mirror: box (64 elements, 128
// tokens, 1, 1), 128-byte swizzled like a 16-bit key page.
msa_status_t make_mirror_map(const msa_index_score_args* a, void* mirror, CUtensorMap* m,
                             bool bf16 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t D = (cuuint64_t)a->D, P = (cuuint64_t)a->P;
  cuuint64_t dims[4] = {D, P, (cuuint64_t)a->H_kv, (cuuint64_t)a->NP};
  cuuint64_t strides[3] = {D * 2, P * D * 2, (cuuint64_t)a->H_kv * P * D * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = encode_cached(enc, m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                             4, mirror, dims, strides, box, es, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "key mirror tensor map: CUresult %d", (int)r);
  return MSA_OK;
}

}  // namespace

namespace msa {
void set_last_error_message(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

uint64_t current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id + 1;
}
}  // namespace msa

extern "C" {

int32_t msa_abi_version(void) { return MSA_ABI_VERSION; }

msa_status_t msa_index_score_out_shape(const msa_index_score_args* args, int64_t shape[3]) {
  // the same shape for FP4 inputs (validated by their own entry point's rules)
  msa_status_t st = validate(args, args && args->q_dtype == MSA_E2M1);
  if (st != MSA_OK) return st;
  if (!shape) return fail(MSA_ERR_INVALID_ARG, "shape is NULL");
  shape[0] = args->H_q;
  shape[1] = args->T;
  shape[2] = round16(args->MB);
  return MSA_OK;
}

msa_status_t msa_index_score_workspace_size(const msa_index_score_args* args, size_t* bytes) {
  msa_status_t st = validate(args);
  if (st != MSA_OK) return st;
  if (!bytes) return fail(MSA_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = msa::workspace_bytes_for(args->B) + mirror_bytes(args);
  return MSA_OK;
}

}  // extern "C"

namespace {

msa_status_t launch_plan_checked(const msa::Params& p, cudaStream_t s) {
  cudaError_t e = msa::launch_plan(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan kernel launch");
  return MSA_OK;
}

// mirror: the fp16 copy of the int8 key pages in the workspace, or null (the
// converter warps then convert each page per query tile).
msa_status_t launch_score_checked(const msa_index_score_args* args, const msa::Params& p,
                                  cudaStream_t s, void* mirror = nullptr) {
  // short-query requests exist only for int8 keys and when a query row group
  // fits 32 MMA columns
  const bool short_ok = args->k_dtype == MSA_I8 && p.g <= msa::kShortRows;
  CUtensorMap tq, tk, tqs, tks;
  msa_status_t st = make_maps(args, p, &tq, &tk, short_ok ? &tqs : nullptr, &tks);
  if (st != MSA_OK) return st;
  const bool i8 = args->k_dtype == MSA_I8;
  const bool bf16 = args->q_dtype == MSA_BF16;
  // a host bound that puts every request in the short class: no tile launch
  // (the plan flags any request longer than the bound)
  const bool short_only =
      short_ok && args->max_seqlen_q > 0 && (int64_t)args->max_seqlen_q * p.g <= msa::kShortRows;
  cudaError_t e = cudaSuccess;
  if (!short_only) {
    if (i8 && mirror) {
      CUtensorMap tm;
      if ((st = make_mirror_map(args, mirror, &tm)) != MSA_OK) return st;
      e = msa::launch_i8_mirror(p, args->key_cache, args->page_stride, mirror, s);
      if (e == cudaSuccess) e = msa::launch_score_i8_mirror(&tq, &tm, p, s);
    } else if (i8)
      e = msa::launch_score_i8(&tq, &tk, p, s);
    else if (is_f8(args->q_dtype))
      e = msa::launch_score_f8(&tq, &tk, p, args->q_dtype == MSA_E5M2, s);
    else
      e = msa::launch_score_16(&tq, &tk, p, bf16, s);
  }
  if (e == cudaSuccess && short_ok) e = msa::launch_short_i8(&tqs, &tks, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "score kernel launch");
  return MSA_OK;
}

// The mirror's place in a workspace of `bytes` (after the plan), or null if
// it is not used or does not fit.
void* mirror_in(const msa_index_score_args* args, void* ws, size_t bytes) {
  const size_t m = mirror_bytes(args), plan = msa::workspace_bytes_for(args->B);
  if (!m || !ws || bytes < plan + m) return nullptr;
  return static_cast<uint8_t*>(ws) + plan;
}

// Shared front half of the entry points: validation, empty-call shortcut,
// workspace and output checks, kernel parameters.
msa_status_t prepare(const msa_index_score_args* args, float* out, bool need_out, void* ws,
                     size_t ws_bytes, msa::Params& p, bool& empty) {
  g_msg[0] = 0;
  msa_status_t st = validate(args);
  if (st != MSA_OK) return st;
  empty = args->T == 0 || args->B == 0;
  if (empty) return MSA_OK;
  if ((st = check_ws(args, ws, ws_bytes)) != MSA_OK) return st;
  if (need_out && (!out || !aligned(out, 16)))
    return fail(MSA_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
  return fill_params(args, out, ws, p);
}

}  // namespace

extern "C" {

msa_status_t msa_index_score_plan(const msa_index_score_args* args, void* workspace,
                                  size_t workspace_bytes, msa_stream_t stream) {
  msa::Params p;
  bool empty = false;
  msa_status_t st = prepare(args, nullptr, false, workspace, workspace_bytes, p, empty);
  if (st != MSA_OK || empty) return st;
  return launch_plan_checked(p, reinterpret_cast<cudaStream_t>(stream));
}

msa_status_t msa_index_score_run(const msa_index_score_args* args, float* out, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream) {
  msa::Params p;
  bool empty = false;
  msa_status_t st = prepare(args, out, true, workspace, workspace_bytes, p, empty);
  if (st != MSA_OK || empty) return st;
  return launch_score_checked(args, p, reinterpret_cast<cudaStream_t>(stream),
                              mirror_in(args, workspace, workspace_bytes));
}

msa_status_t msa_index_score(const msa_index_score_args* args, float* out, void* workspace,
                             size_t workspace_bytes, msa_stream_t stream) {
  msa::Params p;
  bool empty = false;
  msa_status_t st = prepare(args, out, true, workspace, workspace_bytes, p, empty);
  if (st != MSA_OK || empty) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_plan_checked(p, s)) != MSA_OK) return st;
  return launch_score_checked(args, p, s, mirror_in(args, workspace, workspace_bytes));
}

msa_status_t msa_index_score_topk_workspace_size(const msa_index_score_args* args, int32_t k,
                                                 size_t* bytes) {
  msa_status_t st = validate(args);
  if (st != MSA_OK) return st;
  if ((st = validate_select(args, k)) != MSA_OK) return st;
  if (!bytes) return fail(MSA_ERR_INVALID_ARG, "bytes is NULL");
  const SelectPlan sp = select_plan(args, k);
  const size_t mb = mirror_bytes(args);
  *bytes = mb ? (sp.plan_bytes + sp.cand_bytes + 255) / 256 * 256 + mb : sp.plan_bytes + sp.cand_bytes;
  return MSA_OK;
}

msa_status_t msa_index_score_topk(const msa_index_score_args* args, int32_t k, int32_t local_slot,
                                  float* out, int32_t* indices, void* workspace,
                                  size_t workspace_bytes, msa_stream_t stream) {
  g_msg[0] = 0;
  msa_status_t st = validate(args);
  if (st != MSA_OK) return st;
  if ((st = validate_select(args, k)) != MSA_OK) return st;
  if (args->T == 0 || args->B == 0) return MSA_OK;
  if (!indices || !aligned(indices, 4)) return fail(MSA_ERR_INVALID_ARG, "indices must be a 4-byte aligned pointer");
  if (out && !aligned(out, 16)) return fail(MSA_ERR_INVALID_ARG, "out must be 16-byte aligned (or NULL)");
  const SelectPlan sp = select_plan(args, k);
  if (!workspace) return fail(MSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(MSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < sp.plan_bytes + sp.cand_bytes)
    return fail(MSA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", sp.plan_bytes + sp.cand_bytes,
                workspace_bytes);
  msa::Params p;
  if ((st = fill_params(args, out, workspace, p)) != MSA_OK) return st;
  p.topk_k = k;
  p.cand = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + sp.plan_bytes);
  p.cand_parts = sp.parts;
  p.chunk_min[0] = sp.chunk_min[0];
  p.chunk_min[1] = sp.chunk_min[1];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the fp16 mirror of int8 key pages after the candidate lists (256-byte
  // aligned), if it fits
  const size_t mb = mirror_bytes(args);
  const size_t moff = (sp.plan_bytes + sp.cand_bytes + 255) / 256 * 256;
  void* mirror = mb && workspace_bytes >= moff + mb ? static_cast<uint8_t*>(workspace) + moff : nullptr;
  if ((st = launch_plan_checked(p, s)) != MSA_OK) return st;
  if ((st = launch_score_checked(args, p, s, mirror)) != MSA_OK) return st;
  cudaError_t e = msa::launch_group_select(p, local_slot ? 1 : 0, indices, s);
  if (e != cudaSuccess) return cuda_fail(e, "selection kernel launch");
  return MSA_OK;
}

size_t fp4_query_bytes(const msa_index_score_args* a) {
  return ((size_t)a->T * a->H_q * a->D * 2 + 255) / 256 * 256;
}

msa_status_t msa_index_score_fp4_workspace_size(const msa_index_score_args* args, int32_t format,
                                                size_t* bytes) {
  msa_status_t st = validate(args, true);
  if (st != MSA_OK) return st;
  if (format != MSA_FP4_MX && format != MSA_FP4_NV)
    return fail(MSA_ERR_INVALID_ARG, "format must be MSA_FP4_MX or MSA_FP4_NV");
  if (!bytes) return fail(MSA_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = msa::workspace_bytes_for(args->B) + fp4_query_bytes(args) +
           (fp4_mirror_pays(args) ? fp4_mirror_bytes(args) : 0);
  return MSA_OK;
}

}  // extern "C"

namespace {

// Shared checks and parameters of the FP4 entry points.
msa_status_t prepare_fp4(const msa_index_score_args* args, int32_t format, const uint8_t* q_scale,
                         const uint8_t* k_scale, float* out, bool need_out, void* workspace,
                         size_t workspace_bytes, msa::Params& p, bool& empty, void** q16) {
  g_msg[0] = 0;
  msa_status_t st = validate(args, true);
  if (st != MSA_OK) return st;
  if (format != MSA_FP4_MX && format != MSA_FP4_NV)
    return fail(MSA_ERR_INVALID_ARG, "format must be MSA_FP4_MX or MSA_FP4_NV");
  empty = args->T == 0 || args->B == 0;
  if (empty) return MSA_OK;
  if (q_scale && !aligned(q_scale, 16)) return fail(MSA_ERR_INVALID_ARG, "q_scale must be 16-byte aligned");
  if (k_scale && !aligned(k_scale, 16)) return fail(MSA_ERR_INVALID_ARG, "k_scale must be 16-byte aligned");
  if (need_out && (!out || !aligned(out, 16)))
    return fail(MSA_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
  const size_t plan_bytes = msa::workspace_bytes_for(args->B);
  if (!workspace) return fail(MSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(MSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan_bytes + fp4_query_bytes(args))
    return fail(MSA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu",
                plan_bytes + fp4_query_bytes(args), workspace_bytes);
  if ((st = fill_params(args, out, workspace, p)) != MSA_OK) return st;
  p.k_scale8 = k_scale;
  p.fp4_ng = args->D / (format == MSA_FP4_NV ? 16 : 32);
  *q16 = static_cast<uint8_t*>(workspace) + plan_bytes;
  return MSA_OK;
}

}  // namespace

extern "C" {

msa_status_t msa_index_score_fp4_plan(const msa_index_score_args* args, int32_t format,
                                      const uint8_t* q_scale, void* workspace,
                                      size_t workspace_bytes, msa_stream_t stream) {
  msa::Params p;
  bool empty = false;
  void* q16 = nullptr;
  msa_status_t st = prepare_fp4(args, format, q_scale, nullptr, nullptr, false, workspace,
                                workspace_bytes, p, empty, &q16);
  if (st != MSA_OK || empty) return st;
  if (!q_scale) return fail(MSA_ERR_INVALID_ARG, "q_scale is required");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = msa::launch_fp4_dequant_query(static_cast<const uint8_t*>(args->query), q_scale,
                                                args->T * (int64_t)args->H_q,
                                                format == MSA_FP4_NV, q16, s);
  if (e != cudaSuccess) return cuda_fail(e, "FP4 query dequantisation launch");
  return launch_plan_checked(p, s);
}

msa_status_t msa_index_score_fp4_run(const msa_index_score_args* args, int32_t format,
                                     const uint8_t* k_scale, float* out, void* workspace,
                                     size_t workspace_bytes, msa_stream_t stream) {
  msa::Params p;
  bool empty = false;
  void* q16 = nullptr;
  msa_status_t st = prepare_fp4(args, format, nullptr, k_scale, out, true, workspace,
                                workspace_bytes, p, empty, &q16);
  if (st != MSA_OK || empty) return st;
  if (!k_scale) return fail(MSA_ERR_INVALID_ARG, "k_scale is required");
  const bool nv = format == MSA_FP4_NV;
  // short-query requests (Lq * g <= 32 query rows) go to the short-query
  // kernel, the others to the tile kernel; a host length bound that puts
  // every request in the short class leaves the tile launch out
  const bool short_ok = p.g <= msa::kShortRows;
  const bool short_only =
      short_ok && args->max_seqlen_q > 0 && (int64_t)args->max_seqlen_q * p.g <= msa::kShortRows;
  CUtensorMap tq, tk, tqs, tks;
  if ((st = make_maps(args, p, &tq, &tk, short_ok ? &tqs : nullptr, &tks, q16, nv)) != MSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // prefill-heavy calls on paged keys: dequantise the query-tile requests'
  // pages once into the 16-bit mirror after the query, then the 16-bit tile
  // kernel (BNBD order)
  const size_t mb = fp4_mirror_pays(args) ? fp4_mirror_bytes(args) : 0;
  const size_t moff = msa::workspace_bytes_for(args->B) + fp4_query_bytes(args);
  cudaError_t e = cudaSuccess;
  if (short_only) {
    // no query-tile request
  } else if (mb && workspace_bytes >= moff + mb) {
    void* mirror = static_cast<uint8_t*>(workspace) + moff;
    CUtensorMap tm;
    if ((st = make_mirror_map(args, mirror, &tm, !nv)) != MSA_OK) return st;
    e = msa::launch_fp4_mirror(p, args->key_cache, args->page_stride, nv, mirror, s);
    msa::Params pm = p;
    pm.layout = 1;   // the mirror's order; the table and kv_len are read as before
    if (e == cudaSuccess) e = msa::launch_score_16(&tq, &tm, pm, !nv, s);
  } else {
    e = msa::launch_score_fp4(&tq, &tk, p, nv, s);
  }
  if (e == cudaSuccess && short_ok) e = msa::launch_short_fp4(&tqs, &tks, p, nv, s);
  if (e != cudaSuccess) return cuda_fail(e, "score kernel launch");
  return MSA_OK;
}

msa_status_t msa_index_score_fp4(const msa_index_score_args* args, int32_t format,
                                 const uint8_t* q_scale, const uint8_t* k_scale, float* out,
                                 void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  g_msg[0] = 0;
  if (args && args->T > 0 && args->B > 0 && (!q_scale || !k_scale))
    return fail(MSA_ERR_INVALID_ARG, "q_scale and k_scale are required");
  if (args && args->T > 0 && args->B > 0 && (!out || !aligned(out, 16)))
    return fail(MSA_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
  msa_status_t st = msa_index_score_fp4_plan(args, format, q_scale, workspace, workspace_bytes, stream);
  if (st != MSA_OK) return st;
  return msa_index_score_fp4_run(args, format, k_scale, out, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Workspace of a sparse-attention call, each array 256-byte aligned.
struct SparseLayout {
  size_t header, cnt, row_ptr, cursor, unit_ptr, qrec, units, o_part, lse_part, bytes;
  int64_t rows, entries;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

SparseLayout sparse_layout(const msa_index_score_args* a, int k) {
  SparseLayout l;
  l.rows = (int64_t)a->H_kv * a->B * a->MB;
  l.entries = a->T * (int64_t)a->H_kv * k;
  size_t off = 0;
  l.header = off;   off += 256;
  l.cnt = off;      off += up256(4 * (size_t)l.rows);
  l.row_ptr = off;  off += up256(4 * (size_t)(l.rows + 1));
  l.cursor = off;   off += up256(4 * (size_t)l.rows);
  l.unit_ptr = off; off += up256(4 * (size_t)(l.rows + 1));
  l.qrec = off;     off += up256(8 * (size_t)l.entries);
  l.units = off;    off += up256(16 * (size_t)l.entries);
  l.o_part = off;   off += up256(2 * (size_t)a->T * a->H_q * k * a->D);   // 16-bit partials
  l.lse_part = off; off += up256(4 * (size_t)a->T * a->H_q * k);
  l.bytes = off;
  return l;
}

msa_status_t validate_sparse(const msa_index_score_args* a, const msa_sparse_attention_args* sa) {
  msa_status_t st = validate(a);
  if (st != MSA_OK) return st;
  if (!sa) return fail(MSA_ERR_INVALID_ARG, "sparse attention args are NULL");
  if (a->q_dtype != MSA_F16 && a->q_dtype != MSA_BF16)
    return fail(MSA_ERR_INVALID_ARG, "sparse attention takes fp16 or bf16 query, keys and values");
  if (sa->k < 1 || sa->k > 32) return fail(MSA_ERR_INVALID_ARG, "k must be in [1, 32]");
  // a unit descriptor keeps the kv head in 15 bits
  if (a->H_kv > 32767) return fail(MSA_ERR_UNSUPPORTED, "sparse attention takes H_kv <= 32767");
  // an entry record keeps token * 32 + slot in 32 bits
  if (a->T >= (1ll << 27)) return fail(MSA_ERR_UNSUPPORTED, "sparse attention takes T < 2^27");
  if (!(sa->sm_scale >= 0.f)) return fail(MSA_ERR_INVALID_ARG, "sm_scale must be >= 0 (0: 1/sqrt(D))");
  if (a->T > 0 && a->B > 0) {
    if (!sa->value_cache || !sa->selection)
      return fail(MSA_ERR_INVALID_ARG, "value_cache and selection are required");
    if (!aligned(sa->value_cache, 16)) return fail(MSA_ERR_INVALID_ARG, "value_cache must be 16-byte aligned");
    if (!aligned(sa->selection, 4)) return fail(MSA_ERR_INVALID_ARG, "selection must be 4-byte aligned");
  }
  return MSA_OK;
}

}  // namespace

extern "C" {

msa_status_t msa_sparse_attention_workspace_size(const msa_index_score_args* args,
                                                 const msa_sparse_attention_args* sa,
                                                 size_t* bytes) {
  msa_status_t st = validate_sparse(args, sa);
  if (st != MSA_OK) return st;
  if (!bytes) return fail(MSA_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = sparse_layout(args, sa->k).bytes;
  return MSA_OK;
}

msa_status_t msa_sparse_attention(const msa_index_score_args* args,
                                  const msa_sparse_attention_args* sa, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  g_msg[0] = 0;
  msa_status_t st = validate_sparse(args, sa);
  if (st != MSA_OK) return st;
  if (args->T == 0 || args->B == 0) return MSA_OK;
  if (!out || !aligned(out, 16)) return fail(MSA_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
  if (lse && !aligned(lse, 4)) return fail(MSA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const SparseLayout lo = sparse_layout(args, sa->k);
  if (!workspace) return fail(MSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(MSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < lo.bytes)
    return fail(MSA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", lo.bytes, workspace_bytes);
  if (lo.entries > 0x7fffffffLL) return fail(MSA_ERR_UNSUPPORTED, "T * H_kv * k too large");
  msa::SparseParams sp;
  if ((st = fill_params(args, nullptr, workspace, sp.p)) != MSA_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  sp.query = args->query;
  sp.sel = sa->selection;
  sp.k = sa->k;
  sp.qpu = msa::kTileRows / sp.p.g;
  sp.sm_scale = sa->sm_scale > 0.f ? sa->sm_scale : 1.0f / sqrtf((float)args->D);
  sp.pad_ = 0;
  sp.rows = lo.rows;
  sp.cnt = reinterpret_cast<int32_t*>(w + lo.cnt);
  sp.row_ptr = reinterpret_cast<int32_t*>(w + lo.row_ptr);
  sp.cursor = reinterpret_cast<int32_t*>(w + lo.cursor);
  sp.unit_ptr = reinterpret_cast<int32_t*>(w + lo.unit_ptr);
  sp.qrec = reinterpret_cast<int2*>(w + lo.qrec);
  sp.units = reinterpret_cast<int4*>(w + lo.units);
  sp.o_part = reinterpret_cast<uint16_t*>(w + lo.o_part);
  sp.lse_part = reinterpret_cast<float*>(w + lo.lse_part);
  // K and V pages through the key cache's tensor-map recipe; the query maps
  // with a run of one position (a box is one query entry's g heads) and of
  // 128 / g positions (a unit of consecutive query tokens in two boxes)
  CUtensorMap tq, tk, tv, tq_unused, tqr;
  msa::Params p1 = sp.p;
  p1.np = 1;
  if ((st = make_maps(args, p1, &tq, &tk, nullptr, nullptr)) != MSA_OK) return st;
  if ((st = make_maps(args, sp.p, &tqr, &tq_unused, nullptr, nullptr)) != MSA_OK) return st;
  msa_index_score_args va = *args;
  va.key_cache = sa->value_cache;
  if ((st = make_maps(&va, p1, &tq_unused, &tv, nullptr, nullptr)) != MSA_OK) return st;
  cudaError_t e = msa::launch_sparse_attention(&tq, &tk, &tv, &tqr, sp, args->q_dtype == MSA_BF16, out, lse,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention launch");
  return MSA_OK;
}

msa_status_t msa_block_topk(const float* score, int32_t H, int64_t T, int32_t MBp, int32_t MB,
                            int32_t k, int32_t* out, msa_stream_t stream) {
  if (H < 0 || T < 0 || MBp < 0 || MB < 0) return fail(MSA_ERR_INVALID_ARG, "sizes must be >= 0");
  if (MB > MBp) return fail(MSA_ERR_INVALID_ARG, "MB must be <= MBp");
  if (k < 1 || k > 32) return fail(MSA_ERR_INVALID_ARG, "k must be in [1, 32]");
  if ((int64_t)H * T == 0) return MSA_OK;
  if (!out || (!score && MB > 0)) return fail(MSA_ERR_INVALID_ARG, "score and out are required");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = msa::launch_topk(score, H, T, MBp, MB, k, out, sm_count(dev), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-k kernel launch");
  return MSA_OK;
}

msa_status_t msa_get_device_error(const void* workspace, int32_t* bits, msa_stream_t stream) {
  if (!workspace || !bits) return fail(MSA_ERR_INVALID_ARG, "workspace and bits are required");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  const auto* hdr = static_cast<const msa::PlanHeader*>(workspace);
  cudaError_t e = cudaMemcpyAsync(&v, &hdr->err, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *bits = v;
  return MSA_OK;
}

const char* msa_status_string(msa_status_t st) {
  switch (st) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_DEVICE_DATA: return "bad device data";
    case MSA_ERR_WORKSPACE: return "bad workspace";
  }
  return "unknown status";
}

const char* msa_last_error_message(void) { return g_msg; }

msa_status_t msa_set_watchdog(uint64_t wait_limit_ns, int32_t stall) {
  g_wait_limit_ns.store(wait_limit_ns, std::memory_order_relaxed);
  g_wait_stall.store(stall ? 1 : 0, std::memory_order_relaxed);
  return MSA_OK;
}

}  // extern "C"
