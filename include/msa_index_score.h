/*
 * msa_index_score -- MSA (MiniMax Sparse Attention) index-branch block score
 * on NVIDIA GB300 (sm_103a).  C ABI.
 *
 * Operation (feature request "MsaIndexScore",
 * gitcode.com/cann/ops-transformer/issues/4117, section "calculation"):
 *
 *   for token t of request b, head h, logical KV block beta:
 *     score[h, t, beta] = max over visible j in [beta*P, beta*P + P) of
 *                         < query[t, h, :], k~[j, h / g, :] >,   g = H_q / H_kv
 *
 *   k~ is read from the paged cache through block_table (BBND / BNBD) or from
 *   the packed keys (TND).  int8 keys are dequantised by a per-(page, head,
 *   token) fp32 scale applied to the dot product before the mask
 *   (order DOT -> DEQUANT -> MASK -> MAX).  A key j is visible to token t
 *   when j < kv_len[b] and, for sparse_mode 3 (rightDownCausal),
 *   j <= kv_len[b] - Lq[b] + (t - cu_seqlens_q[b]).  sparse_mode 0 has no
 *   causal bound.  A block with no visible key gets -inf.
 *
 *   Local mask (torch API guide "CANN ops-transformer ... msa_index_score",
 *   sec. 2), applied after the max to every row of a request with
 *   kv_len > 0: blocks [0, init_blocks) get 1e30f; blocks
 *   [max(0, start_loc+1-local_blocks), start_loc] get 1e29f (overriding the
 *   init value).  Both clipped to [0, MB).
 *
 *   Output (same guide, sec. 5): fp32 [H_q, T, RoundUp(MB, 16)], row-major.
 *   Columns [MB, RoundUp(MB,16)) hold -inf.  Every element is written, so the
 *   caller need not initialise it.
 *
 * All pointers in msa_index_score_args are DEVICE pointers owned by the
 * caller, except where marked.  Calls are asynchronous on `stream`; the
 * library never synchronises the host inside a compute call and never
 * allocates device memory.  Scratch state lives in a caller-provided
 * workspace (size from msa_index_score_workspace_size, two-phase like the
 * reference op's aclnn interface).  Two calls that share a workspace must be
 * ordered (same stream, or joined by events).
 *
 * Scope of this library: D == 128 and P == 128; g = H_q / H_kv <= 128.
 */
#ifndef MSA_INDEX_SCORE_H_
#define MSA_INDEX_SCORE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_ABI_VERSION 3

/* Same object as cudaStream_t / CUstream (NULL = legacy default stream). */
typedef struct CUstream_st *msa_stream_t;

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1,   /* argument violates the op's rules (layout, dtype, shapes) */
    MSA_ERR_UNSUPPORTED = 2,   /* legal for the op, outside this library (D != 128, P != 128, g > 128) */
    MSA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed; see msa_last_error_message() */
    MSA_ERR_DEVICE_DATA = 4,   /* device-side data check failed; see msa_get_device_error() */
    MSA_ERR_WORKSPACE = 5      /* workspace NULL, too small or misaligned */
} msa_status_t;

typedef enum { MSA_LAYOUT_BBND = 0, MSA_LAYOUT_BNBD = 1, MSA_LAYOUT_TND = 2 } msa_layout_t;
/* Element types.  Query: fp16, bf16, FP8 E4M3 (e4m3fn: finite only) or FP8
 * E5M2.  Key: the query's type, or int8 with an fp16 query and a scale.  FP8
 * query and key must be of the same FP8 type and take no scale (torch API
 * guide "CANN ops-transformer ... msa_index_score", sec. 4 and 7.2; on this
 * GPU they run on tcgen05 kind::f8f6f4 with fp32 accumulation). */
typedef enum { MSA_F16 = 0, MSA_BF16 = 1, MSA_I8 = 2, MSA_E4M3 = 3, MSA_E5M2 = 4,
               MSA_E2M1 = 5 /* FP4, two codes per byte: msa_index_score_fp4 only */ } msa_dtype_t;

/* FP4 group-scale formats (MiniMax Sparse Attention notes, sec. 8.2, "FP4
 * Indexer"): MXFP4 = E2M1 values with one E8M0 scale byte per 32 elements;
 * NVFP4 = E2M1 values with one E4M3 scale byte per 16 elements. */
typedef enum { MSA_FP4_MX = 0, MSA_FP4_NV = 1 } msa_fp4_format_t;

/* Bits of the device error word (msa_get_device_error). */
#define MSA_DEVERR_CU_Q        0x01  /* cu_seqlens_q[0] != 0, decreasing, cu_seqlens_q[B] != T, or a query length above a nonzero max_seqlen_q */
#define MSA_DEVERR_KV_LEN      0x02  /* kv_len < 0, or ceil(kv_len/P) > MB */
#define MSA_DEVERR_CU_K        0x04  /* TND: cu_seqlens_k[0] != 0, decreasing, or beyond T2 */
#define MSA_DEVERR_BLOCK_TABLE 0x08  /* a block_table entry that is read lies outside [0, NP) */
#define MSA_DEVERR_TIMEOUT     0x10  /* an on-chip pipeline wait ran past its limit (kernel returned early) */
#define MSA_DEVERR_SELECTION   0x20  /* sparse attention: a selection entry >= MB, repeated, or not ascending */

typedef struct {
    /* query: [T, H_q, D] contiguous ("TND" query of the guide, sec. 4); fp16, bf16 or
     * FP8 (see msa_dtype_t); E2M1 codes only through msa_index_score_fp4. */
    const void *query;
    msa_dtype_t q_dtype;
    int64_t T;                  /* total query tokens = cu_seqlens_q[B] */
    int32_t H_q;
    int32_t D;                  /* head dim; 128 */

    /* key cache (guide sec. 4, 6, 8.1):
     *   BBND [NP, P, H_kv, D], BNBD [NP, H_kv, P, D]: dim0 may be strided
     *        (page_stride elements, >= the compact page size, multiple of 16 bytes);
     *        the inner three dims are compact.
     *   TND  [T2, H_kv, D] contiguous; page_stride must equal H_kv*D.
     * dtype: same as query, or int8 with fp16 query (then scale is required). */
    const void *key_cache;
    msa_dtype_t k_dtype;
    msa_layout_t layout;
    int64_t NP;                 /* number of pages (paged) or T2 key rows (TND) */
    int32_t P;                  /* block_size = tokens per page; 128 */
    int32_t H_kv;
    int64_t page_stride;        /* elements between consecutive dim0 entries of key_cache */

    /* block_table [B, MB] int32, logical block -> physical page (paged only; NULL for TND).
     * Entries at or beyond ceil(kv_len/P) are never read.  For TND, MB is the
     * caller's max over requests of ceil(kv_len/P), at least 1 (guide sec. 8.5). */
    const int32_t *block_table;
    int32_t B;
    int32_t MB;

    const int32_t *cu_seqlens_q;   /* [B+1] prefix sums of query lengths, cu[0] == 0 */
    const int32_t *kv_len;         /* [B] visible KV length (paged); NULL for TND */
    const int32_t *cu_seqlens_k;   /* [B+1] prefix sums of key lengths (TND); NULL for paged */
    const int32_t *start_loc;      /* [B] logical block index of the current query (local mask only) */
    const float *scale;            /* int8 only: paged [NP, H_kv, P], TND [T2, H_kv]; else NULL */

    int32_t sparse_mode;           /* 0 = no causal mask, 3 = rightDownCausal (default 3) */
    int32_t init_blocks;           /* default 0, <= MB */
    int32_t local_blocks;          /* default 1, <= MB */

    /* Optional host-side upper bound on every request's query length (0 = not
     * known).  An addition of this library, not an argument of the op in the
     * pages: like the max_seqlen_q of varlen attention calls, it lets the host
     * skip the query-tile kernel when every request is a short int8 request
     * (max_seqlen_q * H_q / H_kv <= 32).  A request longer than a nonzero bound
     * is reported as MSA_DEVERR_CU_Q; its scores are then not written. */
    int32_t max_seqlen_q;
} msa_index_score_args;

/* Library ABI version (MSA_ABI_VERSION of the build). */
int32_t msa_abi_version(void);

/* Output shape {H_q, T, RoundUp(MB, 16)} (guide sec. 5, 8.5).  Host-only, validates args. */
msa_status_t msa_index_score_out_shape(const msa_index_score_args *args, int64_t shape[3]);

/* Bytes of device workspace one call needs (>= 256, grows with B).  Host-only.
 * With int8 keys in a paged layout it also holds an fp16 copy of the key pages
 * [NP, H_kv, P, D] (NP * H_kv * P * D * 2 bytes): the pages of requests scored
 * by query tiles are converted into it once per call instead of once per tile
 * (every int8 value is exact in fp16; the scale is applied to the dot products
 * as before).  A workspace of only the plan's size (the value for 16-bit keys
 * with the same B) is also accepted; those pages are then converted per tile. */
msa_status_t msa_index_score_workspace_size(const msa_index_score_args *args, size_t *bytes);

/*
 * Compute the block scores into `out` (device, fp32 [H_q, T, RoundUp(MB,16)],
 * 16-byte aligned).  `workspace` is device memory of at least
 * msa_index_score_workspace_size() bytes, 256-byte aligned, owned by the
 * caller; it need not be initialised.  Equivalent to msa_index_score_plan
 * followed by msa_index_score_run on the same stream.
 *
 * Errors: argument problems return before anything is enqueued.  Bad values
 * inside the device arrays (cu_seqlens, kv_len, block_table) are detected on
 * the device, recorded in the workspace's error word and do not fault; read
 * them with msa_get_device_error.  T == 0 or B == 0 enqueues nothing.
 */
msa_status_t msa_index_score(const msa_index_score_args *args, float *out, void *workspace,
                             size_t workspace_bytes, msa_stream_t stream);

/* First half of msa_index_score: one small kernel that validates the
 * per-request arrays and writes the work plan (request order, unit counts,
 * cleared work counter and error word) into `workspace`. */
msa_status_t msa_index_score_plan(const msa_index_score_args *args, void *workspace,
                                  size_t workspace_bytes, msa_stream_t stream);

/* Second half: the persistent tensor-core kernel that consumes the plan in
 * `workspace` and writes every element of `out`.  `args` must be the ones
 * given to the plan call. */
msa_status_t msa_index_score_run(const msa_index_score_args *args, float *out, void *workspace,
                                 size_t workspace_bytes, msa_stream_t stream);

/*
 * Allocation-free variant of msa_index_score, for callers that cannot
 * allocate device memory (a serving loop that forbids allocator calls after
 * start-up, or a host program without a device allocator of its own).  The
 * pages define no such call: this entry point has no counterpart there.
 *
 * Same arguments and results as msa_index_score, without the workspace: the
 * plan scratch is a fixed array inside the library (MSA_NOALLOC_WORKSPACE_BYTES
 * bytes on every GPU that loads the library, held until the process exits).
 * It handles at most MSA_NOALLOC_MAX_BATCH requests; a larger B returns
 * MSA_ERR_WORKSPACE and enqueues nothing.  No device memory is allocated or
 * freed.
 *
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and caches it; make that
 *   first call before any stream capture on that device.
 *   The cache is keyed by the CUDA context as well: after a device reset,
 *   or when another context is current on that device, the next call looks
 *   the address up again (again outside any stream capture).
 * - Every call uses the same array and leaves its contents behind; each call
 *   clears the parts that must start at zero (work counter, error word) itself.
 * - Calls whose kernels overlap on the GPU (different streams, or several
 *   host threads) race on the array: order them, e.g. on one stream.
 * - The device error word of these calls lives in the library's array; read
 *   it with msa_noalloc_device_error.
 */
#define MSA_NOALLOC_MAX_BATCH 1024
#define MSA_NOALLOC_WORKSPACE_BYTES 41216
msa_status_t msa_index_score_noalloc(const msa_index_score_args *args, float *out,
                                     msa_stream_t stream);

/* Synchronise `stream` and read the device error word that the last
 * msa_index_score_noalloc call on the current device left in the library's
 * array (MSA_DEVERR_* bits; 0 = clean).  Allocates nothing.  Returns MSA_OK,
 * MSA_ERR_INVALID_ARG for a NULL `bits`, or MSA_ERR_CUDA if the copy fails. */
msa_status_t msa_noalloc_device_error(int32_t *bits, msa_stream_t stream);

/*
 * Block top-k selection, the consumer of the block scores (MiniMax Sparse
 * Attention notes, section 4.7: Equation (7) I_i = TopK_b(M_i, k) over a
 * query's block scores, and the selector contract quoted there and in
 * section 5.3).
 *
 *   score  device, fp32 [H, T, MBp] row-major: msa_index_score's output (or
 *          any score tensor of that layout); read only.
 *   MB     valid columns of a row (0 <= MB <= MBp); columns [MB, MBp) are
 *          never selected.
 *   k      blocks per row, 1 <= k <= 32 (the pages' selector fixes 16).
 *   out    device, int32 [T, H, k] row-major, written completely: for row
 *          (h, t), out[t, h, :] lists the k blocks with the highest score in
 *          ascending block-index order (not score order), followed by -1
 *          when fewer than k blocks are valid.
 *
 * A block is valid when its score is above -inf (-inf marks a block with no
 * visible key; a NaN score is never selected).  Equal scores rank the smaller
 * block index first.  The local mask's forced blocks (1e30 / 1e29) therefore
 * always make the selection when k covers them.  When H_q > H_kv the
 * selection is per index head; one selection per GQA group (section 4.3,
 * Equation (3)) is what msa_index_score_topk computes, fused into the scores.
 *
 * Asynchronous on `stream`; no workspace, no allocation.  Returns
 * MSA_ERR_INVALID_ARG for null pointers with work to do, negative sizes,
 * MB > MBp or k outside [1, 32]; MSA_ERR_CUDA if the launch fails.
 */
msa_status_t msa_block_topk(const float *score, int32_t H, int64_t T, int32_t MBp, int32_t MB,
                            int32_t k, int32_t *out, msa_stream_t stream);

/*
 * Block scores with the per-GQA-group block selection fused into the score
 * kernels (MiniMax Sparse Attention notes, section 4.3 Equation (3): the
 * heads of a GQA group share one index set; section 4.7 Equation (7) and the
 * selector contract: top-k blocks, indices ascending, -1 tail; section 10,
 * checklist items 7-9).  The scores are computed exactly as by
 * msa_index_score; the selection never reads them back from memory.
 *
 *   k           blocks per selection, 1 <= k <= 16 (the pages' selector fixes 16).
 *   local_slot  nonzero: each query token's own block -- the block holding its
 *               position kv_len - Lq + i under the rightDownCausal alignment,
 *               when 0 <= that position < kv_len -- always takes one of the k
 *               slots; the other k - 1 go to the best remaining blocks.  Zero:
 *               the plain top-k of the group score.
 *   out         device fp32 [H_q, T, RoundUp(MB, 16)] for the scores, or NULL
 *               to compute the selection without storing the scores.
 *   indices     device int32 [T, H_kv, k], written completely: for token t
 *               and group r (the query heads r*g .. r*g+g-1, g = H_q / H_kv),
 *               the selected blocks in ascending order, then -1.
 *   workspace   device memory of msa_index_score_topk_workspace_size() bytes
 *               (256-byte aligned, caller-owned, need not be initialised): the
 *               plan and each row's partial selections (at most 64 MiB of them).
 *
 * The group score of block beta is the maximum over the group's g index heads
 * of score[h, t, beta]; a block is a candidate when beta < MB and that score
 * is above -inf.  Equal group scores rank the smaller block first.  Forced
 * blocks of the local mask (1e30 / 1e29) outrank every dot product.
 *
 * Errors: as msa_index_score, plus MSA_ERR_INVALID_ARG for k outside [1, 16]
 * or a NULL `indices`, and MSA_ERR_UNSUPPORTED when g = H_q / H_kv does not
 * divide 32 (the heads of a position are combined inside one warp).
 * Asynchronous on `stream`; T == 0 or B == 0 enqueues nothing.
 */
msa_status_t msa_index_score_topk_workspace_size(const msa_index_score_args *args, int32_t k,
                                                 size_t *bytes);
msa_status_t msa_index_score_topk(const msa_index_score_args *args, int32_t k, int32_t local_slot,
                                  float *out, int32_t *indices, void *workspace,
                                  size_t workspace_bytes, msa_stream_t stream);

/*
 * Block scores of an FP4 index branch (the block-scaled FP4 indexer of the
 * MiniMax Sparse Attention notes, sec. 8.2: E2M1 values with group scales,
 * fp32 block scores; its results approximate the real-valued index score, so
 * top-k orders need not match a 16-bit indexer's).  Computes exactly what
 * msa_index_score computes, on the dequantised values
 *     q~[t, h, d] = e2m1(q) * scale(q_scale[t, h, d / G])
 *     k~[j, hk, d] = e2m1(k) * scale(k_scale[.., d / G])   (G = 32 MX, 16 NV)
 * with fp32 accumulation (every dequantised value is exact in the 16-bit
 * operand type: fp16 for NVFP4, bf16 for MXFP4 with E8M0 codes 2 .. 252).
 *
 *   args      q_dtype = k_dtype = MSA_E2M1, args->scale = NULL.  query
 *             [T, H_q, D/2] bytes; key_cache BBND [NP, P, H_kv, D/2], BNBD
 *             [NP, H_kv, P, D/2] (page_stride in bytes) or TND [T2, H_kv, D/2];
 *             element 2i of a row is the low nibble of byte i.  D = 128.
 *   format    MSA_FP4_MX or MSA_FP4_NV.
 *   q_scale   device bytes [T, H_q, D/G], 16-byte aligned.
 *   k_scale   device bytes in logical page order: paged [NP, H_kv, P, D/G]
 *             (compact, even when key_cache has a page stride), TND
 *             [T2, H_kv, D/G]; 16-byte aligned.
 *   out       as msa_index_score.
 *   workspace msa_index_score_fp4_workspace_size() bytes (256-byte aligned,
 *             caller-owned): the plan and the dequantised query, and for a
 *             prefill-heavy call on paged keys (T * g >= 128 * B) a 16-bit copy
 *             of the dequantised key pages [NP, H_kv, P, D] of the query-tile
 *             requests, which lets every page be dequantised once per call
 *             instead of once per query tile (a workspace without it is
 *             accepted: the slower route then).  Requests with Lq * g <= 32
 *             query rows (decode) are scored by the short-query kernel, which
 *             dequantises each page once into tensor memory; a positive
 *             args->max_seqlen_q with max_seqlen_q * g <= 32 leaves the tile
 *             kernel out of the call.
 *
 * Errors as msa_index_score, plus MSA_ERR_INVALID_ARG for a bad format or a
 * missing or misaligned scale array.  Asynchronous on `stream`.
 */
msa_status_t msa_index_score_fp4_workspace_size(const msa_index_score_args *args, int32_t format,
                                                size_t *bytes);
msa_status_t msa_index_score_fp4(const msa_index_score_args *args, int32_t format,
                                 const uint8_t *q_scale, const uint8_t *k_scale, float *out,
                                 void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* The two halves of msa_index_score_fp4, on the same stream and workspace:
 * _plan dequantises the query into the workspace and writes the work plan;
 * _run launches the score kernels that read the key cache and write `out`. */
msa_status_t msa_index_score_fp4_plan(const msa_index_score_args *args, int32_t format,
                                      const uint8_t *q_scale, void *workspace,
                                      size_t workspace_bytes, msa_stream_t stream);
msa_status_t msa_index_score_fp4_run(const msa_index_score_args *args, int32_t format,
                                     const uint8_t *k_scale, float *out, void *workspace,
                                     size_t workspace_bytes, msa_stream_t stream);

/*
 * Sparse main branch (MiniMax Sparse Attention notes, sec. 4.8 Equation (8)):
 * softmax attention of every query head over the keys of the blocks its GQA
 * group selected (sec. 4.3 Equation (3)), computed KV-outer in two phases
 * (sec. 4.11, 5.5-5.10): the selection is inverted into block -> query lists,
 * every selected block's K and V pages are loaded once per unit of gathered
 * queries and give one partial (output, log-sum-exp) per (query, head, block),
 * and the partials are merged exactly:
 *
 *   out[t, h, :] = sum_{j in S} softmax_j(s_j) V[j, h / g, :],  s_j = sm_scale <Q[t, h], K[j, h / g]>
 *   lse[t, h]    = log sum_{j in S} exp(s_j)
 *
 * S holds the keys j of the blocks listed in selection[t, h / g, :] (logical
 * block indices of the token's request; -1 entries and blocks at or beyond
 * ceil(kv_len / P) are skipped) that are visible to t: j < kv_len and, for
 * sparse_mode 3, j <= kv_len - Lq + i.  A token with no such key gets out = 0
 * and lse = -inf.
 *
 *   args   as for msa_index_score: query [T, H_q, D] fp16 / bf16 (the main
 *          branch's query), key_cache the main branch's keys, layout, table,
 *          lengths, sparse_mode; start_loc, init_blocks, local_blocks and
 *          max_seqlen_q are not used; scale must be NULL.
 *   sa     value_cache: device, the same layout, shape, dtype and page stride as
 *          key_cache (one block table serves both); selection: device int32
 *          [T, H_kv, k], ascending with a -1 tail (msa_index_score_topk writes
 *          it); k in [1, 32]; sm_scale: 0 for 1 / sqrt(D).
 *   out    device fp32 [T, H_q, D], 16-byte aligned.
 *   lse    device fp32 [T, H_q], or NULL.
 *   workspace  msa_sparse_attention_workspace_size() bytes (256-byte aligned,
 *          caller-owned): the block -> query lists, the work units and the
 *          per-block partials (T * H_q * k * D outputs in the input's 16-bit
 *          type and T * H_q * k fp32 log-sum-exps).
 *
 * Errors: as msa_index_score, plus MSA_ERR_INVALID_ARG for a missing value
 * cache or selection, k outside [1, 32] or a dtype other than fp16 / bf16,
 * and MSA_ERR_UNSUPPORTED for H_kv > 32767 or T >= 2^27.
 * Selection rows that are out of range, repeated or not ascending set
 * MSA_DEVERR_SELECTION (their outputs are then unspecified); read the error
 * word with msa_get_device_error.  Asynchronous on `stream`.
 */
typedef struct {
    const void *value_cache;
    const int32_t *selection;
    int32_t k;
    float sm_scale;
} msa_sparse_attention_args;

msa_status_t msa_sparse_attention_workspace_size(const msa_index_score_args *args,
                                                 const msa_sparse_attention_args *sa,
                                                 size_t *bytes);
msa_status_t msa_sparse_attention(const msa_index_score_args *args,
                                  const msa_sparse_attention_args *sa, float *out, float *lse,
                                  void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* Synchronise `stream` and read the device error word left in `workspace`
 * by the last call (MSA_DEVERR_* bits; 0 = clean).  Returns MSA_OK, or
 * MSA_ERR_CUDA if the copy fails. */
msa_status_t msa_get_device_error(const void *workspace, int32_t *bits, msa_stream_t stream);

/*
 * Watchdog of the score kernels (process-wide; applies to the calls enqueued
 * after it is set).  Every on-chip pipeline wait has a wall-clock limit,
 * `wait_limit_ns` (0 restores the default of 4 s, far above any legitimate
 * wait).  A wait that runs past it records MSA_DEVERR_TIMEOUT; the kernel then
 * lets its in-flight copies and tensor-core work finish, frees its tensor
 * memory and returns instead of hanging, and that call's scores are
 * incomplete.
 *
 * `stall` != 0 is for tests of that path: in every CTA of the score kernels
 * the warp that feeds the tensor-core issuer first waits on a barrier that
 * nothing completes, as a lost copy would leave it, so the limit runs out on
 * every call.  Set it back to 0 for normal calls.  Returns MSA_OK.
 */
msa_status_t msa_set_watchdog(uint64_t wait_limit_ns, int32_t stall);

/* Static description of a status code. */
const char *msa_status_string(msa_status_t status);

/* Detail of the last failing call on this host thread ("" if none). */
const char *msa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_INDEX_SCORE_H_ */
