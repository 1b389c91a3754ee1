/*
 * CPU oracle for the MSA index-branch block score (test infrastructure only).
 *
 * This file is the plain, slow definition that the CUDA path is checked
 * against.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline load it; the product library never links, includes or calls it,
 * and it includes nothing from the product.
 *
 * Definition followed (the feature request "MsaIndexScore",
 * gitcode.com/cann/ops-transformer/issues/4117, section "calculation"):
 *
 *   for token t of request b, head h, logical block beta:
 *     score[h,t,beta] = max over j in [beta*P, beta*P+P), j <= q_pos(t),
 *                       j < kv_len[b]  of  < q[t,h], k~[j, h/g] >
 *   with k~ gathered from the paged cache through block_table (or the packed
 *   TND keys), optionally int8-dequantised by scale[page, h_kv, j mod P]
 *   applied to the dot product before the mask ("DOT -> DEQUANT -> MASK ->
 *   MAX"), and fill_value (-inf) where no j is visible.
 *
 * Then the local mask of the torch API guide "CANN ops-transformer ...
 * msa_index_score" (sec. 2): blocks [0, init_blocks) take 1e30, the window
 * [max(0, start_loc+1-local_blocks), start_loc] takes 1e29 and overrides the
 * init value.  Output is fp32 [H_q, T, RoundUp(MB, 16)] (same guide, sec. 5),
 * padding columns hold the fill value.
 *
 * Readings taken where the pages are silent or disagree (each one is listed
 * with its reason in the design notes of this repository):
 *   - visibility uses rightDownCausal: q_pos = kv_len - Lq + i (sparse_mode 3);
 *     sparse_mode 0 has no causal bound.  start_loc is a logical block index
 *     used only by the local mask.
 *   - the local mask is applied to every row of a request with kv_len > 0,
 *     columns clipped to [0, MB); a request with kv_len == 0 is all fill.
 *   - arithmetic: products and sums in fp64 (all inputs are exact in fp64),
 *     int8 scale multiplied in fp64, one rounding to fp32 at the end.
 *
 * Element types: 0 = fp16, 1 = bf16, 2 = int8 (keys only), 3 = fp8 e4m3fn,
 * 4 = fp8 e5m2 (query and key of the same FP8 type, no scale: torch API guide,
 * sec. 4 and 7.2), 5 = FP4 E2M1 with group scales, query and key alike (the
 * block-scaled FP4 indexer of the MiniMax Sparse Attention notes, sec. 8.2:
 * MXFP4 = E2M1 values with one E8M0 scale per 32 elements, NVFP4 = E2M1
 * values with one E4M3 scale per 16 elements).  The FP8 decodings follow the
 * OCP 8-bit floating point formats (E4M3: bias 7, no infinities, S.1111.111 is
 * NaN; E5M2: bias 15, IEEE-style infinities and NaNs); E2M1 and E8M0 follow
 * the OCP Microscaling (MX) formats (E2M1: bias 1, no infinities or NaN;
 * E8M0: 2^(e - 127), 0xFF is NaN).  An FP4 row of D elements is D/2 bytes,
 * element 2i in the low nibble of byte i; each element is dequantised as
 * value * scale of its group before the dot product, all in fp64 (exact).
 * Layouts: 0 = BBND [NP,P,H_kv,D], 1 = BNBD [NP,H_kv,P,D], 2 = TND [T2,H_kv,D].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const void *query;          /* [T, H_q, D] contiguous */
    int32_t q_dtype;            /* 0 fp16, 1 bf16, 3 e4m3fn, 4 e5m2 */
    int64_t T;
    int32_t H_q, D;
    const void *key;            /* layout below; dim0 stride = page_stride elements */
    int32_t k_dtype;            /* 0 fp16, 1 bf16, 2 int8, 3 e4m3fn, 4 e5m2 */
    int32_t layout;             /* 0 BBND, 1 BNBD, 2 TND */
    int64_t NP;                 /* pages (paged) or T2 rows (TND) */
    int32_t P, H_kv;
    int64_t page_stride;        /* elements between consecutive dim0 entries */
    const int32_t *block_table; /* [B, MB] (paged) */
    int32_t B, MB;
    const int32_t *cu_q;        /* [B+1] */
    const int32_t *kv_len;      /* [B] (paged) */
    const int32_t *cu_k;        /* [B+1] (TND) */
    const int32_t *start_loc;   /* [B] */
    const float *scale;         /* int8: paged [NP, H_kv, P]; TND [T2, H_kv] */
    int32_t sparse_mode, init_blocks, local_blocks;
    float fill_value;
    /* FP4 (type 5) group scales, one byte per group of G elements:
     * query [T, H_q, D/G]; key paged [NP, H_kv, P, D/G], TND [T2, H_kv, D/G] */
    const uint8_t *q_scale;
    const uint8_t *k_scale;
    int32_t fp4_format;         /* 0: MXFP4 (E8M0, G = 32); 1: NVFP4 (E4M3, G = 16) */
} msa_oracle_args;

/* IEEE binary16 -> double, from the format's definition (1/5/10 bits). */
static double half_to_double(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-14 / 2^10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);   /* (1 + m/2^10) * 2^(e-15) */
    return s ? -v : v;
}

/* bfloat16 -> double: the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (the "fn" variant: finite only) -> double: 1/4/3 bits, bias 7. */
static double e4m3_to_double(uint8_t b)
{
    int s = (b >> 7) & 1, e = (b >> 3) & 0xf, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                /* subnormal: (m/8) * 2^-6 */
    else
        v = ldexp((double)(m + 8), e - 10);      /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* FP8 E5M2 -> double: 1/5/2 bits, bias 15, exponent 31 = inf / NaN. */
static double e5m2_to_double(uint8_t b)
{
    int s = (b >> 7) & 1, e = (b >> 2) & 0x1f, m = b & 3;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -16);               /* subnormal: (m/4) * 2^-14 */
    else
        v = ldexp((double)(m + 4), e - 17);      /* (1 + m/4) * 2^(e-15) */
    return s ? -v : v;
}

/* FP4 E2M1 -> double: 1/2/1 bits, bias 1, no infinities or NaN. */
static double e2m1_to_double(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? ldexp((double)m, -1)           /* subnormal: (m/2) * 2^0 */
                      : ldexp((double)(m + 2), e - 2); /* (1 + m/2) * 2^(e-1) */
    return s ? -v : v;
}

/* E8M0 scale -> double: 2^(e - 127); 0xFF is NaN. */
static double e8m0_to_double(uint8_t b)
{
    return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127);
}

/* Element d of an FP4 row that starts at byte `row`, dequantised by the
 * scale of its group (scales of the row start at `srow`). */
static double fp4_elem(const uint8_t *base, int64_t row, const uint8_t *scales, int64_t srow,
                       int d, int32_t fmt)
{
    const uint8_t byte = base[row + d / 2];
    const double v = e2m1_to_double((uint8_t)((d & 1) ? (byte >> 4) : (byte & 15)));
    const int G = fmt ? 16 : 32;
    const uint8_t sb = scales[srow + d / G];
    return v * (fmt ? e4m3_to_double(sb) : e8m0_to_double(sb));
}

static double load_elem(const void *base, int32_t dtype, int64_t idx)
{
    if (dtype == 2)
        return (double)((const int8_t *)base)[idx];
    if (dtype == 3)
        return e4m3_to_double(((const uint8_t *)base)[idx]);
    if (dtype == 4)
        return e5m2_to_double(((const uint8_t *)base)[idx]);
    uint16_t bits = ((const uint16_t *)base)[idx];
    return dtype == 1 ? bf16_to_double(bits) : half_to_double(bits);
}

/* Request that owns global token t: the b with cu_q[b] <= t < cu_q[b+1]. */
static int request_of(const msa_oracle_args *a, int64_t t)
{
    for (int b = 0; b < a->B; ++b)
        if (a->cu_q[b] <= t && t < a->cu_q[b + 1])
            return b;
    return -1;
}

/* Storage elements of one row of D values: D, or D/2 bytes for FP4. */
static int64_t row_units(const msa_oracle_args *a)
{
    return a->k_dtype == 5 ? a->D / 2 : a->D;
}

/* Storage offset of key row j (logical position in request b), head hk; the
 * row's scale index (int8: one per row; FP4: the row's first group scale is
 * scale_idx * D/G).  Returns -1 if the row cannot be addressed (bad table entry). */
static int64_t key_offset(const msa_oracle_args *a, int b, int64_t j, int hk,
                          int64_t *scale_idx)
{
    const int64_t ru = row_units(a);
    if (a->layout == 2) {                                   /* TND */
        int64_t row = (int64_t)a->cu_k[b] + j;
        if (row < 0 || row >= a->NP)
            return -1;
        *scale_idx = row * a->H_kv + hk;
        return (row * a->H_kv + hk) * ru;
    }
    int64_t beta = j / a->P, off = j % a->P;
    int64_t page = a->block_table[(int64_t)b * a->MB + beta];
    if (page < 0 || page >= a->NP)
        return -1;
    *scale_idx = (page * a->H_kv + hk) * (int64_t)a->P + off;
    if (a->layout == 0)                                      /* BBND */
        return page * a->page_stride + (off * a->H_kv + hk) * ru;
    return page * a->page_stride + ((int64_t)hk * a->P + off) * ru;  /* BNBD */
}

/* One output row (h, t): MBp values. Returns 0, or 1 if a needed key row could
 * not be addressed (the row is then left as computed from the rows that could). */
static int oracle_row(const msa_oracle_args *a, int h, int64_t t, float *dst)
{
    const int64_t MBp = ((int64_t)a->MB + 15) / 16 * 16;
    const int g = a->H_q / a->H_kv;
    const int hk = h / g;
    int bad = 0;
    for (int64_t c = 0; c < MBp; ++c)
        dst[c] = a->fill_value;
    int b = request_of(a, t);
    if (b < 0)
        return 0;
    const int64_t Lq = a->cu_q[b + 1] - a->cu_q[b];
    const int64_t L = a->layout == 2 ? (int64_t)a->cu_k[b + 1] - a->cu_k[b]
                                     : (int64_t)a->kv_len[b];
    const int64_t i = t - a->cu_q[b];
    const int64_t qpos = a->sparse_mode == 3 ? L - Lq + i : INT64_MAX;
    const int64_t qrow = (t * a->H_q + h) * row_units(a);
    const int64_t ng = a->fp4_format ? a->D / 16 : a->D / 32;   /* FP4 groups per row */

    for (int64_t beta = 0; beta < a->MB; ++beta) {
        double best = 0.0;
        int any = 0;
        for (int64_t j = beta * a->P; j < beta * a->P + a->P; ++j) {
            if (j >= L || j > qpos)
                continue;                                    /* MASK */
            int64_t sidx = 0;
            int64_t koff = key_offset(a, b, j, hk, &sidx);
            if (koff < 0) {
                bad = 1;
                continue;
            }
            double s = 0.0;                                  /* DOT */
            if (a->k_dtype == 5) {                           /* FP4: dequantised values */
                for (int d = 0; d < a->D; ++d)
                    s += fp4_elem((const uint8_t *)a->query, qrow, a->q_scale,
                                  (t * a->H_q + h) * ng, d, a->fp4_format) *
                         fp4_elem((const uint8_t *)a->key, koff, a->k_scale, sidx * ng, d,
                                  a->fp4_format);
            } else {
                for (int d = 0; d < a->D; ++d)
                    s += load_elem(a->query, a->q_dtype, qrow + d) *
                         load_elem(a->key, a->k_dtype, koff + d);
            }
            if (a->k_dtype == 2)
                s *= (double)a->scale[sidx];                 /* DEQUANT (column scale) */
            if (!any || s > best)                            /* MAX */
                best = s;
            any = 1;
        }
        dst[beta] = any ? (float)best : a->fill_value;
    }

    /* local mask: forced scores for blocks the downstream top-k must keep */
    if (L > 0 && (a->init_blocks > 0 || a->local_blocks > 0)) {
        for (int64_t beta = 0; beta < a->init_blocks && beta < a->MB; ++beta)
            dst[beta] = 1e30f;
        const int64_t sl = a->start_loc[b];
        int64_t lo = sl + 1 - a->local_blocks;
        if (lo < 0)
            lo = 0;
        for (int64_t beta = lo; beta <= sl && beta < a->MB; ++beta)
            dst[beta] = 1e29f;
    }
    return bad;
}

/*
 * Compute the listed output rows.  rows[r] = h * T + t; out holds
 * nrows x RoundUp(MB,16) floats.  nthreads <= 0 uses the OpenMP default.
 * Returns the number of rows that met an unaddressable key row.
 */
int msa_oracle_rows(const msa_oracle_args *a, const int64_t *rows, int64_t nrows,
                    float *out, int nthreads)
{
    const int64_t MBp = ((int64_t)a->MB + 15) / 16 * 16;
    int nbad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : nbad)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int h = (int)(rows[r] / a->T);
        int64_t t = rows[r] % a->T;
        nbad += oracle_row(a, h, t, out + r * MBp);
    }
    return nbad;
}

/* Full output [H_q, T, RoundUp(MB,16)]. */
int msa_oracle_full(const msa_oracle_args *a, float *out, int nthreads)
{
    const int64_t MBp = ((int64_t)a->MB + 15) / 16 * 16;
    const int64_t n = (int64_t)a->H_q * a->T;
    int nbad = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : nbad)
#endif
    for (int64_t r = 0; r < n; ++r)
        nbad += oracle_row(a, (int)(r / a->T), r % a->T, out + r * MBp);
    return nbad;
}

/* Threads an OpenMP region would use with the given request (for reports). */
int msa_oracle_threads(int nthreads)
{
#ifdef _OPENMP
    int n = 0;
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Decode one element of the given type (for tests of the decoders); 5 is an
 * E2M1 code (low nibble), 6 an E8M0 scale byte. */
double msa_oracle_decode(int32_t dtype, uint32_t bits)
{
    if (dtype == 2) return (double)(int8_t)(uint8_t)bits;
    if (dtype == 3) return e4m3_to_double((uint8_t)bits);
    if (dtype == 4) return e5m2_to_double((uint8_t)bits);
    if (dtype == 5) return e2m1_to_double((uint8_t)(bits & 15));
    if (dtype == 6) return e8m0_to_double((uint8_t)bits);
    return dtype == 1 ? bf16_to_double((uint16_t)bits) : half_to_double((uint16_t)bits);
}
