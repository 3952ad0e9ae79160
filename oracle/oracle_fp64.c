/*
 * FP64 CPU oracle for causal grouped-query softmax attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written
 * definition that the CUDA path is checked against.  It shares no code,
 * header or constant with the CUDA library, and only the test suite, the
 * smoke check and the benchmark's CPU-baseline / reference arm may load it.
 * The product path never calls it and has no CPU fallback.
 *
 * What is computed (one query row at a time, every quantity in double):
 *
 *   TileOPs "Attention Operators", GQADenseFwdOp, stages 1, 4, 5, 7:
 *     r(h)  = floor(h / g),  g = Hq / Hkv           (head grouping)
 *     p_i   = i + Skv - Sq                          (bottom-right alignment)
 *     z_j   = scale * <q_i,h , k_j,r(h)>            (scores)
 *     V_i   = { j : (!causal || j <= p_i) }         (visibility)
 *     O_i,h = sum_{j in V_i} softmax_j(z) * v_j,r(h)
 *   RL-Kernel "Standard Softmax Attention", Tensor Contract / Accuracy:
 *     key_padding_mask[b, j] == 0 removes key j from V_i for every head and
 *     query (the column becomes -inf); scale None -> 1/sqrt(D) is resolved by
 *     the caller, any explicit value (0.0 included) is used as given.
 *   TileOPs "Attention Operators", MHADecodePagedWithKVCacheFwdOp and
 *   GQAPagedFwdOp:  a row with no visible key outputs zeros; paged K/V of
 *     request b at logical position t live in physical page
 *     block_table[b, t / page_size], slot t % page_size.
 *   MATE "QSA", Core Attention: the log-sum-exp is natural-log, of the
 *     scaled logits, and -inf for a row with no visible key.
 *
 * Optional terms (TileOPs "Attention Operators", GQADenseFwdOp stages 5 and
 * 6, and GQAPagedFwdOp's sinks):
 *   window:  with wL = window_left and wR = window_right (negative =
 *            unlimited), key j is visible to row i only if j >= p_i - wL and
 *            j <= p_i + wR, on top of the causal and padding conditions;
 *   softcap: with c > 0 every visible logit z becomes c * tanh(z / c); c = 0
 *            leaves it unchanged;
 *   sinks:   a logit s_h per query head joins the softmax denominator only
 *            (no value, not scaled, not capped): weight_j = exp(z_j) /
 *            (sum_{j in V_i} exp(z_j) + exp(s_h)), and the log-sum-exp
 *            includes exp(s_h).  s_h = -inf adds nothing; s_h = +inf makes
 *            the row's output zero (and its log-sum-exp +inf).  A row with no
 *            visible key still outputs zeros with log-sum-exp -inf (the pages
 *            fix the zero output; -inf keeps "zero row <=> -inf" whether a
 *            sink is given or not).
 *
 * FP8 keys and values (TileOPs "Attention Operators", GQADenseFwdOp stage 2):
 * float8_e4m3fn caches are widened exactly and multiplied by one scale per
 * request and KV head, K^ = K * k_scale[b, r], V' = V * v_scale[b, r], before
 * the definition above (oracle_attn_paged_fp8kv_ex).
 *
 * softmax_j(z) is written out as its definition: with M = max_{j in V_i} z_j
 * and Z = sum_{j in V_i} exp(z_j - M), weight_j = exp(z_j - M) / Z and
 * LSE = M + log Z.  Subtracting M changes nothing mathematically; it only
 * keeps exp() finite.
 *
 * Inputs may be given as IEEE double, as bfloat16 bit patterns or as IEEE
 * half (float16) bit patterns (uint16); both 16-bit types widen to double
 * exactly: a bfloat16 is the top half of a float, and a half is
 * (-1)^s * 2^(e-15) * (1 + m/1024) for a biased exponent e in 1..30,
 * (-1)^s * 2^-14 * (m/1024) for e = 0 (zero and subnormals), and an infinity
 * or NaN for e = 31.  Outputs are always double.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared (OpenMP optional).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F64 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* Exact widening of one element of an input array to double. */
static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == ORACLE_F64) return ((const double*)base)[idx];
    if (dtype == ORACLE_F16) {
        const uint16_t h = ((const uint16_t*)base)[idx];
        const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
        double mag;
        if (e == 0) mag = ldexp((double)m, -24);                  /* 2^-14 * m / 1024 */
        else if (e == 31) mag = m ? NAN : INFINITY;
        else mag = ldexp(1024.0 + m, e - 25);                    /* 2^(e-15) * (1024 + m) / 1024 */
        return sign ? -mag : mag;
    }
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * One query row of the dense definition.
 *   q      : [B, Sq, Hq, D]      k, v : [B, Skv, Hkv, D]      (BSHD)
 *   mask   : [B, Skv] bytes, nonzero = keep, or NULL
 *   z      : scratch of Skv doubles
 *   out    : D doubles; *lse_out : the row's log-sum-exp
 */
/* Optional terms of one call (see the header). */
typedef struct {
    long window_left, window_right;            /* negative = unlimited */
    double softcap;                            /* 0 = off */
    const double* sinks;                       /* [Hq] or NULL */
} oracle_opts;

static const oracle_opts NO_OPTS = {-1, -1, 0.0, NULL};

static void dense_row(const void* q, const void* k, const void* v, int dtype,
                      const uint8_t* mask, int Hq, int Hkv, int Sq, int Skv,
                      int D, int causal, double scale, const oracle_opts* opt,
                      int b, int i, int h, double* z, double* out, double* lse_out) {
    const int g = Hq / Hkv;
    const int r = h / g;                       /* KV head of query head h */
    const long p = (long)i + Skv - Sq;         /* query position on the key axis */
    const size_t q_off = (((size_t)b * Sq + i) * Hq + h) * (size_t)D;

    int any = 0;
    double M = -INFINITY;
    for (int j = 0; j < Skv; ++j) {
        int visible = (!causal || (long)j <= p) &&
                      (opt->window_left < 0 || (long)j >= p - opt->window_left) &&
                      (opt->window_right < 0 || (long)j <= p + opt->window_right) &&
                      (mask == NULL || mask[(size_t)b * Skv + j] != 0);
        if (!visible) { z[j] = -INFINITY; continue; }
        const size_t k_off = (((size_t)b * Skv + j) * Hkv + r) * (size_t)D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load_elem(q, q_off + d, dtype) * load_elem(k, k_off + d, dtype);
        z[j] = scale * dot;
        if (opt->softcap > 0.0) z[j] = opt->softcap * tanh(z[j] / opt->softcap);
        if (!any || z[j] > M) M = z[j];
        any = 1;
    }

    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (!any) {                                /* no visible key: zeros, -inf */
        *lse_out = -INFINITY;
        return;
    }
    /* A sink joins the denominator: it takes part in the maximum that keeps
     * exp() finite, and adds exp(s - M) to Z. */
    const double sink = opt->sinks ? opt->sinks[h] : -INFINITY;
    if (sink == INFINITY) {                    /* the sink takes all the weight */
        *lse_out = INFINITY;
        return;
    }
    if (sink > M) M = sink;
    double Z = sink == -INFINITY ? 0.0 : exp(sink - M);
    for (int j = 0; j < Skv; ++j)
        if (z[j] != -INFINITY) Z += exp(z[j] - M);
    for (int j = 0; j < Skv; ++j) {
        if (z[j] == -INFINITY) continue;
        const double w = exp(z[j] - M) / Z;
        const size_t v_off = (((size_t)b * Skv + j) * Hkv + r) * (size_t)D;
        for (int d = 0; d < D; ++d) out[d] += w * load_elem(v, v_off + d, dtype);
    }
    *lse_out = M + log(Z);
}

static int check_dense_args(int B, int Hq, int Hkv, int Sq, int Skv, int D) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -2;              /* GQA needs Hq divisible by Hkv */
    return 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the next parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Dense attention over every row.  o: [B, Sq, Hq, D]; lse: [B, Sq, Hq].
 * Returns 0, -1 for a bad size, -2 when Hq is not a multiple of Hkv,
 * -3 when scratch memory cannot be had.
 */
static int dense_all(const void* q, const void* k, const void* v, int dtype,
                     const uint8_t* mask, double* o, double* lse, int B,
                     int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                     double scale, const oracle_opts* opt, int nthreads) {
    int rc = check_dense_args(B, Hq, Hkv, Sq, Skv, D);
    if (rc) return rc;
    set_threads(nthreads);
    const long nrows = (long)B * Sq * Hq;
    int failed = 0;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long row = 0; row < nrows; ++row) {
                const int h = (int)(row % Hq);
                const int i = (int)((row / Hq) % Sq);
                const int b = (int)(row / ((long)Hq * Sq));
                dense_row(q, k, v, dtype, mask, Hq, Hkv, Sq, Skv, D, causal,
                          scale, opt, b, i, h, z, o + (size_t)row * D, lse + row);
            }
            free(z);
        }
    }
    return failed ? -3 : 0;
}

static int check_opts(long window_left, long window_right, double softcap) {
    if (window_left < -1 || window_right < -1) return -7;
    if (!(softcap >= 0.0) || softcap == INFINITY) return -8;
    return 0;
}

int oracle_attn_dense(const void* q, const void* k, const void* v, int dtype,
                      const uint8_t* mask, double* o, double* lse, int B,
                      int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                      double scale, int nthreads) {
    return dense_all(q, k, v, dtype, mask, o, lse, B, Hq, Hkv, Sq, Skv, D, causal,
                     scale, &NO_OPTS, nthreads);
}

/*
 * oracle_attn_dense with the optional terms: window_left / window_right
 * (-1 = unlimited), softcap (0 = off), sinks ([Hq] doubles or NULL).
 * Also returns -7 for a window below -1 and -8 for a negative or non-finite
 * softcap.
 */
int oracle_attn_dense_ex(const void* q, const void* k, const void* v, int dtype,
                         const uint8_t* mask, double* o, double* lse, int B,
                         int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                         double scale, long window_left, long window_right,
                         double softcap, const double* sinks, int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    return dense_all(q, k, v, dtype, mask, o, lse, B, Hq, Hkv, Sq, Skv, D, causal,
                     scale, &opt, nthreads);
}

/*
 * Dense attention for a list of rows only.  rows: nrows triples (b, i, h);
 * o_rows: [nrows, D]; lse_rows: [nrows].  Same return codes, plus -4 for a
 * row index out of range.
 */
static int dense_rows(const void* q, const void* k, const void* v,
                      int dtype, const uint8_t* mask, const int32_t* rows,
                      int nrows, double* o_rows, double* lse_rows, int B,
                      int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                      double scale, const oracle_opts* opt, int nthreads) {
    int rc = check_dense_args(B, Hq, Hkv, Sq, Skv, D);
    if (rc) return rc;
    for (int n = 0; n < nrows; ++n) {
        if (rows[3 * n] < 0 || rows[3 * n] >= B || rows[3 * n + 1] < 0 ||
            rows[3 * n + 1] >= Sq || rows[3 * n + 2] < 0 || rows[3 * n + 2] >= Hq)
            return -4;
    }
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int n = 0; n < nrows; ++n)
                dense_row(q, k, v, dtype, mask, Hq, Hkv, Sq, Skv, D, causal,
                          scale, opt, rows[3 * n], rows[3 * n + 1], rows[3 * n + 2],
                          z, o_rows + (size_t)n * D, lse_rows + n);
            free(z);
        }
    }
    return failed ? -3 : 0;
}

int oracle_attn_dense_rows(const void* q, const void* k, const void* v,
                           int dtype, const uint8_t* mask, const int32_t* rows,
                           int nrows, double* o_rows, double* lse_rows, int B,
                           int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                           double scale, int nthreads) {
    return dense_rows(q, k, v, dtype, mask, rows, nrows, o_rows, lse_rows, B, Hq, Hkv,
                      Sq, Skv, D, causal, scale, &NO_OPTS, nthreads);
}

/* oracle_attn_dense_rows with the optional terms (as oracle_attn_dense_ex). */
int oracle_attn_dense_rows_ex(const void* q, const void* k, const void* v,
                              int dtype, const uint8_t* mask, const int32_t* rows,
                              int nrows, double* o_rows, double* lse_rows, int B,
                              int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                              double scale, long window_left, long window_right,
                              double softcap, const double* sinks, int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    return dense_rows(q, k, v, dtype, mask, rows, nrows, o_rows, lse_rows, B, Hq, Hkv,
                      Sq, Skv, D, causal, scale, &opt, nthreads);
}

/*
 * Physical page holding token t of a request whose block_table row is trow
 * (max_pages entries): trow[t / page_size], the token sitting in slot
 * t % page_size of it (the page addressing of the paged ops on the TileOPs
 * page).  -1 when the logical page lies past the row or the page id lies
 * outside [0, num_pages), so that no read leaves the table or the pool.
 */
static long page_of_token(const int32_t* trow, int max_pages, int page_size, int num_pages, int t) {
    const long lp = t / page_size;
    if (lp < 0 || lp >= max_pages) return -1;
    const int32_t phys = trow[lp];
    return (phys < 0 || phys >= num_pages) ? -1 : (long)phys;
}

/*
 * Paged attention, written as "gather the request's cache into a dense
 * sequence, then apply the dense definition" (the paged ops on the TileOPs
 * page read the same logical sequence through block_table).
 *
 *   q            : [B, Sq, Hq, D]
 *   k_cache, v_cache : [num_pages, page_size, Hkv, D]
 *   seqlens      : [B] logical cache length L_b, the Sq query tokens included
 *   block_table  : [B, max_pages] physical page of each logical page
 *   req_mask     : [B] bytes, nonzero = compute request b (NULL = all)
 *   o            : [B, Sq, Hq, D]; lse : [B, Sq, Hq]; rows of requests left
 *                  out by req_mask are not written.
 *
 * Query i of request b sits at key position i + L_b - Sq (end-aligned).
 * Returns 0; -1 bad size; -2 Hq % Hkv != 0; -3 out of memory; -5 a length
 * outside [0, max_pages * page_size]; -6 a needed block_table entry outside
 * [0, num_pages).
 */
static int paged_all(const void* q, const void* k_cache, const void* v_cache,
                     int dtype, const int32_t* seqlens,
                     const int32_t* block_table, int page_size,
                     const uint8_t* req_mask, double* o, double* lse, int B,
                     int Sq, int Hq, int Hkv, int D, int num_pages,
                     int max_pages, int causal, double scale, const oracle_opts* opt,
                     int nthreads) {
    int rc = check_dense_args(B, Hq, Hkv, Sq, 0, D);
    if (rc) return rc;
    if (page_size <= 0 || num_pages < 0 || max_pages < 0) return -1;
    for (int b = 0; b < B; ++b) {
        if (req_mask && !req_mask[b]) continue;
        const int L = seqlens[b];
        if (L < 0 || (long)L > (long)max_pages * page_size) return -5;
        const int npages = (L + page_size - 1) / page_size;
        for (int lp = 0; lp < npages; ++lp) {
            const int32_t phys = block_table[(size_t)b * max_pages + lp];
            if (phys < 0 || phys >= num_pages) return -6;
        }
    }
    const size_t es = dtype == ORACLE_F64 ? sizeof(double) : sizeof(uint16_t);
    for (int b = 0; b < B; ++b) {
        if (req_mask && !req_mask[b]) continue;
        const int L = seqlens[b];
        /* Gather request b's keys and values, token by token, into the dense
         * layout [1, L, Hkv, D]. */
        const size_t tok_elems = (size_t)Hkv * D;
        char* kd = (char*)malloc(es * tok_elems * (size_t)(L > 0 ? L : 1));
        char* vd = (char*)malloc(es * tok_elems * (size_t)(L > 0 ? L : 1));
        if (!kd || !vd) { free(kd); free(vd); return -3; }
        for (int t = 0; t < L; ++t) {
            const long phys = page_of_token(block_table + (size_t)b * max_pages, max_pages, page_size, num_pages, t);
            if (phys < 0) { free(kd); free(vd); return -6; }
            const size_t src = ((size_t)phys * page_size + t % page_size) * tok_elems;
            memcpy(kd + (size_t)t * tok_elems * es, (const char*)k_cache + src * es,
                   tok_elems * es);
            memcpy(vd + (size_t)t * tok_elems * es, (const char*)v_cache + src * es,
                   tok_elems * es);
        }
        const char* qb = (const char*)q + (size_t)b * Sq * Hq * D * es;
        rc = dense_all(qb, kd, vd, dtype, NULL,
                       o + (size_t)b * Sq * Hq * D, lse + (size_t)b * Sq * Hq,
                       1, Hq, Hkv, Sq, L, D, causal, scale, opt, nthreads);
        free(kd);
        free(vd);
        if (rc) return rc;
    }
    return 0;
}

int oracle_attn_paged(const void* q, const void* k_cache, const void* v_cache,
                      int dtype, const int32_t* seqlens,
                      const int32_t* block_table, int page_size,
                      const uint8_t* req_mask, double* o, double* lse, int B,
                      int Sq, int Hq, int Hkv, int D, int num_pages,
                      int max_pages, int causal, double scale, int nthreads) {
    return paged_all(q, k_cache, v_cache, dtype, seqlens, block_table, page_size, req_mask,
                     o, lse, B, Sq, Hq, Hkv, D, num_pages, max_pages, causal, scale,
                     &NO_OPTS, nthreads);
}

/* oracle_attn_paged with the optional terms (as oracle_attn_dense_ex). */
int oracle_attn_paged_ex(const void* q, const void* k_cache, const void* v_cache,
                         int dtype, const int32_t* seqlens,
                         const int32_t* block_table, int page_size,
                         const uint8_t* req_mask, double* o, double* lse, int B,
                         int Sq, int Hq, int Hkv, int D, int num_pages,
                         int max_pages, int causal, double scale, long window_left,
                         long window_right, double softcap, const double* sinks,
                         int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    return paged_all(q, k_cache, v_cache, dtype, seqlens, block_table, page_size, req_mask,
                     o, lse, B, Sq, Hq, Hkv, D, num_pages, max_pages, causal, scale, &opt,
                     nthreads);
}

/*
 * float8_e4m3fn, the 8-bit type the pages name for FP8 keys and values
 * (TileOPs "Attention Operators", GQAVarlenFwdOp), widened to double: sign s,
 * 4-bit exponent e with bias 7, 3-bit mantissa m, no infinities:
 *   e in 1..15 (except e = 15, m = 7):  (-1)^s * 2^(e-7) * (1 + m/8)
 *   e = 0:                              (-1)^s * 2^-6 * (m/8)   (zero, subnormals)
 *   e = 15, m = 7:                      NaN
 */
static double e4m3_to_double(uint8_t x) {
    const int s = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double mag;
    if (e == 15 && m == 7) mag = NAN;
    else if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(8.0 + m, e - 10);
    return s ? -mag : mag;
}

/* e4m3fn codes widened to double, for the tests' check of the table. */
int oracle_e4m3_decode(const uint8_t* codes, double* out, long n) {
    if (n < 0) return -1;
    for (long i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
    return 0;
}

/*
 * Paged attention over float8_e4m3fn key and value caches (TileOPs "Attention
 * Operators", GQADenseFwdOp stage 2, FP8 dequantization): with per-(request,
 * KV head) scales, K^_{j,r} = K_{j,r} * k_scale[b, r] and
 * V'_{j,r} = V_{j,r} * v_scale[b, r]; Q stays 16-bit (its scale is one).
 * The dequantized request is then the dense definition above, in double.
 *   q            : [B, Sq, Hq, D], dtype ORACLE_BF16 or ORACLE_F16 (or F64)
 *   k/v_cache    : [num_pages, page_size, Hkv, D] e4m3fn codes
 *   k/v_scale    : [B, Hkv] doubles, or NULL for all ones
 * Other arguments and return codes as oracle_attn_paged_ex.
 */
int oracle_attn_paged_fp8kv_ex(const void* q, int q_dtype, const uint8_t* k_cache,
                               const uint8_t* v_cache, const double* k_scale,
                               const double* v_scale, const int32_t* seqlens,
                               const int32_t* block_table, int page_size,
                               const uint8_t* req_mask, double* o, double* lse, int B,
                               int Sq, int Hq, int Hkv, int D, int num_pages, int max_pages,
                               int causal, double scale, long window_left, long window_right,
                               double softcap, const double* sinks, int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    rc = check_dense_args(B, Hq, Hkv, Sq, 0, D);
    if (rc) return rc;
    if (page_size <= 0 || num_pages < 0 || max_pages < 0) return -1;
    for (int b = 0; b < B; ++b) {
        if (req_mask && !req_mask[b]) continue;
        const int L = seqlens[b];
        if (L < 0 || (long)L > (long)max_pages * page_size) return -5;
        const int npages = (L + page_size - 1) / page_size;
        for (int lp = 0; lp < npages; ++lp) {
            const int32_t phys = block_table[(size_t)b * max_pages + lp];
            if (phys < 0 || phys >= num_pages) return -6;
        }
    }
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    const size_t tok_elems = (size_t)Hkv * D;
    const size_t q_elems = (size_t)Sq * Hq * D;
    for (int b = 0; b < B; ++b) {
        if (req_mask && !req_mask[b]) continue;
        const int L = seqlens[b];
        /* request b: Q widened, K and V gathered token by token and dequantized */
        double* qd = (double*)malloc(sizeof(double) * (q_elems > 0 ? q_elems : 1));
        double* kd = (double*)malloc(sizeof(double) * tok_elems * (size_t)(L > 0 ? L : 1));
        double* vd = (double*)malloc(sizeof(double) * tok_elems * (size_t)(L > 0 ? L : 1));
        if (!qd || !kd || !vd) { free(qd); free(kd); free(vd); return -3; }
        for (size_t e = 0; e < q_elems; ++e) qd[e] = load_elem(q, (size_t)b * q_elems + e, q_dtype);
        const int32_t* trow = block_table + (size_t)b * max_pages;   /* request b's pages */
        for (int t = 0; t < L; ++t) {
            const long phys = page_of_token(trow, max_pages, page_size, num_pages, t);
            if (phys < 0) { free(qd); free(kd); free(vd); return -6; }
            const size_t src = ((size_t)phys * page_size + t % page_size) * tok_elems;
            for (int r = 0; r < Hkv; ++r) {
                const double ks = k_scale ? k_scale[(size_t)b * Hkv + r] : 1.0;
                const double vs = v_scale ? v_scale[(size_t)b * Hkv + r] : 1.0;
                for (int d = 0; d < D; ++d) {
                    const size_t e = (size_t)r * D + d;
                    kd[(size_t)t * tok_elems + e] = e4m3_to_double(k_cache[src + e]) * ks;
                    vd[(size_t)t * tok_elems + e] = e4m3_to_double(v_cache[src + e]) * vs;
                }
            }
        }
        rc = dense_all(qd, kd, vd, ORACLE_F64, NULL, o + (size_t)b * q_elems, lse + (size_t)b * Sq * Hq,
                       1, Hq, Hkv, Sq, L, D, causal, scale, &opt, nthreads);
        free(qd);
        free(kd);
        free(vd);
        if (rc) return rc;
    }
    return 0;
}

/*
 * Offsets of packed requests: non-decreasing from 0 up to total, B + 1 of them
 * (TileOPs "Attention Operators", GQAVarlenFwdOp: cu_seqlens delimit each
 * request).
 */
static int check_offsets(const int32_t* cu, int B, long total) {
    if (cu[0] != 0 || (long)cu[B] != total) return -9;
    for (int b = 0; b < B; ++b)
        if (cu[b + 1] < cu[b]) return -9;
    return 0;
}

/*
 * Packed variable-length attention (TileOPs "Attention Operators",
 * GQAVarlenFwdOp): request b owns the packed query rows
 * [cu_q[b], cu_q[b + 1]) and the key / value rows [cu_kv[b], cu_kv[b + 1]);
 * every request is the dense definition on its own rows, with its own
 * bottom-right-aligned causal mask (Sq_b queries, Skv_b keys).
 *   q : [total_q, Hq, D]      k, v : [total_kv, Hkv, D]
 *   o : [total_q, Hq, D]      lse  : [total_q, Hq]
 * Returns 0; -1 bad size; -2 Hq % Hkv != 0; -3 out of memory; -7 / -8 bad
 * options; -9 offsets that do not run from 0 up to the total without
 * decreasing.
 */
int oracle_attn_varlen_ex(const void* q, const void* k, const void* v, int dtype,
                          const int32_t* cu_q, const int32_t* cu_kv, double* o,
                          double* lse, int B, int total_q, int total_kv, int Hq,
                          int Hkv, int D, int causal, double scale, long window_left,
                          long window_right, double softcap, const double* sinks,
                          int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    rc = check_dense_args(B, Hq, Hkv, total_q, total_kv, D);
    if (rc) return rc;
    if (check_offsets(cu_q, B, total_q) || check_offsets(cu_kv, B, total_kv)) return -9;
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    const size_t es = dtype == ORACLE_F64 ? sizeof(double) : sizeof(uint16_t);
    for (int b = 0; b < B; ++b) {
        const int qs = cu_q[b], sq = cu_q[b + 1] - qs;
        const int ks = cu_kv[b], skv = cu_kv[b + 1] - ks;
        /* rows [qs, qs + sq) of a [total, H, D] tensor are a [1, sq, H, D] one */
        rc = dense_all((const char*)q + (size_t)qs * Hq * D * es,
                       (const char*)k + (size_t)ks * Hkv * D * es,
                       (const char*)v + (size_t)ks * Hkv * D * es, dtype, NULL,
                       o + (size_t)qs * Hq * D, lse + (size_t)qs * Hq, 1, Hq, Hkv, sq,
                       skv, D, causal, scale, &opt, nthreads);
        if (rc) return rc;
    }
    return 0;
}

/*
 * Paged attention over packed queries (TileOPs "Attention Operators",
 * GQAPagedFwdOp): request b's queries are the packed rows
 * [cu_q[b], cu_q[b + 1]); its cache holds cache_seqlens[b] tokens, its query
 * tokens included, through block_table[b].  Every request is the paged
 * definition above on its own query rows; a request without query rows
 * produces nothing.
 *   q : [total_q, Hq, D]      k_cache, v_cache : [num_pages, page_size, Hkv, D]
 *   o : [total_q, Hq, D]      lse : [total_q, Hq]
 * Returns the codes of paged_all, -7 / -8 for bad options and -9 for bad
 * query offsets.
 */
int oracle_attn_paged_varlen_ex(const void* q, const void* k_cache, const void* v_cache,
                                int dtype, const int32_t* cu_q, const int32_t* cache_seqlens,
                                const int32_t* block_table, int page_size, double* o,
                                double* lse, int B, int total_q, int Hq, int Hkv, int D,
                                int num_pages, int max_pages, int causal, double scale,
                                long window_left, long window_right, double softcap,
                                const double* sinks, int nthreads) {
    int rc = check_opts(window_left, window_right, softcap);
    if (rc) return rc;
    rc = check_dense_args(B, Hq, Hkv, total_q, 0, D);
    if (rc) return rc;
    if (check_offsets(cu_q, B, total_q)) return -9;
    const oracle_opts opt = {window_left, window_right, softcap, sinks};
    const size_t es = dtype == ORACLE_F64 ? sizeof(double) : sizeof(uint16_t);
    for (int b = 0; b < B; ++b) {
        const int qs = cu_q[b], sq = cu_q[b + 1] - qs;
        if (sq == 0) continue;
        rc = paged_all((const char*)q + (size_t)qs * Hq * D * es, k_cache, v_cache, dtype,
                       cache_seqlens + b, block_table + (size_t)b * max_pages, page_size, NULL,
                       o + (size_t)qs * Hq * D, lse + (size_t)qs * Hq, 1, sq, Hq, Hkv, D,
                       num_pages, max_pages, causal, scale, &opt, nthreads);
        if (rc) return rc;
    }
    return 0;
}
