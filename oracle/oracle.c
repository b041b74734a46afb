/*
 * CPU oracle for the sparse-attention prefill indexer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load or run this file.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * It writes out the plain definition of what the indexer returns:
 *
 *   score    s[r,j] = k_scale[j] * sum_h w[r,h] * max(0, sum_d q[r,h,d] k[j,d])
 *            for every visible key ks[r] <= j < ke[r], in fp64, every sum taken
 *            in ascending index order.  Pages: "[sglang] logits를 쓰지 않는
 *            top-k" introduction (an indexer score per query row over every
 *            visible key) and section 1 (the heads are reduced per key); the
 *            page does not print the formula, the ReLU-weighted head sum with a
 *            per-key scale is the stated problem of this library.
 *   select   order the visible keys by (score descending, key index
 *            ascending), keep the first topk, return their row-relative
 *            indices j - ks[r] in ascending order, then -1 up to topk.
 *            Same page, section 1 (candidate indices are stored as
 *            key - ks[row]) and section 3 (a consumer skips negative
 *            positions); "[sglang] ROCm DSA Indexer Top-K 최적화", solution
 *            section (exact top-k at torch.topk-level recall).
 *   page     map a row-relative position p >= 0 to the physical KV slot
 *            table[t, p / P] * P + p % P of a paged cache with page size P,
 *            where t is the page-table row of the query row; negative
 *            positions (the -1 padding) stay as they are.  "[sglang] logits를
 *            쓰지 않는 top-k", section 3 (the page-table transform for paged
 *            output, page size 64).
 *
 * Inputs are decoded exactly to fp64 from the bit formats:
 *   e4m3 (fn):  1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals
 *               at exponent 0, S.1111.111 is NaN, no infinities, max 448.
 *   bfloat16:   1 sign, 8 exponent bits (bias 127), 7 mantissa bits.
 *   MXFP4:      the OCP microscaling format with FP4 elements: every element
 *               is an e2m1 code (1 sign, 2 exponent bits with bias 1, 1
 *               mantissa bit; exponent 0 holds 0 and 0.5; no infinities or
 *               NaN; max 6) times the e8m0 scale of its block of 32
 *               consecutive elements along D (8 exponent bits, bias 127, no
 *               sign or mantissa: 2^(c - 127); 0xFF is NaN).  Two elements per
 *               byte, element 2i in bits 0..3 and element 2i+1 in bits 4..7;
 *               scale bytes [rows, H, D/32] for q and [keys, D/32] for k.
 *               "[sglang] logits를 쓰지 않는 top-k", section 1, names an
 *               mxf4 scoring path with 64-byte keys (128 elements) but not the
 *               scale layout; one scale per 32 elements is the OCP block size.
 *
 * Build: plain C11, no fast-math and no FMA contraction (-ffp-contract=off),
 * so the fp64 results are the same on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 1, ORC_E4M3 = 2, ORC_MXFP4 = 3 };

/* ---------------------------------------------------------------- decoders */

double orc_e4m3_to_f64(uint32_t code) {
    const int sign = (code >> 7) & 1;
    const int expo = (code >> 3) & 0xF;
    const int mant = code & 0x7;
    double v;
    if (expo == 0xF && mant == 0x7) return NAN;
    if (expo == 0)
        v = ldexp((double)mant / 8.0, 1 - 7);          /* subnormal */
    else
        v = ldexp(1.0 + (double)mant / 8.0, expo - 7);  /* normal */
    return sign ? -v : v;
}

double orc_bf16_to_f64(uint32_t code) {
    const int sign = (code >> 15) & 1;
    const int expo = (code >> 7) & 0xFF;
    const int mant = code & 0x7F;
    double v;
    if (expo == 0xFF) v = mant ? NAN : INFINITY;
    else if (expo == 0) v = ldexp((double)mant / 128.0, 1 - 127);
    else v = ldexp(1.0 + (double)mant / 128.0, expo - 127);
    return sign ? -v : v;
}

double orc_e2m1_to_f64(uint32_t code) {
    const int sign = (code >> 3) & 1;
    const int expo = (code >> 1) & 0x3;
    const int mant = code & 0x1;
    double v;
    if (expo == 0)
        v = ldexp((double)mant / 2.0, 1 - 1);          /* subnormal: 0 or 0.5 */
    else
        v = ldexp(1.0 + (double)mant / 2.0, expo - 1);  /* normal */
    return sign ? -v : v;
}

double orc_e8m0_to_f64(uint32_t code) {
    if ((code & 0xFF) == 0xFF) return NAN;
    return ldexp(1.0, (int)(code & 0xFF) - 127);
}

/* Every code of the formats decoded once by the functions above. */
static double tab_e4m3[256];
static double tab_bf16[65536];
static double tab_e2m1[16];
static double tab_e8m0[256];
static pthread_once_t tab_once = PTHREAD_ONCE_INIT;

static void fill_tables(void) {
    for (uint32_t c = 0; c < 256; ++c) tab_e4m3[c] = orc_e4m3_to_f64(c);
    for (uint32_t c = 0; c < 65536; ++c) tab_bf16[c] = orc_bf16_to_f64(c);
    for (uint32_t c = 0; c < 16; ++c) tab_e2m1[c] = orc_e2m1_to_f64(c);
    for (uint32_t c = 0; c < 256; ++c) tab_e8m0[c] = orc_e8m0_to_f64(c);
}

/* Element i of a row-major array of the format (flat index over [..., D]);
 * sf holds the MXFP4 block scales ([..., D/32], so block i / 32). */
static double decode(const void* base, const uint8_t* sf, long long i, int dtype) {
    pthread_once(&tab_once, fill_tables);
    if (dtype == ORC_E4M3) return tab_e4m3[((const uint8_t*)base)[i]];
    if (dtype == ORC_MXFP4) {
        const uint32_t byte = ((const uint8_t*)base)[i >> 1];
        const uint32_t code = (i & 1) ? (byte >> 4) : (byte & 0xF);
        return tab_e2m1[code] * tab_e8m0[sf[i / 32]];
    }
    return tab_bf16[((const uint16_t*)base)[i]];
}

/* ------------------------------------------------------------------ scores */

/* Scores of one row over its visible keys, out[j - ks] for ks <= j < ke.
 * q_sf / k_sf: the block scales of MXFP4 inputs (NULL for the other formats). */
int orc_scores_row(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                   int dtype, const float* k_scale, const float* w, int H, int D,
                   long long r, long long ks, long long ke, double* out) {
    if (ke <= ks) return 0;
    double* qd = (double*)malloc(sizeof(double) * (size_t)H * D);
    double* kd = (double*)malloc(sizeof(double) * (size_t)D);
    double* dot = (double*)malloc(sizeof(double) * (size_t)H);
    if (!qd || !kd || !dot) { free(qd); free(kd); free(dot); return -1; }
    /* qd[d*H + h] = q[r,h,d]: heads contiguous for the inner loop below */
    for (int h = 0; h < H; ++h)
        for (int d = 0; d < D; ++d)
            qd[(size_t)d * H + h] = decode(q, q_sf, (r * (long long)H + h) * D + d, dtype);
    for (long long j = ks; j < ke; ++j) {
        for (int d = 0; d < D; ++d) kd[d] = decode(k, k_sf, j * (long long)D + d, dtype);
        /* q[r,h,:] . k[j,:], summed over d in ascending order for every head */
        for (int h = 0; h < H; ++h) dot[h] = 0.0;
        for (int d = 0; d < D; ++d)
            for (int h = 0; h < H; ++h) dot[h] += qd[(size_t)d * H + h] * kd[d];
        double s = 0.0;
        for (int h = 0; h < H; ++h) {
            const double relu = dot[h] > 0.0 ? dot[h] : 0.0;
            s += (double)w[r * H + h] * relu;
        }
        out[j - ks] = (double)k_scale[j] * s;
    }
    free(qd); free(kd); free(dot);
    return 0;
}

/* --------------------------------------------------------------- selection */

typedef struct { double s; long long j; } orc_item;

/* score descending, then key index ascending */
static int by_score_then_index(const void* a, const void* b) {
    const orc_item* x = (const orc_item*)a;
    const orc_item* y = (const orc_item*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int by_index(const void* a, const void* b) {
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Top-k of s[0..n) (row-relative indices), written ascending into out[topk]
 * and padded with -1.  A full sort: plain and slow on purpose. */
int orc_select_row(const double* s, long long n, int topk, int32_t* out) {
    if (n < 0) n = 0;
    const long long take = n < topk ? n : topk;
    orc_item* it = (orc_item*)malloc(sizeof(orc_item) * (size_t)(n > 0 ? n : 1));
    if (!it) return -1;
    for (long long j = 0; j < n; ++j) { it[j].s = s[j]; it[j].j = j; }
    qsort(it, (size_t)n, sizeof(orc_item), by_score_then_index);
    for (long long i = 0; i < take; ++i) out[i] = (int32_t)it[i].j;
    qsort(out, (size_t)take, sizeof(int32_t), by_index);
    for (long long i = take; i < topk; ++i) out[i] = -1;
    free(it);
    return 0;
}

/* ------------------------------------------------------ row-parallel driver */

typedef struct {
    /* indexer inputs (score_topk) */
    const void* q; const uint8_t* q_sf; const void* k; const uint8_t* k_sf; int dtype;
    const float* k_scale; const float* w;
    int H, D;
    /* given scores (topk_from_scores) */
    const float* scores; long long stride;
    /* common */
    const int32_t* ks; const int32_t* ke; const int32_t* rows; int nrows; int topk;
    int32_t* out;          /* [nrows, topk] */
    double* out_scores;    /* optional [nrows, score_stride] */
    long long score_stride;
    int next; pthread_mutex_t lock; int err;
} orc_job;

static int grab(orc_job* J) {
    pthread_mutex_lock(&J->lock);
    const int i = J->next < J->nrows ? J->next++ : -1;
    pthread_mutex_unlock(&J->lock);
    return i;
}

static void* worker(void* arg) {
    orc_job* J = (orc_job*)arg;
    for (int i = grab(J); i >= 0; i = grab(J)) {
        const long long r = J->rows[i];
        const long long ks = J->ks[r], ke = J->ke[r];
        const long long n = ke > ks ? ke - ks : 0;
        double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!s) { J->err = -1; continue; }
        int e;
        if (J->scores) {
            for (long long j = 0; j < n; ++j) s[j] = (double)J->scores[r * J->stride + ks + j];
            e = 0;
        } else {
            e = orc_scores_row(J->q, J->q_sf, J->k, J->k_sf, J->dtype, J->k_scale, J->w, J->H,
                               J->D, r, ks, ke, s);
        }
        if (!e && J->out) e = orc_select_row(s, n, J->topk, J->out + (long long)i * J->topk);
        if (!e && J->out_scores)
            for (long long j = 0; j < n && j < J->score_stride; ++j)
                J->out_scores[(long long)i * J->score_stride + j] = s[j];
        if (e) J->err = e;
        free(s);
    }
    return NULL;
}

static int run(orc_job* J, int nthreads) {
    J->next = 0; J->err = 0;
    pthread_mutex_init(&J->lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t th[1024];
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, worker, J) == 0) ++started;
    worker(J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J->lock);
    return J->err;
}

/* Exact top-k of the indexer scores for the listed rows.
 * out[i, :] belongs to rows[i]; out_scores (optional) receives the fp64 scores
 * of rows[i] at [i, 0 .. ke-ks) with row pitch score_stride. */
int orc_score_topk(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                   int dtype, const float* k_scale, const float* w, const int32_t* ks,
                   const int32_t* ke, int H, int D, const int32_t* rows, int nrows, int topk,
                   int32_t* out, double* out_scores, long long score_stride, int nthreads) {
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.q_sf = q_sf; J.k = k; J.k_sf = k_sf; J.dtype = dtype; J.k_scale = k_scale; J.w = w; J.H = H; J.D = D;
    J.ks = ks; J.ke = ke; J.rows = rows; J.nrows = nrows; J.topk = topk; J.out = out;
    J.out_scores = out_scores; J.score_stride = score_stride;
    return run(&J, nthreads);
}

/* Exact top-k of given fp32 scores [*, stride] for the listed rows. */
int orc_topk_from_scores(const float* scores, long long stride, const int32_t* ks,
                         const int32_t* ke, const int32_t* rows, int nrows, int topk,
                         int32_t* out, int nthreads) {
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.scores = scores; J.stride = stride;
    J.ks = ks; J.ke = ke; J.rows = rows; J.nrows = nrows; J.topk = topk; J.out = out;
    return run(&J, nthreads);
}

/* Page-table transform of idx [rows, topk] into out (same shape).
 * table is [table_rows, table_stride]; row r uses table row row_map[r]
 * (row_map NULL: row r).  A position whose page lies outside the table row,
 * or whose table row lies outside [0, table_rows), has no physical slot: it
 * becomes -1 and is counted.  Returns that count, or -1 for bad arguments. */
long long orc_page_transform(const int32_t* idx, int rows, int topk, const int32_t* table,
                             long long table_rows, long long table_stride,
                             const int32_t* row_map, int page_size, int32_t* out) {
    if (rows < 0 || topk < 0 || page_size < 1 || table_stride < 0 || table_rows < 0) return -1;
    long long bad = 0;
    for (int r = 0; r < rows; ++r) {
        const long long t = row_map ? (long long)row_map[r] : (long long)r;
        const int row_ok = t >= 0 && t < table_rows;
        for (int i = 0; i < topk; ++i) {
            const long long p = idx[(long long)r * topk + i];
            long long v = p;
            if (p >= 0) {
                const long long page = p / page_size;
                if (row_ok && page < table_stride) {
                    v = (long long)table[t * table_stride + page] * page_size + p % page_size;
                } else {
                    v = -1;
                    ++bad;
                }
            }
            out[(long long)r * topk + i] = (int32_t)v;
        }
    }
    return bad;
}
