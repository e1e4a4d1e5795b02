/*
 * Row-softmax ORACLE -- test infrastructure, not part of the product.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference arm may load this library.  The product path (the CUDA library
 * under memory_bound_row_gb300/) never calls it, and it shares no code,
 * header, table or constant with that path.
 *
 * What it computes is the plain definition of the row softmax, in double
 * precision, one row at a time:
 *
 *     m_r    = max_k x[r][k]
 *     y[r][j] = exp(x[r][j] - m_r) / sum_k exp(x[r][k] - m_r)
 *
 * This is the computation of the fused softmax kernel in
 * "stanleyjacob.dev: Triton", Part II, "Worked example: fused softmax"
 * (load the row, subtract its max, exponentiate, sum, divide, store), and of
 * the "Safe Softmax Pattern" and "Reference Kernel: Softmax" sections of the
 * Hugging Face "triton-kernels" skill page.  Subtracting the max does not
 * change the value in exact arithmetic; it only keeps exp() in range.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - inputs are decoded exactly from their stored format (fp32, fp16, bf16,
 *    or fp64 for hand-made cases) before any arithmetic;
 *  - IEEE semantics are kept as the formula gives them: a row that is all
 *    -inf gives NaN everywhere ((-inf) - (-inf) is NaN); a NaN anywhere in a
 *    row makes the sum NaN and so the whole row NaN; +inf gives NaN through
 *    inf - inf;
 *  - output encoding to fp16 / bf16 is round-to-nearest, ties-to-even, done
 *    directly from the double result (no intermediate fp32 rounding).
 *
 * It also holds the plain definitions of RMSNorm and LayerNorm, the row
 * softmax over a prefix of every row (a causal attention mask: row r keeps its
 * first L_r elements, the rest is treated as -inf and never read), and the
 * three steps of the softmax of a row split by columns into shards (partial
 * pairs, their merge, the finish; end of file).
 *
 * Parity pins for this file live in tests/test_oracle_pins.py,
 * tests/test_oracle_norm_pins.py, tests/test_oracle_prefix_pins.py and
 * tests/test_oracle_split_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The oracle's own storage-format codes. */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };

/* ---------------------------------------------------------------------------
 * Exact decoding of the stored formats.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * bfloat16: the upper 16 bits of an IEEE binary32 value (1, 8 (bias 127), 7).
 * ------------------------------------------------------------------------- */
double orc_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0x1f) {
        v = f ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    } else {
        v = ldexp((double)(f + 1024), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

double orc_decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0xff) {
        v = f ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)f, -133);             /* f * 2^(1-127-7) */
    } else {
        v = ldexp((double)(f + 128), e - 134);  /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* ---------------------------------------------------------------------------
 * Round-to-nearest-even encoding of a double into a small binary format with
 * `eb` exponent bits and `mb` fraction bits (binary16: 5/10, bfloat16: 8/7).
 * The value is scaled by the spacing of representable numbers at its
 * magnitude, rounded to an integer with ties to even, and the integer is laid
 * into the exponent/fraction fields; a carry out of the fraction moves into
 * the exponent field by itself because the encoding is monotonic.
 * ------------------------------------------------------------------------- */
static uint16_t orc_encode_small(double v, int eb, int mb)
{
    const int bias = (1 << (eb - 1)) - 1;
    const int emin = 1 - bias;                    /* smallest normal exponent */
    const uint32_t inf_bits = ((1u << eb) - 1u) << mb;
    uint32_t sign = signbit(v) ? (1u << (eb + mb)) : 0u;
    if (isnan(v)) return (uint16_t)(inf_bits | (1u << (mb - 1)));   /* quiet NaN */
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | inf_bits);
    if (a == 0.0) return (uint16_t)sign;

    int k;
    frexp(a, &k);                 /* a = f * 2^k, f in [0.5, 1): exponent k-1 */
    int e = k - 1;
    if (e < emin) e = emin;       /* subnormal range shares the min spacing */
    double q = ldexp(1.0, e - mb);/* spacing at this magnitude */
    double r = rint(a / q);       /* a/q is exact (power-of-two divide)       */
    uint32_t bits;
    if (r < ldexp(1.0, mb)) {
        bits = (uint32_t)r;                        /* subnormal (e == emin) */
    } else {
        bits = ((uint32_t)(e + bias) << mb) + (uint32_t)(r - ldexp(1.0, mb));
    }
    if (bits >= inf_bits) bits = inf_bits;         /* overflow to infinity */
    return (uint16_t)(sign | bits);
}

uint16_t orc_encode_f16(double v) { return orc_encode_small(v, 5, 10); }
uint16_t orc_encode_bf16(double v) { return orc_encode_small(v, 8, 7); }

static double orc_load(const void* base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float*)base)[idx];
    case ORC_F16: return orc_decode_f16(((const uint16_t*)base)[idx]);
    case ORC_BF16: return orc_decode_bf16(((const uint16_t*)base)[idx]);
    case ORC_F64: return ((const double*)base)[idx];
    default: return NAN;
    }
}

static void orc_store(void* base, int dtype, int64_t idx, double v)
{
    switch (dtype) {
    case ORC_F32: ((float*)base)[idx] = (float)v; break;
    case ORC_F16: ((uint16_t*)base)[idx] = orc_encode_f16(v); break;
    case ORC_BF16: ((uint16_t*)base)[idx] = orc_encode_bf16(v); break;
    case ORC_F64: ((double*)base)[idx] = v; break;
    default: break;
    }
}

/* Batch helpers for the pins: decode n stored values to double, or encode n
 * doubles into a stored format. */
void orc_decode_array(const void* x, int dtype, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_load(x, dtype, i);
}

void orc_encode_array(const double* v, int dtype, int64_t n, void* out)
{
    for (int64_t i = 0; i < n; ++i) orc_store(out, dtype, i, v[i]);
}

/* One row of the definition.  `xr` holds N decoded values, `yr` receives N
 * doubles.  The max starts at -inf and a NaN never wins the comparison, so a
 * NaN input reaches the sum through exp(NaN - m) and spreads to the row. */
static void orc_row(const double* xr, int64_t N, double* yr)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (xr[j] > m) m = xr[j];
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j)
        s += exp(xr[j] - m);
    for (int64_t j = 0; j < N; ++j)
        yr[j] = exp(xr[j] - m) / s;
}

static int orc_check(int dtype, int64_t M, int64_t N, int64_t ldx, int64_t ldy)
{
    if (dtype < ORC_F32 || dtype > ORC_F64) return 1;
    if (M < 0 || N < 0) return 1;
    if (M > 0 && N > 0 && (ldx < N || ldy < N)) return 1;
    return 0;
}

/* y (double, row stride ldy) = softmax of each of the M rows of x (stored
 * format `dtype`, row stride ldx, unit column stride).  Returns 0 on success,
 * 1 on bad arguments, 2 when scratch memory cannot be had. */
int orc_softmax_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx,
                    double* y, int64_t ldy)
{
    if (orc_check(dtype, M, N, ldx, ldy)) return 1;
    if (M == 0 || N == 0) return 0;
    double* xr = (double*)malloc((size_t)N * sizeof(double));
    if (!xr) return 2;
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < N; ++j) xr[j] = orc_load(x, dtype, r * ldx + j);
        orc_row(xr, N, y + r * ldy);
    }
    free(xr);
    return 0;
}

/* ---------------------------------------------------------------------------
 * The row softmax under a causal mask, the attention-score example of the
 * mohakchugh.is-a.dev post ("How Flash Attention Uses Triton": a softmax that
 * skips the fully masked causal region).  For scores [B, H, S_q, S_k] viewed
 * as (B*H*S_q) x S_k rows, row r is query position q = r mod S_q and may see
 * keys k <= q + (S_k - S_q).  In general, with period P > 0 and diagonal
 * offset D, row r keeps
 *     L_r = min(N, max(0, (r mod P) + 1 + D))
 * elements; the masked ones are -inf by definition, so
 *     y[r][j] = exp(x[r][j] - m_r) / sum_{k < L_r} exp(x[r][k] - m_r)  (j < L_r)
 *     y[r][j] = 0                                                      (j >= L_r)
 * with m_r the max of the kept elements; L_r = 0 is an all -inf row: NaN.
 * The masked elements are never read (they may hold anything).
 * ------------------------------------------------------------------------- */
int64_t orc_prefix_len(int64_t r, int64_t N, int64_t period, int64_t offset)
{
    int64_t L = r % period + 1 + offset;
    if (L < 0) L = 0;
    if (L > N) L = N;
    return L;
}

/* Rows r = row0 .. row0 + M - 1 of the masked tensor (x and y point at row row0). */
int orc_softmax_prefix_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx, int64_t row0,
                           int64_t period, int64_t offset, double* y, int64_t ldy)
{
    if (orc_check(dtype, M, N, ldx, ldy) || period <= 0 || row0 < 0) return 1;
    if (M == 0 || N == 0) return 0;
    double* xr = (double*)malloc((size_t)N * sizeof(double));
    if (!xr) return 2;
    for (int64_t r = 0; r < M; ++r) {
        const int64_t L = orc_prefix_len(row0 + r, N, period, offset);
        double* yr = y + r * ldy;
        if (L == 0) {
            for (int64_t j = 0; j < N; ++j) yr[j] = NAN;
            continue;
        }
        for (int64_t j = 0; j < L; ++j) xr[j] = orc_load(x, dtype, r * ldx + j);
        orc_row(xr, L, yr);
        for (int64_t j = L; j < N; ++j) yr[j] = 0.0;
    }
    free(xr);
    return 0;
}

/* Same definition, but the result is encoded into the stored format `dtype`
 * (the output format equals the input format) and the rows are split into
 * contiguous blocks over `nthreads` POSIX threads (nthreads <= 1: the calling
 * thread does all rows).  Used for the timed CPU baseline. */
typedef struct {
    const void* x; void* y; int dtype;
    int64_t r0, r1, N, ldx, ldy;
    int status;
} orc_job;

static void* orc_worker(void* p)
{
    orc_job* jb = (orc_job*)p;
    double* buf = (double*)malloc((size_t)jb->N * 2 * sizeof(double));
    if (!buf) { jb->status = 2; return NULL; }
    double* xr = buf;
    double* yr = buf + jb->N;
    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        for (int64_t j = 0; j < jb->N; ++j) xr[j] = orc_load(jb->x, jb->dtype, r * jb->ldx + j);
        orc_row(xr, jb->N, yr);
        for (int64_t j = 0; j < jb->N; ++j) orc_store(jb->y, jb->dtype, r * jb->ldy + j, yr[j]);
    }
    free(buf);
    jb->status = 0;
    return NULL;
}

int orc_softmax_store(const void* x, void* y, int dtype, int64_t M, int64_t N,
                      int64_t ldx, int64_t ldy, int nthreads)
{
    if (orc_check(dtype, M, N, ldx, ldy)) return 1;
    if (M == 0 || N == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > M) nthreads = (int)M;
    orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 2; }
    int64_t per = M / nthreads, extra = M % nthreads, r = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t cnt = per + (t < extra ? 1 : 0);
        jobs[t] = (orc_job){x, y, dtype, r, r + cnt, N, ldx, ldy, 2};
        r += cnt;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, orc_worker, &jobs[t]) != 0) break;
        started = t;
    }
    orc_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    /* rows of threads that could not be started are done here */
    for (int t = started + 1; t < nthreads; ++t) orc_worker(&jobs[t]);
    int status = 0;
    for (int t = 0; t < nthreads; ++t) if (jobs[t].status) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* ---------------------------------------------------------------------------
 * Row normalisations (the next operation on the same row engine).
 *
 * RMSNorm, as the "Reference Kernel: RMSNorm" of the Hugging Face
 * "triton-kernels" skill page computes it:
 *     r_r = sqrt( (1/N) sum_k x[r][k]^2 + eps ),   y[r][j] = x[r][j] / r_r * w[j]
 * LayerNorm (the pages name it, next to softmax, as a memory-bound row kernel,
 * without a formula; the plain definition is taken: population variance,
 * eps inside the square root, optional elementwise weight and bias):
 *     mu_r = (1/N) sum_k x[r][k],   var_r = (1/N) sum_k (x[r][k] - mu_r)^2,
 *     y[r][j] = (x[r][j] - mu_r) / sqrt(var_r + eps) * w[j] + b[j]
 * w (and b) are N stored values of the same format as x; a NULL w means 1,
 * a NULL b means 0.  Results are double; sums are plain recursive sums.
 * ------------------------------------------------------------------------- */
static double orc_vec(const void* v, int dtype, int64_t j, double dflt)
{
    return v ? orc_load(v, dtype, j) : dflt;
}

int orc_rmsnorm_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx, const void* w, double eps,
                    double* y, int64_t ldy)
{
    if (orc_check(dtype, M, N, ldx, ldy)) return 1;
    for (int64_t r = 0; r < M; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double v = orc_load(x, dtype, r * ldx + j);
            ss += v * v;
        }
        const double rms = sqrt(ss / (double)N + eps);
        for (int64_t j = 0; j < N; ++j)
            y[r * ldy + j] = orc_load(x, dtype, r * ldx + j) / rms * orc_vec(w, dtype, j, 1.0);
    }
    return 0;
}

int orc_layernorm_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx, const void* w, const void* b,
                      double eps, double* y, int64_t ldy)
{
    if (orc_check(dtype, M, N, ldx, ldy)) return 1;
    for (int64_t r = 0; r < M; ++r) {
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += orc_load(x, dtype, r * ldx + j);
        const double mu = s / (double)N;
        double d = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double v = orc_load(x, dtype, r * ldx + j) - mu;
            d += v * v;
        }
        const double sd = sqrt(d / (double)N + eps);
        for (int64_t j = 0; j < N; ++j)
            y[r * ldy + j] = (orc_load(x, dtype, r * ldx + j) - mu) / sd * orc_vec(w, dtype, j, 1.0) +
                             orc_vec(b, dtype, j, 0.0);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * A row split by columns into shards (the vocabulary-parallel softmax, where
 * each device holds a block of columns of every row).  The online normaliser
 * of the mohakchugh.is-a.dev post ("How Flash Attention Uses Triton") carries
 * a running pair (m, l) -- the max seen so far and the sum of exp(x - m) over
 * the values seen -- and combines two pairs as
 *     m = max(m1, m2),   l = l1 exp(m1 - m) + l2 exp(m2 - m),
 * starting from (-inf, 0).  Here:
 *   partial: each shard reduces its columns of row r to (m, l) with
 *            m = max_j x_j, l = sum_j exp(x_j - m);
 *   merge:   the R shards' pairs of a row are combined with the rule above,
 *            shard 0 first;
 *   finish:  each shard writes y_j = exp(x_j - m) / l for its columns with the
 *            merged pair.
 * In exact arithmetic this is the row softmax of the whole row, however the
 * columns are split.  Readings where the recurrence leaves a case open: a
 * shard with no column, or whose entries are all -inf, contributes the
 * starting pair (-inf, 0) (it holds no mass of the row; the plain formula's
 * (-inf) - (-inf) would otherwise turn a well-defined row into NaN); a pair
 * whose max is -inf enters a merge with weight 0 times its sum, so a NaN sum
 * still reaches the result; NaN entries never win the max and make the sum
 * NaN; the finish of a row whose merged max is -inf is NaN (the whole row is
 * -inf: the plain formula's NaN row).
 * Pairs are stored as two doubles (m, l) per row.
 * ------------------------------------------------------------------------- */
static void orc_partial_row(const void* x, int dtype, int64_t off, int64_t N, double* m_out, double* l_out)
{
    double m = -INFINITY;
    int any_nan = 0;
    for (int64_t j = 0; j < N; ++j) {
        const double v = orc_load(x, dtype, off + j);
        if (v > m) m = v;
        if (v != v) any_nan = 1;
    }
    double l = 0.0;
    if (m == -INFINITY) {
        l = any_nan ? NAN : 0.0;  /* all -inf (or empty): the starting pair */
    } else {
        for (int64_t j = 0; j < N; ++j) l += exp(orc_load(x, dtype, off + j) - m);
    }
    *m_out = m;
    *l_out = l;
}

/* ml[2 r] = m_r, ml[2 r + 1] = l_r for the M rows of x (N columns, stride ldx). */
int orc_softmax_partial_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx, double* ml)
{
    if (orc_check(dtype, M, N, ldx, N) || (M > 0 && ldx < N)) return 1;
    for (int64_t r = 0; r < M; ++r) orc_partial_row(x, dtype, r * ldx, N, &ml[2 * r], &ml[2 * r + 1]);
    return 0;
}

/* One step of the online normaliser: (m, l) absorbs (m2, l2). */
static void orc_absorb(double* m, double* l, double m2, double l2)
{
    const double mn = m2 > *m ? m2 : *m;
    const double a = *m == -INFINITY ? *l * 0.0 : *l * exp(*m - mn);
    const double b = m2 == -INFINITY ? l2 * 0.0 : l2 * exp(m2 - mn);
    *m = mn;
    *l = a + b;
}

/* ml_in: R x M pairs, shard-major (pair of shard s, row r at ml_in[2 (s M + r)]);
 * ml_out: the M merged pairs. */
int orc_merge_pairs_f64(const double* ml_in, int64_t R, int64_t M, double* ml_out)
{
    if (R < 0 || M < 0) return 1;
    for (int64_t r = 0; r < M; ++r) {
        double m = -INFINITY, l = 0.0;
        for (int64_t s = 0; s < R; ++s) orc_absorb(&m, &l, ml_in[2 * (s * M + r)], ml_in[2 * (s * M + r) + 1]);
        ml_out[2 * r] = m;
        ml_out[2 * r + 1] = l;
    }
    return 0;
}

/* y[r][j] = exp(x[r][j] - m_r) / l_r with the merged pairs ml (two doubles a row). */
int orc_softmax_finish_f64(const void* x, int dtype, int64_t M, int64_t N, int64_t ldx, const double* ml,
                           double* y, int64_t ldy)
{
    if (orc_check(dtype, M, N, ldx, ldy)) return 1;
    for (int64_t r = 0; r < M; ++r) {
        const double m = ml[2 * r], l = ml[2 * r + 1];
        for (int64_t j = 0; j < N; ++j) y[r * ldy + j] = exp(orc_load(x, dtype, r * ldx + j) - m) / l;
    }
    return 0;
}
