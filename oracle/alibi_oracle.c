/*
 * fp64 CPU oracle for causal multi-head attention with ALiBi linear biases.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: it is used by tests/, by the smoke check and by the benchmark's
 * CPU-baseline leg. It shares no code, header, table or constant with the CUDA
 * library.
 *
 * Everything is the plain definition, one query row at a time, in fp64 from the
 * exact input values (bf16 and fp32 inputs are passed widened to fp32, which
 * holds both exactly):
 *
 *   a_ij = (q_i . k_j) / sqrt(d)                      scaled content score
 *   x_ij = a_ij - m_h * D_ij                          ALiBi bias, D_ij = i - j
 *   keys j > i are excluded (causal mask)
 *   M_i = max_j x_ij, Z_i = sum_j exp(x_ij - M_i)     stable softmax
 *   w_ij = exp(x_ij - M_i) / Z_i,  o_i = sum_j w_ij v_j,  LSE_i = M_i + ln Z_i
 *
 * Sources (page title, then section / equation):
 *  - "When Attention Goes Blind: Numerical Failure in ALiBi Positional
 *    Encodings" (arXiv 2608.03994): sec. 3.1 eq. 1-3 (A = QK^T/sqrt(d_k),
 *    B = -m D); sec. 3.2 eq. 4 and the blindness distance; sec. 3.4 (clamping,
 *    log-scaled distances, soft capping); App. A Table 4; App. B.1 (stable
 *    softmax).
 *  - "ALiBi: Attention with Linear Biases" (abhik.ai): "From distance to a
 *    normalized weight" (distance i - j for j <= i, future keys masked, weights
 *    sum to one); "Different heads, different distance penalties" (slope
 *    schedule for power-of-two and other head counts); the KV-cache paragraph
 *    after the full-sequence example (true sequence positions).
 *  - "ALiBi and Relative Position Bias" (quantmemo.com), "The mechanics" and
 *    "ALiBi in Attention: Complete Implementation" (mbrenndoerfer.com): the
 *    symmetric |i - j| distance used when causal == 0.
 *
 * Every function is pinned by the tests in tests/test_oracle_pins.py against
 * values the pages print, closed forms, invariants and brute force; the
 * backward pass (oracle_attn_bwd) by tests/test_oracle_bwd_pins.py against
 * finite differences of the forward and gradient identities.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

/* Variant flags: the mitigations of "When Attention Goes Blind", sec. 3.4. */
#define ORACLE_CLAMP 1   /* B* = max(B, c_clamp)          ("Clamping")          */
#define ORACLE_LOGDIST 2 /* D* = log(D + 1)               ("Log-scaled Distances") */
#define ORACLE_SOFTCAP 4 /* A* = z * tanh(A / z)          ("Soft Capping")      */

/* ------------------------------------------------------------------ slopes */

/* Largest power of two c <= H. */
static int pow2_floor(int H)
{
    int c = 1;
    while (c <= H / 2) c *= 2;
    return c;
}

/*
 * Slope of head h as 2^(-num/den).
 * "ALiBi: Attention with Linear Biases", "Different heads, different distance
 * penalties": for a power-of-two head count H the schedule is
 * m_h = 2^(-8(h+1)/H), h = 0..H-1 (ratio 2^(-8/H)). For other H, keep the
 * schedule of the largest smaller power of two c, then append alternating
 * entries (the 1st, 3rd, 5th, ...) of the schedule for 2c heads; the six-head
 * table on that page fixes the order (0.25, 0.0625, 0.015625, 0.00390625, 0.5,
 * 0.125).
 */
int oracle_slope_exponent(int H, int h, int *num, int *den)
{
    if (H < 1 || h < 0 || h >= H || !num || !den) return ORACLE_EINVAL;
    int c = pow2_floor(H);
    if (h < c) {
        *num = 8 * (h + 1);
        *den = c;
    } else {
        int t = h - c;           /* t-th appended head                      */
        *num = 8 * (2 * t + 1);  /* entry 2t (0-based) of the 2c schedule    */
        *den = 2 * c;
    }
    return ORACLE_OK;
}

/* fp64 slopes (the schedule evaluated in long double, then rounded to double). */
int oracle_slopes(int H, double *m)
{
    if (H < 1 || !m) return ORACLE_EINVAL;
    for (int h = 0; h < H; ++h) {
        int num, den;
        oracle_slope_exponent(H, h, &num, &den);
        m[h] = (double)exp2l(-(long double)num / (long double)den);
    }
    return ORACLE_OK;
}

/* Slopes rounded once to fp32 (round to nearest even) from long double. */
int oracle_slopes_f32(int H, float *m)
{
    if (H < 1 || !m) return ORACLE_EINVAL;
    for (int h = 0; h < H; ++h) {
        int num, den;
        oracle_slope_exponent(H, h, &num, &den);
        m[h] = (float)exp2l(-(long double)num / (long double)den);
    }
    return ORACLE_OK;
}

/*
 * Slopes chosen from target blindness distances ("When Attention Goes Blind",
 * sec. 3.4 "Robust Slopes"; sec. 4.2 "Positional Encoding Configurations";
 * sec. 4.3 for the log-distance adaptation; App. F Table 8 for the schedules).
 * The targets run geometrically from delta_first (head 0) to delta_last
 * (head H - 1):
 *   delta_h = delta_first * (delta_last / delta_first)^(h / (H - 1)),
 * and each slope puts the zero-logit crossing exactly at its target, i.e.
 * solves -m delta_h = tau (linear distances) or -m log(delta_h + 1) = tau
 * (log-scaled distances, the E+L combination). H = 1 takes delta_first.
 */
int oracle_slopes_explicit(int H, double delta_first, double delta_last, double tau, int log_distance, double *m)
{
    if (H < 1 || !m || !(delta_first > 0.0) || !(delta_last > 0.0) || !(tau < 0.0)) return ORACLE_EINVAL;
    if (!isfinite(delta_first) || !isfinite(delta_last) || !isfinite(tau)) return ORACLE_EINVAL;
    for (int h = 0; h < H; ++h) {
        double t = H > 1 ? (double)h / (double)(H - 1) : 0.0;
        double delta = delta_first * pow(delta_last / delta_first, t);
        double dist = log_distance ? log(delta + 1.0) : delta;
        m[h] = -tau / dist;
    }
    return ORACLE_OK;
}

/* -------------------------------------------------------------------- bias */

/*
 * ALiBi bias of query i and key j for slope m.
 * causal != 0: -m (i - j) for j <= i, -inf for j > i ("When Attention Goes
 * Blind" eq. 2-3 with the causal mask of "ALiBi: Attention with Linear Biases").
 * causal == 0: -m |i - j| ("ALiBi and Relative Position Bias", "The mechanics").
 * Variants: ORACLE_LOGDIST replaces the distance D by log(D + 1);
 * ORACLE_CLAMP replaces the bias B by max(B, c_clamp).
 */
double oracle_bias_ex(double m, long i, long j, int causal, int variant, double c_clamp)
{
    if (causal && j > i) return -INFINITY;
    double D = (double)(i >= j ? i - j : j - i);
    if (variant & ORACLE_LOGDIST) D = log(D + 1.0);
    double B = -m * D;
    if ((variant & ORACLE_CLAMP) && B < c_clamp) B = c_clamp;
    return B;
}

double oracle_bias(double m, long i, long j, int causal)
{
    return oracle_bias_ex(m, i, j, causal, 0, 0.0);
}

/* Soft capping of a content logit: z tanh(A / z) ("When Attention Goes Blind", sec. 3.4). */
static double softcap(double a, double z)
{
    return z * tanh(a / z);
}

/* --------------------------------------------------------------- threading */

typedef void (*row_fn)(void *ctx, long r, double *scratch);

typedef struct {
    row_fn fn;
    void *ctx;
    long nrows;
    int tid, nthreads;
    long scratch_len;
    int status;
} worker_t;

static void *worker_main(void *arg)
{
    worker_t *w = (worker_t *)arg;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(w->scratch_len > 0 ? w->scratch_len : 1));
    if (!scratch) {
        w->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (long r = w->tid; r < w->nrows; r += w->nthreads) w->fn(w->ctx, r, scratch);
    free(scratch);
    w->status = ORACLE_OK;
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run_rows(row_fn fn, void *ctx, long nrows, long scratch_len, int nthreads)
{
    int T = resolve_threads(nthreads);
    if (T > nrows) T = (int)(nrows > 0 ? nrows : 1);
    worker_t *ws = (worker_t *)calloc((size_t)T, sizeof(worker_t));
    pthread_t *th = (pthread_t *)calloc((size_t)T, sizeof(pthread_t));
    if (!ws || !th) {
        free(ws);
        free(th);
        return ORACLE_ENOMEM;
    }
    int status = ORACLE_OK;
    for (int t = 0; t < T; ++t) {
        ws[t] = (worker_t){fn, ctx, nrows, t, T, scratch_len, ORACLE_OK};
        if (T == 1) {
            worker_main(&ws[t]);
        } else if (pthread_create(&th[t], NULL, worker_main, &ws[t]) != 0) {
            ws[t].status = ORACLE_ENOMEM;
            th[t] = 0;
        }
    }
    if (T > 1)
        for (int t = 0; t < T; ++t)
            if (th[t]) pthread_join(th[t], NULL);
    for (int t = 0; t < T; ++t)
        if (ws[t].status != ORACLE_OK) status = ws[t].status;
    free(ws);
    free(th);
    return status;
}

/* ------------------------------------------------------- attention (rows) */

typedef struct {
    const float *q, *k, *v;
    const double *m;
    int B, H, N, d, causal, variant;
    double c_clamp, z_cap;
    const long *rows; /* flat (b*H + h)*N + i, or NULL for all rows in order */
    double *out, *lse, *w;
} attn_ctx;

/* Scaled content score a_ij = q_i . k_j / sqrt(d) ("When Attention Goes Blind" eq. 1). */
static double content_score(const float *qi, const float *kj, int d)
{
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += (double)qi[t] * (double)kj[t];
    return s / sqrt((double)d);
}

static void attn_row(void *vctx, long r, double *x)
{
    const attn_ctx *c = (const attn_ctx *)vctx;
    long flat = c->rows ? c->rows[r] : r;
    long bh = flat / c->N;
    long i = flat % c->N;
    int h = (int)(bh % c->H);
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    const float *qi = c->q + base + (size_t)i * c->d;
    const double m = c->m[h];
    long jend = c->causal ? i : (long)c->N - 1;

    /* logits of the allowed keys */
    double M = -INFINITY;
    for (long j = 0; j <= jend; ++j) {
        double a = content_score(qi, c->k + base + (size_t)j * c->d, c->d);
        if (c->variant & ORACLE_SOFTCAP) a = softcap(a, c->z_cap);
        x[j] = a + oracle_bias_ex(m, i, j, c->causal, c->variant, c->c_clamp);
        if (x[j] > M) M = x[j];
    }
    /* stable softmax ("When Attention Goes Blind", App. B.1) */
    double Z = 0.0;
    for (long j = 0; j <= jend; ++j) {
        x[j] = exp(x[j] - M);
        Z += x[j];
    }
    double *o = c->out + (size_t)r * c->d;
    for (int t = 0; t < c->d; ++t) o[t] = 0.0;
    for (long j = 0; j <= jend; ++j) {
        double wij = x[j] / Z;
        const float *vj = c->v + base + (size_t)j * c->d;
        for (int t = 0; t < c->d; ++t) o[t] += wij * (double)vj[t];
        if (c->w) c->w[(size_t)r * c->N + j] = wij;
    }
    if (c->w)
        for (long j = jend + 1; j < c->N; ++j) c->w[(size_t)r * c->N + j] = 0.0;
    if (c->lse) c->lse[r] = M + log(Z);
}

/*
 * Attention output, LSE and (optionally) full weight rows for the requested
 * query rows. rows == NULL means all B*H*N rows in [b][h][i] order.
 * out: nrows x d; lse: nrows (may be NULL); w: nrows x N (may be NULL).
 */
int oracle_attn_rows(const float *q, const float *k, const float *v, const double *m,
                     int B, int H, int N, int d, int causal, int variant,
                     double c_clamp, double z_cap, const long *rows, long nrows,
                     double *out, double *lse, double *w, int nthreads)
{
    if (!q || !k || !v || !m || !out || B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_EINVAL;
    long total = (long)B * H * N;
    if (!rows) nrows = total;
    if (nrows < 0) return ORACLE_EINVAL;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return ORACLE_EINVAL;
    attn_ctx c = {q, k, v, m, B, H, N, d, causal, variant, c_clamp, z_cap, rows, out, lse, w};
    return run_rows(attn_row, &c, nrows, N, nthreads);
}

/* --------------------------------------------------------------- backward */

/*
 * Gradients of the attention above for an upstream gradient dO, written out
 * from the definition (the forward of "When Attention Goes Blind" sec. 3.1
 * eq. 1-4; its sec. 5.1 remarks that only nonzero weights carry gradient):
 *
 *   w_ij  = softmax_j(x_ij)                      (allowed keys only)
 *   g_ij  = dO_i . v_j                           d loss / d w_ij
 *   dx_ij = w_ij (g_ij - sum_t w_it g_it)        softmax Jacobian applied to g
 *   da_ij = dx_ij                                (z (1 - tanh^2(a_ij / z)) / z
 *                                                 factor with ORACLE_SOFTCAP)
 *   dQ_i  = sum_j da_ij k_j / sqrt(d)
 *   dK_j  = sum_i da_ij q_i / sqrt(d)
 *   dV_j  = sum_i w_ij dO_i
 *
 * The bias has no trainable parameter, so it only enters through w. Three
 * passes, each a plain loop: per query row the weights' normaliser and the
 * sum_t w_it g_it; dQ per query row; dK and dV per key (column of w).
 */
typedef struct {
    const float *q, *k, *v, *dout;
    const double *m;
    int B, H, N, d, causal, variant;
    double c_clamp, z_cap;
    double *lse, *rowdot; /* per (b, h, i): ln sum_j e^{x_ij}, sum_j w_ij g_ij */
    double *dq, *dk, *dv;
} bwd_ctx;

/* Logit x_ij of the forward (with its variants); -inf for masked keys. If araw
 * is given it receives the scaled content score a_ij before soft capping. */
static double bwd_logit(const bwd_ctx *c, long bh, long i, long j, double *araw)
{
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    double b = oracle_bias_ex(c->m[bh % c->H], i, j, c->causal, c->variant, c->c_clamp);
    if (b == -INFINITY) return -INFINITY;
    double a = content_score(c->q + base + (size_t)i * c->d, c->k + base + (size_t)j * c->d, c->d);
    if (araw) *araw = a;
    if (c->variant & ORACLE_SOFTCAP) a = softcap(a, c->z_cap);
    return a + b;
}

static double bwd_g(const bwd_ctx *c, long bh, long i, long j)
{
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    const float *o = c->dout + base + (size_t)i * c->d, *vj = c->v + base + (size_t)j * c->d;
    double g = 0.0;
    for (int t = 0; t < c->d; ++t) g += (double)o[t] * (double)vj[t];
    return g;
}

/* d x_ij / d a_ij: 1, or 1 - tanh^2(a / z) under soft capping. */
static double bwd_cap_factor(const bwd_ctx *c, double a)
{
    if (!(c->variant & ORACLE_SOFTCAP)) return 1.0;
    double t = tanh(a / c->z_cap);
    return 1.0 - t * t;
}

/* pass 1, per query row: normaliser (as an LSE) and sum_t w_it g_it */
static void bwd_row_stats(void *vctx, long r, double *x)
{
    const bwd_ctx *c = (const bwd_ctx *)vctx;
    long bh = r / c->N, i = r % c->N;
    double M = -INFINITY;
    for (long j = 0; j < c->N; ++j) {
        x[j] = bwd_logit(c, bh, i, j, NULL);
        if (x[j] > M) M = x[j];
    }
    double Z = 0.0;
    for (long j = 0; j < c->N; ++j) Z += exp(x[j] - M);
    double s = 0.0;
    for (long j = 0; j < c->N; ++j)
        if (x[j] != -INFINITY) s += exp(x[j] - M) / Z * bwd_g(c, bh, i, j);
    c->lse[r] = M + log(Z);
    c->rowdot[r] = s;
}

/* pass 2, per query row: dQ_i */
static void bwd_dq_row(void *vctx, long r, double *x)
{
    (void)x;
    const bwd_ctx *c = (const bwd_ctx *)vctx;
    long bh = r / c->N, i = r % c->N;
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    double *dq = c->dq + (size_t)r * c->d;
    for (int t = 0; t < c->d; ++t) dq[t] = 0.0;
    for (long j = 0; j < c->N; ++j) {
        double a = 0.0, xij = bwd_logit(c, bh, i, j, &a);
        if (xij == -INFINITY) continue;
        double w = exp(xij - c->lse[r]);
        double da = w * (bwd_g(c, bh, i, j) - c->rowdot[r]) * bwd_cap_factor(c, a);
        const float *kj = c->k + base + (size_t)j * c->d;
        for (int t = 0; t < c->d; ++t) dq[t] += da * (double)kj[t];
    }
    for (int t = 0; t < c->d; ++t) dq[t] /= sqrt((double)c->d);
}

/* pass 3, per key (column): dK_j and dV_j */
static void bwd_dkv_col(void *vctx, long r, double *x)
{
    (void)x;
    const bwd_ctx *c = (const bwd_ctx *)vctx;
    long bh = r / c->N, j = r % c->N;
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    double *dk = c->dk + (size_t)r * c->d, *dv = c->dv + (size_t)r * c->d;
    for (int t = 0; t < c->d; ++t) dk[t] = dv[t] = 0.0;
    for (long i = 0; i < c->N; ++i) {
        double a = 0.0, xij = bwd_logit(c, bh, i, j, &a);
        if (xij == -INFINITY) continue;
        long ri = bh * c->N + i;
        double w = exp(xij - c->lse[ri]);
        double da = w * (bwd_g(c, bh, i, j) - c->rowdot[ri]) * bwd_cap_factor(c, a);
        const float *qi = c->q + base + (size_t)i * c->d, *oi = c->dout + base + (size_t)i * c->d;
        for (int t = 0; t < c->d; ++t) {
            dk[t] += da * (double)qi[t];
            dv[t] += w * (double)oi[t];
        }
    }
    for (int t = 0; t < c->d; ++t) dk[t] /= sqrt((double)c->d);
}

/*
 * dq, dk, dv: B*H*N x d each (fp64). lse, rowdot: optional outputs of pass 1
 * (B*H*N each); pass NULL to use internal buffers.
 */
int oracle_attn_bwd(const float *q, const float *k, const float *v, const float *dout, const double *m,
                    int B, int H, int N, int d, int causal, int variant, double c_clamp, double z_cap,
                    double *dq, double *dk, double *dv, double *lse, double *rowdot, int nthreads)
{
    if (!q || !k || !v || !dout || !m || !dq || !dk || !dv || B < 1 || H < 1 || N < 1 || d < 1)
        return ORACLE_EINVAL;
    long rows = (long)B * H * N;
    double *l = lse ? lse : (double *)malloc(sizeof(double) * (size_t)rows);
    double *rd = rowdot ? rowdot : (double *)malloc(sizeof(double) * (size_t)rows);
    int st = ORACLE_ENOMEM;
    if (l && rd) {
        bwd_ctx c = {q, k, v, dout, m, B, H, N, d, causal, variant, c_clamp, z_cap, l, rd, dq, dk, dv};
        st = run_rows(bwd_row_stats, &c, rows, N, nthreads);
        if (st == ORACLE_OK) st = run_rows(bwd_dq_row, &c, rows, 1, nthreads);
        if (st == ORACLE_OK) st = run_rows(bwd_dkv_col, &c, rows, 1, nthreads);
    }
    if (!lse) free(l);
    if (!rowdot) free(rd);
    return st;
}

/* ----------------------------------------------------------------- decode */

typedef struct {
    const float *q, *kc, *vc;
    const double *m;
    int H, L, d;
    double *out, *lse;
} decode_ctx;

/*
 * One new token per (b, h) against a KV cache of L positions. The query sits
 * at its true sequence position L - 1, so key j has distance L - 1 - j
 * ("ALiBi: Attention with Linear Biases", the KV-cache paragraph after the
 * full-sequence example).
 */
static void decode_row(void *vctx, long bh, double *x)
{
    const decode_ctx *c = (const decode_ctx *)vctx;
    int h = (int)(bh % c->H);
    const float *qv = c->q + (size_t)bh * c->d;
    const float *K = c->kc + (size_t)bh * c->L * c->d;
    const float *V = c->vc + (size_t)bh * c->L * c->d;
    const long pos = (long)c->L - 1;
    double M = -INFINITY;
    for (long j = 0; j < c->L; ++j) {
        double a = 0.0;
        for (int t = 0; t < c->d; ++t) a += (double)qv[t] * (double)K[(size_t)j * c->d + t];
        a /= sqrt((double)c->d);
        x[j] = a - c->m[h] * (double)(pos - j);
        if (x[j] > M) M = x[j];
    }
    double Z = 0.0;
    for (long j = 0; j < c->L; ++j) {
        x[j] = exp(x[j] - M);
        Z += x[j];
    }
    double *o = c->out + (size_t)bh * c->d;
    for (int t = 0; t < c->d; ++t) o[t] = 0.0;
    for (long j = 0; j < c->L; ++j)
        for (int t = 0; t < c->d; ++t) o[t] += (x[j] / Z) * (double)V[(size_t)j * c->d + t];
    if (c->lse) c->lse[bh] = M + log(Z);
}

int oracle_attn_decode(const float *q, const float *kc, const float *vc, const double *m,
                       int B, int H, int L, int d, double *out, double *lse, int nthreads)
{
    if (!q || !kc || !vc || !m || !out || B < 1 || H < 1 || L < 1 || d < 1) return ORACLE_EINVAL;
    decode_ctx c = {q, kc, vc, m, H, L, d, out, lse};
    return run_rows(decode_row, &c, (long)B * H, L, nthreads);
}

/* -------------------------------------------------------------- underflow */

typedef struct {
    const float *q, *k;
    const double *m;
    int H, N, d;
    double tau, band;
    const long *rows;
    unsigned long long *count, *near;
} uf_ctx;

/*
 * Per query row: the number of allowed keys whose max-subtracted exponent
 * x_ij - M_i is <= tau (the entry underflows; "When Attention Goes Blind",
 * sec. 3.2: e^{tau} = 0 and the blindness distance uses "<= tau"), and the
 * number within +-band of tau (entries whose classification depends on
 * rounding).
 */
static void uf_row(void *vctx, long r, double *x)
{
    const uf_ctx *c = (const uf_ctx *)vctx;
    long flat = c->rows ? c->rows[r] : r;
    long bh = flat / c->N;
    long i = flat % c->N;
    int h = (int)(bh % c->H);
    const size_t base = (size_t)bh * (size_t)c->N * (size_t)c->d;
    const float *qi = c->q + base + (size_t)i * c->d;
    double M = -INFINITY;
    for (long j = 0; j <= i; ++j) {
        x[j] = content_score(qi, c->k + base + (size_t)j * c->d, c->d) - c->m[h] * (double)(i - j);
        if (x[j] > M) M = x[j];
    }
    unsigned long long cnt = 0, nr = 0;
    for (long j = 0; j <= i; ++j) {
        double e = x[j] - M;
        if (e <= c->tau) ++cnt;
        if (fabs(e - c->tau) <= c->band) ++nr;
    }
    c->count[r] = cnt;
    if (c->near) c->near[r] = nr;
}

int oracle_underflow_rows(const float *q, const float *k, const double *m, int B, int H, int N,
                          int d, double tau, double band, const long *rows, long nrows,
                          unsigned long long *count, unsigned long long *near, int nthreads)
{
    if (!q || !k || !m || !count || B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_EINVAL;
    long total = (long)B * H * N;
    if (!rows) nrows = total;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return ORACLE_EINVAL;
    uf_ctx c = {q, k, m, H, N, d, tau, band, rows, count, near};
    return run_rows(uf_row, &c, nrows, N, nthreads);
}

/* ---------------------------------------------------- analytic quantities */

/*
 * Floating-point thresholds of "When Attention Goes Blind", App. A Table 4, as
 * natural logs of format limits:
 *   [0] underflow bf16  = ln(smallest bf16 subnormal) = ln 2^-133
 *   [1] underflow fp32  = ln(smallest fp32 subnormal) = ln 2^-149
 *   [2] denorm bf16 = [3] denorm fp32 = ln(smallest normal) = ln 2^-126
 *   [4] overflow bf16 = ln((2 - 2^-7) 2^127), [5] overflow fp32 = ln((2 - 2^-23) 2^127)
 */
void oracle_thresholds(double *t)
{
    const double ln2 = log(2.0);
    t[0] = -133.0 * ln2;
    t[1] = -149.0 * ln2;
    t[2] = -126.0 * ln2;
    t[3] = -126.0 * ln2;
    t[4] = 127.0 * ln2 + log(2.0 - ldexp(1.0, -7));
    t[5] = 127.0 * ln2 + log(2.0 - ldexp(1.0, -23));
}

/*
 * Blindness distance ("When Attention Goes Blind", sec. 3.2):
 * Delta_h(eps) = min{ D in N : eps - m_h D* <= tau }, D* = D or log(D + 1).
 * oracle_blindness_real returns the real-valued crossing point D with
 * eps - m D* = tau (the tables print it rounded to the nearest integer);
 * oracle_blindness_int returns the integer minimum of the definition.
 */
double oracle_blindness_real(double m, double eps, double tau, int log_distance)
{
    double t = (eps - tau) / m; /* required (log-)distance */
    if (t <= 0.0) return 0.0;
    return log_distance ? expm1(t) : t;
}

double oracle_blindness_int(double m, double eps, double tau, int log_distance)
{
    double t = (eps - tau) / m;
    if (t <= 0.0) return 0.0;
    double D = log_distance ? ceil(expm1(t)) : ceil(t);
    /* step forward while D does not satisfy the condition (rounding of t) */
    for (;;) {
        double Ds = log_distance ? log(D + 1.0) : D;
        if (eps - m * Ds <= tau) break;
        D += 1.0;
    }
    /* step back while the predecessor already satisfies the condition */
    while (D > 0.0) {
        double Dm = D - 1.0;
        double Ds = log_distance ? log(Dm + 1.0) : Dm;
        if (eps - m * Ds <= tau) D = Dm; else break;
    }
    return D;
}
