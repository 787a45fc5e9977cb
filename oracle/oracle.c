/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the APEX-1 attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA path is
 * checked against; it is not part of the product.  Only the test suite, the
 * smoke check of the package entry file and the CPU-baseline leg of the bench
 * may load it.  It shares no code, header, table or constant with the CUDA
 * library: it is written straight from the formulas of the two APEX-1
 * "Mathematical Reference" pages, in double precision, with no blocking,
 * fusion or reordering beyond what those formulas state.
 *
 * What it computes, for every batch b, query head h and query row r:
 *
 *   1. group  g = floor(h / G),  G = H_q / H_kv
 *        (Part 2, §8.2 "Formula" and the §8.4 worked assignment: query heads
 *         Q0,Q1 share KV head 0, Q2,Q3 share KV head 1 -- contiguous groups)
 *   2. query position m = q_pos0 + r; key j sits at position j
 *        (Part 1, §1 symbol table: m is the token position index 0..S-1)
 *   3. RoPE on the query at m and on every key at j
 *        (Part 1, §4.2 pairwise rotation, §4.3 theta_i = base^(-2i/d_h),
 *         §4.4 compact form x*cos + rotate_half(x)*sin with
 *         rotate_half([x0,x1,x2,x3]) = [-x1,x0,-x3,x2], §4.7 cos/sin cache)
 *   4. scores s_j = <q', k'_j> / sqrt(d_h) for the visible keys
 *        (Part 2, §6.2 softmax(Q K^T / sqrt(d_h)) V)
 *      visibility (Part 2, §10.2): j <= m and, with a window W > 0,
 *      0 <= m - j < W.  Without the causal flag every key is visible (used only
 *      to reproduce the unmasked worked example of Part 2, §6.4).
 *   5. softmax over the visible keys, written as the three plain passes
 *      M = max_j s_j ; Z = sum_j exp(s_j - M) ; o = sum_j exp(s_j - M)/Z * v_j
 *        (Part 2, §6.4 steps 3 and 4: exponentiate, normalise, weight V)
 *
 * Options beyond the plain block (all off by default):
 *   - YaRN frequency scaling with factor s (Part 1, §5.3-§5.4): with the
 *     wavelength lambda_i = 2 pi / theta_i, pairs with lambda_i < beta_fast keep
 *     theta_i, pairs with lambda_i > beta_slow * s use theta_i / s, the others
 *     use theta_i / (t s + 1 - t) with t = (lambda_i / beta_slow - 1) / (s - 1)
 *     clamped to [0, 1]; and the attention temperature 0.1 ln(s) + 1 multiplied
 *     into the scores (§5.5).
 *   - a bidirectional prefix of P positions (Part 2, §11.1): a query at m < P
 *     sees exactly the keys j < P; queries at m >= P follow the causal/window rule.
 *   - keys given already rotated (a KV cache holding RoPE(k, j)): the keys are
 *     used as they are.
 *   - decoupled RoPE of multi-head latent attention (Part 2, §9.3): query and
 *     key rows are [content (d_h) | rope part (d_r)] with length d_h + d_r,
 *     value and output rows have length d_h; only the trailing d_r entries are
 *     rotated, as a d_r-dimensional RoPE vector (theta_i = base^(-2i/d_r)),
 *     and the scores are divided by sqrt(d_h + d_r), the length of the vectors
 *     being dotted.  The plain block is the case d_r = d_h + d_r = row length,
 *     i.e. no content part and value rows as long as query rows.
 *
 * Inputs are either raw bf16 bit patterns (widened exactly to double) or
 * doubles.  A rope_base <= 0 switches RoPE off (again only for the §6.4
 * example, which has none).  The cos/sin cache of §4.7 is built here, in
 * double precision with libm, for every position the call touches.
 *
 * Parallelism is a plain split of independent (batch, kv-head, row-chunk)
 * tasks over POSIX threads; every output element is computed by exactly one
 * thread with the same sequential sums, so results do not depend on the
 * thread count.
 */
#include <math.h>
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_NOMEM = 2 };
enum { ELEM_BF16 = 0, ELEM_F64 = 1 };

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, size_t idx, int kind)
{
    if (kind == ELEM_BF16)
        return widen_bf16(((const uint16_t *)base)[idx]);
    return ((const double *)base)[idx];
}

/* Part 1, §4.3: theta_i = 1 / base^(2i/d_h), i = 0 .. d_h/2 - 1. */
static double rope_theta(int i, int d, double base)
{
    return pow(base, -2.0 * (double)i / (double)d);
}

typedef struct {
    double yarn_s;      /* YaRN scale factor s; <= 1: no scaling */
    double beta_fast;   /* wavelength below which a pair is not scaled (32)  */
    double beta_slow;   /* beta_slow * s: wavelength above which it is fully scaled (1) */
    int prefix_len;     /* P: bidirectional prefix [0, P); 0: none */
    int keys_prerotated;/* keys already carry their rotation */
} oracle_opts;

/* Part 1, §5.3-§5.4: the YaRN-scaled value of one frequency theta. */
static double yarn_scale(double th, const oracle_opts *o)
{
    if (!o || o->yarn_s <= 1.0)
        return th;
    const double s = o->yarn_s;
    const double lambda = 2.0 * M_PI / th;           /* wavelength */
    if (lambda < o->beta_fast)                       /* high frequency: unchanged */
        return th;
    if (lambda > o->beta_slow * s)                   /* low frequency: full scaling */
        return th / s;
    double t = (lambda / o->beta_slow - 1.0) / (s - 1.0);  /* mid: interpolate */
    if (t < 0.0) t = 0.0;
    if (t > 1.0) t = 1.0;
    return th / (t * s + (1.0 - t));
}

static double yarn_theta(int i, int d, double base, const oracle_opts *o)
{
    return yarn_scale(rope_theta(i, d, base), o);
}

/* Part 1, §5.5: attention temperature, multiplied into the scores. */
static double yarn_attn_factor(const oracle_opts *o)
{
    if (!o || o->yarn_s <= 1.0)
        return 1.0;
    return 0.1 * log(o->yarn_s) + 1.0;
}

/* Part 1, §4.7: cos/sin cache, one (cos, sin) pair per (position, pair i). */
typedef struct {
    long n_pos;
    int half;
    double *cs; /* [n_pos][half][2] */
} rope_cache;

static int rope_cache_build(rope_cache *c, long n_pos, int d, double base, const oracle_opts *o)
{
    c->n_pos = n_pos;
    c->half = d / 2;
    c->cs = NULL;
    if (base <= 0.0 || n_pos <= 0)
        return ORACLE_OK;
    c->cs = (double *)malloc(sizeof(double) * 2 * (size_t)n_pos * (size_t)c->half);
    if (!c->cs)
        return ORACLE_ERR_NOMEM;
    for (int i = 0; i < c->half; ++i) {
        double th = yarn_theta(i, d, base, o);
        for (long m = 0; m < n_pos; ++m) {
            double ang = (double)m * th;
            c->cs[((size_t)m * c->half + i) * 2 + 0] = cos(ang);
            c->cs[((size_t)m * c->half + i) * 2 + 1] = sin(ang);
        }
    }
    return ORACLE_OK;
}

/*
 * Part 1, §4.2 / §4.4: rotate each pair (x_2i, x_2i+1) by angle m*theta_i:
 *   x'_2i   = x_2i * cos - x_2i+1 * sin
 *   x'_2i+1 = x_2i * sin + x_2i+1 * cos
 * over the trailing d_rope entries of the length-d vector (the whole vector in
 * the plain block; the rope part of Part 2, §9.3 otherwise), whose pairs are
 * numbered from the start of that part.  The leading d - d_rope entries are
 * copied.  With no cache (RoPE switched off) the vector is copied unchanged.
 */
static void rope_apply(const rope_cache *c, long m, const double *x, double *out, int d, int d_rope)
{
    memcpy(out, x, sizeof(double) * (size_t)d);
    if (!c->cs)
        return;
    const double *xr = x + (d - d_rope);
    double *outr = out + (d - d_rope);
    for (int i = 0; i < d_rope / 2; ++i) {
        double cs = c->cs[((size_t)m * c->half + i) * 2 + 0];
        double sn = c->cs[((size_t)m * c->half + i) * 2 + 1];
        double x0 = xr[2 * i], x1 = xr[2 * i + 1];
        outr[2 * i] = x0 * cs - x1 * sn;
        outr[2 * i + 1] = x0 * sn + x1 * cs;
    }
}

/* Part 2, §10.2 (with the causal part of the same formula), and the
 * bidirectional prefix of Part 2, §11.1. */
static int key_visible(long m, long j, int window, int causal, int prefix_len)
{
    if (!causal)
        return 1;
    if (m < prefix_len)
        return j < prefix_len;
    if (j > m)
        return 0;
    if (window > 0 && m - j >= (long)window)
        return 0;
    return 1;
}

typedef struct {
    /* problem */
    const void *q, *k, *v;
    int kind;
    double *out;
    int B, H_q, H_kv, S_q, S_k, window, causal, prefix_len, keys_prerotated;
    int d;      /* query / key row length */
    int d_v;    /* value / output row length */
    int d_rope; /* trailing query / key entries that RoPE rotates */
    double score_factor; /* 1 / sqrt(d), times the YaRN temperature */
    long q_pos0;
    const int *rows;
    int n_rows;
    const rope_cache *cache;
    /* task list: (b, g, row chunk) */
    int chunk;
    int n_chunks;
    long n_tasks;
    long next_task;
    pthread_mutex_t lock;
    int status;
} attn_job;

static long take_task(attn_job *job)
{
    long t;
    pthread_mutex_lock(&job->lock);
    t = job->next_task++;
    pthread_mutex_unlock(&job->lock);
    return t;
}

static int row_index(const attn_job *job, int i)
{
    return job->rows ? job->rows[i] : i;
}

static void run_task(attn_job *job, long task, double *kbuf, double *qraw, double *qrot,
                     double *kraw, double *scores, double *acc)
{
    const int d = job->d, d_v = job->d_v, d_rope = job->d_rope;
    const int G = job->H_q / job->H_kv;
    const int chunk_id = (int)(task % job->n_chunks);
    const int g = (int)((task / job->n_chunks) % job->H_kv);
    const int b = (int)(task / ((long)job->n_chunks * job->H_kv));
    const int i0 = chunk_id * job->chunk;
    const int i1 = (i0 + job->chunk < job->n_rows) ? i0 + job->chunk : job->n_rows;
    const double score_factor = job->score_factor;

    /* keys this chunk can see: the union of its rows' visible ranges */
    long j_lo = 0, j_hi = job->S_k - 1;
    if (job->causal) {
        long lo_all = job->S_k, hi_all = -1;
        for (int i = i0; i < i1; ++i) {
            long m = job->q_pos0 + row_index(job, i);
            long lo, hi;
            if (m < job->prefix_len) {
                lo = 0;
                hi = job->prefix_len - 1;
            } else {
                hi = m;
                lo = (job->window > 0 && m - job->window + 1 > 0) ? m - job->window + 1 : 0;
            }
            if (lo < lo_all) lo_all = lo;
            if (hi > hi_all) hi_all = hi;
        }
        j_lo = lo_all;
        if (hi_all < j_hi) j_hi = hi_all;
    }

    /* step 3 for the keys: k'_j = RoPE(k_j, j) */
    const size_t kv_head = (size_t)b * job->H_kv + g;
    for (long j = j_lo; j <= j_hi; ++j) {
        size_t base = (kv_head * job->S_k + (size_t)j) * d;
        for (int e = 0; e < d; ++e)
            kraw[e] = load_elem(job->k, base + e, job->kind);
        if (job->keys_prerotated)
            memcpy(kbuf + (size_t)(j - j_lo) * d, kraw, sizeof(double) * (size_t)d);
        else
            rope_apply(job->cache, j, kraw, kbuf + (size_t)(j - j_lo) * d, d, d_rope);
    }

    for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh; /* step 1: head h reads KV head floor(h/G) = g */
        for (int i = i0; i < i1; ++i) {
            const int r = row_index(job, i);
            const long m = job->q_pos0 + r;
            size_t qbase = (((size_t)b * job->H_q + h) * job->S_q + (size_t)r) * d;
            for (int e = 0; e < d; ++e)
                qraw[e] = load_elem(job->q, qbase + e, job->kind);
            rope_apply(job->cache, m, qraw, qrot, d, d_rope);

            /* step 4: scaled scores of the visible keys (times the YaRN temperature) */
            double M = -INFINITY;
            int any = 0;
            for (long j = j_lo; j <= j_hi; ++j) {
                if (!key_visible(m, j, job->window, job->causal, job->prefix_len))
                    continue;
                const double *kr = kbuf + (size_t)(j - j_lo) * d;
                double dot = 0.0;
                for (int e = 0; e < d; ++e)
                    dot += qrot[e] * kr[e];
                double s = dot * score_factor;
                scores[j - j_lo] = s;
                if (!any || s > M) M = s;
                any = 1;
            }
            double *o = job->out + (((size_t)b * job->H_q + h) * job->n_rows + (size_t)i) * d_v;
            if (!any) { /* no visible key: left as NaN, the API forbids it */
                for (int e = 0; e < d_v; ++e) o[e] = NAN;
                continue;
            }
            /* step 5: Z = sum exp(s - M), then o = sum exp(s - M)/Z * v */
            double Z = 0.0;
            for (long j = j_lo; j <= j_hi; ++j)
                if (key_visible(m, j, job->window, job->causal, job->prefix_len))
                    Z += exp(scores[j - j_lo] - M);
            for (int e = 0; e < d_v; ++e) acc[e] = 0.0;
            for (long j = j_lo; j <= j_hi; ++j) {
                if (!key_visible(m, j, job->window, job->causal, job->prefix_len))
                    continue;
                double p = exp(scores[j - j_lo] - M) / Z;
                size_t vbase = (kv_head * job->S_k + (size_t)j) * d_v;
                for (int e = 0; e < d_v; ++e)
                    acc[e] += p * load_elem(job->v, vbase + e, job->kind);
            }
            for (int e = 0; e < d_v; ++e) o[e] = acc[e];
        }
    }
}

static void *worker(void *arg)
{
    attn_job *job = (attn_job *)arg;
    const int d = job->d;
    double *kbuf = (double *)malloc(sizeof(double) * (size_t)job->S_k * d);
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(3 * d + job->d_v + job->S_k));
    if (!kbuf || !scratch) {
        pthread_mutex_lock(&job->lock);
        job->status = ORACLE_ERR_NOMEM;
        pthread_mutex_unlock(&job->lock);
        free(kbuf);
        free(scratch);
        return NULL;
    }
    double *qraw = scratch, *qrot = scratch + d, *kraw = scratch + 2 * d, *acc = scratch + 3 * d;
    double *scores = scratch + 3 * d + job->d_v;
    for (;;) {
        long t = take_task(job);
        if (t >= job->n_tasks)
            break;
        run_task(job, t, kbuf, qraw, qrot, kraw, scores, acc);
    }
    free(kbuf);
    free(scratch);
    return NULL;
}

static int attn_common(const void *q, const void *k, const void *v, int kind, double *out,
                       int B, int H_q, int H_kv, int S_q, int S_k, int d, int d_v, int d_rope,
                       int window, long q_pos0, double rope_base, int causal, const int *rows,
                       int n_rows, int n_threads, const oracle_opts *opts)
{
    if (opts && (opts->prefix_len < 0 || opts->prefix_len > S_k ||
                 (opts->yarn_s > 1.0 && (opts->beta_fast <= 0.0 || opts->beta_slow <= 0.0))))
        return ORACLE_ERR_ARG;
    if (!q || !k || !v || !out || B <= 0 || H_q <= 0 || H_kv <= 0 || S_q <= 0 || S_k <= 0 ||
        d <= 0 || d_v <= 0 || d_rope <= 0 || (d_rope & 1) || d_rope > d || H_q % H_kv != 0 ||
        q_pos0 < 0)
        return ORACLE_ERR_ARG;
    if (!rows)
        n_rows = S_q;
    if (n_rows <= 0)
        return ORACLE_ERR_ARG;
    long max_pos = S_k;
    for (int i = 0; i < n_rows; ++i) {
        int r = rows ? rows[i] : i;
        if (r < 0 || r >= S_q)
            return ORACLE_ERR_ARG;
        if (q_pos0 + r + 1 > max_pos)
            max_pos = q_pos0 + r + 1;
    }

    rope_cache cache;
    if (rope_cache_build(&cache, max_pos, d_rope, rope_base, opts) != ORACLE_OK)
        return ORACLE_ERR_NOMEM;

    attn_job job;
    memset(&job, 0, sizeof job);
    job.q = q; job.k = k; job.v = v; job.kind = kind; job.out = out;
    job.B = B; job.H_q = H_q; job.H_kv = H_kv; job.S_q = S_q; job.S_k = S_k; job.d = d;
    job.d_v = d_v; job.d_rope = d_rope;
    job.window = window; job.causal = causal; job.q_pos0 = q_pos0;
    job.prefix_len = opts ? opts->prefix_len : 0;
    job.keys_prerotated = opts ? opts->keys_prerotated : 0;
    job.score_factor = yarn_attn_factor(opts) / sqrt((double)d);
    job.rows = rows; job.n_rows = n_rows; job.cache = &cache;
    if (n_threads <= 0)
        n_threads = 1;
    /* enough chunks to keep every thread busy, at most 64 rows each */
    long units = (long)B * H_kv;
    int chunk = n_rows;
    while (chunk > 64 || (units * ((n_rows + chunk - 1) / chunk) < 4L * n_threads && chunk > 1))
        chunk = (chunk + 1) / 2;
    job.chunk = chunk;
    job.n_chunks = (n_rows + chunk - 1) / chunk;
    job.n_tasks = units * job.n_chunks;
    pthread_mutex_init(&job.lock, NULL);

    if (n_threads > job.n_tasks)
        n_threads = (int)job.n_tasks;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!tid) {
        free(cache.cs);
        return ORACLE_ERR_NOMEM;
    }
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&tid[t], NULL, worker, &job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        worker(&job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    free(cache.cs);
    return job.status;
}

/*
 * RoPE of n_vec vectors of length d, vector n at position pos[n]
 * (Part 1, §4.2-§4.4).  out may not alias x.
 */
int oracle_rope_f64(const double *x, double *out, long n_vec, int d, const long *pos, double base)
{
    if (!x || !out || !pos || n_vec < 0 || d <= 0 || (d & 1) || base <= 0.0)
        return ORACLE_ERR_ARG;
    for (long n = 0; n < n_vec; ++n) {
        if (pos[n] < 0)
            return ORACLE_ERR_ARG;
        for (int i = 0; i < d / 2; ++i) {
            double ang = (double)pos[n] * rope_theta(i, d, base);
            double cs = cos(ang), sn = sin(ang);
            double x0 = x[n * d + 2 * i], x1 = x[n * d + 2 * i + 1];
            out[n * d + 2 * i] = x0 * cs - x1 * sn;
            out[n * d + 2 * i + 1] = x0 * sn + x1 * cs;
        }
    }
    return ORACLE_OK;
}

/* theta_i for i = 0 .. d/2-1 (Part 1, §4.3). */
int oracle_rope_theta_f64(int d, double base, double *theta)
{
    if (d <= 0 || (d & 1) || base <= 0.0 || !theta)
        return ORACLE_ERR_ARG;
    for (int i = 0; i < d / 2; ++i)
        theta[i] = rope_theta(i, d, base);
    return ORACLE_OK;
}

/*
 * Attention block on bf16 inputs given as raw 16-bit patterns.
 *   q   [B, H_q,  S_q, d]      k, v [B, H_kv, S_k, d]     (row-major)
 *   out [B, H_q,  n_rows, d]   doubles; n_rows = S_q when rows == NULL,
 *                              otherwise row i of out is query row rows[i].
 * The _ex forms take the options above (NULL: none).
 */
int oracle_attn_ex_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                        int B, int H_q, int H_kv, int S_q, int S_k, int d, int window,
                        long q_pos0, double rope_base, int causal, const int *rows, int n_rows,
                        int n_threads, const oracle_opts *opts)
{
    return attn_common(q, k, v, ELEM_BF16, out, B, H_q, H_kv, S_q, S_k, d, d, d, window, q_pos0,
                       rope_base, causal, rows, n_rows, n_threads, opts);
}

int oracle_attn_ex_f64(const double *q, const double *k, const double *v, double *out, int B,
                       int H_q, int H_kv, int S_q, int S_k, int d, int window, long q_pos0,
                       double rope_base, int causal, const int *rows, int n_rows, int n_threads,
                       const oracle_opts *opts)
{
    return attn_common(q, k, v, ELEM_F64, out, B, H_q, H_kv, S_q, S_k, d, d, d, window, q_pos0,
                       rope_base, causal, rows, n_rows, n_threads, opts);
}

int oracle_attn_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                     int B, int H_q, int H_kv, int S_q, int S_k, int d, int window,
                     long q_pos0, double rope_base, int causal, const int *rows, int n_rows,
                     int n_threads)
{
    return attn_common(q, k, v, ELEM_BF16, out, B, H_q, H_kv, S_q, S_k, d, d, d, window, q_pos0,
                       rope_base, causal, rows, n_rows, n_threads, NULL);
}

/* The same on double inputs (worked examples and brute-force checks). */
int oracle_attn_f64(const double *q, const double *k, const double *v, double *out, int B,
                    int H_q, int H_kv, int S_q, int S_k, int d, int window, long q_pos0,
                    double rope_base, int causal, const int *rows, int n_rows, int n_threads)
{
    return attn_common(q, k, v, ELEM_F64, out, B, H_q, H_kv, S_q, S_k, d, d, d, window, q_pos0,
                       rope_base, causal, rows, n_rows, n_threads, NULL);
}

/*
 * Multi-head latent attention with decoupled RoPE (Part 2, §9.3):
 *   q   [B, H_q,  S_q, d_h + d_r]   k [B, H_kv, S_k, d_h + d_r]
 *   v   [B, H_kv, S_k, d_h]         out [B, H_q, n_rows, d_h]
 * Rows of q and k are [content | rope part]; RoPE (of dimension d_r) turns
 * only the rope part, scores are divided by sqrt(d_h + d_r).
 */
int oracle_mla_attn_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                         int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r, int window,
                         long q_pos0, double rope_base, int causal, const int *rows, int n_rows,
                         int n_threads, const oracle_opts *opts)
{
    if (d_h <= 0 || d_r <= 0)
        return ORACLE_ERR_ARG;
    return attn_common(q, k, v, ELEM_BF16, out, B, H_q, H_kv, S_q, S_k, d_h + d_r, d_h, d_r,
                       window, q_pos0, rope_base, causal, rows, n_rows, n_threads, opts);
}

int oracle_mla_attn_f64(const double *q, const double *k, const double *v, double *out, int B,
                        int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r, int window,
                        long q_pos0, double rope_base, int causal, const int *rows, int n_rows,
                        int n_threads, const oracle_opts *opts)
{
    if (d_h <= 0 || d_r <= 0)
        return ORACLE_ERR_ARG;
    return attn_common(q, k, v, ELEM_F64, out, B, H_q, H_kv, S_q, S_k, d_h + d_r, d_h, d_r,
                       window, q_pos0, rope_base, causal, rows, n_rows, n_threads, opts);
}

/* YaRN-scaled frequencies theta'_i, i < d/2 (Part 1, §5.3-§5.4), and the
 * attention temperature (§5.5). */
int oracle_yarn_theta_f64(int d, double base, double s, double beta_fast, double beta_slow,
                          double *theta)
{
    if (d <= 0 || (d & 1) || base <= 0.0 || !theta || beta_fast <= 0.0 || beta_slow <= 0.0)
        return ORACLE_ERR_ARG;
    oracle_opts o;
    memset(&o, 0, sizeof o);
    o.yarn_s = s;
    o.beta_fast = beta_fast;
    o.beta_slow = beta_slow;
    for (int i = 0; i < d / 2; ++i)
        theta[i] = yarn_theta(i, d, base, &o);
    return ORACLE_OK;
}

/* The YaRN rule applied to arbitrary frequencies (the worked example of
 * Part 1, §5.6 quotes rounded theta values). */
int oracle_yarn_scale_theta_f64(const double *theta, int n, double s, double beta_fast,
                                double beta_slow, double *out)
{
    if (!theta || !out || n < 0 || beta_fast <= 0.0 || beta_slow <= 0.0)
        return ORACLE_ERR_ARG;
    oracle_opts o;
    memset(&o, 0, sizeof o);
    o.yarn_s = s;
    o.beta_fast = beta_fast;
    o.beta_slow = beta_slow;
    for (int i = 0; i < n; ++i)
        out[i] = yarn_scale(theta[i], &o);
    return ORACLE_OK;
}

double oracle_yarn_attn_factor(double s)
{
    oracle_opts o;
    memset(&o, 0, sizeof o);
    o.yarn_s = s;
    return yarn_attn_factor(&o);
}
