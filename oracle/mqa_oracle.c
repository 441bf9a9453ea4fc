/*
 * CPU oracle for the fused FP8 MQA-logits + per-row top-k prefill selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously correct: it writes the
 * definition out in fp64 and shares no code, header, table or constant with
 * the CUDA library.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may call it.
 *
 * What it computes (sources, cited by page and section):
 *  - Op contract and output convention: vLLM API page
 *    `vllm.model_executor.kernels.attention.dsa.fused_mqa_topk`,
 *    `fused_mqa_topk_prefill` docstring: q [rows, 32, 128] fp8 e4m3,
 *    k [keys, 128] fp8 e4m3, per-key fp32 scales, weights [rows, 32] fp32,
 *    visible range [start, end) per row; output indices are relative to the
 *    row's start (key - start), unordered, -1 padded when fewer than k keys
 *    are visible.
 *  - Score: for a visible key j of row r,
 *        S(r, j) = scale_j * sum_h w[r,h] * relu(q[r,h,:] . k[j,:])
 *    (the indexer's ReLU-weighted multi-head score; vLLM pull request #60618,
 *    section "What this PR does", Scoring bullet, states the relu form).
 *  - Key scales: same API page, `fused_mqa_topk_key_scales` docstring: the
 *    [keys, 4] uint8 UE8M0 group carries exponent e in its first byte; the
 *    fp32 scale is the float whose bit pattern is e << 23.
 *  - Selection: the k largest S over the row's visible keys; the pull
 *    request's Summary and Performance table define the target as the exact
 *    fp32 top-k up to ties at the boundary.  For determinism the oracle
 *    breaks ties by key index ascending (any tie choice is correct).
 *  - Block selection (the two-level candidate selection of the pull request's
 *    "Limitations of this PR -- TODOs": a source layer also writes, per row,
 *    the top blocks of 8 keys ranked by their maximum score): block b holds
 *    keys [8b, 8b + 8) of the key array; its score is the largest S over the
 *    row's visible keys in it.  The output lists the chosen blocks as
 *    b - floor(start / 8), ties by block index ascending, -1 padded.
 *  - Masked selection (the consumer layers of the same two-level selection
 *    mask their scores to the source's blocks before their top-k): a key j of
 *    row r is visible only if it lies in [start, end) and bit (j / 8) % 32 of
 *    word j / 256 of row r's block mask is set; the selection is then the
 *    one above over the visible keys.
 *
 * Arithmetic: every e4m3 value is an integer multiple of 2^-9 with magnitude
 * at most 448, so each q.k product is a multiple of 2^-18 below 2^18 and a
 * 128-term dot product is exact in fp64 in any order.  The weighted sum and
 * the scale are rounded once per step in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- e4m3fn decode: an exhaustive 256-entry table ------------------------ */
/* Bit fields: s eeee mmm, exponent bias 7.  e == 0 is subnormal (m * 2^-9);
 * e == 15 with m == 7 is NaN (0x7F / 0xFF); there are no infinities. */
static double e4m3_decode_bits(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 0xFu, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

static double g_e4m3[256];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;
static void build_table(void) {
    for (unsigned c = 0; c < 256; ++c) g_e4m3[c] = e4m3_decode_bits(c);
}

void oracle_e4m3_table(double *out256) {
    pthread_once(&g_table_once, build_table);
    memcpy(out256, g_e4m3, sizeof(g_e4m3));
}

/* ---- UE8M0 key-scale decode ---------------------------------------------- */
/* scale = the fp32 whose bits are (byte 0 of the group) << 23, i.e. 2^(e-127)
 * for 1 <= e <= 254 (e == 0 gives +0, e == 255 gives +inf under this rule). */
void oracle_ue8m0_decode(const uint8_t *groups, float *out, int64_t keys) {
    for (int64_t j = 0; j < keys; ++j) {
        uint32_t bits = ((uint32_t)groups[4 * j]) << 23;
        float f;
        memcpy(&f, &bits, sizeof f);
        out[j] = f;
    }
}

/* ---- per-head dot products ------------------------------------------------ */
/* dots[h] = sum_d E(q[row,h,d]) * E(k[key,d])  (exact in fp64) */
void oracle_head_dots(const uint8_t *q, const uint8_t *k, int heads, int dim,
                      int64_t row, int64_t key, double *dots) {
    pthread_once(&g_table_once, build_table);
    const uint8_t *kr = k + key * (int64_t)dim;
    for (int h = 0; h < heads; ++h) {
        const uint8_t *qr = q + (row * heads + h) * (int64_t)dim;
        double acc = 0.0;
        for (int d = 0; d < dim; ++d) acc += g_e4m3[qr[d]] * g_e4m3[kr[d]];
        dots[h] = acc;
    }
}

/* S(r, j) for one visible pair, in fp64. */
static double score_pair(const double *qd /* [heads*dim] decoded row */, const uint8_t *k,
                         int heads, int dim, const float *w_row, double scale, int64_t key) {
    const uint8_t *kr = k + key * (int64_t)dim;
    double kd[1024];
    for (int d = 0; d < dim; ++d) kd[d] = g_e4m3[kr[d]];
    double s = 0.0;
    for (int h = 0; h < heads; ++h) {
        const double *qh = qd + (int64_t)h * dim;
        double dot = 0.0;
        for (int d = 0; d < dim; ++d) dot += qh[d] * kd[d];
        double relu = dot > 0.0 ? dot : 0.0;
        s += (double)w_row[h] * relu;
    }
    return scale * s;
}

typedef struct {
    double score;
    int64_t key;
} scored_key;

/* order: larger score first; equal scores by smaller key first */
static int cmp_scored(const void *a, const void *b) {
    const scored_key *x = (const scored_key *)a, *y = (const scored_key *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->key > y->key) - (x->key < y->key);
}

/* order: larger block score first; equal scores by smaller block first */
typedef struct {
    double score;
    int64_t block;
} scored_block;

static int cmp_block(const void *a, const void *b) {
    const scored_block *x = (const scored_block *)a, *y = (const scored_block *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->block > y->block) - (x->block < y->block);
}

typedef struct {
    const uint8_t *q, *k, *scale_groups;
    const float *w;
    const int32_t *starts, *ends;
    const int64_t *row_list; /* rows to process (indices into q/w/starts/ends) */
    int64_t nlist, keys;
    int heads, dim, topk;
    int32_t *out;           /* [nlist, topk] */
    double *scores_out;     /* optional [nlist, keys] dense scores (-inf outside) */
    int block_mode;         /* select blocks of 8 keys by their largest score */
    const uint32_t *mask;   /* optional [rows, mask_words] block mask (masked selection) */
    int64_t mask_words;
    int64_t next;           /* shared work counter */
    pthread_mutex_t lock;
    int status;
} job_t;

static int64_t take_row(job_t *J) {
    pthread_mutex_lock(&J->lock);
    int64_t i = J->next++;
    pthread_mutex_unlock(&J->lock);
    return i;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    int64_t hd = (int64_t)J->heads * J->dim;
    double *qd = (double *)malloc(sizeof(double) * hd);
    scored_key *buf = NULL;
    int64_t cap = 0;
    if (!qd) { J->status = -1; return NULL; }
    for (;;) {
        int64_t i = take_row(J);
        if (i >= J->nlist) break;
        int64_t r = J->row_list[i];
        for (int64_t t = 0; t < hd; ++t) qd[t] = g_e4m3[J->q[r * hd + t]];
        int64_t s = J->starts[r], e = J->ends[r];
        /* an empty or reversed range sees no key */
        int64_t n = e > s ? e - s : 0;
        if (J->scores_out) {
            double *row = J->scores_out + i * J->keys;
            for (int64_t j = 0; j < J->keys; ++j) row[j] = -INFINITY;
        }
        if (n > cap) {
            free(buf);
            cap = n;
            buf = (scored_key *)malloc(sizeof(scored_key) * (size_t)cap);
            if (!buf) { J->status = -1; free(qd); return NULL; }
        }
        int64_t nv = 0; /* visible keys written to buf */
        for (int64_t t = 0; t < n; ++t) {
            int64_t j = s + t;
            if (J->mask) {
                const uint32_t word = J->mask[r * J->mask_words + (j >> 8)];
                if (!((word >> ((j >> 3) & 31)) & 1u)) continue;
            }
            uint32_t bits = ((uint32_t)J->scale_groups[4 * j]) << 23;
            float sc;
            memcpy(&sc, &bits, sizeof sc);
            double v = score_pair(qd, J->k, J->heads, J->dim, J->w + r * J->heads, (double)sc, j);
            if (buf) { buf[nv].score = v; buf[nv].key = j; }
            ++nv;
            if (J->scores_out) J->scores_out[i * J->keys + j] = v;
        }
        if (J->out && J->block_mode) {
            /* blocks [s / 8, (e - 1) / 8]; buf holds the row's visible keys */
            int64_t b0 = s >> 3, nb = n > 0 ? ((e - 1) >> 3) - b0 + 1 : 0;
            scored_block *blk = nb > 0 ? (scored_block *)malloc(sizeof(scored_block) * (size_t)nb) : NULL;
            if (nb > 0 && !blk) { J->status = -1; break; }
            for (int64_t b = 0; b < nb; ++b) { blk[b].score = -INFINITY; blk[b].block = b0 + b; }
            for (int64_t t = 0; t < nv; ++t) {
                int64_t b = (buf[t].key >> 3) - b0;
                if (buf[t].score > blk[b].score) blk[b].score = buf[t].score;
            }
            if (nb > 0) qsort(blk, (size_t)nb, sizeof(scored_block), cmp_block);
            int64_t c = nb < J->topk ? nb : J->topk;
            int32_t *o = J->out + i * J->topk;
            for (int64_t t = 0; t < c; ++t) o[t] = (int32_t)(blk[t].block - b0);
            for (int64_t t = c; t < J->topk; ++t) o[t] = -1;
            free(blk);
        } else if (J->out) {
            if (nv > 0) qsort(buf, (size_t)nv, sizeof(scored_key), cmp_scored);
            int64_t c = nv < J->topk ? nv : J->topk;
            int32_t *o = J->out + i * J->topk;
            for (int64_t t = 0; t < c; ++t) o[t] = (int32_t)(buf[t].key - s);
            for (int64_t t = c; t < J->topk; ++t) o[t] = -1;
        }
    }
    free(buf);
    free(qd);
    return NULL;
}

static int run_jobs(job_t *J, int nthreads) {
    pthread_once(&g_table_once, build_table);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    pthread_mutex_init(&J->lock, NULL);
    J->next = 0;
    J->status = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, J) != 0) break;
        ++started;
    }
    if (started == 0) worker(J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J->lock);
    return J->status;
}

/* Top-k and/or dense scores of the listed rows.
 *  out    (nullable) [nlist, topk]: indices relative to the row's start, the
 *         c = min(topk, n) selected keys first (by score, ties by key), then -1.
 *  scores (nullable) [nlist, keys]: fp64 S(r, j), -inf outside [start, end).
 * A row whose range is empty or reversed sees no key.  A non-empty range that
 * leaves [0, keys) is rejected (-3).  Returns 0 on success. */
static int run_mode(const uint8_t *q, const uint8_t *k, const uint8_t *scale_groups,
                    const float *w, const int32_t *starts, const int32_t *ends,
                    const int64_t *row_list, int64_t nlist, int64_t keys,
                    int heads, int dim, int topk, int32_t *out, double *scores, int nthreads,
                    int block_mode, const uint32_t *mask, int64_t mask_words) {
    if (dim > 1024 || heads < 1 || dim < 1 || (out && topk < 1)) return -2;
    for (int64_t i = 0; i < nlist; ++i) {
        int64_t r = row_list[i];
        if ((starts[r] < 0 || ends[r] > keys) && ends[r] > starts[r]) return -3;
    }
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.scale_groups = scale_groups; J.w = w;
    J.starts = starts; J.ends = ends; J.row_list = row_list; J.nlist = nlist;
    J.keys = keys; J.heads = heads; J.dim = dim; J.topk = topk > 0 ? topk : 1;
    J.out = out; J.scores_out = scores; J.block_mode = block_mode;
    J.mask = mask; J.mask_words = mask_words;
    return run_jobs(&J, nthreads);
}

int oracle_run(const uint8_t *q, const uint8_t *k, const uint8_t *scale_groups,
               const float *w, const int32_t *starts, const int32_t *ends,
               const int64_t *row_list, int64_t nlist, int64_t keys,
               int heads, int dim, int topk, int32_t *out, double *scores, int nthreads) {
    return run_mode(q, k, scale_groups, w, starts, ends, row_list, nlist, keys, heads, dim, topk,
                    out, scores, nthreads, 0, NULL, 0);
}

/* Masked selection (see the header): mask [rows, mask_words] indexed by the
 * row's position in q, mask_words >= ceil(keys / 256).  out and scores as
 * oracle_run, scores of masked keys are -inf. */
int oracle_run_masked(const uint8_t *q, const uint8_t *k, const uint8_t *scale_groups,
                      const float *w, const int32_t *starts, const int32_t *ends,
                      const int64_t *row_list, int64_t nlist, int64_t keys,
                      int heads, int dim, int topk, const uint32_t *mask, int64_t mask_words,
                      int32_t *out, double *scores, int nthreads) {
    if (!mask || mask_words * 256 < keys) return -2;
    return run_mode(q, k, scale_groups, w, starts, ends, row_list, nlist, keys, heads, dim, topk,
                    out, scores, nthreads, 0, mask, mask_words);
}

/* Top `btopk` blocks of 8 keys per listed row by block score (see the header):
 * out_blocks [nlist, btopk] receives b - floor(start / 8), -1 padded. */
int oracle_run_blocks(const uint8_t *q, const uint8_t *k, const uint8_t *scale_groups,
                      const float *w, const int32_t *starts, const int32_t *ends,
                      const int64_t *row_list, int64_t nlist, int64_t keys,
                      int heads, int dim, int btopk, int32_t *out_blocks, int nthreads) {
    if (!out_blocks) return -2;
    return run_mode(q, k, scale_groups, w, starts, ends, row_list, nlist, keys, heads, dim, btopk,
                    out_blocks, NULL, nthreads, 1, NULL, 0);
}


/* ---- the fold --------------------------------------------------------------
 * vLLM pull request #60618, "What this PR does", Scoring bullet: since
 * relu(s) = (s + |s|) / 2, the weighted sum of the heads' linear halves is one
 * query (the heads folded with their weights) times the key, which can run on
 * the tensor core, leaving only the |s| terms to the math warps:
 *     sum_h w_h relu(s_h) = ( v . k + sum_h w_h |s_h| ) / 2,  v = sum_h w_h q_h.
 * The pages give no format for v on the tensor core.  Reading: v is formed in
 * fp32 with one fused multiply-add per head, heads in order (the e4m3 codes
 * below are decided in that precision, the kernel's), and written as `terms`
 * e4m3 vectors with power-of-two scales: term t has exponent e_t, the
 * smallest integer with max_d |r_t[d]| * 2^-e_t <= 448 (0 when r_t is zero),
 * codes u_t[d] = e4m3 round-to-nearest-even of r_t[d] * 2^-e_t, and
 * r_{t+1} = r_t - 2^e_t * E(u_t) (exact in fp32).  beta is the 2-norm of the
 * last residual: |v . k - sum_t 2^e_t E(u_t) . k| <= beta * |k|_2. */

/* e4m3fn code nearest to x (|x| <= 448), ties to the even code, by search over
 * the table; the sign of a zero result follows x. */
uint8_t oracle_e4m3_encode(double x) {
    pthread_once(&g_table_once, build_table);
    const int neg = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 0x7F; ++c) { /* non-negative finite codes 0x00..0x7E */
        const double d = fabs(g_e4m3[c] - a);
        if (d < bd || (d == bd && (c & 1u) == 0u)) {
            bd = d;
            best = c;
        }
    }
    return (uint8_t)(best | (neg ? 0x80u : 0u));
}

/* smallest integer e with m * 2^-e <= 448, for m > 0 */
static int fold_exponent(double m) {
    int ex;
    const double f = frexp(m, &ex); /* m = f * 2^ex, f in [0.5, 1) */
    return ex - 9 + (f > 0.875 ? 1 : 0);
}

void oracle_fold_prep(const uint8_t *q, const float *w, int64_t rows, int heads, int dim, int terms,
                      uint8_t *codes, int32_t *exps, float *v_out, double *beta) {
    pthread_once(&g_table_once, build_table);
    float *r = (float *)malloc(sizeof(float) * (size_t)dim);
    for (int64_t row = 0; row < rows; ++row) {
        for (int d = 0; d < dim; ++d) {
            float acc = 0.0f;
            for (int h = 0; h < heads; ++h)
                acc = fmaf(w[row * heads + h], (float)g_e4m3[q[(row * heads + h) * (int64_t)dim + d]], acc);
            r[d] = acc;
            if (v_out) v_out[row * dim + d] = acc;
        }
        for (int t = 0; t < terms; ++t) {
            float m = 0.0f;
            for (int d = 0; d < dim; ++d) m = fmaxf(m, fabsf(r[d]));
            const int e = m > 0.0f ? fold_exponent((double)m) : 0;
            exps[row * terms + t] = e;
            uint8_t *u = codes + (row * terms + t) * (int64_t)dim;
            for (int d = 0; d < dim; ++d) {
                u[d] = oracle_e4m3_encode(ldexp((double)r[d], -e));
                r[d] = r[d] - (float)ldexp(g_e4m3[u[d]], e);
            }
        }
        double s = 0.0;
        for (int d = 0; d < dim; ++d) s += (double)r[d] * (double)r[d];
        beta[row] = sqrt(s);
    }
    free(r);
}

/* Score of one pair through the fold (what a folded kernel computes, in fp64):
 * scale_j * ( sum_t 2^e_t E(u_t) . E(k_j) + sum_h w_h |s_h| ) / 2. */
double oracle_fold_score(const uint8_t *q, const uint8_t *k, const uint8_t *scale_groups, const float *w,
                         const uint8_t *codes, const int32_t *exps, int heads, int dim, int terms,
                         int64_t row, int64_t key) {
    pthread_once(&g_table_once, build_table);
    const uint8_t *kr = k + key * (int64_t)dim;
    double lin = 0.0;
    for (int t = 0; t < terms; ++t) {
        const uint8_t *u = codes + (row * terms + t) * (int64_t)dim;
        double acc = 0.0;
        for (int d = 0; d < dim; ++d) acc += g_e4m3[u[d]] * g_e4m3[kr[d]];
        lin += ldexp(acc, exps[row * terms + t]);
    }
    double ab = 0.0;
    for (int h = 0; h < heads; ++h) {
        const uint8_t *qr = q + (row * heads + h) * (int64_t)dim;
        double acc = 0.0;
        for (int d = 0; d < dim; ++d) acc += g_e4m3[qr[d]] * g_e4m3[kr[d]];
        ab += (double)w[row * heads + h] * fabs(acc);
    }
    uint32_t bits = ((uint32_t)scale_groups[4 * key]) << 23;
    float sc;
    memcpy(&sc, &bits, sizeof sc);
    return (double)sc * 0.5 * (lin + ab);
}
