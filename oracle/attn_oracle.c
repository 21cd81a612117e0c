/*
 * attn_oracle.c -- plain fp64 CPU attention, the parity oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * path under split_flash_decoding_gb300/csrc.
 *
 * What it computes (the plain definition, no blocking, no online softmax, no
 * split-K):
 *
 *   For sequence b, query row i (0 <= i < n_b), query head h, KV head
 *   k = h / group (group counts the query heads that share one KV head,
 *   mha_sm100_dispatch, Parameters; mha_decoding_single_batch_pipelined,
 *   Parameters):
 *
 *     J      = { j : 0 <= j < L_b, and j <= L_b - n_b + i when causal }
 *     s_j    = scale * sum_c q[c] * K[j, k, c]         (scale multiplies
 *              Q K^T ahead of the softmax, mha_sm100_dispatch, Args)
 *     t      = sink[h] if sinks are given, else -inf
 *     M      = max(max_{j in J} s_j, t)
 *     Z      = sum_{j in J} exp(s_j - M) + exp(t - M)
 *     out[c] = sum_{j in J} exp(s_j - M) * V[j, k, c] / Z
 *     lse    = M + ln Z
 *
 *   An empty J with no sink gives out = 0 and lse = -inf.  MLA is the same
 *   with one KV head, a 576-deep K and V = K[:, :512], passed here as a V
 *   operand that aliases K with dim_v = 512 (V is the leading depth_v
 *   channels of K, flare_mla_decoding_dispatch, Args: k).
 *
 *   Logical token t of sequence b lives at physical row
 *   page_table[b][t / page_size] * page_size + t % page_size of the cache
 *   (the KV operand type carries the page size, mha_sm100_dispatch,
 *   Parameters: KVType); with no page table the page index is b.
 *
 *   Sparse top-k (flare_mla_decoding_dispatch, Parameters: sparse; Args:
 *   d_indices, indices_stride, topk_lengths): sequence b attends only to the
 *   L_b = topk_lengths[b] cache rows that its index list names.  Its logical
 *   token t (t < L_b) is physical row r = indices[b * indices_stride + t],
 *   which sits in slot r % page_size of page r / page_size; entries past L_b
 *   are never read.  With that mapping the definition above applies as it
 *   stands (kv_len = topk_lengths, no causal mask for a single query row).
 *
 * oracle_partials computes the per-partition statistics that the split-K
 * method keeps (each key slice leaves its running maximum and exponential
 * sum behind, mha_decoding_single_batch_pipelined, summary): for a key slice S,
 *   m_S = max_{j in S cap J} s_j,  l_S = sum exp(s_j - m_S),
 *   O_S[c] = sum exp(s_j - m_S) V[j, c]   (unnormalised),
 * and (-inf, 0, 0) for an empty slice.
 *
 * oracle_spread gives, for the exact result above, the quantities that bound
 * how far an implementation that rounds its weights may land from it (the
 * tolerance of the parity tests is stated in terms of them; they are not part
 * of the attention definition).  With the exact weights w_j = exp(s_j - M) / Z
 * (Z includes the sink, so the w_j sum to at most 1):
 *   sd[c]  = sqrt( sum_{j in J} w_j (V[j, k, c] - out[c])^2 ),
 *   am[c]  = sum_{j in J} w_j |V[j, k, c]|,
 * and per (row, head): the visible key count |J|, the largest magnitude sum
 * scale * sum_c |q[c] K[j, k, c]| over J, and the largest |s_j|.
 *
 * Inputs are bf16 bit patterns (uint16); each one is widened exactly to
 * double.  All arithmetic is double; exp/log are the C library's.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const uint16_t *base;   /* bf16 bits */
    int64_t page_stride;    /* elements between pages (or sequences) */
    int64_t token_stride;   /* elements between tokens inside a page */
    int64_t head_stride;    /* elements between KV heads */
    int32_t page_size;      /* tokens per page */
    int32_t _pad;
    const int32_t *page_table; /* [batch][max_pages] or NULL: page = b */
    int64_t max_pages;
    const int32_t *indices;    /* sparse: [batch][indices_stride] physical rows, or NULL */
    int64_t indices_stride;
} oracle_kv;

typedef struct {
    const uint16_t *q;          /* [rows][num_q_heads][dim_qk] bf16 bits */
    const oracle_kv *k;
    const oracle_kv *v;
    const int32_t *kv_len;      /* [batch] */
    const int32_t *q_row_offsets; /* [batch+1] or NULL (one row per seq) */
    int32_t batch, num_q_heads, group, dim_qk, dim_v, causal;
    double scale;
    const double *sink;         /* [num_q_heads] or NULL */
} oracle_problem;

static double bf16_to_double(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static const uint16_t *kv_row(const oracle_kv *kv, int b, int64_t t, int head) {
    int64_t page, slot;
    if (kv->indices) {
        int64_t r = kv->indices[(int64_t)b * kv->indices_stride + t];
        page = r / kv->page_size;
        slot = r % kv->page_size;
    } else if (kv->page_table) {
        page = kv->page_table[(int64_t)b * kv->max_pages + t / kv->page_size];
        slot = t % kv->page_size;
    } else {
        page = b;
        slot = t;
    }
    return kv->base + page * kv->page_stride + slot * kv->token_stride +
           (int64_t)head * kv->head_stride;
}

static void row_of(const oracle_problem *pr, int64_t row, int *b_out, int *i_out, int *n_out) {
    if (!pr->q_row_offsets) {
        *b_out = (int)row; *i_out = 0; *n_out = 1;
        return;
    }
    int lo = 0, hi = pr->batch; /* find b with off[b] <= row < off[b+1] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (pr->q_row_offsets[mid] <= row) lo = mid; else hi = mid;
    }
    *b_out = lo;
    *i_out = (int)(row - pr->q_row_offsets[lo]);
    *n_out = pr->q_row_offsets[lo + 1] - pr->q_row_offsets[lo];
}

/* Number of visible keys of query row i of a sequence with n rows and L keys. */
static int64_t visible_keys(const oracle_problem *pr, int64_t L, int i, int n) {
    if (!pr->causal) return L;
    int64_t lim = L - n + i + 1;  /* keys j <= L - n + i */
    if (lim < 0) lim = 0;
    return lim < L ? lim : L;
}

/* Scores s_j for j in [0, nvis) into s[]. */
static void scores(const oracle_problem *pr, int b, int64_t row, int h, int64_t nvis,
                   double *s, double *qd) {
    int kh = h / pr->group;
    const uint16_t *qp = pr->q + (row * pr->num_q_heads + h) * (int64_t)pr->dim_qk;
    for (int c = 0; c < pr->dim_qk; ++c) qd[c] = bf16_to_double(qp[c]);
    for (int64_t j = 0; j < nvis; ++j) {
        const uint16_t *kp = kv_row(pr->k, b, j, kh);
        double acc = 0.0;
        for (int c = 0; c < pr->dim_qk; ++c) acc += qd[c] * bf16_to_double(kp[c]);
        s[j] = pr->scale * acc;
    }
}

typedef struct {
    const oracle_problem *pr;
    /* full attention */
    const int64_t *rows;   /* sample rows or NULL */
    const int32_t *heads;  /* sample heads or NULL */
    int64_t num_items;
    double *out, *lse;
    /* error-bound statistics (oracle_spread) */
    double *sd, *am, *stats;
    /* partials */
    const int64_t *bounds; /* [num_parts+1] key boundaries, or NULL */
    int32_t num_parts;
    int64_t num_rows;
    double *ws_o, *ws_m, *ws_l;
    /* threading */
    int tid, nthreads;
    int64_t max_keys;
    int status;
} worker_arg;

static void attention_item(worker_arg *a, int64_t item, double *s, double *qd) {
    const oracle_problem *pr = a->pr;
    int64_t row;
    int h;
    if (a->rows) { row = a->rows[item]; h = a->heads[item]; }
    else { row = item / pr->num_q_heads; h = (int)(item % pr->num_q_heads); }
    int b, i, n;
    row_of(pr, row, &b, &i, &n);
    int64_t L = pr->kv_len[b];
    int64_t nvis = visible_keys(pr, L, i, n);
    scores(pr, b, row, h, nvis, s, qd);

    double t = pr->sink ? pr->sink[h] : -INFINITY;
    double M = t;
    for (int64_t j = 0; j < nvis; ++j) if (s[j] > M) M = s[j];

    double *o = a->out + item * (int64_t)pr->dim_v;
    for (int c = 0; c < pr->dim_v; ++c) o[c] = 0.0;
    if (M == -INFINITY) {           /* nothing visible and no sink */
        a->lse[item] = -INFINITY;
        return;
    }
    double Z = exp(t - M);          /* exp(-inf) = 0 when there is no sink */
    int kh = h / pr->group;
    for (int64_t j = 0; j < nvis; ++j) {
        double w = exp(s[j] - M);
        Z += w;
        const uint16_t *vp = kv_row(pr->v, b, j, kh);
        for (int c = 0; c < pr->dim_v; ++c) o[c] += w * bf16_to_double(vp[c]);
    }
    for (int c = 0; c < pr->dim_v; ++c) o[c] /= Z;
    a->lse[item] = M + log(Z);
}

static void spread_item(worker_arg *a, int64_t item, double *s, double *qd) {
    const oracle_problem *pr = a->pr;
    int64_t row = a->rows[item];
    int h = a->heads[item];
    int b, i, n;
    row_of(pr, row, &b, &i, &n);
    int64_t L = pr->kv_len[b];
    int64_t nvis = visible_keys(pr, L, i, n);
    scores(pr, b, row, h, nvis, s, qd);
    int kh = h / pr->group;

    /* magnitudes of the scores and of their products */
    double sabs = 0.0, smax = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const uint16_t *kp = kv_row(pr->k, b, j, kh);
        double acc = 0.0;
        for (int c = 0; c < pr->dim_qk; ++c) acc += fabs(qd[c] * bf16_to_double(kp[c]));
        acc *= fabs(pr->scale);
        if (acc > sabs) sabs = acc;
        if (fabs(s[j]) > smax) smax = fabs(s[j]);
    }
    double *st = a->stats + item * 3;
    st[0] = (double)nvis;
    st[1] = sabs;
    st[2] = smax;

    double *sd = a->sd + item * (int64_t)pr->dim_v;
    double *am = a->am + item * (int64_t)pr->dim_v;
    for (int c = 0; c < pr->dim_v; ++c) { sd[c] = 0.0; am[c] = 0.0; }
    double t = pr->sink ? pr->sink[h] : -INFINITY;
    double M = t;
    for (int64_t j = 0; j < nvis; ++j) if (s[j] > M) M = s[j];
    if (M == -INFINITY) return;     /* no weights at all */
    double Z = exp(t - M);
    for (int64_t j = 0; j < nvis; ++j) Z += exp(s[j] - M);
    /* out[c] first (am holds it for now), then the spread around it */
    for (int64_t j = 0; j < nvis; ++j) {
        double w = exp(s[j] - M) / Z;
        const uint16_t *vp = kv_row(pr->v, b, j, kh);
        for (int c = 0; c < pr->dim_v; ++c) am[c] += w * bf16_to_double(vp[c]);
    }
    for (int64_t j = 0; j < nvis; ++j) {
        double w = exp(s[j] - M) / Z;
        const uint16_t *vp = kv_row(pr->v, b, j, kh);
        for (int c = 0; c < pr->dim_v; ++c) {
            double d = bf16_to_double(vp[c]) - am[c];
            sd[c] += w * d * d;
        }
    }
    for (int c = 0; c < pr->dim_v; ++c) { sd[c] = sqrt(sd[c]); am[c] = 0.0; }
    for (int64_t j = 0; j < nvis; ++j) {
        double w = exp(s[j] - M) / Z;
        const uint16_t *vp = kv_row(pr->v, b, j, kh);
        for (int c = 0; c < pr->dim_v; ++c) am[c] += w * fabs(bf16_to_double(vp[c]));
    }
}

static void partials_item(worker_arg *a, int64_t item, double *s, double *qd) {
    const oracle_problem *pr = a->pr;
    int64_t row = item / pr->num_q_heads;
    int h = (int)(item % pr->num_q_heads);
    int b, i, n;
    row_of(pr, row, &b, &i, &n);
    int64_t L = pr->kv_len[b];
    int64_t nvis = visible_keys(pr, L, i, n);
    scores(pr, b, row, h, nvis, s, qd);
    int kh = h / pr->group;
    for (int p = 0; p < a->num_parts; ++p) {
        int64_t lo = a->bounds[p], hi = a->bounds[p + 1];
        if (hi > nvis) hi = nvis;
        int64_t idx = ((int64_t)p * a->num_rows + row) * pr->num_q_heads + h;
        double *o = a->ws_o + idx * pr->dim_v;
        for (int c = 0; c < pr->dim_v; ++c) o[c] = 0.0;
        double m = -INFINITY, l = 0.0;
        for (int64_t j = lo; j < hi; ++j) if (s[j] > m) m = s[j];
        if (m != -INFINITY) {
            for (int64_t j = lo; j < hi; ++j) {
                double w = exp(s[j] - m);
                l += w;
                const uint16_t *vp = kv_row(pr->v, b, j, kh);
                for (int c = 0; c < pr->dim_v; ++c) o[c] += w * bf16_to_double(vp[c]);
            }
        }
        a->ws_m[idx] = m;
        a->ws_l[idx] = l;
    }
}

static void *worker(void *p) {
    worker_arg *a = (worker_arg *)p;
    double *s = (double *)malloc(sizeof(double) * (size_t)(a->max_keys > 0 ? a->max_keys : 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)a->pr->dim_qk);
    if (!s || !qd) { a->status = 1; free(s); free(qd); return NULL; }
    for (int64_t it = a->tid; it < a->num_items; it += a->nthreads) {
        if (a->bounds) partials_item(a, it, s, qd);
        else if (a->sd) spread_item(a, it, s, qd);
        else attention_item(a, it, s, qd);
    }
    free(s);
    free(qd);
    return NULL;
}

static int run(worker_arg *proto, int nthreads) {
    const oracle_problem *pr = proto->pr;
    int64_t max_keys = 0;
    for (int b = 0; b < pr->batch; ++b) if (pr->kv_len[b] > max_keys) max_keys = pr->kv_len[b];
    proto->max_keys = max_keys;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if (nthreads > proto->num_items && proto->num_items > 0) nthreads = (int)proto->num_items;
    worker_arg *args = (worker_arg *)calloc((size_t)nthreads, sizeof(worker_arg));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!args || !th) { free(args); free(th); return 1; }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t] = *proto;
        args[t].tid = t;
        args[t].nthreads = nthreads;
        args[t].status = 0;
    }
    if (nthreads == 1) {
        worker(&args[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &args[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t) status |= args[t].status;
    free(args);
    free(th);
    return status;
}

static int check_problem(const oracle_problem *pr) {
    if (!pr || !pr->q || !pr->k || !pr->v || !pr->kv_len) return 2;
    if (pr->batch < 0 || pr->num_q_heads <= 0 || pr->group <= 0) return 2;
    if (pr->num_q_heads % pr->group) return 2;
    if (pr->dim_qk <= 0 || pr->dim_v <= 0) return 2;
    if (pr->k->page_table && pr->k->page_size <= 0) return 2;
    if (pr->v->page_table && pr->v->page_size <= 0) return 2;
    return 0;
}

/*
 * Full attention.  With num_items == 0 every (row, head) is computed and out
 * is [rows][num_q_heads][dim_v], lse [rows][num_q_heads]; otherwise only the
 * listed (rows[i], heads[i]) pairs, and out is [num_items][dim_v].
 */
int oracle_attention(const oracle_problem *pr, const int64_t *rows, const int32_t *heads,
                     int64_t num_items, double *out, double *lse, int nthreads) {
    int st = check_problem(pr);
    if (st) return st;
    int64_t total_rows = pr->q_row_offsets ? pr->q_row_offsets[pr->batch] : pr->batch;
    worker_arg a;
    memset(&a, 0, sizeof a);
    a.pr = pr;
    if (num_items > 0) {
        a.rows = rows; a.heads = heads; a.num_items = num_items;
    } else {
        a.num_items = total_rows * pr->num_q_heads;
    }
    a.out = out;
    a.lse = lse;
    return run(&a, nthreads);
}

/*
 * Per-partition statistics for every (row, head): key slice p is
 * [bounds[p], bounds[p+1]) intersected with the row's visible keys.
 * ws_o is [num_parts][rows][num_q_heads][dim_v]; ws_m, ws_l are
 * [num_parts][rows][num_q_heads].
 */
int oracle_partials(const oracle_problem *pr, const int64_t *bounds, int num_parts,
                    double *ws_o, double *ws_m, double *ws_l, int nthreads) {
    int st = check_problem(pr);
    if (st) return st;
    if (!bounds || num_parts <= 0) return 2;
    int64_t total_rows = pr->q_row_offsets ? pr->q_row_offsets[pr->batch] : pr->batch;
    worker_arg a;
    memset(&a, 0, sizeof a);
    a.pr = pr;
    a.num_items = total_rows * pr->num_q_heads;
    a.bounds = bounds;
    a.num_parts = num_parts;
    a.num_rows = total_rows;
    a.ws_o = ws_o; a.ws_m = ws_m; a.ws_l = ws_l;
    return run(&a, nthreads);
}

/*
 * Error-bound statistics of the exact result for the listed (rows[i],
 * heads[i]) pairs: sd and am are [num_items][dim_v], stats [num_items][3] =
 * (visible keys, max_j scale * sum_c |q[c] K[j, c]|, max_j |s_j|).
 */
int oracle_spread(const oracle_problem *pr, const int64_t *rows, const int32_t *heads,
                  int64_t num_items, double *sd, double *am, double *stats, int nthreads) {
    int st = check_problem(pr);
    if (st) return st;
    if (num_items < 0 || (num_items > 0 && (!rows || !heads || !sd || !am || !stats)))
        return 2;
    if (num_items == 0) return 0;
    worker_arg a;
    memset(&a, 0, sizeof a);
    a.pr = pr;
    a.rows = rows; a.heads = heads; a.num_items = num_items;
    a.sd = sd; a.am = am; a.stats = stats;
    return run(&a, nthreads);
}
