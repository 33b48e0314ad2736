/*
 * attention_ref.c -- TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library. The product path (the CUDA library and its Python
 * binding) never calls it and shares no code, header or table with it.
 *
 * What it computes is the plain definition of exact scaled-dot-product
 * attention, written out row by row, in double precision, from the exact
 * values of the (fp16/bf16) inputs:
 *
 *   S_ij   = scale * sum_c Q_ic K_jc                 ("Flash Attention:
 *            revolutionizing transformer efficiency", standard attention
 *            listing: scores = Q K^T / sqrt(d_k))
 *   S_ij   = -inf where key j is masked for query i (causal: j > i;
 *            key padding: j >= kv_len[b]; block-sparse: the 128x128 block
 *            (i/blk, j/blk) has a zero mask entry)
 *   LSE_i  = ln sum_j exp(S_ij)    (evaluated as m + ln sum exp(S_ij - m),
 *            m = max_j S_ij: the softmax decomposition of the same page,
 *            section "The Math Behind Flash Attention", formula 1)
 *   P_ij   = exp(S_ij - LSE_i)     (softmax(scores), same listing)
 *   O_i    = sum_j P_ij V_j        (attention_weights @ V, same listing)
 *
 * A row with no kept key has O_i = 0 and LSE_i = -inf, and contributes
 * nothing to any gradient (the pages leave this case open; this is the
 * reading used throughout).
 *
 * Backward: the pages only say that the backward pass recomputes the
 * attention matrix instead of storing it ("Flash Attention:
 * revolutionizing transformer efficiency", key idea 2, Recomputation).
 * What it must produce is the gradient of the forward definition, which in
 * closed form (chain rule through softmax) is
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i
 *
 * Every loop below follows these lines directly. Work is split across
 * threads only over independent (head, row-range) tasks; the per-row
 * arithmetic is the same whatever the split, and partial dK/dV sums of the
 * row ranges are added in a fixed order, so results do not depend on the
 * thread count.
 *
 * Layout: every tensor is [B, H, N, d] row-major (d fastest), LSE and D
 * are [B, H, N]. kv_len is int32 [B] or NULL. block_mask is uint8
 * [nb * nb], nb = ceil(N / blk), row = query block, column = key block,
 * nonzero = keep, shared by all (b, h); NULL means no block mask.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    int B, H, N, d;
    double scale;
    int causal;
    const int32_t *kv_len;
    const uint8_t *block_mask;
    int blk;
} problem_t;

/* Is key j visible to query i of batch b? */
static int kept(const problem_t *p, int b, int i, int j)
{
    if (p->causal && j > i) return 0;
    if (p->kv_len && j >= p->kv_len[b]) return 0;
    if (p->block_mask) {
        int nb = (p->N + p->blk - 1) / p->blk;
        if (!p->block_mask[(size_t)(i / p->blk) * nb + (j / p->blk)]) return 0;
    }
    return 1;
}

/*
 * Scores, LSE and probabilities of one query row i of head (b, h).
 * s_row and p_row have N entries; masked keys get P = 0.
 * Returns LSE_i (-inf when the row has no kept key).
 */
static double row_probs(const problem_t *p, int b, const double *qh, const double *kh,
                        int i, double *s_row, double *p_row)
{
    const int N = p->N, d = p->d;
    const double *qi = qh + (size_t)i * d;
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (!kept(p, b, i, j)) { s_row[j] = -INFINITY; continue; }
        const double *kj = kh + (size_t)j * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s_row[j] = p->scale * acc;
        if (s_row[j] > m) m = s_row[j];
    }
    if (m == -INFINITY) {
        for (int j = 0; j < N; ++j) p_row[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int j = 0; j < N; ++j)
        if (s_row[j] != -INFINITY) l += exp(s_row[j] - m);
    const double lse = m + log(l);
    for (int j = 0; j < N; ++j)
        p_row[j] = (s_row[j] == -INFINITY) ? 0.0 : exp(s_row[j] - lse);
    return lse;
}

/* ------------------------------------------------------------------ */
/* forward                                                              */
/* ------------------------------------------------------------------ */

typedef struct {
    const problem_t *p;
    double *o, *lse;
    /* task list: rows [r0, r1) of head bh */
    int ntask, next;
    pthread_mutex_t mu;
    int rows_per_task;
} fwd_job_t;

static void fwd_rows(const problem_t *p, int bh, int r0, int r1, double *o, double *lse)
{
    const int N = p->N, d = p->d, b = bh / p->H;
    const size_t head = (size_t)bh * N * d;
    const double *qh = p->q + head, *kh = p->k + head, *vh = p->v + head;
    double *s_row = (double *)malloc(sizeof(double) * N);
    double *p_row = (double *)malloc(sizeof(double) * N);
    for (int i = r0; i < r1; ++i) {
        double l = row_probs(p, b, qh, kh, i, s_row, p_row);
        double *oi = o + head + (size_t)i * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = 0; j < N; ++j) {
            if (p_row[j] == 0.0) continue;
            const double *vj = vh + (size_t)j * d;
            for (int c = 0; c < d; ++c) oi[c] += p_row[j] * vj[c];
        }
        lse[(size_t)bh * N + i] = l;
    }
    free(s_row);
    free(p_row);
}

static void *fwd_worker(void *arg)
{
    fwd_job_t *job = (fwd_job_t *)arg;
    const problem_t *p = job->p;
    const int per_head = (p->N + job->rows_per_task - 1) / job->rows_per_task;
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int t = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (t >= job->ntask) break;
        int bh = t / per_head, chunk = t % per_head;
        int r0 = chunk * job->rows_per_task;
        int r1 = r0 + job->rows_per_task;
        if (r1 > p->N) r1 = p->N;
        fwd_rows(p, bh, r0, r1, job->o, job->lse);
    }
    return NULL;
}

static int run_threads(int nthreads, void *(*fn)(void *), void *arg)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) { fn(arg); return 0; }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, fn, arg) == 0) ++started;
    if (started == 0) fn(arg);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    return 0;
}

static int check_args(int B, int H, int N, int d, int blk)
{
    if (B < 0 || H < 0 || N < 0 || d < 1 || blk < 1) return -1;
    return 0;
}

/*
 * Full forward: o [B,H,N,d], lse [B,H,N]. Returns 0, or -1 on bad sizes.
 */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    int B, int H, int N, int d, double scale, int causal,
                    const int32_t *kv_len, const uint8_t *block_mask, int blk,
                    double *o, double *lse, int nthreads)
{
    if (check_args(B, H, N, d, blk)) return -1;
    if ((size_t)B * H * N == 0) return 0;
    problem_t p = {q, k, v, NULL, B, H, N, d, scale, causal, kv_len, block_mask, blk};
    fwd_job_t job;
    job.p = &p;
    job.o = o;
    job.lse = lse;
    job.rows_per_task = 64;
    job.ntask = B * H * ((N + 63) / 64);
    job.next = 0;
    pthread_mutex_init(&job.mu, NULL);
    run_threads(nthreads, fwd_worker, &job);
    pthread_mutex_destroy(&job.mu);
    return 0;
}

/*
 * Forward of selected rows of ONE head (arrays q, k, v are [N, d]).
 * kv_len_b < 0 means no key padding. rows[r] are query indices; outputs
 * o_rows [nrows, d], lse_rows [nrows].
 */
typedef struct {
    const problem_t *p;
    int b, nrows, next;
    const int64_t *rows;
    double *o_rows, *lse_rows;
    pthread_mutex_t mu;
} fwd_rows_job_t;

static void *fwd_rows_worker(void *arg)
{
    fwd_rows_job_t *job = (fwd_rows_job_t *)arg;
    const problem_t *p = job->p;
    const int N = p->N, d = p->d;
    double *s_row = (double *)malloc(sizeof(double) * N);
    double *p_row = (double *)malloc(sizeof(double) * N);
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int r = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (r >= job->nrows) break;
        int i = (int)job->rows[r];
        double l = row_probs(p, job->b, p->q, p->k, i, s_row, p_row);
        double *oi = job->o_rows + (size_t)r * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = 0; j < N; ++j) {
            if (p_row[j] == 0.0) continue;
            for (int c = 0; c < d; ++c) oi[c] += p_row[j] * p->v[(size_t)j * d + c];
        }
        job->lse_rows[r] = l;
    }
    free(s_row);
    free(p_row);
    return NULL;
}

int oracle_attn_fwd_rows(const double *q, const double *k, const double *v,
                         int N, int d, double scale, int causal, int kv_len_b,
                         const uint8_t *block_mask, int blk,
                         int nrows, const int64_t *rows,
                         double *o_rows, double *lse_rows, int nthreads)
{
    if (check_args(1, 1, N, d, blk) || nrows < 0) return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    int32_t len = kv_len_b;
    problem_t p = {q, k, v, NULL, 1, 1, N, d, scale, causal,
                   kv_len_b >= 0 ? &len : NULL, block_mask, blk};
    fwd_rows_job_t job;
    job.p = &p;
    job.b = 0;
    job.nrows = nrows;
    job.next = 0;
    job.rows = rows;
    job.o_rows = o_rows;
    job.lse_rows = lse_rows;
    pthread_mutex_init(&job.mu, NULL);
    run_threads(nthreads, fwd_rows_worker, &job);
    pthread_mutex_destroy(&job.mu);
    return 0;
}

/* ------------------------------------------------------------------ */
/* backward                                                             */
/* ------------------------------------------------------------------ */

/*
 * One task = rows [r0, r1) of head bh. It writes dQ and D of its rows
 * directly and accumulates its rows' contributions to dK and dV into its
 * own partial buffers (pk, pv, each [N, d]); the caller adds the partial
 * buffers of a head in task order.
 */
typedef struct {
    const problem_t *p;
    double *dq, *delta;
    double *part_k, *part_v; /* [ntask][N*d] */
    int ntask, next, rows_per_task;
    pthread_mutex_t mu;
} bwd_job_t;

static void bwd_rows(const problem_t *p, int bh, int r0, int r1,
                     double *dq, double *delta, double *pk, double *pv)
{
    const int N = p->N, d = p->d, b = bh / p->H;
    const size_t head = (size_t)bh * N * d;
    const double *qh = p->q + head, *kh = p->k + head, *vh = p->v + head;
    const double *doh = p->dout + head;
    double *s_row = (double *)malloc(sizeof(double) * N);
    double *p_row = (double *)malloc(sizeof(double) * N);
    double *dp_row = (double *)malloc(sizeof(double) * N);
    for (int j = 0; j < N * d; ++j) { pk[j] = 0.0; pv[j] = 0.0; }
    for (int i = r0; i < r1; ++i) {
        const double *qi = qh + (size_t)i * d;
        const double *doi = doh + (size_t)i * d;
        double *dqi = dq + head + (size_t)i * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        row_probs(p, b, qh, kh, i, s_row, p_row);
        /* dP_ij = dO_i . V_j and D_i = sum_j P_ij dP_ij */
        double D = 0.0;
        for (int j = 0; j < N; ++j) {
            const double *vj = vh + (size_t)j * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += doi[c] * vj[c];
            dp_row[j] = acc;
            D += p_row[j] * acc;
        }
        if (delta) delta[(size_t)bh * N + i] = D;
        for (int j = 0; j < N; ++j) {
            if (p_row[j] == 0.0) continue;
            const double ds = p_row[j] * (dp_row[j] - D);
            const double *kj = kh + (size_t)j * d;
            double *pkj = pk + (size_t)j * d, *pvj = pv + (size_t)j * d;
            for (int c = 0; c < d; ++c) {
                dqi[c] += p->scale * ds * kj[c];
                pkj[c] += p->scale * ds * qi[c];
                pvj[c] += p_row[j] * doi[c];
            }
        }
    }
    free(s_row);
    free(p_row);
    free(dp_row);
}

static void *bwd_worker(void *arg)
{
    bwd_job_t *job = (bwd_job_t *)arg;
    const problem_t *p = job->p;
    const int per_head = (p->N + job->rows_per_task - 1) / job->rows_per_task;
    const size_t nd = (size_t)p->N * p->d;
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int t = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (t >= job->ntask) break;
        int bh = t / per_head, chunk = t % per_head;
        int r0 = chunk * job->rows_per_task;
        int r1 = r0 + job->rows_per_task;
        if (r1 > p->N) r1 = p->N;
        bwd_rows(p, bh, r0, r1, job->dq, job->delta,
                 job->part_k + (size_t)t * nd, job->part_v + (size_t)t * nd);
    }
    return NULL;
}

/*
 * Full backward. Outputs dq, dk, dv [B,H,N,d]; delta [B,H,N] (may be NULL)
 * receives D_i = sum_j P_ij dP_ij. rows_per_task sets the row range of one
 * task (<= 0: whole heads). Returns 0, -1 on bad sizes, -2 if out of memory.
 */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int B, int H, int N, int d, double scale, int causal,
                    const int32_t *kv_len, const uint8_t *block_mask, int blk,
                    double *dq, double *dk, double *dv, double *delta,
                    int rows_per_task, int nthreads)
{
    if (check_args(B, H, N, d, blk)) return -1;
    if ((size_t)B * H * N == 0) return 0;
    problem_t p = {q, k, v, dout, B, H, N, d, scale, causal, kv_len, block_mask, blk};
    if (rows_per_task <= 0 || rows_per_task > N) rows_per_task = N;
    const int per_head = (N + rows_per_task - 1) / rows_per_task;
    const size_t nd = (size_t)N * d;
    bwd_job_t job;
    job.p = &p;
    job.dq = dq;
    job.delta = delta;
    job.rows_per_task = rows_per_task;
    job.ntask = B * H * per_head;
    job.next = 0;
    job.part_k = (double *)malloc(sizeof(double) * nd * job.ntask);
    job.part_v = (double *)malloc(sizeof(double) * nd * job.ntask);
    if (!job.part_k || !job.part_v) {
        free(job.part_k);
        free(job.part_v);
        return -2;
    }
    pthread_mutex_init(&job.mu, NULL);
    run_threads(nthreads, bwd_worker, &job);
    pthread_mutex_destroy(&job.mu);
    for (int bh = 0; bh < B * H; ++bh) {
        double *dkh = dk + (size_t)bh * nd, *dvh = dv + (size_t)bh * nd;
        for (size_t e = 0; e < nd; ++e) { dkh[e] = 0.0; dvh[e] = 0.0; }
        for (int c = 0; c < per_head; ++c) {
            const double *pk = job.part_k + (size_t)(bh * per_head + c) * nd;
            const double *pv = job.part_v + (size_t)(bh * per_head + c) * nd;
            for (size_t e = 0; e < nd; ++e) { dkh[e] += pk[e]; dvh[e] += pv[e]; }
        }
    }
    free(job.part_k);
    free(job.part_v);
    return 0;
}

/* ------------------------------------------------------------------ */
/* backward on sampled rows / columns of ONE head                       */
/* ------------------------------------------------------------------ */

/*
 * For large heads the full backward is too slow, but single outputs are
 * cheap once every row's LSE_i and D_i is known:
 *   dQ_i = scale * sum_j P_ij (dP_ij - D_i) K_j           (one row i)
 *   dK_j = scale * sum_i P_ij (dP_ij - D_i) Q_i            (one key j)
 *   dV_j = sum_i P_ij dO_i                                 (one key j)
 * with P_ij = exp(S_ij - LSE_i) for kept (i, j), else 0. Arrays are [N, d]
 * of one head; kv_len_b < 0 means no key padding.
 */
typedef struct {
    const problem_t *p;
    double *lse, *D;
    int next;
    pthread_mutex_t mu;
} stats_job_t;

static void *stats_worker(void *arg)
{
    stats_job_t *job = (stats_job_t *)arg;
    const problem_t *p = job->p;
    const int N = p->N, d = p->d;
    double *s_row = (double *)malloc(sizeof(double) * N);
    double *p_row = (double *)malloc(sizeof(double) * N);
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int i0 = job->next;
        job->next += 16;
        pthread_mutex_unlock(&job->mu);
        if (i0 >= N) break;
        for (int i = i0; i < i0 + 16 && i < N; ++i) {
            job->lse[i] = row_probs(p, 0, p->q, p->k, i, s_row, p_row);
            const double *doi = p->dout + (size_t)i * d;
            double D = 0.0;
            for (int j = 0; j < N; ++j) {
                if (p_row[j] == 0.0) continue;
                const double *vj = p->v + (size_t)j * d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += doi[c] * vj[c];
                D += p_row[j] * acc;
            }
            job->D[i] = D;
        }
    }
    free(s_row);
    free(p_row);
    return NULL;
}

typedef struct {
    const problem_t *p;
    const double *lse, *D;
    int nq, nk, next;
    const int64_t *qrows, *kcols;
    double *dq_rows, *dk_rows, *dv_rows;
    pthread_mutex_t mu;
} sample_job_t;

static void *sample_worker(void *arg)
{
    sample_job_t *job = (sample_job_t *)arg;
    const problem_t *p = job->p;
    const int N = p->N, d = p->d;
    double *s_row = (double *)malloc(sizeof(double) * N);
    double *p_row = (double *)malloc(sizeof(double) * N);
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int t = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (t >= job->nq + job->nk) break;
        if (t < job->nq) {
            const int i = (int)job->qrows[t];
            const double *doi = p->dout + (size_t)i * d;
            double *dqi = job->dq_rows + (size_t)t * d;
            for (int c = 0; c < d; ++c) dqi[c] = 0.0;
            row_probs(p, 0, p->q, p->k, i, s_row, p_row);
            for (int j = 0; j < N; ++j) {
                if (p_row[j] == 0.0) continue;
                const double *vj = p->v + (size_t)j * d;
                double dp = 0.0;
                for (int c = 0; c < d; ++c) dp += doi[c] * vj[c];
                const double ds = p_row[j] * (dp - job->D[i]);
                for (int c = 0; c < d; ++c) dqi[c] += p->scale * ds * p->k[(size_t)j * d + c];
            }
        } else {
            const int u = t - job->nq;
            const int j = (int)job->kcols[u];
            const double *kj = p->k + (size_t)j * d, *vj = p->v + (size_t)j * d;
            double *dkj = job->dk_rows + (size_t)u * d, *dvj = job->dv_rows + (size_t)u * d;
            for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
            for (int i = 0; i < N; ++i) {
                if (!kept(p, 0, i, j) || job->lse[i] == -INFINITY) continue;
                const double *qi = p->q + (size_t)i * d, *doi = p->dout + (size_t)i * d;
                double s = 0.0, dp = 0.0;
                for (int c = 0; c < d; ++c) { s += qi[c] * kj[c]; dp += doi[c] * vj[c]; }
                const double P = exp(p->scale * s - job->lse[i]);
                const double ds = P * (dp - job->D[i]);
                for (int c = 0; c < d; ++c) {
                    dkj[c] += p->scale * ds * qi[c];
                    dvj[c] += P * doi[c];
                }
            }
        }
    }
    free(s_row);
    free(p_row);
    return NULL;
}

int oracle_attn_bwd_sampled(const double *q, const double *k, const double *v, const double *dout,
                            int N, int d, double scale, int causal, int kv_len_b,
                            const uint8_t *block_mask, int blk,
                            int nq, const int64_t *qrows, double *dq_rows,
                            int nk, const int64_t *kcols, double *dk_rows, double *dv_rows,
                            double *lse_out, double *delta_out, int nthreads)
{
    if (check_args(1, 1, N, d, blk) || nq < 0 || nk < 0) return -1;
    for (int r = 0; r < nq; ++r) if (qrows[r] < 0 || qrows[r] >= N) return -1;
    for (int r = 0; r < nk; ++r) if (kcols[r] < 0 || kcols[r] >= N) return -1;
    if (N == 0) return 0;
    int32_t len = kv_len_b;
    problem_t p = {q, k, v, dout, 1, 1, N, d, scale, causal,
                   kv_len_b >= 0 ? &len : NULL, block_mask, blk};
    double *lse = (double *)malloc(sizeof(double) * N);
    double *D = (double *)malloc(sizeof(double) * N);
    if (!lse || !D) { free(lse); free(D); return -2; }
    stats_job_t sj;
    sj.p = &p;
    sj.lse = lse;
    sj.D = D;
    sj.next = 0;
    pthread_mutex_init(&sj.mu, NULL);
    run_threads(nthreads, stats_worker, &sj);
    pthread_mutex_destroy(&sj.mu);
    sample_job_t job;
    job.p = &p;
    job.lse = lse;
    job.D = D;
    job.nq = nq;
    job.nk = nk;
    job.next = 0;
    job.qrows = qrows;
    job.kcols = kcols;
    job.dq_rows = dq_rows;
    job.dk_rows = dk_rows;
    job.dv_rows = dv_rows;
    pthread_mutex_init(&job.mu, NULL);
    run_threads(nthreads, sample_worker, &job);
    pthread_mutex_destroy(&job.mu);
    if (lse_out) memcpy(lse_out, lse, sizeof(double) * N);
    if (delta_out) memcpy(delta_out, D, sizeof(double) * N);
    free(lse);
    free(D);
    return 0;
}
