/*
 * Exact softmax attention, plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the plain definition, no tiling, no online recurrence):
 *   for every query row i of every (b, h):
 *     s_j   = scale * sum_t q[i,t] * k[j,t]            for all keys j < N
 *             ("understand-flashattention", forward-pass formulas S = Q K^T;
 *              the scale is applied to the scores after the matmul and before
 *              the mask, as in "PyTorch profiling part 3: attention",
 *              section "Naive attention", steps 1-3)
 *     vis_j = (!causal || j <= i) && j < key_len[b]    (same section, step 3:
 *              masked scores are -inf; the key-padding form follows the
 *              "Linear Attention CUDA kernel" page, key_lengths mask on K)
 *     m     = max over visible j of s_j                 ("understand-flashattention",
 *     l     = sum over visible j of exp(s_j - m)         section "numerically stable
 *     p_j   = exp(s_j - m) / l  (0 for masked j)         softmax", key statistics)
 *     o     = sum_j p_j v[j,:]                          (forward pass, O = P V)
 *     lse   = m + log(l)   (natural log)                ("understand-flashattention",
 *                                                        logsumexp derivation, step 8)
 *   A row with no visible key gets o = 0 and lse = -inf: the "safe softmax"
 *   convention of "PyTorch profiling part 3: attention", section "The safe softmax".
 *
 * Masked terms are left out of the max and the sum rather than carried as
 * -inf; the two readings give the same numbers and this one needs no inf
 * arithmetic.
 *
 * Inputs are bfloat16 bit patterns; each is widened to double exactly
 * (a bf16 value is the upper half of an IEEE binary32).
 *
 * Threads: plain pthreads over independent query rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t B, H, N, d;
    double scale;
    int causal;
    const int32_t *key_len;
    const int64_t *rows;   /* flat row ids into [B*H*N], or NULL for all */
    int64_t n_rows;
    double *o, *lse;
    int64_t begin, end;    /* this worker's slice of [0, n_rows) */
    int status;
} oracle_job;

/* One query row, the plain definition written out. */
static void one_row(const oracle_job *J, int64_t flat, double *s, double *qrow,
                    double *o_out, double *lse_out)
{
    const int64_t N = J->N, d = J->d;
    const int64_t bh = flat / N;
    const int64_t i = flat % N;
    const int64_t b = bh / J->H;
    const uint16_t *qp = J->q + flat * d;
    const uint16_t *kp = J->k + bh * N * d;
    const uint16_t *vp = J->v + bh * N * d;

    int64_t klen = N;
    if (J->key_len) {
        klen = J->key_len[b];
        if (klen < 0) klen = 0;
        if (klen > N) klen = N;
    }

    for (int64_t t = 0; t < d; ++t) qrow[t] = bf16_bits_to_double(qp[t]);

    /* 1. the full score row, scaled */
    for (int64_t j = 0; j < N; ++j) {
        double acc = 0.0;
        const uint16_t *kj = kp + j * d;
        for (int64_t t = 0; t < d; ++t) acc += qrow[t] * bf16_bits_to_double(kj[t]);
        s[j] = J->scale * acc;
    }

    /* 2.-3. visibility, row max, normaliser */
    int any = 0;
    double m = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        int vis = (!J->causal || j <= i) && j < klen;
        if (!vis) continue;
        if (!any || s[j] > m) m = s[j];
        any = 1;
    }
    for (int64_t t = 0; t < d; ++t) o_out[t] = 0.0;
    if (!any) {
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        int vis = (!J->causal || j <= i) && j < klen;
        if (vis) l += exp(s[j] - m);
    }

    /* 4. o = sum_j p_j v_j */
    for (int64_t j = 0; j < N; ++j) {
        int vis = (!J->causal || j <= i) && j < klen;
        if (!vis) continue;
        double p = exp(s[j] - m) / l;
        const uint16_t *vj = vp + j * d;
        for (int64_t t = 0; t < d; ++t) o_out[t] += p * bf16_bits_to_double(vj[t]);
    }

    /* 5. natural-log LSE */
    *lse_out = m + log(l);
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->N);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)J->d);
    if (!s || !qrow) {
        free(s);
        free(qrow);
        J->status = 2;
        return NULL;
    }
    for (int64_t r = J->begin; r < J->end; ++r) {
        int64_t flat = J->rows ? J->rows[r] : r;
        one_row(J, flat, s, qrow, J->o + r * J->d, J->lse + r);
    }
    free(s);
    free(qrow);
    J->status = 0;
    return NULL;
}

/*
 * q, k, v : bf16 bits, [B, H, N, d] contiguous.
 * key_len : int32 [B] or NULL (all N keys).
 * rows    : flat row ids (b*H + h)*N + i to evaluate, or NULL for every row.
 * o       : double [n_rows, d] (n_rows = B*H*N when rows is NULL).
 * lse     : double [n_rows].
 * Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 */
int fattn_oracle_forward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                         int causal, const int32_t *key_len, const int64_t *rows,
                         int64_t n_rows, double *o, double *lse, int n_threads)
{
    if (!q || !k || !v || !o || !lse || B < 0 || H < 0 || N < 0 || d <= 0) return 1;
    const int64_t total = B * H * N;
    if (!rows) n_rows = total;
    if (n_rows < 0) return 1;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return 1;
    if (n_rows == 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > n_rows) n_threads = (int)n_rows;

    oracle_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int w = 0; w < n_threads; ++w) {
        oracle_job *J = &jobs[w];
        J->q = q; J->k = k; J->v = v;
        J->B = B; J->H = H; J->N = N; J->d = d;
        J->scale = scale; J->causal = causal; J->key_len = key_len;
        J->rows = rows; J->n_rows = n_rows; J->o = o; J->lse = lse;
        /* contiguous blocks: every row costs the same (a full score row) */
        J->begin = n_rows * w / n_threads;
        J->end = n_rows * (w + 1) / n_threads;
        J->status = 0;
    }
    int rc = 0;
    for (int w = 0; w < n_threads; ++w) {
        started[w] = (n_threads > 1) && pthread_create(&tids[w], NULL, worker, &jobs[w]) == 0;
        if (!started[w]) worker(&jobs[w]);
    }
    for (int w = 0; w < n_threads; ++w) {
        if (started[w]) pthread_join(tids[w], NULL);
        if (jobs[w].status) rc = jobs[w].status;
    }
    return rc;
}

/*
 * The full probability matrix P (and the scaled score matrix S) of one
 * (b, h), for small N: p[i*N + j] = softmax row i, 0 where masked; a row with
 * no visible key is all zero.  s may be NULL.  Same definition as above.
 */
int fattn_oracle_probs(const uint16_t *q, const uint16_t *k, int64_t B, int64_t H,
                       int64_t N, int64_t d, double scale, int causal,
                       const int32_t *key_len, int64_t b, int64_t h, double *p, double *s)
{
    if (!q || !k || !p || b < 0 || b >= B || h < 0 || h >= H || N < 0 || d <= 0) return 1;
    int64_t klen = N;
    if (key_len) {
        klen = key_len[b];
        if (klen < 0) klen = 0;
        if (klen > N) klen = N;
    }
    const uint16_t *qp = q + (b * H + h) * N * d;
    const uint16_t *kp = k + (b * H + h) * N * d;
    for (int64_t i = 0; i < N; ++i) {
        double *prow = p + i * N;
        int any = 0;
        double m = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t)
                acc += bf16_bits_to_double(qp[i * d + t]) * bf16_bits_to_double(kp[j * d + t]);
            prow[j] = scale * acc;
            if (s) s[i * N + j] = prow[j];
            int vis = (!causal || j <= i) && j < klen;
            if (vis && (!any || prow[j] > m)) m = prow[j];
            if (vis) any = 1;
        }
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            int vis = (!causal || j <= i) && j < klen;
            prow[j] = (vis && any) ? exp(prow[j] - m) : 0.0;
            l += prow[j];
        }
        for (int64_t j = 0; j < N; ++j) prow[j] = any ? prow[j] / l : 0.0;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Backward pass (gradients of a scalar loss L through O), plain fp64.
 *
 * "understand-flashattention", section "Attention forward and backward
 * formulas", backward pass, steps 1-5, with the scale of S = scale * Q K^T
 * carried through the chain rule (it multiplies dQ and dK once):
 *   dV   = P^T dO                                      (step 1)
 *   dP   = dO V^T                                      (step 2)
 *   dS_ij = P_ij (dP_ij - sum_k dP_ik P_ik)            (step 3, the row form)
 *   dQ   = scale * dS K                                (step 4)
 *   dK   = scale * dS^T Q                              (step 5)
 * P is the forward's softmax of the masked, scaled scores (same definition as
 * fattn_oracle_forward); masked entries have P = 0 and so contribute nothing.
 * A row with no visible key has P = 0: its dQ row is 0 and it adds nothing to
 * dK or dV.
 *
 * Threads: whole heads per worker when there are at least as many heads as
 * workers; otherwise the rows of each head are split over the workers, each
 * with private dK / dV accumulators that are summed after the join.
 */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int64_t H, N, d;
    double scale;
    int causal;
    const int32_t *key_len;
    const int64_t *heads;   /* flat b*H + h of each requested head */
    int64_t n_heads;
    double *dq, *dk, *dv;   /* [n_heads, N, d] */
    int64_t head_begin, head_end;  /* whole-head mode: this worker's heads */
    int64_t head, row_begin, row_end;  /* row mode: one head, this worker's rows */
    double *dk_priv, *dv_priv;  /* row mode: private [N, d] accumulators */
    int row_mode;
    int status;
} bwd_job;

/* Rows [r0, r1) of head slot `hs` (flat head bh): dQ rows into dq_head,
 * dK / dV contributions added into dk_acc / dv_acc ([N, d]). */
static void bwd_rows(const bwd_job *J, int64_t hs, int64_t r0, int64_t r1, double *dk_acc, double *dv_acc,
                     double *s, double *p, double *dp, double *qrow, double *grow)
{
    const int64_t N = J->N, d = J->d;
    const int64_t bh = J->heads ? J->heads[hs] : hs;
    const int64_t b = bh / J->H;
    const uint16_t *qp = J->q + bh * N * d;
    const uint16_t *kp = J->k + bh * N * d;
    const uint16_t *vp = J->v + bh * N * d;
    const uint16_t *gp = J->dout + bh * N * d;
    double *dq_head = J->dq + hs * N * d;
    int64_t klen = N;
    if (J->key_len) {
        klen = J->key_len[b];
        if (klen < 0) klen = 0;
        if (klen > N) klen = N;
    }
    for (int64_t i = r0; i < r1; ++i) {
        for (int64_t t = 0; t < d; ++t) {
            qrow[t] = bf16_bits_to_double(qp[i * d + t]);
            grow[t] = bf16_bits_to_double(gp[i * d + t]);
        }
        /* forward: scaled scores, visibility, softmax row */
        int any = 0;
        double m = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t) acc += qrow[t] * bf16_bits_to_double(kp[j * d + t]);
            s[j] = J->scale * acc;
            int vis = (!J->causal || j <= i) && j < klen;
            if (vis && (!any || s[j] > m)) m = s[j];
            if (vis) any = 1;
        }
        double *dqi = dq_head + i * d;
        for (int64_t t = 0; t < d; ++t) dqi[t] = 0.0;
        if (!any) continue;
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            int vis = (!J->causal || j <= i) && j < klen;
            p[j] = vis ? exp(s[j] - m) : 0.0;
            l += p[j];
        }
        for (int64_t j = 0; j < N; ++j) p[j] /= l;
        /* step 2: dP row = dO_i . v_j */
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < d; ++t) acc += grow[t] * bf16_bits_to_double(vp[j * d + t]);
            dp[j] = acc;
        }
        /* step 3: dS_ij = P_ij (dP_ij - sum_k dP_ik P_ik) */
        double r = 0.0;
        for (int64_t j = 0; j < N; ++j) r += dp[j] * p[j];
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            const double ds = p[j] * (dp[j] - r);
            const uint16_t *kj = kp + j * d;
            for (int64_t t = 0; t < d; ++t) {
                dqi[t] += J->scale * ds * bf16_bits_to_double(kj[t]);  /* step 4 */
                dk_acc[j * d + t] += J->scale * ds * qrow[t];          /* step 5 */
                dv_acc[j * d + t] += p[j] * grow[t];                   /* step 1 */
            }
        }
    }
}

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    const int64_t N = J->N, d = J->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(3 * N + 2 * d));
    if (!s) {
        J->status = 2;
        return NULL;
    }
    double *p = s + N, *dp = p + N, *qrow = dp + N, *grow = qrow + d;
    if (J->row_mode) {
        bwd_rows(J, J->head, J->row_begin, J->row_end, J->dk_priv, J->dv_priv, s, p, dp, qrow, grow);
    } else {
        for (int64_t hs = J->head_begin; hs < J->head_end; ++hs) {
            double *dk = J->dk + hs * N * d, *dv = J->dv + hs * N * d;
            for (int64_t x = 0; x < N * d; ++x) dk[x] = dv[x] = 0.0;
            bwd_rows(J, hs, 0, N, dk, dv, s, p, dp, qrow, grow);
        }
    }
    free(s);
    J->status = 0;
    return NULL;
}

/*
 * q, k, v, dout : bf16 bits, [B, H, N, d] contiguous (dout = dL/dO).
 * key_len       : int32 [B] or NULL.
 * heads         : flat b*H + h of the heads to evaluate, or NULL for all B*H.
 * dq, dk, dv    : double [n_heads, N, d] (n_heads = B*H when heads is NULL).
 * Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 */
int fattn_oracle_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                          int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                          const int32_t *key_len, const int64_t *heads, int64_t n_heads,
                          double *dq, double *dk, double *dv, int n_threads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 0 || H < 0 || N < 0 || d <= 0) return 1;
    if (!heads) n_heads = B * H;
    if (n_heads < 0) return 1;
    if (heads)
        for (int64_t x = 0; x < n_heads; ++x)
            if (heads[x] < 0 || heads[x] >= B * H) return 1;
    if (n_heads == 0 || N == 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;

    bwd_job proto;
    memset(&proto, 0, sizeof proto);
    proto.q = q; proto.k = k; proto.v = v; proto.dout = dout;
    proto.H = H; proto.N = N; proto.d = d; proto.scale = scale; proto.causal = causal;
    proto.key_len = key_len; proto.heads = heads; proto.n_heads = n_heads;
    proto.dq = dq; proto.dk = dk; proto.dv = dv;

    bwd_job jobs[256];
    pthread_t tids[256];
    int started[256];
    int rc = 0;
    if (n_heads >= n_threads) {
        for (int w = 0; w < n_threads; ++w) {
            jobs[w] = proto;
            jobs[w].head_begin = n_heads * w / n_threads;
            jobs[w].head_end = n_heads * (w + 1) / n_threads;
        }
        for (int w = 0; w < n_threads; ++w) {
            started[w] = (n_threads > 1) && pthread_create(&tids[w], NULL, bwd_worker, &jobs[w]) == 0;
            if (!started[w]) bwd_worker(&jobs[w]);
        }
        for (int w = 0; w < n_threads; ++w) {
            if (started[w]) pthread_join(tids[w], NULL);
            if (jobs[w].status) rc = jobs[w].status;
        }
        return rc;
    }
    int nw = n_threads;
    if ((int64_t)nw > N) nw = (int)N;
    double *priv = (double *)malloc(sizeof(double) * (size_t)(2 * nw) * (size_t)(N * d));
    if (!priv) return 2;
    for (int64_t hs = 0; hs < n_heads && rc == 0; ++hs) {
        for (int w = 0; w < nw; ++w) {
            jobs[w] = proto;
            jobs[w].row_mode = 1;
            jobs[w].head = hs;
            jobs[w].row_begin = N * w / nw;
            jobs[w].row_end = N * (w + 1) / nw;
            jobs[w].dk_priv = priv + (size_t)(2 * w) * (size_t)(N * d);
            jobs[w].dv_priv = jobs[w].dk_priv + N * d;
            for (int64_t x = 0; x < 2 * N * d; ++x) jobs[w].dk_priv[x] = 0.0;
        }
        for (int w = 0; w < nw; ++w) {
            started[w] = (nw > 1) && pthread_create(&tids[w], NULL, bwd_worker, &jobs[w]) == 0;
            if (!started[w]) bwd_worker(&jobs[w]);
        }
        for (int w = 0; w < nw; ++w) {
            if (started[w]) pthread_join(tids[w], NULL);
            if (jobs[w].status) rc = jobs[w].status;
        }
        double *dkh = dk + hs * N * d, *dvh = dv + hs * N * d;
        for (int64_t x = 0; x < N * d; ++x) {
            double a = 0.0, c = 0.0;
            for (int w = 0; w < nw; ++w) {
                a += jobs[w].dk_priv[x];
                c += jobs[w].dv_priv[x];
            }
            dkh[x] = a;
            dvh[x] = c;
        }
    }
    free(priv);
    return rc;
}

/*
 * Causal linear attention, plain fp64 CPU oracle (the second workload).
 *
 * What it computes ("Linear Attention CUDA kernel" page: the kernel feature
 * map phi(x) = elu(x) + 1 of the linear transformer, the key-length mask of
 * CausalLinearAttention.forward, which multiplies the mapped keys by the
 * per-position 0/1 length matrix, and the causal dot product of its CPU
 * implementation, which walks the sequence keeping a running outer-product
 * state), for every (b, h):
 *     kt_j = phi(k_j) if j < key_len[b] else 0,   qt_i = phi(q_i)
 *     state S_i = sum_{j <= i} kt_j v_j^T   (E x M),   s_i = sum_{j <= i} kt_j
 *     out_i = (qt_i^T S_i) / (qt_i . s_i + eps)
 * -- the page's numerator V'_i = sum_{j <= i} (qt_i . kt_j) v_j times its
 * normaliser Z_i = 1 / (qt_i . cumsum(kt)_i + eps).
 * Inputs are float32 (the page's kernels take float tensors), widened to double.
 */
typedef struct {
    const float *q, *k, *v;
    int64_t H, N, E, M;
    const int32_t *key_len;
    double eps;
    double *out;
    int64_t head_begin, head_end;
    int status;
} lin_job;

static double phi_elu1(double x) { return x > 0.0 ? x + 1.0 : exp(x); } /* elu(x) + 1 */

static void *lin_worker(void *arg) {
    lin_job *J = (lin_job *)arg;
    const int64_t E = J->E, M = J->M, N = J->N;
    double *S = (double *)malloc((size_t)(E * M + 2 * E) * sizeof(double));
    if (!S) {
        J->status = 2;
        return NULL;
    }
    double *s = S + E * M, *kt = s + E;
    for (int64_t hs = J->head_begin; hs < J->head_end; ++hs) {
        const int64_t b = hs / J->H;
        int64_t kl = J->key_len ? J->key_len[b] : N;
        if (kl < 0) kl = 0;
        if (kl > N) kl = N;
        for (int64_t x = 0; x < E * M + E; ++x) S[x] = 0.0;
        const float *qh = J->q + hs * N * E, *kh = J->k + hs * N * E, *vh = J->v + hs * N * M;
        double *oh = J->out + hs * N * M;
        for (int64_t i = 0; i < N; ++i) {
            /* the state takes row i's key and value (a masked key adds nothing) */
            for (int64_t e = 0; e < E; ++e) kt[e] = i < kl ? phi_elu1((double)kh[i * E + e]) : 0.0;
            for (int64_t e = 0; e < E; ++e) {
                s[e] += kt[e];
                for (int64_t m = 0; m < M; ++m) S[e * M + m] += kt[e] * (double)vh[i * M + m];
            }
            /* row i's output from the state */
            double den = J->eps;
            for (int64_t m = 0; m < M; ++m) oh[i * M + m] = 0.0;
            for (int64_t e = 0; e < E; ++e) {
                const double qt = phi_elu1((double)qh[i * E + e]);
                den += qt * s[e];
                for (int64_t m = 0; m < M; ++m) oh[i * M + m] += qt * S[e * M + m];
            }
            for (int64_t m = 0; m < M; ++m) oh[i * M + m] /= den;
        }
    }
    free(S);
    return NULL;
}

int fattn_oracle_linear(const float *q, const float *k, const float *v, int64_t B, int64_t H, int64_t N, int64_t E,
                        int64_t M, const int32_t *key_len, double eps, double *out, int threads) {
    if (B < 0 || H < 0 || N < 0 || E <= 0 || M <= 0) return 1;
    const int64_t heads = B * H;
    if (heads == 0 || N == 0) return 0;
    int nw = threads < 1 ? 1 : threads;
    if (nw > 256) nw = 256;
    if (nw > heads) nw = (int)heads;
    lin_job jobs[256];
    pthread_t tids[256];
    int started[256];
    int rc = 0;
    for (int w = 0; w < nw; ++w) {
        jobs[w] = (lin_job){q, k, v, H, N, E, M, key_len, eps, out, heads * w / nw, heads * (w + 1) / nw, 0};
        started[w] = (nw > 1) && pthread_create(&tids[w], NULL, lin_worker, &jobs[w]) == 0;
        if (!started[w]) lin_worker(&jobs[w]);
    }
    for (int w = 0; w < nw; ++w) {
        if (started[w]) pthread_join(tids[w], NULL);
        if (jobs[w].status) rc = jobs[w].status;
    }
    return rc;
}
