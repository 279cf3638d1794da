/*
 * attn_oracle.c - fp64 CPU oracle for the exact-attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct definition that the GPU
 * path is checked against.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  The product path never calls it, and it shares no code, header, constant or
 * helper with the CUDA library.
 *
 * What it computes.  Exact (dense) softmax attention, which the tiled online-softmax method
 * reaches up to rounding order:
 *   - "Attention Kernel 实现与正确性验证" (walkerchi.com), section 1.1: block-wise evaluation with an
 *     online softmax is equivalent to the softmax over the full sequence; section 1.2: GQA head map
 *     h_kv = h_q * H_kv // H_q and the causal condition offs_m >= offs_n.
 *   - "Triton-CUDA Attention" (skillmd.com), "GQA" variant: the map uses integer division, never a
 *     modulus; "Causal Attention" variant: the same top-left causal condition.
 *   - "Flash Attention 与 Kernel 优化" (fangpin.github.io), "输出与保存状态": the saved per-row
 *     statistic is the log-sum-exp m + log(l); read here as the natural log of the sum of exp of
 *     the scaled scores, with no epsilon (l >= 1 because the maximum contributes exp(0) = 1).
 *
 * For every batch b, query head hq and query row i:
 *     h_kv    = (hq * Hkv) / Hq                                   (integer division)
 *     J(i)    = causal ? {0, ..., i} : {0, ..., N-1}
 *     s_j     = sm_scale * sum_d Q[b,hq,i,d] * K[b,h_kv,j,d]        for j in J(i)
 *     m       = max_{j in J(i)} s_j
 *     Z       = sum_{j in J(i)} exp(s_j - m)
 *     O[b,hq,i,:] = sum_{j in J(i)} exp(s_j - m) * V[b,h_kv,j,:] / Z
 *     LSE[b,hq,i] = m + ln Z
 *
 * Two passes per row (maximum, then exponentials), no tiling, no online rescaling.  All
 * arithmetic is in double precision on the exact values of the bf16 inputs.  Inputs are the raw
 * bf16 bit patterns (uint16), layout [B, H, N, D] contiguous.
 *
 * Threads only split the rows between them; every row is computed by exactly the code above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NOMEM (-2)

/* bf16 is the upper half of an IEEE binary32; widening it to double is exact. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, Hq, Hkv, N, D, causal;
    double sm_scale;
    const int32_t *rows; /* NULL: every row of every head */
    int n_rows;          /* rows per (b, hq) */
    double *out, *lse;   /* out [B*Hq, n_rows, D], lse [B*Hq, n_rows] */
    double *probs;       /* optional: [B*Hq, n_rows, N] normalised probabilities */
    long first, last;    /* this worker's share of the flattened (b*Hq + hq, r) index */
    int status;
} job_t;

/* One query row: the definition above, written out. */
static int one_row(const job_t *J, long flat, double *s, double *qrow, double *acc) {
    const int N = J->N, D = J->D;
    const long bh = flat / J->n_rows;
    const int r = (int)(flat % J->n_rows);
    const int b = (int)(bh / J->Hq), hq = (int)(bh % J->Hq);
    const int hkv = (int)(((long)hq * J->Hkv) / J->Hq);
    const int i = J->rows ? J->rows[flat] : r;
    if (i < 0 || i >= N) return ORACLE_ERR_ARG;

    const uint16_t *qi = J->q + (((long)b * J->Hq + hq) * N + i) * D;
    const uint16_t *kh = J->k + ((long)b * J->Hkv + hkv) * (long)N * D;
    const uint16_t *vh = J->v + ((long)b * J->Hkv + hkv) * (long)N * D;
    const int n_vis = J->causal ? i + 1 : N; /* J(i) = {0, ..., n_vis - 1} */

    for (int d = 0; d < D; ++d) qrow[d] = bf16_to_f64(qi[d]);

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int j = 0; j < n_vis; ++j) {
        const uint16_t *kj = kh + (long)j * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * bf16_to_f64(kj[d]);
        s[j] = J->sm_scale * dot;
        if (s[j] > m) m = s[j];
    }

    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double Z = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j < n_vis; ++j) {
        const double e = exp(s[j] - m);
        s[j] = e;
        Z += e;
        const uint16_t *vj = vh + (long)j * D;
        for (int d = 0; d < D; ++d) acc[d] += e * bf16_to_f64(vj[d]);
    }

    double *o = J->out + flat * D;
    for (int d = 0; d < D; ++d) o[d] = acc[d] / Z;
    J->lse[flat] = m + log(Z);

    if (J->probs) {
        double *p = J->probs + flat * (long)N;
        for (int j = 0; j < N; ++j) p[j] = (j < n_vis) ? s[j] / Z : 0.0;
    }
    return ORACLE_OK;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->N);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)J->D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->D);
    J->status = ORACLE_OK;
    if (!s || !qrow || !acc) {
        J->status = ORACLE_ERR_NOMEM;
    } else {
        for (long f = J->first; f < J->last; ++f) {
            const int st = one_row(J, f, s, qrow, acc);
            if (st != ORACLE_OK) { J->status = st; break; }
        }
    }
    free(s);
    free(qrow);
    free(acc);
    return NULL;
}

static int run(const job_t *proto, int n_threads) {
    const long total = (long)proto->B * proto->Hq * proto->n_rows;
    if (total == 0) return ORACLE_OK;
    if (n_threads <= 0) {
        long hw = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = hw > 0 ? (int)hw : 1;
    }
    if (n_threads > total) n_threads = (int)total;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    char *threaded = (char *)calloc((size_t)n_threads, 1);
    if (!jobs || !tid || !threaded) {
        free(jobs); free(tid); free(threaded);
        return ORACLE_ERR_NOMEM;
    }
    for (int t = 0; t < n_threads; ++t) {
        jobs[t] = *proto;
        jobs[t].first = total * t / n_threads;
        jobs[t].last = total * (t + 1) / n_threads;
        if (n_threads > 1 && pthread_create(&tid[t], NULL, worker, &jobs[t]) == 0)
            threaded[t] = 1;
        else
            worker(&jobs[t]); /* single thread, or a thread could not be created */
    }
    int status = ORACLE_OK;
    for (int t = 0; t < n_threads; ++t) {
        if (threaded[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    }
    free(jobs); free(tid); free(threaded);
    return status;
}

static int check_args(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                      int Hkv, int N, int D, double sm_scale, const double *out,
                      const double *lse) {
    if (!q || !k || !v || !out || !lse) return ORACLE_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0) return ORACLE_ERR_ARG;
    if (Hq % Hkv != 0) return ORACLE_ERR_ARG;
    if (!(sm_scale == sm_scale)) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/*
 * Full or row-subset oracle.
 *   rows == NULL : every row; out is [B, Hq, N, D] and lse is [B, Hq, N].
 *   rows != NULL : rows[(b*Hq + hq)*n_rows + r] is the query row for output slot r of head (b, hq);
 *                  out is [B*Hq, n_rows, D] and lse is [B*Hq, n_rows].
 * n_threads <= 0 uses every online core.  Returns 0, or a negative code on bad arguments.
 */
int oracle_attn_fwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                        int Hkv, int N, int D, int causal, double sm_scale, const int32_t *rows,
                        int n_rows, double *out, double *lse, int n_threads) {
    const int st = check_args(q, k, v, B, Hq, Hkv, N, D, sm_scale, out, lse);
    if (st != ORACLE_OK) return st;
    if (rows && n_rows < 0) return ORACLE_ERR_ARG;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.N = N; J.D = D; J.causal = causal ? 1 : 0;
    J.sm_scale = sm_scale;
    J.rows = rows;
    J.n_rows = rows ? n_rows : N;
    J.out = out; J.lse = lse; J.probs = NULL;
    return run(&J, n_threads);
}

/*
 * The same definition, also returning the normalised probability rows p[b,hq,i,j] =
 * exp(s_j - m) / Z for j in J(i) and 0 elsewhere, as [B, Hq, N, N].  Meant for tiny N only.
 */
int oracle_attn_probs_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                          int Hkv, int N, int D, int causal, double sm_scale, double *out,
                          double *lse, double *probs, int n_threads) {
    const int st = check_args(q, k, v, B, Hq, Hkv, N, D, sm_scale, out, lse);
    if (st != ORACLE_OK) return st;
    if (!probs) return ORACLE_ERR_ARG;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.N = N; J.D = D; J.causal = causal ? 1 : 0;
    J.sm_scale = sm_scale;
    J.rows = NULL;
    J.n_rows = N;
    J.out = out; J.lse = lse; J.probs = probs;
    return run(&J, n_threads);
}

/* Number of online cores the oracle uses when asked for n_threads <= 0. */
int oracle_default_threads(void) {
    long hw = sysconf(_SC_NPROCESSORS_ONLN);
    return hw > 0 ? (int)hw : 1;
}

/*
 * Backward of the same definition (test infrastructure as well).
 *
 * The pages train through this attention by recomputing the scores and probabilities from the
 * saved log-sum-exp instead of storing them ("Attention Kernel 实现与正确性验证", section 1.1,
 * third idea; "Flash Attention 与 Kernel 优化", section on autograd and backward: rebuild
 * s = qk^T * scale, apply the causal mask, rebuild p = softmax(s), then dv, dp, ds, dq, dk).  The
 * oracle writes that chain rule out densely, in double precision, per query row i of head
 * (b, hq) and visible key j of its KV head:
 *     p_ij  = exp(s_ij - LSE_i)             with s_ij = sm_scale * <q_i, k_j>, LSE from above
 *     dp_ij = <dO_i, v_j>
 *     D_i   = sum_j p_ij dp_ij
 *     ds_ij = p_ij (dp_ij - D_i)
 *     dQ_i  = sm_scale * sum_j ds_ij k_j
 *     dK_j  = sm_scale * sum over (hq in the group, i) of ds_ij q_i
 *     dV_j  = sum over (hq in the group, i) of p_ij dO_i
 * Inputs are bf16 bit patterns; outputs are doubles: dq [B,Hq,N,D], dk and dv [B,Hkv,N,D].
 * Threads split the query heads; each thread keeps private dK/dV sums for its heads, and the
 * per-head sums are added in head order afterwards (the result does not depend on the threads).
 */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int B, Hq, Hkv, N, D, causal;
    double sm_scale;
    double *dq;            /* [B*Hq, N, D] */
    double *dk_h, *dv_h;   /* per query head: [B*Hq, N, D] */
    int first, last;       /* query heads (b*Hq + hq) of this worker */
    int status;
} bjob_t;

static void *bworker(void *arg) {
    bjob_t *J = (bjob_t *)arg;
    const int N = J->N, D = J->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *qi = (double *)malloc(sizeof(double) * (size_t)D);
    double *gi = (double *)malloc(sizeof(double) * (size_t)D);
    J->status = ORACLE_OK;
    if (!s || !dp || !qi || !gi) { J->status = ORACLE_ERR_NOMEM; goto done; }
    for (int bh = J->first; bh < J->last; ++bh) {
        const int b = bh / J->Hq, hq = bh % J->Hq;
        const int hkv = (int)(((long)hq * J->Hkv) / J->Hq);
        const uint16_t *kh = J->k + ((long)b * J->Hkv + hkv) * (long)N * D;
        const uint16_t *vh = J->v + ((long)b * J->Hkv + hkv) * (long)N * D;
        double *dkh = J->dk_h + (long)bh * N * D, *dvh = J->dv_h + (long)bh * N * D;
        for (int i = 0; i < N; ++i) {
            const uint16_t *q_row = J->q + ((long)bh * N + i) * D;
            const uint16_t *do_row = J->dout + ((long)bh * N + i) * D;
            const int n_vis = J->causal ? i + 1 : N;
            for (int d = 0; d < D; ++d) { qi[d] = bf16_to_f64(q_row[d]); gi[d] = bf16_to_f64(do_row[d]); }
            /* scores and the log-sum-exp (two passes, as in the forward) */
            double m = -INFINITY;
            for (int j = 0; j < n_vis; ++j) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qi[d] * bf16_to_f64(kh[(long)j * D + d]);
                s[j] = J->sm_scale * dot;
                if (s[j] > m) m = s[j];
            }
            double Z = 0.0;
            for (int j = 0; j < n_vis; ++j) Z += exp(s[j] - m);
            const double lse = m + log(Z);
            /* p, dp and D_i */
            double Di = 0.0;
            for (int j = 0; j < n_vis; ++j) {
                s[j] = exp(s[j] - lse); /* now p_ij */
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += gi[d] * bf16_to_f64(vh[(long)j * D + d]);
                dp[j] = dot;
                Di += s[j] * dp[j];
            }
            double *dq_row = J->dq + ((long)bh * N + i) * D;
            for (int d = 0; d < D; ++d) dq_row[d] = 0.0;
            for (int j = 0; j < n_vis; ++j) {
                const double ds = s[j] * (dp[j] - Di);
                for (int d = 0; d < D; ++d) {
                    dq_row[d] += J->sm_scale * ds * bf16_to_f64(kh[(long)j * D + d]);
                    dkh[(long)j * D + d] += J->sm_scale * ds * qi[d];
                    dvh[(long)j * D + d] += s[j] * gi[d];
                }
            }
        }
    }
done:
    free(s); free(dp); free(qi); free(gi);
    return NULL;
}

/*
 * Gradients of the forward above for an output gradient `dout` [B,Hq,N,D] (bf16 bits).
 * dq [B,Hq,N,D], dk [B,Hkv,N,D], dv [B,Hkv,N,D] in double.  Returns 0 or a negative code.
 */
int oracle_attn_bwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *dout, int B, int Hq, int Hkv, int N, int D, int causal,
                        double sm_scale, double *dq, double *dk, double *dv, int n_threads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return ORACLE_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || D <= 0 || Hq % Hkv != 0) return ORACLE_ERR_ARG;
    const long heads = (long)B * Hq;
    const long per_head = (long)N * D;
    for (long x = 0; x < (long)B * Hkv * per_head; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
    if (heads == 0 || N == 0) return ORACLE_OK;
    double *dk_h = (double *)calloc((size_t)(heads * per_head), sizeof(double));
    double *dv_h = (double *)calloc((size_t)(heads * per_head), sizeof(double));
    if (!dk_h || !dv_h) { free(dk_h); free(dv_h); return ORACLE_ERR_NOMEM; }
    if (n_threads <= 0) n_threads = oracle_default_threads();
    if (n_threads > heads) n_threads = (int)heads;
    bjob_t *jobs = (bjob_t *)calloc((size_t)n_threads, sizeof(bjob_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    char *threaded = (char *)calloc((size_t)n_threads, 1);
    int status = ORACLE_OK;
    if (!jobs || !tid || !threaded) { status = ORACLE_ERR_NOMEM; goto out; }
    for (int t = 0; t < n_threads; ++t) {
        bjob_t *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->dout = dout;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->N = N; J->D = D; J->causal = causal ? 1 : 0;
        J->sm_scale = sm_scale; J->dq = dq; J->dk_h = dk_h; J->dv_h = dv_h;
        J->first = (int)(heads * t / n_threads);
        J->last = (int)(heads * (t + 1) / n_threads);
        if (n_threads > 1 && pthread_create(&tid[t], NULL, bworker, J) == 0)
            threaded[t] = 1;
        else
            bworker(J);
    }
    for (int t = 0; t < n_threads; ++t) {
        if (threaded[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    }
    /* dK, dV of a KV head: the sum over its query heads, in head order */
    for (long bh = 0; bh < heads; ++bh) {
        const long b = bh / Hq, hq = bh % Hq;
        const long hkv = (hq * Hkv) / Hq;
        double *dkk = dk + (b * Hkv + hkv) * per_head, *dvv = dv + (b * Hkv + hkv) * per_head;
        for (long x = 0; x < per_head; ++x) {
            dkk[x] += dk_h[bh * per_head + x];
            dvv[x] += dv_h[bh * per_head + x];
        }
    }
out:
    free(jobs); free(tid); free(threaded); free(dk_h); free(dv_h);
    return status;
}
