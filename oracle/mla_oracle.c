/*
 * mla_oracle.c - fp64 CPU oracle for absorbed multi-head latent attention (MLA) decode.
 *
 * TEST INFRASTRUCTURE ONLY, like attn_oracle.c: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it, and it shares nothing with the CUDA library.
 *
 * What it computes ("Attention Kernel 实现与正确性验证" (walkerchi.com), section 2.1, the absorption
 * trick, and section 2.2, the absorbed reference).  With W_uk folded into the query beforehand
 * (q_abs = q_nope W_uk, one vector of d_c numbers per head), the KV cache of a sequence is the
 * compressed c_kv (d_c numbers per token) followed by the decoupled RoPE key k_pe (d_r numbers per
 * token), shared by every head.  For one decode query per head (batch b, head h) and the T cached
 * tokens t:
 *     s_t   = sm_scale * ( q_abs[b,h,:] . c_kv[b,t,:]  +  q_pe[b,h,:] . k_pe[b,t,:] )
 *     m     = max_t s_t ,  Z = sum_t exp(s_t - m)
 *     out_c[b,h,:] = sum_t exp(s_t - m) * c_kv[b,t,:] / Z          (d_c numbers, compressed space)
 *     LSE[b,h]     = m + ln Z
 * The up-projection out = out_c W_uv^T and the query absorption are plain matrix products around
 * this core; the tests apply them in float64 to tie this oracle to the page's un-absorbed form.
 *
 * Layout: q is [B, H, d_c + d_r] (q_abs then q_pe), kv is [B, T, d_c + d_r] (c_kv then k_pe),
 * out is [B, H, d_c], lse is [B, H]; all float64, contiguous.  Two passes per (b, h), no tiling.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *kv;
    int B, H, T, d_c, d_r;
    double sm_scale;
    double *out, *lse;
    long first, last; /* this worker's share of the flattened b*H + h index */
    int status;
} mla_job_t;

static void *mla_worker(void *arg) {
    mla_job_t *J = (mla_job_t *)arg;
    const int dq = J->d_c + J->d_r;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->T > 0 ? J->T : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->d_c);
    J->status = 0;
    if (!s || !acc) {
        J->status = -2;
        free(s);
        free(acc);
        return NULL;
    }
    for (long f = J->first; f < J->last; ++f) {
        const long b = f / J->H;
        const double *qh = J->q + f * dq;
        const double *kvb = J->kv + b * (long)J->T * dq;
        /* pass 1: scores over the compressed and the RoPE parts, and their maximum */
        double m = -INFINITY;
        for (int t = 0; t < J->T; ++t) {
            const double *row = kvb + (long)t * dq;
            double nope = 0.0, pe = 0.0;
            for (int d = 0; d < J->d_c; ++d) nope += qh[d] * row[d];
            for (int d = 0; d < J->d_r; ++d) pe += qh[J->d_c + d] * row[J->d_c + d];
            s[t] = J->sm_scale * (nope + pe);
            if (s[t] > m) m = s[t];
        }
        /* pass 2: exponentials, their sum, and the weighted sum of the c_kv rows */
        double Z = 0.0;
        for (int d = 0; d < J->d_c; ++d) acc[d] = 0.0;
        for (int t = 0; t < J->T; ++t) {
            const double e = exp(s[t] - m);
            const double *row = kvb + (long)t * dq;
            Z += e;
            for (int d = 0; d < J->d_c; ++d) acc[d] += e * row[d];
        }
        double *o = J->out + f * J->d_c;
        for (int d = 0; d < J->d_c; ++d) o[d] = acc[d] / Z;
        J->lse[f] = m + log(Z);
    }
    free(s);
    free(acc);
    return NULL;
}

/*
 * Absorbed MLA decode oracle (see the header).  T >= 1.  n_threads <= 0 uses every online core.
 * Returns 0, -1 on bad arguments, -2 if memory ran out.
 */
int oracle_mla_decode_f64(const double *q, const double *kv, int B, int H, int T, int d_c, int d_r,
                          double sm_scale, double *out, double *lse, int n_threads) {
    if (!q || !kv || !out || !lse) return -1;
    if (B < 0 || H <= 0 || T <= 0 || d_c <= 0 || d_r < 0) return -1;
    if (!(sm_scale == sm_scale)) return -1;
    const long total = (long)B * H;
    if (total == 0) return 0;
    if (n_threads <= 0) {
        long hw = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = hw > 0 ? (int)hw : 1;
    }
    if (n_threads > total) n_threads = (int)total;
    mla_job_t *jobs = (mla_job_t *)calloc((size_t)n_threads, sizeof(mla_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    char *threaded = (char *)calloc((size_t)n_threads, 1);
    if (!jobs || !tid || !threaded) {
        free(jobs); free(tid); free(threaded);
        return -2;
    }
    for (int t = 0; t < n_threads; ++t) {
        mla_job_t *J = &jobs[t];
        J->q = q; J->kv = kv; J->B = B; J->H = H; J->T = T; J->d_c = d_c; J->d_r = d_r;
        J->sm_scale = sm_scale; J->out = out; J->lse = lse;
        J->first = total * t / n_threads;
        J->last = total * (t + 1) / n_threads;
        if (n_threads > 1 && pthread_create(&tid[t], NULL, mla_worker, J) == 0)
            threaded[t] = 1;
        else
            mla_worker(J);
    }
    int status = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (threaded[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status != 0) status = jobs[t].status;
    }
    free(jobs); free(tid); free(threaded);
    return status;
}
