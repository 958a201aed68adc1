/*
 * fw_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 CPU statement of the delta-rule fast-weight
 * layer core with the DPFP feature map.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this code; the product path never
 * does.  It shares no code, header or table with the CUDA library.
 *
 * Sources (all on the Fast Weights Transformer guide, xdnf.cn/news/308600,
 * a walk-through of "Linear Transformers Are Secretly Fast Weight Memory
 * Systems", arXiv:2102.11174):
 *   - section "DPFP: projection formula and hyper-parameters": the feature
 *     map phi over ReLU([k,-k]) and its cyclic shifts, output size
 *     2*d_key*nu, nu in 1..2*d_key-1;
 *   - section "normalisation" and the DPFP source listed with it: phi is
 *     divided by (sum of its entries + eps), eps = 1e-6 by default, and the
 *     shift is torch.roll(shifts=i), i.e. the rolled vector at position j
 *     holds x[(j - i) mod 2*d_key];
 *   - section "FastWeightsAttention: the new update rule": retrieve
 *     vbar = W_{i-1} phi(k_i), write W_i = W_{i-1} + beta_i (v_i - vbar)
 *     outer phi(k_i), read y_i = W_i phi(q_i) with the updated W;
 *   - section "forward pass", the loop over steps: W starts at zero with
 *     shape [batch, heads, d_value, d_dot] and phi is applied to query and
 *     key, not to value;
 *   - section "token_wise variant": one token at a time against a W that
 *     persists across calls (the decode step);
 *   - the backward of the recurrence (the gradients the guide's training
 *     loop takes through it by autograd; the pages print no backward): the
 *     chain rule applied to the steps above in reverse order, with the whole
 *     history of W kept (see fwo_delta_backward);
 *   - section "linear self-attention, the fast form" (the sum rule the
 *     delta rule replaces): W_i = W_{i-1} + v_i outer phi(k_i),
 *     z_i = z_{i-1} + phi(k_i), y_i = W_i phi(q_i) / (z_i . phi(q_i)) -- the
 *     kernel-attention ratio written as a recurrence; the unnormalised form
 *     drops the division.  The pages give no guard for a zero denominator;
 *     here y_i = 0 when z_i . phi(q_i) == 0 (then every phi(k_j) . phi(q_i)
 *     is 0, the numerator too, as all phi >= 0).
 *
 * Every routine below follows those steps in that order, one token at a time,
 * with no blocking, fusion or reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define FWO_OK 0
#define FWO_BAD_ARG 1

/* DPFP of one vector k (length d_key) into phi (length 2*d_key*nu).
 * x = ReLU([k, -k]); phi[(i-1)*2*d_key + j] = x[j] * x[(j - i) mod 2*d_key]
 * for i = 1..nu and j = 0..2*d_key-1; then phi /= (sum(phi) + eps).
 * x is a caller-provided scratch of length 2*d_key. */
static void dpfp_one(const double *k, double *phi, double *x, int d_key, int nu, double eps)
{
    const int n = 2 * d_key;
    for (int j = 0; j < d_key; ++j) {
        x[j] = k[j] > 0.0 ? k[j] : 0.0;
        x[d_key + j] = -k[j] > 0.0 ? -k[j] : 0.0;
    }
    double s = 0.0;
    for (int i = 1; i <= nu; ++i) {
        for (int j = 0; j < n; ++j) {
            int src = ((j - i) % n + n) % n;
            double p = x[j] * x[src];
            phi[(size_t)(i - 1) * n + j] = p;
            s += p;
        }
    }
    const int d_dot = n * nu;
    for (int m = 0; m < d_dot; ++m)
        phi[m] = phi[m] / (s + eps);
}

int fwo_dpfp(const double *x, double *phi, int64_t rows, int d_key, int nu, double eps)
{
    if (!x || !phi || rows < 0 || d_key <= 0 || nu < 1 || nu > 2 * d_key - 1)
        return FWO_BAD_ARG;
    const int d_dot = 2 * d_key * nu;
    double *scratch = (double *)malloc(sizeof(double) * 2 * (size_t)d_key);
    if (!scratch)
        return FWO_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r)
        dpfp_one(x + r * d_key, phi + r * d_dot, scratch, d_key, nu, eps);
    free(scratch);
    return FWO_OK;
}

/* ---------------------------------------------------------------------- */
/* The recurrence for one (batch, head) pair over L tokens.               */
/*   q, k: [L, d_key]; v, y: [L, d_v]; beta: [L]; W: [d_v, d_dot] in/out.  */
/* ---------------------------------------------------------------------- */
static void recurrence_one(const double *q, const double *k, const double *v, const double *beta,
                           double *W, double *y, int64_t L, int d_key, int nu, int d_v, double eps)
{
    const int d_dot = 2 * d_key * nu;
    double *pk = (double *)malloc(sizeof(double) * d_dot);
    double *pq = (double *)malloc(sizeof(double) * d_dot);
    double *x = (double *)malloc(sizeof(double) * 2 * d_key);
    double *vbar = (double *)malloc(sizeof(double) * d_v);
    for (int64_t t = 0; t < L; ++t) {
        /* phi is applied to the key and the query of this step */
        dpfp_one(k + t * d_key, pk, x, d_key, nu, eps);
        dpfp_one(q + t * d_key, pq, x, d_key, nu, eps);
        /* retrieve: vbar = W_{t-1} phi(k_t) */
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int m = 0; m < d_dot; ++m)
                acc += W[(size_t)r * d_dot + m] * pk[m];
            vbar[r] = acc;
        }
        /* write: W_t = W_{t-1} + beta_t (v_t - vbar) outer phi(k_t) */
        for (int r = 0; r < d_v; ++r) {
            double u = beta[t] * (v[t * d_v + r] - vbar[r]);
            for (int m = 0; m < d_dot; ++m)
                W[(size_t)r * d_dot + m] += u * pk[m];
        }
        /* read with the updated weights: y_t = W_t phi(q_t) */
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int m = 0; m < d_dot; ++m)
                acc += W[(size_t)r * d_dot + m] * pq[m];
            y[t * d_v + r] = acc;
        }
    }
    free(pk);
    free(pq);
    free(x);
    free(vbar);
}

typedef struct {
    const double *q, *k, *v, *beta, *W0;
    double *W_final, *y;
    int64_t BH, L;
    int d_key, nu, d_v;
    double eps;
    int64_t first, last; /* half-open range of (b,h) indices */
} job_t;

static void *run_job(void *arg)
{
    job_t *j = (job_t *)arg;
    const int d_dot = 2 * j->d_key * j->nu;
    const size_t wsz = (size_t)j->d_v * d_dot;
    for (int64_t bh = j->first; bh < j->last; ++bh) {
        double *W = j->W_final + bh * wsz;
        if (j->W0 && j->W0 + bh * wsz != W)
            memcpy(W, j->W0 + bh * wsz, sizeof(double) * wsz);
        else if (j->W0)
            ; /* in place: W already holds W_0 */
        else
            memset(W, 0, sizeof(double) * wsz); /* W_0 = 0 */
        recurrence_one(j->q + bh * j->L * j->d_key, j->k + bh * j->L * j->d_key,
                       j->v + bh * j->L * j->d_v, j->beta + bh * j->L, W,
                       j->y + bh * j->L * j->d_v, j->L, j->d_key, j->nu, j->d_v, j->eps);
    }
    return NULL;
}

/* The sequential forward: inputs q, k [B,H,L,d_key]; v [B,H,L,d_v];
 * beta [B,H,L]; W0 [B,H,d_v,d_dot] or NULL (zeros).  Outputs y [B,H,L,d_v]
 * and W_final [B,H,d_v,d_dot] (both required; W_final may equal W0).
 * nthreads > 1 splits the independent (b,h) pairs over POSIX threads. */
int fwo_delta_forward(const double *q, const double *k, const double *v, const double *beta,
                      const double *W0, double *W_final, double *y, int64_t B, int64_t H, int64_t L,
                      int d_key, int nu, int d_v, double eps, int nthreads)
{
    if (!q || !k || !v || !beta || !W_final || !y || B < 0 || H < 0 || L < 0 || d_key <= 0 ||
        d_v <= 0 || nu < 1 || nu > 2 * d_key - 1)
        return FWO_BAD_ARG;
    const int64_t BH = B * H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > BH)
        nthreads = BH > 0 ? (int)BH : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        job_t *j = &jobs[i];
        j->q = q; j->k = k; j->v = v; j->beta = beta; j->W0 = W0;
        j->W_final = W_final; j->y = y; j->BH = BH; j->L = L;
        j->d_key = d_key; j->nu = nu; j->d_v = d_v; j->eps = eps;
        j->first = BH * i / nthreads;
        j->last = BH * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        run_job(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&tids[i], NULL, run_job, &jobs[i]);
        for (int i = 0; i < nthreads; ++i)
            pthread_join(tids[i], NULL);
    }
    free(jobs);
    free(tids);
    return FWO_OK;
}

/* One decode step of the token-wise variant: q, k [B,H,d_key]; v, y
 * [B,H,d_v]; beta [B,H]; W [B,H,d_v,d_dot] updated in place.  It is the
 * recurrence above over a single token with W carried in from the caller. */
int fwo_delta_decode_step(const double *q, const double *k, const double *v, const double *beta,
                          double *W, double *y, int64_t B, int64_t H, int d_key, int nu, int d_v,
                          double eps, int nthreads)
{
    return fwo_delta_forward(q, k, v, beta, W, W, y, B, H, 1, d_key, nu, d_v, eps, nthreads);
}

/* ---------------------------------------------------------------------- */
/* The sum rule (linear attention) for one (batch, head) pair.            */
/*   q, k: [L, d_key]; v, y: [L, d_v]; W: [d_v, d_dot], z: [d_dot] in/out.*/
/* ---------------------------------------------------------------------- */
static void linear_one(const double *q, const double *k, const double *v, double *W, double *z,
                       double *y, int64_t L, int d_key, int nu, int d_v, int normalize, double eps)
{
    const int d_dot = 2 * d_key * nu;
    double *pk = (double *)malloc(sizeof(double) * d_dot);
    double *pq = (double *)malloc(sizeof(double) * d_dot);
    double *x = (double *)malloc(sizeof(double) * 2 * d_key);
    for (int64_t t = 0; t < L; ++t) {
        dpfp_one(k + t * d_key, pk, x, d_key, nu, eps);
        dpfp_one(q + t * d_key, pq, x, d_key, nu, eps);
        /* W_t = W_{t-1} + v_t outer phi(k_t);  z_t = z_{t-1} + phi(k_t) */
        for (int r = 0; r < d_v; ++r)
            for (int m = 0; m < d_dot; ++m)
                W[(size_t)r * d_dot + m] += v[t * d_v + r] * pk[m];
        for (int m = 0; m < d_dot; ++m)
            z[m] += pk[m];
        /* y_t = W_t phi(q_t), divided by z_t . phi(q_t) when normalising */
        double den = 1.0;
        if (normalize) {
            den = 0.0;
            for (int m = 0; m < d_dot; ++m)
                den += z[m] * pq[m];
        }
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int m = 0; m < d_dot; ++m)
                acc += W[(size_t)r * d_dot + m] * pq[m];
            y[t * d_v + r] = den != 0.0 ? acc / den : 0.0;
        }
    }
    free(pk);
    free(pq);
    free(x);
}

typedef struct {
    const double *q, *k, *v, *W0, *z0;
    double *W_final, *z_final, *y;
    int64_t L;
    int d_key, nu, d_v, normalize;
    double eps;
    int64_t first, last;
} ljob_t;

static void *run_ljob(void *arg)
{
    ljob_t *j = (ljob_t *)arg;
    const int d_dot = 2 * j->d_key * j->nu;
    const size_t wsz = (size_t)j->d_v * d_dot;
    double *z = (double *)malloc(sizeof(double) * d_dot);
    for (int64_t bh = j->first; bh < j->last; ++bh) {
        double *W = j->W_final + bh * wsz;
        if (j->W0 && j->W0 + bh * wsz != W)
            memcpy(W, j->W0 + bh * wsz, sizeof(double) * wsz);
        else if (!j->W0)
            memset(W, 0, sizeof(double) * wsz);
        for (int m = 0; m < d_dot; ++m)
            z[m] = j->z0 ? j->z0[bh * d_dot + m] : 0.0;
        linear_one(j->q + bh * j->L * j->d_key, j->k + bh * j->L * j->d_key, j->v + bh * j->L * j->d_v, W, z,
                   j->y + bh * j->L * j->d_v, j->L, j->d_key, j->nu, j->d_v, j->normalize, j->eps);
        if (j->z_final)
            memcpy(j->z_final + bh * d_dot, z, sizeof(double) * d_dot);
    }
    free(z);
    return NULL;
}

/* The sum rule over [B,H,L,*] inputs: q, k [B,H,L,d_key]; v [B,H,L,d_v];
 * W0 [B,H,d_v,d_dot] and z0 [B,H,d_dot] or NULL (zeros).  Outputs y
 * [B,H,L,d_v], W_final (required; may equal W0) and z_final (or NULL).
 * normalize = 1 divides by z . phi(q), 0 does not. */
int fwo_linear_forward(const double *q, const double *k, const double *v, const double *W0, const double *z0,
                       double *W_final, double *z_final, double *y, int64_t B, int64_t H, int64_t L, int d_key,
                       int nu, int d_v, int normalize, double eps, int nthreads)
{
    if (!q || !k || !v || !W_final || !y || B < 0 || H < 0 || L < 0 || d_key <= 0 || d_v <= 0 || nu < 1 ||
        nu > 2 * d_key - 1 || (normalize != 0 && normalize != 1))
        return FWO_BAD_ARG;
    const int64_t BH = B * H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > BH)
        nthreads = BH > 0 ? (int)BH : 1;
    ljob_t *jobs = (ljob_t *)calloc((size_t)nthreads, sizeof(ljob_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        ljob_t *j = &jobs[i];
        j->q = q; j->k = k; j->v = v; j->W0 = W0; j->z0 = z0;
        j->W_final = W_final; j->z_final = z_final; j->y = y; j->L = L;
        j->d_key = d_key; j->nu = nu; j->d_v = d_v; j->normalize = normalize; j->eps = eps;
        j->first = BH * i / nthreads;
        j->last = BH * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        run_ljob(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&tids[i], NULL, run_ljob, &jobs[i]);
        for (int i = 0; i < nthreads; ++i)
            pthread_join(tids[i], NULL);
    }
    free(jobs);
    free(tids);
    return FWO_OK;
}

/* ---------------------------------------------------------------------- */
/* Backward of the delta rule for one (batch, head) pair.                 */
/* Forward, per token: pk = phi(k_t), pq = phi(q_t), a = W_{t-1} pk,        */
/* u = beta_t (v_t - a), W_t = W_{t-1} + u pk^T, y_t = W_t pq.              */
/* Given gy_t = dL/dy_t and gW = dL/dW_L, the chain rule in reverse order:  */
/*   gW += gy_t pq^T;  gpq = W_t^T gy_t;  gu = gW pk;                       */
/*   gbeta_t = gu . (v_t - a);  gv_t = beta_t gu;                           */
/*   gpk = gW^T u - W_{t-1}^T (beta_t gu);  gW -= (beta_t gu) pk^T;         */
/* then through phi: with p the unnormalised products and s their sum,      */
/* phi = p/(s+eps): gp_l = gphi_l/(s+eps) - (gphi . p)/(s+eps)^2;           */
/* p_{(i-1)n+j} = x_j x_{(j-i) mod n} sends gp to x_j and x_{(j-i) mod n};  */
/* x = ReLU([k, -k]) sends gx_j to k_j (k_j > 0) and -gx_{d_key+j} to k_j   */
/* (-k_j > 0).  gW after token 1 is dL/dW_0.                                */
/* ---------------------------------------------------------------------- */
static void dpfp_backward_one(const double *k, const double *gphi, double *gk, double *x, double *p,
                              int d_key, int nu, double eps)
{
    const int n = 2 * d_key;
    const int d_dot = n * nu;
    for (int j = 0; j < d_key; ++j) {
        x[j] = k[j] > 0.0 ? k[j] : 0.0;
        x[d_key + j] = -k[j] > 0.0 ? -k[j] : 0.0;
    }
    double s = 0.0;
    for (int i = 1; i <= nu; ++i)
        for (int j = 0; j < n; ++j) {
            p[(size_t)(i - 1) * n + j] = x[j] * x[((j - i) % n + n) % n];
            s += p[(size_t)(i - 1) * n + j];
        }
    double gp_dot_p = 0.0;
    for (int m = 0; m < d_dot; ++m)
        gp_dot_p += gphi[m] * p[m];
    double *gx = (double *)calloc((size_t)n, sizeof(double));
    for (int i = 1; i <= nu; ++i)
        for (int j = 0; j < n; ++j) {
            const int m = (i - 1) * n + j, src = ((j - i) % n + n) % n;
            const double gp = gphi[m] / (s + eps) - gp_dot_p / ((s + eps) * (s + eps));
            gx[j] += gp * x[src];
            gx[src] += gp * x[j];
        }
    for (int j = 0; j < d_key; ++j)
        gk[j] = (k[j] > 0.0 ? gx[j] : 0.0) - (-k[j] > 0.0 ? gx[d_key + j] : 0.0);
    free(gx);
}

static void backward_one(const double *q, const double *k, const double *v, const double *beta, const double *W0,
                         const double *gy, const double *gWL, double *gq, double *gk, double *gv, double *gbeta,
                         double *gW0, int64_t L, int d_key, int nu, int d_v, double eps)
{
    const int d_dot = 2 * d_key * nu;
    const size_t wsz = (size_t)d_v * d_dot;
    /* the forward, keeping W_0 .. W_L, phi(k_t), phi(q_t) and a_t = W_{t-1} phi(k_t) */
    double *Ws = (double *)malloc(sizeof(double) * wsz * (size_t)(L + 1));
    double *pk = (double *)malloc(sizeof(double) * d_dot * (size_t)(L > 0 ? L : 1));
    double *pq = (double *)malloc(sizeof(double) * d_dot * (size_t)(L > 0 ? L : 1));
    double *a = (double *)malloc(sizeof(double) * d_v * (size_t)(L > 0 ? L : 1));
    double *x = (double *)malloc(sizeof(double) * 2 * d_key);
    double *p = (double *)malloc(sizeof(double) * d_dot);
    for (size_t e = 0; e < wsz; ++e)
        Ws[e] = W0 ? W0[e] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        double *Wp = Ws + (size_t)t * wsz, *Wn = Ws + (size_t)(t + 1) * wsz;
        dpfp_one(k + t * d_key, pk + t * d_dot, x, d_key, nu, eps);
        dpfp_one(q + t * d_key, pq + t * d_dot, x, d_key, nu, eps);
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int m = 0; m < d_dot; ++m)
                acc += Wp[(size_t)r * d_dot + m] * pk[t * d_dot + m];
            a[t * d_v + r] = acc;
        }
        for (int r = 0; r < d_v; ++r) {
            const double u = beta[t] * (v[t * d_v + r] - a[t * d_v + r]);
            for (int m = 0; m < d_dot; ++m)
                Wn[(size_t)r * d_dot + m] = Wp[(size_t)r * d_dot + m] + u * pk[t * d_dot + m];
        }
    }
    /* the reverse sweep */
    double *gW = (double *)malloc(sizeof(double) * wsz);
    double *gu = (double *)malloc(sizeof(double) * d_v);
    double *gpq = (double *)malloc(sizeof(double) * d_dot);
    double *gpk = (double *)malloc(sizeof(double) * d_dot);
    for (size_t e = 0; e < wsz; ++e)
        gW[e] = gWL ? gWL[e] : 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
        const double *Wp = Ws + (size_t)t * wsz, *Wn = Ws + (size_t)(t + 1) * wsz;
        const double *pkt = pk + t * d_dot, *pqt = pq + t * d_dot;
        /* y_t = W_t pq */
        for (int r = 0; r < d_v; ++r)
            for (int m = 0; m < d_dot; ++m)
                gW[(size_t)r * d_dot + m] += gy[t * d_v + r] * pqt[m];
        for (int m = 0; m < d_dot; ++m) {
            double acc = 0.0;
            for (int r = 0; r < d_v; ++r)
                acc += Wn[(size_t)r * d_dot + m] * gy[t * d_v + r];
            gpq[m] = acc;
        }
        /* W_t = W_{t-1} + u pk^T */
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int m = 0; m < d_dot; ++m)
                acc += gW[(size_t)r * d_dot + m] * pkt[m];
            gu[r] = acc;
        }
        double gb = 0.0;
        for (int r = 0; r < d_v; ++r)
            gb += gu[r] * (v[t * d_v + r] - a[t * d_v + r]);
        gbeta[t] = gb;
        for (int r = 0; r < d_v; ++r)
            gv[t * d_v + r] = beta[t] * gu[r];
        for (int m = 0; m < d_dot; ++m) {
            double acc = 0.0;
            for (int r = 0; r < d_v; ++r) {
                const double u = beta[t] * (v[t * d_v + r] - a[t * d_v + r]);
                acc += gW[(size_t)r * d_dot + m] * u - Wp[(size_t)r * d_dot + m] * beta[t] * gu[r];
            }
            gpk[m] = acc;
        }
        for (int r = 0; r < d_v; ++r)
            for (int m = 0; m < d_dot; ++m)
                gW[(size_t)r * d_dot + m] -= beta[t] * gu[r] * pkt[m];
        dpfp_backward_one(q + t * d_key, gpq, gq + t * d_key, x, p, d_key, nu, eps);
        dpfp_backward_one(k + t * d_key, gpk, gk + t * d_key, x, p, d_key, nu, eps);
    }
    if (gW0)
        memcpy(gW0, gW, sizeof(double) * wsz);
    free(Ws); free(pk); free(pq); free(a); free(x); free(p);
    free(gW); free(gu); free(gpq); free(gpk);
}

typedef struct {
    const double *q, *k, *v, *beta, *W0, *gy, *gWL;
    double *gq, *gk, *gv, *gbeta, *gW0;
    int64_t L;
    int d_key, nu, d_v;
    double eps;
    int64_t first, last;
} bjob_t;

static void *run_bjob(void *arg)
{
    bjob_t *j = (bjob_t *)arg;
    const int d_dot = 2 * j->d_key * j->nu;
    const size_t wsz = (size_t)j->d_v * d_dot;
    for (int64_t bh = j->first; bh < j->last; ++bh)
        backward_one(j->q + bh * j->L * j->d_key, j->k + bh * j->L * j->d_key, j->v + bh * j->L * j->d_v,
                     j->beta + bh * j->L, j->W0 ? j->W0 + bh * wsz : NULL, j->gy + bh * j->L * j->d_v,
                     j->gWL ? j->gWL + bh * wsz : NULL, j->gq + bh * j->L * j->d_key, j->gk + bh * j->L * j->d_key,
                     j->gv + bh * j->L * j->d_v, j->gbeta + bh * j->L, j->gW0 ? j->gW0 + bh * wsz : NULL, j->L,
                     j->d_key, j->nu, j->d_v, j->eps);
    return NULL;
}

/* Gradients of L = sum(gy * y) + sum(gWL * W_final) with respect to q, k, v,
 * beta and W0, for the forward fwo_delta_forward computes.  gWL and W0 may
 * be NULL (zeros); gW0 may be NULL (not returned). */
int fwo_delta_backward(const double *q, const double *k, const double *v, const double *beta, const double *W0,
                       const double *gy, const double *gWL, double *gq, double *gk, double *gv, double *gbeta,
                       double *gW0, int64_t B, int64_t H, int64_t L, int d_key, int nu, int d_v, double eps,
                       int nthreads)
{
    if (!q || !k || !v || !beta || !gy || !gq || !gk || !gv || !gbeta || B < 0 || H < 0 || L < 0 ||
        d_key <= 0 || d_v <= 0 || nu < 1 || nu > 2 * d_key - 1)
        return FWO_BAD_ARG;
    const int64_t BH = B * H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > BH)
        nthreads = BH > 0 ? (int)BH : 1;
    bjob_t *jobs = (bjob_t *)calloc((size_t)nthreads, sizeof(bjob_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        bjob_t *j = &jobs[i];
        j->q = q; j->k = k; j->v = v; j->beta = beta; j->W0 = W0; j->gy = gy; j->gWL = gWL;
        j->gq = gq; j->gk = gk; j->gv = gv; j->gbeta = gbeta; j->gW0 = gW0; j->L = L;
        j->d_key = d_key; j->nu = nu; j->d_v = d_v; j->eps = eps;
        j->first = BH * i / nthreads;
        j->last = BH * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        run_bjob(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&tids[i], NULL, run_bjob, &jobs[i]);
        for (int i = 0; i < nthreads; ++i)
            pthread_join(tids[i], NULL);
    }
    free(jobs);
    free(tids);
    return FWO_OK;
}
