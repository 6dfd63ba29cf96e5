/*
 * ttt_oracle.c -- fp64 CPU oracle for the Test-Time-Training (TTT) layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file; only the test-suite, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the definition, token by token, in the "primal" form):
 *   hidden state = weights W of an inner model f(x; W), reset to W0 for every
 *   (batch, head) sequence ("Fast weights 与 TTT layers", section 4: fast weights
 *   are reset at each sequence boundary);
 *   reconstruction loss  l_t(W) = 1/2 || f(k_t; W) - v_t ||^2
 *   ("Fast weights 与 TTT layers", opening formula; "TTT：Test-Time Training",
 *   section TTT / MSE loss);
 *   mini-batch gradient descent: the sequence is cut into consecutive blocks of b
 *   tokens; every token of a block takes its gradient at the W the previous block
 *   left, and W moves by -eta_s * grad l_s for each token s in order, so the
 *   running W after token t holds the cumulative sum of the block's writes
 *   ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2, formula 6 and
 *   the cumsum / gradient-operator channels);
 *   output rule z_t = f(q_t; W_t) (same walkthrough, section 1.2, formula 1/5;
 *   "TTT：Test-Time Training", section TTT general form).
 *   causal = 1: W_t includes the writes of all tokens s <= t of t's block.
 *   causal = 0: every query of a block reads the W at the end of that block
 *   (b = T gives the single full-batch step of the vision variant, ViT3 article,
 *   observation 2).
 *   norm (linear): f(x; W) = x + LN(x W), LN(y) = gamma * (y - mean(y)) /
 *   sqrt(var(y) + eps) + beta over the d outputs (the walkthrough's TTT-Linear,
 *   section 2.2.1: the inner model always carries a layer norm and a residual
 *   connection); gamma, beta per head are inputs, not trained by the inner step.
 *   With e = f(k; Ws) - v, yh = (y - mean) / s (s = sqrt(var + eps)) and
 *   g = gamma * e, the gradient is dW = k^T dy with
 *   dy = (g - mean(g) - yh * mean(g * yh)) / s.
 *   epochs (linear, causal = 0 with one block b >= T only): the block's gradient
 *   step is taken `epochs` times, each pass with its gradients at the W the
 *   previous pass left, before the queries read W (the ViT3 article, observation
 *   2: one epoch of full-batch inner training is one update over all N tokens,
 *   further epochs repeat it).
 *
 * Inner models (walkthrough section 2.2.1; ViT3 article observation 4):
 *   linear: f(x; W) = x W, W in R^{d x d} (row convention, x is a 1 x d row).
 *   norm (mlp): f(x) = x + LN(act(x W1 + c1) W2 + c2) with the same LN and gradient
 *   rule (the walkthrough's TTT-MLP carries the norm and residual too); the MLP's
 *   backward then starts from dy instead of e.
 *   mlp   : f(x) = act(x W1 + c1) W2 + c2, W1 d x m, c1 1 x m, W2 m x d, c2 1 x d,
 *           act = SiLU, SiLU(h) = h * sigma(h) (ViT3 article, observation 4), or
 *           act = GELU, GELU(h) = h * Phi(h) with Phi the standard normal CDF
 *           (the walkthrough's TTT-MLP, section 2.2.1; exact erf form).
 * Gradients are written out by hand from the chain rule:
 *   linear mse: e = k W - v,   dW = k^T e
 *   linear dot (negative dot-product loss l = -(k W) v^T, "TTT：Test-Time Training",
 *              section "如何理解"): dW = -k^T v
 *   mlp: h = k W1 + c1, a = act(h), e = a W2 + c2 - v,
 *        dW2 = a^T e, dc2 = e, g = (e W2^T) * act'(h), dW1 = k^T g, dc1 = g,
 *        SiLU'(h) = sigma(h) (1 + h (1 - sigma(h))), GELU'(h) = Phi(h) + h phi(h)
 *        with phi the standard normal density.
 *
 * Layouts: all arrays are C-contiguous double.  q, k, v, z: [B,H,T,d];
 * eta: [B,H,T] or NULL (then eta_scalar is used for every token);
 * W0 (linear) [.., H, d, d] with batch stride w0_bstride elements (0 = shared over
 * the batch); W_out [B,H,d,d] or NULL.  MLP: W1 [.., H, d, m], c1 [.., H, m],
 * W2 [.., H, m, d], c2 [.., H, d]; per_batch = 0 means one parameter set per head
 * shared over the batch ([H,...]), 1 means one per (batch, head) ([B,H,...]);
 * outputs [B,H,...] or NULL.
 * Returns 0 on success, -1 on bad arguments.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ linear */

typedef struct {
    int B, H, T, d, b, causal, loss, epochs;
    const double *q, *k, *v, *eta;
    double eta_scalar;
    const double *W0;
    long long w0_bstride;
    double *z, *W_out;
    const double *ln_gamma, *ln_beta;  /* [H][d] each, or NULL: no norm / residual */
    double ln_eps;
    int next;               /* next (batch, head) chain to process */
    pthread_mutex_t lock;
} linear_job;

/* y -> LN(y) in place over d entries; returns s = sqrt(var + eps) and leaves the
 * normalised values in yh */
static double layer_norm(int d, const double *gamma, const double *beta, double eps, const double *y,
                         double *yh, double *out)
{
    double mu = 0.0, var = 0.0;
    for (int j = 0; j < d; ++j) mu += y[j];
    mu /= d;
    for (int j = 0; j < d; ++j) var += (y[j] - mu) * (y[j] - mu);
    var /= d;
    const double s = sqrt(var + eps);
    for (int j = 0; j < d; ++j) {
        yh[j] = (y[j] - mu) / s;
        out[j] = gamma[j] * yh[j] + beta[j];
    }
    return s;
}

/* z_t = f(q_t; W): q_t W, or q_t + LN(q_t W) with the norm */
static void linear_out(const linear_job *J, int hi, const double *qt, const double *W, double *zt,
                       double *tmp, double *tmp2)
{
    const int d = J->d;
    for (int j = 0; j < d; ++j) {
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += qt[i] * W[i * d + j];
        tmp[j] = s;
    }
    if (!J->ln_gamma) {
        for (int j = 0; j < d; ++j) zt[j] = tmp[j];
        return;
    }
    layer_norm(d, J->ln_gamma + (size_t)hi * d, J->ln_beta + (size_t)hi * d, J->ln_eps, tmp, tmp2, zt);
    for (int j = 0; j < d; ++j) zt[j] += qt[j];
}

static void linear_chain(const linear_job *J, int bh)
{
    const int T = J->T, d = J->d, b = J->b;
    const int bi = bh / J->H, hi = bh % J->H;
    const double *q = J->q + (size_t)bh * T * d;
    const double *k = J->k + (size_t)bh * T * d;
    const double *v = J->v + (size_t)bh * T * d;
    const double *eta = J->eta ? J->eta + (size_t)bh * T : NULL;
    double *z = J->z + (size_t)bh * T * d;
    const double *W0 = J->W0 + (size_t)bi * J->w0_bstride + (size_t)hi * d * d;

    double *W = malloc(sizeof(double) * d * d);    /* running weights          */
    double *Ws = malloc(sizeof(double) * d * d);   /* block's gradient point   */
    double *e = malloc(sizeof(double) * d);
    double *y = malloc(sizeof(double) * d), *yh = malloc(sizeof(double) * d);
    double *ln = malloc(sizeof(double) * d);
    memcpy(W, W0, sizeof(double) * d * d);

    for (int n0 = 0; n0 < T; n0 += b) {
        const int n1 = (n0 + b < T) ? n0 + b : T;
        for (int ep = 0; ep < J->epochs; ++ep) {
        memcpy(Ws, W, sizeof(double) * d * d);
        for (int t = n0; t < n1; ++t) {
            const double *kt = k + (size_t)t * d, *vt = v + (size_t)t * d;
            const double et = eta ? eta[t] : J->eta_scalar;
            if (J->loss == 0 && J->ln_gamma) {
                /* e = k_t + LN(k_t Ws) - v_t; the gradient w.r.t. y = k_t Ws
                 * through the layer norm replaces e below */
                const double *gam = J->ln_gamma + (size_t)hi * d, *bet = J->ln_beta + (size_t)hi * d;
                for (int j = 0; j < d; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < d; ++i) s += kt[i] * Ws[i * d + j];
                    y[j] = s;
                }
                const double sd = layer_norm(d, gam, bet, J->ln_eps, y, yh, ln);
                double mg = 0.0, mgy = 0.0;
                for (int j = 0; j < d; ++j) {
                    const double g = gam[j] * (kt[j] + ln[j] - vt[j]);
                    mg += g;
                    mgy += g * yh[j];
                    e[j] = g;
                }
                mg /= d;
                mgy /= d;
                for (int j = 0; j < d; ++j) e[j] = (e[j] - mg - yh[j] * mgy) / sd;
            } else if (J->loss == 0) {
                /* e = k_t Ws - v_t */
                for (int j = 0; j < d; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < d; ++i) s += kt[i] * Ws[i * d + j];
                    e[j] = s - vt[j];
                }
            } else {
                /* gradient of -(k W) v^T is -k^T v: use e = -v */
                for (int j = 0; j < d; ++j) e[j] = -vt[j];
            }
            /* W -= eta_t k_t^T e */
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j) W[i * d + j] -= et * kt[i] * e[j];
            if (J->causal) linear_out(J, hi, q + (size_t)t * d, W, z + (size_t)t * d, y, yh);
        }
        }  /* epochs */
        if (!J->causal)
            for (int t = n0; t < n1; ++t) linear_out(J, hi, q + (size_t)t * d, W, z + (size_t)t * d, y, yh);
    }
    if (J->W_out) memcpy(J->W_out + (size_t)bh * d * d, W, sizeof(double) * d * d);
    free(W); free(Ws); free(e); free(y); free(yh); free(ln);
}

static void *linear_worker(void *arg)
{
    linear_job *J = (linear_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int bh = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (bh >= J->B * J->H) break;
        linear_chain(J, bh);
    }
    return NULL;
}

int ttt_oracle_linear(int B, int H, int T, int d, int b, int causal, int loss, int epochs,
                      const double *q, const double *k, const double *v,
                      const double *eta, double eta_scalar,
                      const double *W0, long long w0_bstride,
                      double *z, double *W_out, int nthreads,
                      const double *ln_gamma, const double *ln_beta, double ln_eps)
{
    if ((ln_gamma == NULL) != (ln_beta == NULL) || (ln_gamma && loss != 0)) return -1;
    if (B < 0 || H < 0 || T < 0 || d <= 0 || b <= 0 || !W0 || (T > 0 && (!q || !k || !v || !z)))
        return -1;
    if (loss != 0 && loss != 1) return -1;
    if (epochs < 1 || (epochs > 1 && (causal || b < T))) return -1;
    linear_job J = {B, H, T, d, b, causal ? 1 : 0, loss, epochs, q, k, v, eta, eta_scalar,
                    W0, w0_bstride, z, W_out, ln_gamma, ln_beta, ln_eps, 0};
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, linear_worker, &J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* --------------------------------------------------------------------- mlp */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* act(h) and act'(h); act 0 = SiLU, 1 = GELU (erf form) */
static double act_f(int act, double h)
{
    if (act == 0) return h * sigmoid(h);
    return h * 0.5 * (1.0 + erf(h / sqrt(2.0)));
}

static double act_d(int act, double h)
{
    if (act == 0) {
        const double sg = sigmoid(h);
        return sg * (1.0 + h * (1.0 - sg));
    }
    const double Phi = 0.5 * (1.0 + erf(h / sqrt(2.0)));
    const double phi = exp(-0.5 * h * h) / sqrt(2.0 * 3.14159265358979323846);
    return Phi + h * phi;
}

typedef struct {
    int B, H, T, d, m, b, causal, act;
    const double *q, *k, *v, *eta;
    double eta_scalar;
    const double *W1, *c1, *W2, *c2;
    int per_batch;
    double *z, *W1o, *c1o, *W2o, *c2o;
    const double *ln_gamma, *ln_beta;  /* [H][d] inner norm x + LN(mlp(x)), or NULL */
    double ln_eps;
    int next;
    pthread_mutex_t lock;
} mlp_job;

/* With the inner norm, f(x) = x + LN(y), y = the MLP's output row (length d):
 * replaces the residual row r = y - v by dL/dy for l = 1/2 ||x + LN(y) - v||^2, in
 * place (the same formula as the linear model's norm: g = gamma e,
 * dy = (g - mean(g) - yh mean(g yh)) / s with e = x + LN(y) - v); yh is scratch. */
static void mlp_ln_grad(int d, const double *gm, const double *bt, double eps, const double *x,
                        const double *vt, double *r, double *yh)
{
    double mu = 0.0, var = 0.0;
    for (int j = 0; j < d; ++j) r[j] += vt[j];  /* back to y */
    for (int j = 0; j < d; ++j) mu += r[j];
    mu /= d;
    for (int j = 0; j < d; ++j) var += (r[j] - mu) * (r[j] - mu);
    var /= d;
    const double sd = sqrt(var + eps);
    double mg = 0.0, mgy = 0.0;
    for (int j = 0; j < d; ++j) {
        yh[j] = (r[j] - mu) / sd;
        const double e = x[j] + gm[j] * yh[j] + bt[j] - vt[j];
        r[j] = gm[j] * e;
        mg += r[j];
        mgy += r[j] * yh[j];
    }
    mg /= d;
    mgy /= d;
    for (int j = 0; j < d; ++j) r[j] = (r[j] - mg - yh[j] * mgy) / sd;
}

/* z = x + LN(y) in place of the MLP output row y */
static void mlp_ln_out(int d, const double *gm, const double *bt, double eps, const double *x, double *y)
{
    double mu = 0.0, var = 0.0;
    for (int j = 0; j < d; ++j) mu += y[j];
    mu /= d;
    for (int j = 0; j < d; ++j) var += (y[j] - mu) * (y[j] - mu);
    var /= d;
    const double sd = sqrt(var + eps);
    for (int j = 0; j < d; ++j) y[j] = x[j] + gm[j] * (y[j] - mu) / sd + bt[j];
}

/* z = act(x W1 + c1) W2 + c2 with scratch h (length m) */
static void mlp_forward(int act, int d, int m, const double *x, const double *W1, const double *c1,
                        const double *W2, const double *c2, double *h, double *out)
{
    for (int j = 0; j < m; ++j) {
        double s = c1[j];
        for (int i = 0; i < d; ++i) s += x[i] * W1[i * m + j];
        h[j] = act_f(act, s);
    }
    for (int j = 0; j < d; ++j) {
        double s = c2[j];
        for (int i = 0; i < m; ++i) s += h[i] * W2[i * d + j];
        out[j] = s;
    }
}

static void mlp_chain(const mlp_job *J, int bh)
{
    const int T = J->T, d = J->d, m = J->m, b = J->b;
    const int hi = bh % J->H;
    const size_t hp = J->per_batch ? (size_t)bh : (size_t)hi;   /* parameter-set index */
    const double *q = J->q + (size_t)bh * T * d;
    const double *k = J->k + (size_t)bh * T * d;
    const double *v = J->v + (size_t)bh * T * d;
    const double *eta = J->eta ? J->eta + (size_t)bh * T : NULL;
    double *z = J->z + (size_t)bh * T * d;

    double *W1 = malloc(sizeof(double) * d * m), *W1s = malloc(sizeof(double) * d * m);
    double *W2 = malloc(sizeof(double) * m * d), *W2s = malloc(sizeof(double) * m * d);
    double *c1 = malloc(sizeof(double) * m), *c1s = malloc(sizeof(double) * m);
    double *c2 = malloc(sizeof(double) * d), *c2s = malloc(sizeof(double) * d);
    double *h = malloc(sizeof(double) * m), *a = malloc(sizeof(double) * m);
    double *g = malloc(sizeof(double) * m), *e = malloc(sizeof(double) * d);
    double *yh = malloc(sizeof(double) * d);
    const double *gm = J->ln_gamma ? J->ln_gamma + (size_t)hi * d : NULL;
    const double *bt = J->ln_beta ? J->ln_beta + (size_t)hi * d : NULL;
    memcpy(W1, J->W1 + hp * d * m, sizeof(double) * d * m);
    memcpy(c1, J->c1 + hp * m, sizeof(double) * m);
    memcpy(W2, J->W2 + hp * m * d, sizeof(double) * m * d);
    memcpy(c2, J->c2 + hp * d, sizeof(double) * d);

    for (int n0 = 0; n0 < T; n0 += b) {
        const int n1 = (n0 + b < T) ? n0 + b : T;
        memcpy(W1s, W1, sizeof(double) * d * m);
        memcpy(c1s, c1, sizeof(double) * m);
        memcpy(W2s, W2, sizeof(double) * m * d);
        memcpy(c2s, c2, sizeof(double) * d);
        for (int t = n0; t < n1; ++t) {
            const double *kt = k + (size_t)t * d, *vt = v + (size_t)t * d;
            const double et = eta ? eta[t] : J->eta_scalar;
            /* forward at the block's gradient point */
            for (int j = 0; j < m; ++j) {
                double s = c1s[j];
                for (int i = 0; i < d; ++i) s += kt[i] * W1s[i * m + j];
                h[j] = s;
                a[j] = act_f(J->act, s);
            }
            for (int j = 0; j < d; ++j) {
                double s = c2s[j];
                for (int i = 0; i < m; ++i) s += a[i] * W2s[i * d + j];
                e[j] = s - vt[j];
            }
            if (gm) mlp_ln_grad(d, gm, bt, J->ln_eps, kt, vt, e, yh);  /* e := dL/dy */
            /* backward: g = (e W2s^T) * act'(h) */
            for (int i = 0; i < m; ++i) {
                double s = 0.0;
                for (int j = 0; j < d; ++j) s += e[j] * W2s[i * d + j];
                if (J->act == 0) {
                    const double sg = sigmoid(h[i]);
                    g[i] = s * sg * (1.0 + h[i] * (1.0 - sg));
                } else {
                    g[i] = s * act_d(J->act, h[i]);
                }
            }
            /* descent step of token t */
            for (int i = 0; i < m; ++i)
                for (int j = 0; j < d; ++j) W2[i * d + j] -= et * a[i] * e[j];
            for (int j = 0; j < d; ++j) c2[j] -= et * e[j];
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < m; ++j) W1[i * m + j] -= et * kt[i] * g[j];
            for (int j = 0; j < m; ++j) c1[j] -= et * g[j];
            if (J->causal) {
                mlp_forward(J->act, d, m, q + (size_t)t * d, W1, c1, W2, c2, h, z + (size_t)t * d);
                if (gm) mlp_ln_out(d, gm, bt, J->ln_eps, q + (size_t)t * d, z + (size_t)t * d);
            }
        }
        if (!J->causal)
            for (int t = n0; t < n1; ++t) {
                mlp_forward(J->act, d, m, q + (size_t)t * d, W1, c1, W2, c2, h, z + (size_t)t * d);
                if (gm) mlp_ln_out(d, gm, bt, J->ln_eps, q + (size_t)t * d, z + (size_t)t * d);
            }
    }
    if (J->W1o) memcpy(J->W1o + (size_t)bh * d * m, W1, sizeof(double) * d * m);
    if (J->c1o) memcpy(J->c1o + (size_t)bh * m, c1, sizeof(double) * m);
    if (J->W2o) memcpy(J->W2o + (size_t)bh * m * d, W2, sizeof(double) * m * d);
    if (J->c2o) memcpy(J->c2o + (size_t)bh * d, c2, sizeof(double) * d);
    free(W1); free(W1s); free(W2); free(W2s); free(c1); free(c1s); free(c2); free(c2s);
    free(h); free(a); free(g); free(e); free(yh);
}

static void *mlp_worker(void *arg)
{
    mlp_job *J = (mlp_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int bh = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (bh >= J->B * J->H) break;
        mlp_chain(J, bh);
    }
    return NULL;
}

int ttt_oracle_mlp(int B, int H, int T, int d, int m, int b, int causal,
                   const double *q, const double *k, const double *v,
                   const double *eta, double eta_scalar,
                   const double *W1, const double *c1, const double *W2, const double *c2,
                   int per_batch,
                   double *z, double *W1o, double *c1o, double *W2o, double *c2o,
                   int nthreads, int act, const double *ln_gamma, const double *ln_beta, double ln_eps)
{
    if (B < 0 || H < 0 || T < 0 || d <= 0 || m <= 0 || b <= 0 || !W1 || !c1 || !W2 || !c2 ||
        (T > 0 && (!q || !k || !v || !z)) || (act != 0 && act != 1) || (!ln_gamma != !ln_beta))
        return -1;
    mlp_job J = {B, H, T, d, m, b, causal ? 1 : 0, act, q, k, v, eta, eta_scalar,
                 W1, c1, W2, c2, per_batch ? 1 : 0, z, W1o, c1o, W2o, c2o, ln_gamma, ln_beta, ln_eps, 0};
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, mlp_worker, &J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------- depthwise conv */
/*
 * Depthwise 3x3 convolution as the inner model (ViT3 article, observation 6: the
 * inner model of vision TTT can be a small convolution; the ViT3 block uses a
 * depthwise one).  The N = height * width tokens of a sequence are the pixels of a
 * height x width grid in row-major order; f(X; W)[p][c] = sum over the 3 x 3
 * offsets (di, dj) in {-1,0,1}^2 of X[p + (di, dj)][c] * W[(di+1)*3 + (dj+1)][c],
 * with zero outside the grid (cross-correlation, "same" padding).  One full-batch
 * inner step per epoch over all N tokens (observation 2), non-causal: every query
 * reads the final W.  loss 0: l_p = 1/2 || f(K)[p] - v_p ||^2, gradient
 * dW[o][c] = sum_p eta_p e[p][c] K[p + o][c] with e = f(K) - V at the epoch's start
 * weights; loss 1: l_p = -f(K)[p] . v_p, e = -V.
 * Layouts: q, k, v, z [B,H,N,d]; eta [B,H,N] or NULL; W0 [.., H, 9, d] with batch
 * stride w0_bstride elements (0 = shared over the batch); W_out [B,H,9,d] or NULL.
 */
typedef struct {
    int B, H, hh, ww, d, loss, epochs;
    const double *q, *k, *v, *eta;
    double eta_scalar;
    const double *W0;
    long long w0_bstride;
    double *z, *W_out;
    int next;
    pthread_mutex_t lock;
} dwconv_job;

/* X[p + o][c] for offset o = (di+1)*3 + (dj+1), zero outside the grid */
static double dw_tap(const double *X, int hh, int ww, int d, int p, int o, int c)
{
    const int y = p / ww + o / 3 - 1, x = p % ww + o % 3 - 1;
    if (y < 0 || y >= hh || x < 0 || x >= ww) return 0.0;
    return X[((size_t)y * ww + x) * d + c];
}

static void dwconv_chain(const dwconv_job *J, int bh)
{
    const int N = J->hh * J->ww, d = J->d, hh = J->hh, ww = J->ww;
    const int bi = bh / J->H, hi = bh % J->H;
    const double *q = J->q + (size_t)bh * N * d, *k = J->k + (size_t)bh * N * d;
    const double *v = J->v + (size_t)bh * N * d;
    const double *eta = J->eta ? J->eta + (size_t)bh * N : NULL;
    double *W = malloc(sizeof(double) * 9 * d), *Ws = malloc(sizeof(double) * 9 * d);
    double *e = malloc(sizeof(double) * (size_t)N * d);
    memcpy(W, J->W0 + (size_t)bi * J->w0_bstride + (size_t)hi * 9 * d, sizeof(double) * 9 * d);
    for (int ep = 0; ep < J->epochs; ++ep) {
        memcpy(Ws, W, sizeof(double) * 9 * d);
        for (int p = 0; p < N; ++p)
            for (int c = 0; c < d; ++c) {
                double f = 0.0;
                if (J->loss == 0)
                    for (int o = 0; o < 9; ++o) f += dw_tap(k, hh, ww, d, p, o, c) * Ws[o * d + c];
                e[(size_t)p * d + c] = f - v[(size_t)p * d + c];
            }
        for (int o = 0; o < 9; ++o)
            for (int c = 0; c < d; ++c) {
                double g = 0.0;
                for (int p = 0; p < N; ++p)
                    g += (eta ? eta[p] : J->eta_scalar) * e[(size_t)p * d + c] * dw_tap(k, hh, ww, d, p, o, c);
                W[o * d + c] -= g;
            }
    }
    double *z = J->z + (size_t)bh * N * d;
    for (int p = 0; p < N; ++p)
        for (int c = 0; c < d; ++c) {
            double s = 0.0;
            for (int o = 0; o < 9; ++o) s += dw_tap(q, hh, ww, d, p, o, c) * W[o * d + c];
            z[(size_t)p * d + c] = s;
        }
    if (J->W_out) memcpy(J->W_out + (size_t)bh * 9 * d, W, sizeof(double) * 9 * d);
    free(W); free(Ws); free(e);
}

static void *dwconv_worker(void *arg)
{
    dwconv_job *J = (dwconv_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int bh = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (bh >= J->B * J->H) break;
        dwconv_chain(J, bh);
    }
    return NULL;
}

int ttt_oracle_dwconv(int B, int H, int hh, int ww, int d, int loss, int epochs,
                      const double *q, const double *k, const double *v,
                      const double *eta, double eta_scalar,
                      const double *W0, long long w0_bstride,
                      double *z, double *W_out, int nthreads)
{
    if (B < 0 || H < 0 || hh < 0 || ww < 0 || d <= 0 || epochs < 1 || !W0 || (loss != 0 && loss != 1) ||
        (hh * ww > 0 && (!q || !k || !v || !z)))
        return -1;
    dwconv_job J = {B, H, hh, ww, d, loss, epochs, q, k, v, eta, eta_scalar, W0, w0_bstride, z, W_out, 0};
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, dwconv_worker, &J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/*
 * Input-dependent inner learning rate ("Learning to (Learn at Test Time)"
 * walkthrough, section 2.2.3, the learnable rate): eta(x) = eta_base * sigma(theta_lr . x)
 * with theta_lr a learnable vector of the outer loop, sigma the logistic function
 * 1 / (1 + e^-a) and eta_base the base rate (1 for TTT-Linear, 0.1 for TTT-MLP).
 * x is the layer's input token; each head carries its own vector (the passage names
 * one vector; a multi-head layer gates each head's rate).
 *   x: [B,T,dm], theta: [H,dm], eta: [B,H,T] (the layout the TTT layer reads).
 */
int ttt_oracle_eta_gate(int B, int T, int H, int dm, const double *x, const double *theta,
                        double eta_base, double *eta)
{
    if (B < 0 || T < 0 || H < 1 || dm < 1 || !x || !theta || !eta) return -1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int t = 0; t < T; ++t) {
                const double *xt = x + ((size_t)b * T + t) * dm, *th = theta + (size_t)h * dm;
                double a = 0.0;
                for (int i = 0; i < dm; ++i) a += th[i] * xt[i];
                eta[((size_t)b * H + h) * T + t] = eta_base / (1.0 + exp(-a));
            }
    return 0;
}
