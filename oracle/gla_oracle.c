/*
 * gla_oracle.c -- fp64 CPU oracle for the Simple GLA mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * CUDA path is checked against.  Only the test suite, the package's smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Source: "Beyond the KV cache: Training and serving i14's Laplace 3B linear
 * attention model on AWS Trainium2 with native PyTorch" (AWS ML blog), section
 * "i14 and the Laplace 3B architecture", paragraphs "GLA mixer" and "Decay
 * schedule" (the equations there are images; the text fixes the reading used
 * here), and section "Challenge 3" (the backward differentiates through every
 * sequential state update).
 *
 * Everything is the definition written out token by token, in double
 * precision, with no blocking, chunking or reordering:
 *
 *   S_0 = init_state (or 0)
 *   S_t = lambda_h * S_{t-1} + k_t v_t^T            (rank-1 write, fixed decay)
 *   z_t = sum_c a_{h,c} q_{t,c} k_{t,c}             (per-channel rescaled key)
 *   o_t = S_t^T q_t + sigmoid(z_t) v_t              (readout after the update,
 *                                                    plus the self-augmentation)
 *
 * Layouts (all row-major, contiguous):
 *   q, k     [B, T, H, dk]       v, o   [B, T, H, dv]
 *   state    [B, H, dk, dv]      a      [H, dk]        gamma [H]  (natural log)
 * Work is threaded over the independent (b, h) pairs; every reduction over
 * (b, h) is summed afterwards in a fixed order, so results do not depend on
 * the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* Decay schedule ("Decay schedule" paragraph and "Decay schedule's reach"):
 * half-lives geometric from t_min to t_max across the H heads,
 *   T_h = t_min * (t_max / t_min)^(h / (H - 1)),
 * lambda_h = 2^(-1/T_h), so gamma_h = ln(lambda_h) = -ln(2) / T_h.
 * With t_min = 1 this gives lambda_0 = 0.5 (one-token half-life).            */
void oracle_decay_schedule(int H, double t_min, double t_max, double *gamma)
{
    for (int h = 0; h < H; ++h) {
        double frac = (H > 1) ? (double)h / (double)(H - 1) : 0.0;
        double half_life = t_min * pow(t_max / t_min, frac);
        gamma[h] = -log(2.0) / half_life;
    }
}

/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v, *gamma, *a, *init, *dO, *dfin;
    double *o, *fin, *dq, *dk, *dv, *da_part, *dinit;
    long B, T, H, dk_, dv_;
    long next;              /* next (b,h) pair to take */
    pthread_mutex_t lock;
} job_t;

static long take(job_t *j)
{
    pthread_mutex_lock(&j->lock);
    long p = j->next++;
    pthread_mutex_unlock(&j->lock);
    return p;
}

static int nthreads_or_default(int n)
{
    if (n > 0) return n;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

static void run_threads(void *(*fn)(void *), job_t *j, int nthreads, long npairs)
{
    int n = nthreads_or_default(nthreads);
    if (n > npairs) n = (int)(npairs > 0 ? npairs : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
    for (int i = 0; i < n; ++i) pthread_create(&th[i], NULL, fn, j);
    for (int i = 0; i < n; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* Row pointers into the token-major tensors. */
#define QROW(X, b, t, h, d) ((X) + ((((b) * T + (t)) * H + (h)) * (d)))

/* ------------------------------------------------------------------------ */
/* Forward: the token-by-token recurrence. */
static void *fwd_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const long B = j->B, T = j->T, H = j->H, dk = j->dk_, dv = j->dv_;
    double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
    for (;;) {
        long p = take(j);
        if (p >= B * H) break;
        long b = p / H, h = p % H;
        double lam = exp(j->gamma[h]);
        const double *a = j->a + h * dk;
        if (j->init) memcpy(S, j->init + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        for (long t = 0; t < T; ++t) {
            const double *q = QROW(j->q, b, t, h, dk);
            const double *k = QROW(j->k, b, t, h, dk);
            const double *v = QROW(j->v, b, t, h, dv);
            double *o = QROW(j->o, b, t, h, dv);
            /* S_t = lambda S_{t-1} + k_t v_t^T */
            for (long i = 0; i < dk; ++i)
                for (long n = 0; n < dv; ++n)
                    S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];
            /* z_t and the sigmoid gate */
            double z = 0.0;
            for (long i = 0; i < dk; ++i) z += a[i] * q[i] * k[i];
            double g = sigmoid(z);
            /* o_t = S_t^T q_t + g v_t */
            for (long n = 0; n < dv; ++n) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += S[i * dv + n] * q[i];
                o[n] = acc + g * v[n];
            }
        }
        if (j->fin) memcpy(j->fin + p * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
    }
    free(S);
    return NULL;
}

int oracle_fwd(const double *q, const double *k, const double *v, const double *gamma,
               const double *a, const double *init_state, double *o, double *final_state,
               long B, long T, long H, long dk, long dv, int nthreads)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    job_t j;
    memset(&j, 0, sizeof(j));
    j.q = q; j.k = k; j.v = v; j.gamma = gamma; j.a = a; j.init = init_state;
    j.o = o; j.fin = final_state;
    j.B = B; j.T = T; j.H = H; j.dk_ = dk; j.dv_ = dv;
    pthread_mutex_init(&j.lock, NULL);
    run_threads(fwd_worker, &j, nthreads, B * H);
    pthread_mutex_destroy(&j.lock);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward, derived by hand from the recurrence (the pages only say that the
 * backward differentiates through all sequential state updates).  With the
 * scalar loss L = sum_t dO_t . o_t + <dS_final, S_T>:
 *
 *   G_T = q_T dO_T^T + dS_final,   G_t = q_t dO_t^T + lambda G_{t+1}
 *   r_t = sigmoid'(z_t) (dO_t . v_t)
 *   dq_t = S_t dO_t + r_t (a * k_t)
 *   dk_t = G_t v_t + r_t (a * q_t)
 *   dv_t = G_t^T k_t + sigmoid(z_t) dO_t
 *   da   = sum_{b,t} r_t (q_t * k_t)
 *   dS_0 = lambda G_1
 *
 * A forward sweep rebuilds S_t for dq; a reverse sweep carries G_t.          */
static void *bwd_worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const long B = j->B, T = j->T, H = j->H, dk = j->dk_, dv = j->dv_;
    double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
    double *G = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
    for (;;) {
        long p = take(j);
        if (p >= B * H) break;
        long b = p / H, h = p % H;
        double lam = exp(j->gamma[h]);
        const double *a = j->a + h * dk;
        double *da = j->da_part + p * dk;
        for (long i = 0; i < dk; ++i) da[i] = 0.0;

        /* forward sweep: S_t, then dq_t = S_t dO_t + r_t (a*k_t) */
        if (j->init) memcpy(S, j->init + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        for (long t = 0; t < T; ++t) {
            const double *q = QROW(j->q, b, t, h, dk);
            const double *k = QROW(j->k, b, t, h, dk);
            const double *v = QROW(j->v, b, t, h, dv);
            const double *dO = QROW(j->dO, b, t, h, dv);
            double *dq = QROW(j->dq, b, t, h, dk);
            for (long i = 0; i < dk; ++i)
                for (long n = 0; n < dv; ++n)
                    S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];
            double z = 0.0, dov = 0.0;
            for (long i = 0; i < dk; ++i) z += a[i] * q[i] * k[i];
            for (long n = 0; n < dv; ++n) dov += dO[n] * v[n];
            double s = sigmoid(z);
            double r = s * (1.0 - s) * dov;
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long n = 0; n < dv; ++n) acc += S[i * dv + n] * dO[n];
                dq[i] = acc + r * a[i] * k[i];
            }
        }

        /* reverse sweep: G_t, then dk_t, dv_t, da */
        if (j->dfin) memcpy(G, j->dfin + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(G, 0, sizeof(double) * (size_t)(dk * dv));
        for (long t = T - 1; t >= 0; --t) {
            const double *q = QROW(j->q, b, t, h, dk);
            const double *k = QROW(j->k, b, t, h, dk);
            const double *v = QROW(j->v, b, t, h, dv);
            const double *dO = QROW(j->dO, b, t, h, dv);
            double *dk_out = QROW(j->dk, b, t, h, dk);
            double *dv_out = QROW(j->dv, b, t, h, dv);
            /* G_T = q_T dO_T^T + dS_final;  G_t = q_t dO_t^T + lambda G_{t+1} */
            if (t < T - 1)
                for (long i = 0; i < dk * dv; ++i) G[i] *= lam;
            for (long i = 0; i < dk; ++i)
                for (long n = 0; n < dv; ++n)
                    G[i * dv + n] += q[i] * dO[n];
            double z = 0.0, dov = 0.0;
            for (long i = 0; i < dk; ++i) z += a[i] * q[i] * k[i];
            for (long n = 0; n < dv; ++n) dov += dO[n] * v[n];
            double s = sigmoid(z);
            double r = s * (1.0 - s) * dov;
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long n = 0; n < dv; ++n) acc += G[i * dv + n] * v[n];
                dk_out[i] = acc + r * a[i] * q[i];
                da[i] += r * q[i] * k[i];
            }
            for (long n = 0; n < dv; ++n) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += G[i * dv + n] * k[i];
                dv_out[n] = acc + s * dO[n];
            }
        }
        /* dS_0 = lambda G_1 */
        if (j->dinit)
            for (long i = 0; i < dk * dv; ++i) j->dinit[p * dk * dv + i] = lam * G[i];
    }
    free(S);
    free(G);
    return NULL;
}

int oracle_bwd(const double *q, const double *k, const double *v, const double *gamma,
               const double *a, const double *init_state, const double *dO,
               const double *d_final_state, double *dq, double *dk, double *dv, double *d_a,
               double *d_init_state, long B, long T, long H, long dk_, long dv_, int nthreads)
{
    if (B < 0 || T < 0 || H <= 0 || dk_ <= 0 || dv_ <= 0) return 1;
    job_t j;
    memset(&j, 0, sizeof(j));
    j.q = q; j.k = k; j.v = v; j.gamma = gamma; j.a = a; j.init = init_state;
    j.dO = dO; j.dfin = d_final_state;
    j.dq = dq; j.dk = dk; j.dv = dv; j.dinit = d_init_state;
    j.B = B; j.T = T; j.H = H; j.dk_ = dk_; j.dv_ = dv_;
    j.da_part = (double *)calloc((size_t)(B * H * dk_ + 1), sizeof(double));
    pthread_mutex_init(&j.lock, NULL);
    run_threads(bwd_worker, &j, nthreads, B * H);
    pthread_mutex_destroy(&j.lock);
    /* d_a[h] = sum over b of the per-(b,h) partial sums, in order of b. */
    for (long h = 0; h < H; ++h)
        for (long i = 0; i < dk_; ++i) {
            double s = 0.0;
            for (long b = 0; b < B; ++b) s += j.da_part[(b * H + h) * dk_ + i];
            d_a[h * dk_ + i] = s;
        }
    free(j.da_part);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One recurrent decode step for many sequences (section "Inference
 * optimization on Trainium2": the state is read and written in the serving
 * pool, one fixed state per sequence, O(1) per token).  It is one token of the
 * recurrence above, applied in place:
 *   S' = lambda_h S + k v^T,  o = S'^T q + sigmoid(q . (a * k)) v
 * Layouts: state [N, L, H, dk, dv], q/k [N, L, H, dk], v/o [N, L, H, dv],
 *          a [L, H, dk], gamma [H].                                          */
typedef struct {
    double *state, *o;
    const double *q, *k, *v, *gamma, *a;
    long N, L, H, dk, dv, next;
    pthread_mutex_t lock;
} dec_t;

static void *dec_worker(void *arg)
{
    dec_t *j = (dec_t *)arg;
    const long dk = j->dk, dv = j->dv;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        long s = j->next++;
        pthread_mutex_unlock(&j->lock);
        if (s >= j->N * j->L * j->H) break;
        long h = s % j->H, l = (s / j->H) % j->L;
        double lam = exp(j->gamma[h]);
        const double *a = j->a + (l * j->H + h) * dk;
        const double *q = j->q + s * dk, *k = j->k + s * dk, *v = j->v + s * dv;
        double *S = j->state + s * dk * dv, *o = j->o + s * dv;
        for (long i = 0; i < dk; ++i)
            for (long n = 0; n < dv; ++n) S[i * dv + n] = lam * S[i * dv + n] + k[i] * v[n];
        double z = 0.0;
        for (long i = 0; i < dk; ++i) z += a[i] * q[i] * k[i];
        double g = sigmoid(z);
        for (long n = 0; n < dv; ++n) {
            double acc = 0.0;
            for (long i = 0; i < dk; ++i) acc += S[i * dv + n] * q[i];
            o[n] = acc + g * v[n];
        }
    }
    return NULL;
}

int oracle_decode_step(double *state, const double *q, const double *k, const double *v,
                       const double *gamma, const double *a, double *o, long N, long L, long H,
                       long dk, long dv, int nthreads)
{
    if (N < 0 || L <= 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    dec_t j;
    memset(&j, 0, sizeof(j));
    j.state = state; j.o = o; j.q = q; j.k = k; j.v = v; j.gamma = gamma; j.a = a;
    j.N = N; j.L = L; j.H = H; j.dk = dk; j.dv = dv;
    pthread_mutex_init(&j.lock, NULL);
    long n = N * L * H;
    int nt = nthreads_or_default(nthreads);
    if (nt > n) nt = (int)(n > 0 ? n : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, dec_worker, &j);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    return 0;
}
