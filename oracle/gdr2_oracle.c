/*
 * Sequential fp64 CPU oracle for the Gated Delta Rule-2 recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  The product (the CUDA
 * library under gated_delta_rule_166_b300/) never links, calls or includes it,
 * and this file includes nothing from the product.
 *
 * What it computes (the plain definition, no chunking, no reordering):
 *
 *   "Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention" page,
 *   section "Gated Delta Rule-2 update equation":
 *
 *       S_t = (I - k_t (b_t (.) k_t)^T) D_t S_{t-1} + k_t (w_t (.) v_t)^T
 *
 *   with the symbol table that follows it on the same page: S_t the d_k x d_v
 *   memory matrix, k_t the (normalised) key, b_t the erase gate over the KEY
 *   channels, w_t the write gate over the VALUE channels, D_t a diagonal
 *   channel-wise decay.  D_t = diag(exp(log_decay_t)) (d_k x d_k, because it
 *   left-multiplies S).  Readout: o_t = S_t^T q_t, taken after the update (the
 *   standard linear-attention convention; the page prints no readout).
 *
 * Per (batch, head), for t = 0 .. T-1:
 *     P   = D_t S                       (decay each key row i by exp(g_t[i]))
 *     x   = (b_t (.) k_t)^T P           (1 x d_v erase read)
 *     S   = P - k_t x + k_t (w_t (.) v_t)^T
 *     o_t = S^T q_t
 *
 * Layouts (row-major, contiguous):
 *   q, k, b, g : [B, T, H, dk]      v, w, o : [B, T, H, dv]
 *   S0, ST     : [B, H, dk, dv]     (S0 == NULL means a zero initial state)
 *
 * Gate values are used exactly as given (no sigmoid, no clamp: the page's
 * ablation widens the erase range to [0, 2]); keys are not normalised here.
 *
 * The (batch, head) pairs are independent; they are spread over nthreads
 * POSIX threads.  Each pair is computed by the same sequential loop, so the
 * result does not depend on nthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *b, *w, *g, *S0;
    double *o, *ST;
    long B, T, H, dk, dv;
    long next_pair;          /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
} job_t;

/* One (batch, head) pair: the literal recurrence above. */
static void run_pair(const job_t* J, long bh, double* S, double* x) {
    const long H = J->H, T = J->T, dk = J->dk, dv = J->dv;
    const long bi = bh / H, h = bh % H;

    if (J->S0)
        memcpy(S, J->S0 + bh * dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (long t = 0; t < T; ++t) {
        const long tok = (bi * T + t) * H + h;
        const double* qt = J->q + tok * dk;
        const double* kt = J->k + tok * dk;
        const double* bt = J->b + tok * dk;
        const double* gt = J->g + tok * dk;
        const double* vt = J->v + tok * dv;
        const double* wt = J->w + tok * dv;
        double* ot = J->o + tok * dv;

        /* P = D_t S : row i of S scaled by exp(g_t[i]). */
        for (long i = 0; i < dk; ++i) {
            const double a = exp(gt[i]);
            double* row = S + i * dv;
            for (long j = 0; j < dv; ++j) row[j] *= a;
        }
        /* x = (b_t (.) k_t)^T P */
        for (long j = 0; j < dv; ++j) x[j] = 0.0;
        for (long i = 0; i < dk; ++i) {
            const double c = bt[i] * kt[i];
            const double* row = S + i * dv;
            for (long j = 0; j < dv; ++j) x[j] += c * row[j];
        }
        /* S = P - k_t x + k_t (w_t (.) v_t)^T */
        for (long i = 0; i < dk; ++i) {
            double* row = S + i * dv;
            for (long j = 0; j < dv; ++j)
                row[j] = row[j] - kt[i] * x[j] + kt[i] * (wt[j] * vt[j]);
        }
        /* o_t = S_t^T q_t */
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
        for (long i = 0; i < dk; ++i) {
            const double* row = S + i * dv;
            for (long j = 0; j < dv; ++j) ot[j] += qt[i] * row[j];
        }
    }
    if (J->ST) memcpy(J->ST + bh * dk * dv, S, sizeof(double) * dk * dv);
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    double* S = (double*)malloc(sizeof(double) * J->dk * J->dv);
    double* x = (double*)malloc(sizeof(double) * J->dv);
    if (!S || !x) { free(S); free(x); return (void*)1; }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const long bh = J->next_pair++;
        pthread_mutex_unlock(&J->lock);
        if (bh >= J->B * J->H) break;
        run_pair(J, bh, S, x);
    }
    free(S);
    free(x);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure.
 * o must hold B*T*H*dv doubles; ST (optional) B*H*dk*dv doubles. */
int gdr2_oracle_forward(const double* q, const double* k, const double* v,
                        const double* b, const double* w, const double* g,
                        const double* S0, double* o, double* ST,
                        long B, long T, long H, long dk, long dv, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    if (T > 0 && (!q || !k || !v || !b || !w || !g || !o)) return -1;
    job_t J;
    J.q = q; J.k = k; J.v = v; J.b = b; J.w = w; J.g = g; J.S0 = S0;
    J.o = o; J.ST = ST;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.next_pair = 0;
    pthread_mutex_init(&J.lock, NULL);
    long pairs = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = (int)(pairs > 0 ? pairs : 1);
    int rc = 0;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    if (!th) rc = -2;
    for (int i = 1; rc == 0 && i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) { rc = -2; break; }
        ++started;
    }
    if (rc == 0 && worker(&J) != NULL) rc = -2;   /* the calling thread works too */
    for (int i = 1; i <= started; ++i) {
        void* ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
