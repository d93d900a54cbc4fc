/*
 * kda_oracle.c -- FP64 CPU oracle of the KDA forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it computes (plain definitions, written out token by token):
 *
 *   gate   g[t,h,c] = -exp(A_log[h]) * softplus(f[t,h,c] + dt_bias[h,c])
 *          beta[t,h] = sigmoid(b[t,h])
 *     The gate is computed outside the chunk kernel, with FP32 A_log/dt_bias
 *     ("GLM-5.3-Flash F6.2: KDA correctness and FLA sequence parallelism",
 *     fused-gate commit: gate computed externally before the kernel, matching
 *     the HF reference forward; beta passes through a sigmoid).
 *
 *   forward, for each packed sequence n (rows cu[n] .. cu[n+1]-1) and head h,
 *   from S = initial_state[n,h] (a K x V matrix; zero when none is given):
 *          q^ = q / sqrt(sum q^2 + eps),  k^ likewise   (L2 normalisation
 *               inside the op: "Add opt-in FP32 KDA chunk computation",
 *               section Change)
 *          S  <- Diag(exp(g_t)) S                      (per-channel decay)
 *          S  <- S + beta_t k^_t (v_t - S^T k^_t)^T     (delta-rule write; this
 *               is (I - beta k k^T) D S + beta k v^T expanded)
 *          o_t = scale * S^T q^_t
 *   final_state[n,h] = S after the last token of the sequence.
 *     The per-token FP64 recurrence is the reference the pages validate the
 *     chunked kernel against ("Add opt-in FP32 KDA chunk computation",
 *     sections Problem and Validation).
 *
 * Everything is double precision; inputs are passed as doubles (activations
 * that the GPU sees in BF16/FP32 are upcast exactly by the caller).
 *
 * The `mutation` argument plants one deliberate mistake (0 = none).  It exists
 * so that the tests can show that the oracle's pins catch plausible errors; no
 * caller outside the tests sets it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum {
    MUT_NONE = 0,
    MUT_NO_ERASE = 1,        /* drop the -beta k k^T S erase term           */
    MUT_DECAY_AFTER = 2,     /* apply Diag(exp g) after the delta write      */
    MUT_READ_BEFORE = 3,     /* read o_t from S_{t-1} instead of S_t          */
    MUT_TRANSPOSED_READ = 4, /* o_t = scale * S q instead of S^T q            */
    MUT_NO_L2NORM = 5,       /* skip the q/k normalisation                    */
    MUT_BETA_ON_V_ONLY = 6,  /* S += k (beta v - S^T k)^T                     */
    MUT_GATE_NO_ALOG = 7,    /* gate without the -exp(A_log) factor (= -softplus) */
    MUT_GATE_BIAS_HEAD0 = 8, /* gate uses dt_bias of head 0 for every head    */
    MUT_SKIP_SCALE = 9,      /* drop the output scale                         */
    MUT_IGNORE_INIT = 10     /* start every sequence from zero despite an initial state */
};

static double softplus(double x) { return x > 30.0 ? x : log1p(exp(x)); }

/* g and beta from the raw draws.  f: [T,H,K], A_log: [H], dt_bias: [H,K],
 * b: [T,H]  ->  g: [T,H,K], beta: [T,H]. */
void kda_oracle_gate(const double* f, const double* A_log, const double* dt_bias,
                     const double* b, int64_t T, int32_t H, int32_t K,
                     double* g, double* beta, int32_t mutation)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            const double lam = (mutation == MUT_GATE_NO_ALOG) ? 1.0 : exp(A_log[h]);
            const int32_t hb = (mutation == MUT_GATE_BIAS_HEAD0) ? 0 : h;
            for (int32_t c = 0; c < K; ++c) {
                const int64_t i = (t * H + h) * (int64_t)K + c;
                g[i] = -lam * softplus(f[i] + dt_bias[(int64_t)hb * K + c]);
            }
            beta[t * H + h] = 1.0 / (1.0 + exp(-b[t * H + h]));
        }
    }
}

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int32_t* cu;
    const double* init;
    int32_t N, H, K, V;
    double scale, eps;
    int32_t l2norm, mutation;
    double *o, *final_state;
    int64_t n_units;
    int64_t next_unit;           /* shared work counter */
    pthread_mutex_t lock;
} job_t;

static void normalise(const double* x, int32_t n, double eps, int32_t on, double* out)
{
    double ss = 0.0;
    for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
    const double inv = on ? 1.0 / sqrt(ss + eps) : 1.0;
    for (int32_t i = 0; i < n; ++i) out[i] = x[i] * inv;
}

/* One (sequence, head) unit: the token loop. */
static void run_unit(job_t* J, int64_t unit, double* S, double* r, double* qn, double* kn,
                     double* Sprev)
{
    const int32_t n = (int32_t)(unit / J->H), h = (int32_t)(unit % J->H);
    const int32_t K = J->K, V = J->V, H = J->H;
    const int mut = J->mutation;
    if (J->init && mut != MUT_IGNORE_INIT)
        memcpy(S, J->init + unit * (int64_t)K * V, sizeof(double) * (size_t)K * V);
    else
        memset(S, 0, sizeof(double) * (size_t)K * V);
    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double* qt = J->q + (t * H + h) * (int64_t)K;
        const double* kt = J->k + (t * H + h) * (int64_t)K;
        const double* vt = J->v + (t * H + h) * (int64_t)V;
        const double* gt = J->g + (t * H + h) * (int64_t)K;
        const double bt = J->beta[t * H + h];
        const int32_t on = J->l2norm && mut != MUT_NO_L2NORM;
        normalise(qt, K, J->eps, on, qn);
        normalise(kt, K, J->eps, on, kn);
        if (mut == MUT_READ_BEFORE) memcpy(Sprev, S, sizeof(double) * (size_t)K * V);

        if (mut != MUT_DECAY_AFTER) {
            for (int32_t c = 0; c < K; ++c) {
                const double a = exp(gt[c]);
                for (int32_t m = 0; m < V; ++m) S[c * V + m] *= a;
            }
        }
        /* r = S^T k^ */
        for (int32_t m = 0; m < V; ++m) r[m] = 0.0;
        for (int32_t c = 0; c < K; ++c)
            for (int32_t m = 0; m < V; ++m) r[m] += S[c * V + m] * kn[c];
        if (mut == MUT_NO_ERASE)
            for (int32_t m = 0; m < V; ++m) r[m] = 0.0;
        /* S += beta k^ (v - r)^T */
        for (int32_t c = 0; c < K; ++c) {
            for (int32_t m = 0; m < V; ++m) {
                const double w = (mut == MUT_BETA_ON_V_ONLY) ? (bt * vt[m] - r[m])
                                                             : bt * (vt[m] - r[m]);
                S[c * V + m] += kn[c] * w;
            }
        }
        if (mut == MUT_DECAY_AFTER) {
            for (int32_t c = 0; c < K; ++c) {
                const double a = exp(gt[c]);
                for (int32_t m = 0; m < V; ++m) S[c * V + m] *= a;
            }
        }
        /* o = scale * S^T q^ */
        const double* Sr = (mut == MUT_READ_BEFORE) ? Sprev : S;
        const double sc = (mut == MUT_SKIP_SCALE) ? 1.0 : J->scale;
        double* ot = J->o + (t * H + h) * (int64_t)V;
        if (mut == MUT_TRANSPOSED_READ && K == V) {
            for (int32_t m = 0; m < V; ++m) {
                double acc = 0.0;
                for (int32_t c = 0; c < K; ++c) acc += Sr[m * V + c] * qn[c];
                ot[m] = sc * acc;
            }
        } else {
            for (int32_t m = 0; m < V; ++m) {
                double acc = 0.0;
                for (int32_t c = 0; c < K; ++c) acc += Sr[c * V + m] * qn[c];
                ot[m] = sc * acc;
            }
        }
    }
    if (J->final_state)
        memcpy(J->final_state + unit * (int64_t)K * V, S, sizeof(double) * (size_t)K * V);
}

static void* worker(void* arg)
{
    job_t* J = (job_t*)arg;
    const size_t KV = (size_t)J->K * J->V;
    double* S = (double*)malloc(sizeof(double) * KV);
    double* Sp = (double*)malloc(sizeof(double) * KV);
    double* r = (double*)malloc(sizeof(double) * (size_t)J->V);
    double* qn = (double*)malloc(sizeof(double) * (size_t)J->K);
    double* kn = (double*)malloc(sizeof(double) * (size_t)J->K);
    if (S && Sp && r && qn && kn) {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int64_t u = J->next_unit++;
            pthread_mutex_unlock(&J->lock);
            if (u >= J->n_units) break;
            run_unit(J, u, S, r, qn, kn, Sp);
        }
    }
    free(S); free(Sp); free(r); free(qn); free(kn);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments.  o: [T,H,V]; initial_state and
 * final_state: [N,H,K,V] or NULL.  nthreads <= 0 uses every online core. */
int kda_oracle_forward(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const int32_t* cu_seqlens, int32_t N, int64_t T,
                       int32_t H, int32_t K, int32_t V, double scale, int32_t l2norm,
                       double eps, const double* initial_state, double* o,
                       double* final_state, int32_t nthreads, int32_t mutation)
{
    if (N < 0 || H <= 0 || K <= 0 || V <= 0 || T < 0) return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return -1;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    job_t J;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.cu = cu_seqlens; J.init = initial_state;
    J.N = N; J.H = H; J.K = K; J.V = V; J.scale = scale; J.eps = eps;
    J.l2norm = l2norm; J.mutation = mutation; J.o = o; J.final_state = final_state;
    J.n_units = (int64_t)N * H; J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    long nt = nthreads > 0 ? nthreads : sysconf(_SC_NPROCESSORS_ONLN);
    if (nt < 1) nt = 1;
    if (nt > J.n_units) nt = J.n_units > 0 ? J.n_units : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    long started = 0;
    for (long i = 0; i < nt; ++i)
        if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
    if (started == 0) worker(&J);
    for (long i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* Number of worker threads kda_oracle_forward uses for nthreads <= 0. */
int32_t kda_oracle_default_threads(void) { return (int32_t)sysconf(_SC_NPROCESSORS_ONLN); }
