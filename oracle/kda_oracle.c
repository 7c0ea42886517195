/*
 * KDA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the Kimi Delta Attention (KDA)
 * recurrence, one token at a time.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path (the
 * CUDA library) shares no code, header, table or helper with it.
 *
 * Sources (web pages, cited by title and section/equation):
 *   [W] "Kimi K3：从三条信息流到完整系统" (wineandchord.com)
 *       - §KDA 是带逐通道遗忘的 delta rule, eq. (1) and its expanded form:
 *           S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *               = Diag(alpha_t) S_{t-1} + beta_t k_t (v_t^T - k_t^T Diag(alpha_t) S_{t-1})
 *           o_t = S_t^T q_t
 *         The steps below are read off this expanded form: D = Diag(alpha_t)
 *         S_{t-1} scales the key-channel rows and appears in both terms, the
 *         residual is e = v_t - D^T k_t, the write is S_t = D + beta_t k_t e^T,
 *         and o_t reads S_t, the state after this token's write.  (The
 *         worked numbers printed under the equation are a test fixture,
 *         tests/golden/kda_step_worked_example.json, not a template.)
 *       - §下界 log-decay 是一个 kernel 设计, eq. (5):
 *           g_t = g_min * Sigmoid(e^A z_t),  alpha_t = e^{g_t},  g_min = -5.
 *         and, in the same section, the gate it replaced: Kimi Linear's
 *         unbounded negative-softplus log-decay.
 *   [K] "Kimi K3: Two point eight trillion parameters, open weights, and
 *       forty-seven pages of how", §What changed between the paper and the
 *       model (the negative softplus) and the four update rules before it:
 *       the delta rule (no decay), gated delta (one scalar decay per step),
 *       KDA (one decay per key channel).
 *
 * Gate variants (gate_mode), the readings taken where the pages give no
 * formula:
 *   0  bounded:       g = g_min * Sigmoid(e^A z)                 (eq. (5))
 *   1  log-decay:     the gate input is g itself
 *   2  neg-softplus:  g = -Softplus(e^A z) = -log(1 + e^{e^A z}), unbounded
 *                     (the per-head scale enters as in eq. (5))
 *   3  none:          g = 0, alpha = 1: the plain delta rule (gate unused)
 * gate_scalar = 1: one gate value per (token, head), shared by every key
 * channel (gated delta); the gate array is then [total_T, H].
 *
 * Layout: token-major packed sequences, [total_T, H, d] row-major, with
 * cu_seqlens[N+1] (host) splitting the token axis into N independent
 * sequences.  State S is [N, H, dk, dv] row-major: row = key channel c,
 * column = value channel j.  Everything is computed in fp64.
 *
 * Readings where the pages are silent (the same readings the CUDA library
 * takes): the query scale multiplies o_t (1.0 = the pages' plain S_t^T q_t);
 * A_log is one scalar per head; q, k arrive already normalised and beta
 * already in (0,1), so the operator applies neither L2Norm nor Sigmoid to
 * them; packed sequences are independent, each starting from its own
 * initial state.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* eq. (5): the bounded log-decay for one channel. */
double kda_oracle_gate(double z, double A_log, double g_min)
{
    double x = exp(A_log) * z;
    double sig = 1.0 / (1.0 + exp(-x));
    return g_min * sig;
}

/* log(1 + e^x) without overflow: max(x, 0) + log(1 + e^{-|x|}). */
static double softplus(double x)
{
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* The log-decay g of one gate input under each gate mode. */
double kda_oracle_log_decay(int gate_mode, double z, double A_log, double g_min)
{
    switch (gate_mode) {
    case 0: return kda_oracle_gate(z, A_log, g_min);
    case 1: return z;
    case 2: return -softplus(exp(A_log) * z);
    default: return 0.0;
    }
}

/*
 * One (sequence, head) chain, tokens t = 0..len-1.
 *   q, k       : element (t, c) at [t * tok_stride + c]
 *   gate       : element (t, c) at [t * gate_stride + c * gate_cstride]
 *                (gate_cstride = 0: one value per token, all channels)
 *   v          : element (t, j) at [t * tok_stride_v + j]
 *   beta       : element t at [t * beta_stride]
 *   out        : element (t, j) at [t * tok_stride_v + j]
 *   S          : dk x dv row-major, updated in place (entering -> final state)
 * gate_mode: see the header (0 = eq. (5)).
 */
static void chain(int len, int dk, int dv,
                  const double *q, const double *k, const double *v,
                  const double *gate, const double *beta,
                  ptrdiff_t tok_stride, ptrdiff_t tok_stride_v, ptrdiff_t beta_stride,
                  ptrdiff_t gate_stride, ptrdiff_t gate_cstride,
                  double A_log, double g_min, double scale, int gate_mode,
                  double *S, double *out, double *alpha, double *e)
{
    for (int t = 0; t < len; ++t) {
        const double *qt = q + (ptrdiff_t)t * tok_stride;
        const double *kt = k + (ptrdiff_t)t * tok_stride;
        const double *vt = v + (ptrdiff_t)t * tok_stride_v;
        const double *zt = gate ? gate + (ptrdiff_t)t * gate_stride : NULL;
        const double bt = beta[(ptrdiff_t)t * beta_stride];

        /* eq. (5): per-channel retention alpha_c = exp(g_c) */
        for (int c = 0; c < dk; ++c) {
            double g = zt ? kda_oracle_log_decay(gate_mode, zt[(ptrdiff_t)c * gate_cstride], A_log, g_min)
                          : 0.0;
            alpha[c] = exp(g);
        }
        /* D = Diag(alpha) S_{t-1}: row c (key channel c) scaled by alpha_c */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j)
                S[(ptrdiff_t)c * dv + j] *= alpha[c];
        /* residual of the expanded eq. (1): e = v_t - D^T k_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c)
                acc += S[(ptrdiff_t)c * dv + j] * kt[c];
            e[j] = vt[j] - acc;
        }
        /* S_t = D + beta_t k_t e^T */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j)
                S[(ptrdiff_t)c * dv + j] += bt * kt[c] * e[j];
        /* o_t = scale * S_t^T q_t (the state after this token's write) */
        double *ot = out + (ptrdiff_t)t * tok_stride_v;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c)
                acc += S[(ptrdiff_t)c * dv + j] * qt[c];
            ot[j] = scale * acc;
        }
    }
}

typedef struct {
    int H, dk, dv, N;
    const double *q, *k, *v, *gate, *beta, *init_state, *A_log;
    const int32_t *cu;
    double g_min, scale;
    int gate_mode, gate_scalar;
    double *out, *final_state;
    const int *order;       /* chain indices, longest sequence first */
    int n_chains;
    int next;               /* shared work counter */
} job_t;

static void run_one(job_t *J, int ch, double *alpha, double *e)
{
    const int n = ch / J->H, h = ch % J->H;
    const int bos = J->cu[n], len = J->cu[n + 1] - J->cu[n];
    const ptrdiff_t sdk = (ptrdiff_t)J->dk, sdv = (ptrdiff_t)J->dv;
    double *S = J->final_state + ((ptrdiff_t)n * J->H + h) * sdk * sdv;
    if (J->init_state)
        memcpy(S, J->init_state + ((ptrdiff_t)n * J->H + h) * sdk * sdv,
               sizeof(double) * (size_t)(sdk * sdv));
    else
        memset(S, 0, sizeof(double) * (size_t)(sdk * sdv));
    const ptrdiff_t tok = (ptrdiff_t)J->H * sdk, tokv = (ptrdiff_t)J->H * sdv;
    const ptrdiff_t base = (ptrdiff_t)bos * tok + (ptrdiff_t)h * sdk;
    const ptrdiff_t basev = (ptrdiff_t)bos * tokv + (ptrdiff_t)h * sdv;
    const double *gate = NULL;
    ptrdiff_t gstride = tok, gcstride = 1;
    if (J->gate_mode != 3) {
        if (J->gate_scalar) {
            gate = J->gate + (ptrdiff_t)bos * J->H + h;
            gstride = J->H;
            gcstride = 0;
        } else {
            gate = J->gate + base;
        }
    }
    chain(len, J->dk, J->dv, J->q + base, J->k + base, J->v + basev, gate,
          J->beta + (ptrdiff_t)bos * J->H + h, tok, tokv, J->H, gstride, gcstride,
          J->A_log ? J->A_log[h] : 0.0, J->g_min, J->scale, J->gate_mode,
          S, J->out + basev, alpha, e);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *alpha = (double *)malloc(sizeof(double) * (size_t)J->dk);
    double *e = (double *)malloc(sizeof(double) * (size_t)J->dv);
    for (;;) {
        int i = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (i >= J->n_chains) break;
        run_one(J, J->order[i], alpha, e);
    }
    free(alpha);
    free(e);
    return NULL;
}

typedef struct { int len, idx; } chain_key_t;
static int cmp_longest_first(const void *a, const void *b)
{
    const chain_key_t *x = (const chain_key_t *)a, *y = (const chain_key_t *)b;
    if (x->len != y->len) return y->len - x->len;
    return x->idx - y->idx;
}

/*
 * Forward over packed sequences.  Returns 0 on success, nonzero on a bad
 * argument.  out [total_T, H, dv] and final_state [N, H, dk, dv] are written.
 * nthreads <= 0 means 1.
 */
int kda_oracle_fwd(int total_T, int H, int dk, int dv,
                   const double *q, const double *k, const double *v,
                   const double *gate, const double *beta,
                   const int32_t *cu_seqlens, int N,
                   const double *init_state, const double *A_log,
                   double g_min, double scale, int gate_mode, int gate_scalar,
                   double *out, double *final_state, int nthreads)
{
    if (total_T < 0 || H <= 0 || dk <= 0 || dv <= 0 || N <= 0 || !cu_seqlens ||
        !final_state || gate_mode < 0 || gate_mode > 3 ||
        (total_T > 0 && (!q || !k || !v || (!gate && gate_mode != 3) || !beta || !out)))
        return 1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != total_T) return 2;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;

    job_t J;
    J.H = H; J.dk = dk; J.dv = dv; J.N = N;
    J.q = q; J.k = k; J.v = v; J.gate = gate; J.beta = beta;
    J.init_state = init_state; J.A_log = A_log; J.cu = cu_seqlens;
    J.g_min = g_min; J.scale = scale; J.gate_mode = gate_mode; J.gate_scalar = gate_scalar;
    J.out = out; J.final_state = final_state;
    J.n_chains = N * H;
    J.next = 0;
    chain_key_t *keys = (chain_key_t *)malloc(sizeof(chain_key_t) * (size_t)J.n_chains);
    int *order = (int *)malloc(sizeof(int) * (size_t)J.n_chains);
    for (int i = 0; i < J.n_chains; ++i) {
        keys[i].idx = i;
        keys[i].len = cu_seqlens[i / H + 1] - cu_seqlens[i / H];
    }
    qsort(keys, (size_t)J.n_chains, sizeof(chain_key_t), cmp_longest_first);
    for (int i = 0; i < J.n_chains; ++i) order[i] = keys[i].idx;
    free(keys);
    J.order = order;

    if (nthreads <= 1) {
        worker(&J);
    } else {
        if (nthreads > J.n_chains) nthreads = J.n_chains;
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
            ++started;
        }
        if (started == 0) worker(&J);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    free(order);
    return 0;
}
