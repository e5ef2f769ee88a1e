/*
 * Exact softmax attention in fp64: the oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * path.
 *
 * What it computes is the plain definition of attention that the FlashAttention
 * pages take as the target of their tiled algorithm:
 *
 *   s_j   = scale * <q_i, k_j>                       for j in J_i
 *   m     = max_{j in J_i} s_j                       (pass 1)
 *   l     = sum_{j in J_i} exp(s_j - m)              (pass 2)
 *   o_i   = sum_{j in J_i} exp(s_j - m) v_j / l      (pass 3)
 *   LSE_i = m + ln l
 *
 * Sources:
 *  - three-pass safe softmax: "6. FlashAttention 分块逻辑", section 1.1; the
 *    same formula in "9.4 FlashAttention 与 FlashMLA", section 9.4.2;
 *  - S includes the scale: "6. FlashAttention 分块逻辑", section 3.1 code
 *    (Sij = Qi Kj^T * scale) and "08. Triton Flash Attention", TODO 1;
 *  - LSE = m + log(l), natural log: "9.4 FlashAttention 与 FlashMLA",
 *    section 9.4.5 (the kernel stores lse = m_i + log(l_i));
 *  - causal visibility j <= i with absolute (top-left) indices:
 *    "6. FlashAttention 分块逻辑", sections 3.2 and 4.1 (q_pos >= k_pos);
 *  - keys at index >= Nk do not exist (no zero-filled phantom keys).
 *
 * Inputs are the bf16 bit patterns the GPU receives, widened exactly to
 * fp64; `scale` is the fp32 value the GPU receives, widened to fp64.
 * Layout: Q [B,H,Nq,d], K and V [B,H,Nk,d], all contiguous row-major.
 * Outputs: O [rows, d] and LSE [rows] in fp64.
 *
 * Rows are independent, so the row list is split over `nthreads` POSIX
 * threads; each row is computed by the same sequential loops.
 *
 * oracle_attention_rows_f64 is the same computation on inputs given directly
 * as fp64 arrays (used for inputs that are not bf16, e.g. dequantised FP8).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row: the three passes above, over the visible keys 0..nvis-1. */
static void attend_one_row(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                           int64_t nvis, int64_t d, double scale,
                           double *s, double *o, double *lse)
{
    for (int64_t j = 0; j < nvis; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += widen_bf16(q[c]) * widen_bf16(K[j * d + c]);
        s[j] = scale * acc;
    }

    double m = -INFINITY;                         /* pass 1: the maximum */
    for (int64_t j = 0; j < nvis; ++j)
        if (s[j] > m) m = s[j];

    double l = 0.0;                               /* pass 2: the sum */
    for (int64_t j = 0; j < nvis; ++j)
        l += exp(s[j] - m);

    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;   /* pass 3: weighted sum */
    for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * widen_bf16(V[j * d + c]);
    }
    *lse = m + log(l);
}

/* The same three passes on fp64 inputs. */
static void attend_one_row_f64(const double *q, const double *K, const double *V,
                               int64_t nvis, int64_t d, double scale,
                               double *s, double *o, double *lse)
{
    for (int64_t j = 0; j < nvis; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += q[c] * K[j * d + c];
        s[j] = scale * acc;
    }

    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j)
        if (s[j] > m) m = s[j];

    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        l += exp(s[j] - m);

    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * V[j * d + c];
    }
    *lse = m + log(l);
}

typedef struct {
    const uint16_t *Q, *K, *V;
    const double *Qd, *Kd, *Vd;   /* fp64 inputs instead of bf16 when non-NULL */
    int64_t H, Nq, Nk, d;
    double scale;
    int causal;
    const int64_t *rows;   /* flat row ids r = (b*H + h)*Nq + i, or NULL for 0..n-1 */
    int64_t first, last;   /* this worker's slice of the row list */
    double *O, *LSE;
    int failed;
} job_t;

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!s) { jb->failed = 1; return NULL; }
    for (int64_t n = jb->first; n < jb->last; ++n) {
        int64_t r = jb->rows ? jb->rows[n] : n;
        int64_t bh = r / jb->Nq, i = r % jb->Nq;
        /* visible keys J_i: j < Nk, and j <= i when causal */
        int64_t nvis = jb->Nk;
        if (jb->causal && i + 1 < nvis) nvis = i + 1;
        if (jb->Qd)
            attend_one_row_f64(jb->Qd + r * jb->d,
                               jb->Kd + bh * jb->Nk * jb->d,
                               jb->Vd + bh * jb->Nk * jb->d,
                               nvis, jb->d, jb->scale, s,
                               jb->O + n * jb->d, jb->LSE + n);
        else
            attend_one_row(jb->Q + r * jb->d,
                           jb->K + bh * jb->Nk * jb->d,
                           jb->V + bh * jb->Nk * jb->d,
                           nvis, jb->d, jb->scale, s,
                           jb->O + n * jb->d, jb->LSE + n);
    }
    free(s);
    return NULL;
}

/*
 * Attention for the listed rows (all rows when `rows` is NULL, nrows = B*H*Nq).
 * Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure.
 */
static int run_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                    const double *Qd, const double *Kd, const double *Vd,
                    int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                    double scale, int causal,
                    const int64_t *rows, int64_t nrows,
                    double *O, double *LSE, int nthreads)
{
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || nrows < 0) return -1;
    if (rows) {
        for (int64_t n = 0; n < nrows; ++n)
            if (rows[n] < 0 || rows[n] >= B * H * Nq) return -1;
    } else if (nrows != B * H * Nq) {
        return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }

    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        job_t *jb = &jobs[t];
        jb->Q = Q; jb->K = K; jb->V = V;
        jb->Qd = Qd; jb->Kd = Kd; jb->Vd = Vd;
        jb->H = H; jb->Nq = Nq; jb->Nk = Nk; jb->d = d;
        jb->scale = scale;
        jb->causal = causal != 0;
        jb->rows = rows;
        jb->first = nrows * t / nthreads;
        jb->last = nrows * (t + 1) / nthreads;
        jb->O = O; jb->LSE = LSE;
        if (t == 0) continue;   /* worker 0 runs on the calling thread */
        if (pthread_create(&tids[t], NULL, worker, jb) != 0) { rc = -2; break; }
        started = t;
    }
    if (rc == 0) worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = 0; t < nthreads && rc == 0; ++t)
        if (jobs[t].failed) rc = -2;
    free(jobs);
    free(tids);
    return rc;
}

int oracle_attention_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                          int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                          float scale, int causal,
                          const int64_t *rows, int64_t nrows,
                          double *O, double *LSE, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return -1;
    return run_rows(Q, K, V, NULL, NULL, NULL, B, H, Nq, Nk, d, (double)scale, causal, rows, nrows, O, LSE,
                    nthreads);
}

/* Inputs as fp64 arrays with the same layouts; `scale` is taken as given. */
int oracle_attention_rows_f64(const double *Q, const double *K, const double *V,
                              int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                              double scale, int causal,
                              const int64_t *rows, int64_t nrows,
                              double *O, double *LSE, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return -1;
    return run_rows(NULL, NULL, NULL, Q, K, V, B, H, Nq, Nk, d, scale, causal, rows, nrows, O, LSE, nthreads);
}
