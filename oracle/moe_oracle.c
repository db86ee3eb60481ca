/*
 * moe_oracle.c -- FP64 CPU oracle for the routed Mixture-of-Experts SwiGLU FFN
 * forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library and includes nothing from it.
 *
 * What it computes, per token t (plain definition, no blocking, no fusion):
 *   1. selection: k rounds; each round takes the not-yet-chosen expert with the
 *      largest router logit, the smaller expert index winning a tie.  Slot j is
 *      the j-th pick.  ("expert routing" is named in the warp-decode article,
 *      "Cursor warp decode 공개 ... 1.84x 가속", section 배경 및 맥락; the
 *      top-k/tie/renormalise details are the layer's problem statement.)
 *   2. weights: softmax over the k chosen logits only, w_j = exp(l_j - l_0) / S.
 *   3. per chosen expert e = s_j:  g_i = W[e,i,:].x,  u_i = W[e,I+i,:].x,
 *      a_i = g_i * sigmoid(g_i) * u_i   (gate rows 0..I-1, up rows I..2I-1),
 *      y_j[h] = W_down[e,h,:].a
 *   4. combine: out[t,h] = sum_j w_j * y_j[h], slots in ascending order.
 * All arithmetic is IEEE double; BF16 inputs convert to double exactly; the
 * FP32 logits convert to double exactly.  The warp-decode article (section
 * 핵심 내용, and section 경쟁 구도 / 비교 on dropping intermediate
 * activation quantisation) fixes that routed contributions are summed per
 * output dimension with no intermediate quantisation; the oracle keeps every
 * intermediate in double.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread, never -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2
#define ORACLE_EMISSING 3 /* a selected expert has no weights in the map */

/* BF16 is the top half of an IEEE binary32: shifting the 16 bits up gives the
 * float exactly, and float -> double is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Step 1 and 2 for one token.  taken has E bytes of scratch. */
static void route_token(const float *logits, int64_t E, int64_t k,
                        int32_t *idx, double *w, unsigned char *taken)
{
    memset(taken, 0, (size_t)E);
    for (int64_t j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            /* strict '>' keeps the earlier (smaller) index on equal values;
             * -0.0 == +0.0 under this comparison */
            if (best < 0 || logits[e] > logits[best])
                best = e;
        }
        taken[best] = 1;
        idx[j] = (int32_t)best;
    }
    double m = (double)logits[idx[0]];
    double s = 0.0;
    for (int64_t j = 0; j < k; ++j) {
        w[j] = exp((double)logits[idx[j]] - m);
        s += w[j];
    }
    for (int64_t j = 0; j < k; ++j)
        w[j] = w[j] / s;
}

int oracle_route(const float *logits, int64_t T, int64_t E, int64_t k,
                 int32_t *idx_out, double *w_out)
{
    if (!logits || !idx_out || !w_out || T < 0 || E < 1 || k < 1 || k > E)
        return ORACLE_EINVAL;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!taken)
        return ORACLE_ENOMEM;
    for (int64_t t = 0; t < T; ++t)
        route_token(logits + t * E, E, k, idx_out + t * k, w_out + t * k, taken);
    free(taken);
    return ORACLE_OK;
}

/* Step 3 for one (token, expert): y[H] = W_down_e . (silu(W_gate_e x) * (W_up_e x)).
 * wgu_e points at the expert's [2I, H] block, wd_e at its [H, I] block.
 * a has I doubles of scratch. */
static void expert_ffn(const uint16_t *x, const uint16_t *wgu_e,
                       const uint16_t *wd_e, int64_t H, int64_t I,
                       double *a, double *y)
{
    for (int64_t i = 0; i < I; ++i) {
        const uint16_t *gate_row = wgu_e + i * H;
        const uint16_t *up_row = wgu_e + (I + i) * H;
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xh = bf16_to_double(x[h]);
            g += bf16_to_double(gate_row[h]) * xh;
            u += bf16_to_double(up_row[h]) * xh;
        }
        double silu_g = g / (1.0 + exp(-g));
        a[i] = silu_g * u;
    }
    for (int64_t h = 0; h < H; ++h) {
        const uint16_t *down_row = wd_e + h * I;
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i)
            acc += bf16_to_double(down_row[i]) * a[i];
        y[h] = acc;
    }
}

typedef struct {
    const uint16_t *x;
    const float *logits;
    const uint16_t *wgu;
    const uint16_t *wd;
    const int32_t *emap; /* expert id -> block index in wgu/wd, or NULL */
    int64_t T, H, I, E, k;
    double *out;
    int32_t *idx_out; /* may be NULL */
    double *w_out;    /* may be NULL */
    int64_t t_begin, t_end;
    int status;
} oracle_job;

static void *forward_tokens(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t H = job->H, I = job->I, E = job->E, k = job->k;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    int32_t *idx = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    double *w = (double *)malloc((size_t)k * sizeof(double));
    double *a = (double *)malloc((size_t)I * sizeof(double));
    double *y = (double *)malloc((size_t)H * sizeof(double));
    job->status = ORACLE_OK;
    if (!taken || !idx || !w || !a || !y) {
        job->status = ORACLE_ENOMEM;
        goto done;
    }
    for (int64_t t = job->t_begin; t < job->t_end; ++t) {
        route_token(job->logits + t * E, E, k, idx, w, taken);
        double *out = job->out + t * H;
        for (int64_t h = 0; h < H; ++h)
            out[h] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            int64_t blk = job->emap ? job->emap[idx[j]] : idx[j];
            if (blk < 0) {
                job->status = ORACLE_EMISSING;
                goto done;
            }
            expert_ffn(job->x + t * H, job->wgu + blk * (2 * I * H),
                       job->wd + blk * (H * I), H, I, a, y);
            for (int64_t h = 0; h < H; ++h)
                out[h] += w[j] * y[h];
        }
        if (job->idx_out)
            memcpy(job->idx_out + t * k, idx, (size_t)k * sizeof(int32_t));
        if (job->w_out)
            memcpy(job->w_out + t * k, w, (size_t)k * sizeof(double));
    }
done:
    free(taken);
    free(idx);
    free(w);
    free(a);
    free(y);
    return NULL;
}

/*
 * Full forward pass.  x [T,H] bf16 bits, logits [T,E] f32, wgu [Eb,2I,H] bf16
 * bits, wd [Eb,H,I] bf16 bits, out [T,H] double.  emap (nullable, length E)
 * maps an expert id to its block in wgu/wd, -1 meaning "not supplied"; with a
 * NULL map Eb == E and block e is expert e.  This lets a caller hand over only
 * the experts that some tokens select.  idx_out [T,k] and w_out [T,k] are
 * optional.  Tokens are split over nthreads host threads (one token is never
 * split), so the result does not depend on nthreads.
 */
int oracle_forward(const uint16_t *x, const float *logits, const uint16_t *wgu,
                   const uint16_t *wd, const int32_t *emap, int64_t T,
                   int64_t H, int64_t I, int64_t E, int64_t k, double *out,
                   int32_t *idx_out, double *w_out, int nthreads)
{
    if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || k > E)
        return ORACLE_EINVAL;
    if (T == 0)
        return ORACLE_OK;
    if (!x || !logits || !wgu || !wd || !out)
        return ORACLE_EINVAL;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > T)
        nthreads = (int)T;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    int64_t per = T / nthreads, rem = T % nthreads, t0 = 0;
    for (int n = 0; n < nthreads; ++n) {
        oracle_job *j = &jobs[n];
        j->x = x;
        j->logits = logits;
        j->wgu = wgu;
        j->wd = wd;
        j->emap = emap;
        j->T = T;
        j->H = H;
        j->I = I;
        j->E = E;
        j->k = k;
        j->out = out;
        j->idx_out = idx_out;
        j->w_out = w_out;
        j->t_begin = t0;
        t0 += per + (n < rem ? 1 : 0);
        j->t_end = t0;
    }
    int started = 0;
    for (int n = 1; n < nthreads; ++n) {
        if (pthread_create(&tids[n], NULL, forward_tokens, &jobs[n]) != 0)
            break;
        started = n;
    }
    forward_tokens(&jobs[0]);
    /* threads that failed to start: run their share here */
    for (int n = started + 1; n < nthreads; ++n)
        forward_tokens(&jobs[n]);
    for (int n = 1; n <= started; ++n)
        pthread_join(tids[n], NULL);
    int status = ORACLE_OK;
    for (int n = 0; n < nthreads; ++n)
        if (jobs[n].status != ORACLE_OK)
            status = jobs[n].status;
    free(jobs);
    free(tids);
    return status;
}

/* One expert on one token, exposed so the tests can pin step 3 on its own. */
int oracle_expert_ffn(const uint16_t *x, const uint16_t *wgu_e,
                      const uint16_t *wd_e, int64_t H, int64_t I, double *y)
{
    if (!x || !wgu_e || !wd_e || !y || H < 1 || I < 1)
        return ORACLE_EINVAL;
    double *a = (double *)malloc((size_t)I * sizeof(double));
    if (!a)
        return ORACLE_ENOMEM;
    expert_ffn(x, wgu_e, wd_e, H, I, a, y);
    free(a);
    return ORACLE_OK;
}
