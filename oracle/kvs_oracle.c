/*
 * kvs_oracle.c -- plain, slow fp64 CPU oracle for paged GQA decode and the
 * per-(sequence, block) attention mass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never
 * does.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definitions, no blocking, fusion or split):
 *
 *   Decode attention ("KV-Cache Offloading for LLM Inference -- Visual
 *   Reference", section 2, Diagram 2.2 and section 4, Diagram 4.1: a decode
 *   step reads every cached key and value of the sequence):
 *       s_t  = sigma * sum_i q_i k_{t,i},   sigma = 1/sqrt(d)
 *       LSE  = m + log sum_t exp(s_t - m),  m = max_t s_t
 *       p_t  = exp(s_t - LSE)
 *       o_i  = sum_t p_t v_{t,i}
 *   Query head h reads KV head floor(h / G), G = Hq / Hkv ("GQA per-head
 *   attention as scoring streams", section 1: Q0..Q7 map to KV head 0, ...).
 *
 *   Block mass (same GQA page, section 2: the per-(layer, KV head) streams
 *   are aggregated into one score per (sequence, 16-token block)):
 *       mu_{l,h}(b)  = sum_{t in block b} p_t
 *       m_{l,g}(b)   = (1/G) sum_{h in group g} mu_{l,h}(b)     (stream mass)
 *       M(b)         = (1/(L*Hkv)) sum_{l,g} m_{l,g}(b)
 *   The pages give no operator for "aggregated"; the mean is taken so that
 *   M sums to 1 over the blocks and "mass >= 1/num_blocks" reads as "at or
 *   above the uniform share".
 *
 * All arithmetic is IEEE double in the order written; build with
 * -ffp-contract=off so no multiply-add is fused.  bf16 inputs are widened
 * exactly (a bf16 is the top 16 bits of an IEEE single).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_bf16_to_f64(uint16_t h) { return bf16_to_f64(h); }

/*
 * One query head against n tokens of its KV head.
 *   q        : d bf16 values
 *   k, v     : token t at k + t*tok_stride (bf16, d contiguous values)
 *   out      : d doubles (may be NULL to skip the value product)
 *   lse      : 1 double
 *   bmass    : ceil(n / block_tokens) doubles, mu(b) (may be NULL)
 *   sbuf     : n doubles of scratch
 */
/* K and V elements: bf16 bit patterns, float32 values (e.g. dequantised
 * 2-bit groups beside unquantised tokens), or 8-bit codes read through a
 * 256-entry table of values (code value x scale), e.g. for FP8 pages. */
typedef struct {
    const uint16_t *p16;      /* bf16 elements, or NULL    */
    const uint8_t *p8;        /* 8-bit codes, or NULL      */
    const double *lut;        /* value of each code        */
    const float *p32;         /* float32 elements, or NULL */
} elems_t;

static double elem_at(const elems_t *e, int64_t idx)
{
    if (e->p16)
        return bf16_to_f64(e->p16[idx]);
    if (e->p32)
        return (double)e->p32[idx];
    return e->lut[e->p8[idx]];
}

static void attend_head(const uint16_t *q, const elems_t *k, const elems_t *v, int64_t off,
                        int64_t tok_stride, int64_t n, int d, int block_tokens,
                        double *sbuf, double *out, double *lse, double *bmass)
{
    const double sigma = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t kt = off + t * tok_stride;
        double dot = 0.0;
        for (int i = 0; i < d; ++i)
            dot += bf16_to_f64(q[i]) * elem_at(k, kt + i);
        sbuf[t] = sigma * dot;
        if (sbuf[t] > m)
            m = sbuf[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t)
        z += exp(sbuf[t] - m);
    const double L = m + log(z);
    *lse = L;
    for (int64_t t = 0; t < n; ++t)
        sbuf[t] = exp(sbuf[t] - L);          /* p_t */
    if (out) {
        for (int i = 0; i < d; ++i)
            out[i] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            const int64_t vt = off + t * tok_stride;
            for (int i = 0; i < d; ++i)
                out[i] += sbuf[t] * elem_at(v, vt + i);
        }
    }
    if (bmass) {
        const int64_t nb = (n + block_tokens - 1) / block_tokens;
        for (int64_t b = 0; b < nb; ++b) {
            double s = 0.0;
            int64_t t1 = (b + 1) * block_tokens < n ? (b + 1) * block_tokens : n;
            for (int64_t t = b * block_tokens; t < t1; ++t)
                s += sbuf[t];
            bmass[b] = s;
        }
    }
}

typedef struct {
    const uint16_t *q;
    elems_t k, v;
    int64_t n;
    int L, Hq, Hkv, d, block_tokens;
    const int32_t *heads;   /* flat (l*Hq + h) indices to compute */
    int nheads;
    int tid, nthreads;
    int want_out;
    double *out, *lse, *head_mass;
    int failed;
} job_t;

static void *run_job(void *arg)
{
    job_t *j = (job_t *)arg;
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)(j->n > 0 ? j->n : 1));
    if (!sbuf) {
        j->failed = 1;
        return NULL;
    }
    const int G = j->Hq / j->Hkv;
    const int64_t nb = (j->n + j->block_tokens - 1) / j->block_tokens;
    const int64_t tok_stride = (int64_t)j->L * j->Hkv * j->d;
    for (int idx = j->tid; idx < j->nheads; idx += j->nthreads) {
        const int lh = j->heads[idx];
        const int l = lh / j->Hq, h = lh % j->Hq, g = h / G;
        const uint16_t *qh = j->q + ((int64_t)l * j->Hq + h) * j->d;
        const int64_t off = ((int64_t)l * j->Hkv + g) * j->d;
        attend_head(qh, &j->k, &j->v, off, tok_stride, j->n, j->d,
                    j->block_tokens, sbuf,
                    j->want_out ? j->out + (int64_t)idx * j->d : NULL,
                    j->lse + idx, j->head_mass ? j->head_mass + (int64_t)idx * nb : NULL);
    }
    free(sbuf);
    return NULL;
}

/*
 * Decode attention of one sequence for a list of (layer, query head) pairs.
 *   q     : [L][Hq][d] bf16
 *   k, v  : [n][L][Hkv][d] bf16, logical token order
 *   heads : nheads flat indices l*Hq + h (NULL = all L*Hq in order)
 *   out   : [nheads][d] doubles or NULL;  lse : [nheads];
 *   head_mass : [nheads][nb] or NULL
 * Heads are spread over nthreads threads; every output slot is written by
 * exactly one thread, so the result does not depend on the thread count.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
static int decode_heads(const uint16_t *q, elems_t k, elems_t v,
                        int64_t n, int L, int Hq, int Hkv, int d, int block_tokens,
                        const int32_t *heads, int nheads, int nthreads,
                        double *out, double *lse, double *head_mass)
{
    if (n < 1 || L < 1 || Hkv < 1 || Hq % Hkv || d < 1 || block_tokens < 1 ||
        (heads && nheads < 1))
        return -1;
    int32_t *all = NULL;
    if (!heads) {
        nheads = L * Hq;
        all = (int32_t *)malloc(sizeof(int32_t) * (size_t)nheads);
        if (!all)
            return -1;
        for (int i = 0; i < nheads; ++i)
            all[i] = i;
        heads = all;
    }
    for (int i = 0; i < nheads; ++i)
        if (heads[i] < 0 || heads[i] >= L * Hq) {
            free(all);
            return -1;
        }
    if (nheads < 1 || nheads > (1 << 30)) {
        free(all);
        return -1;
    }
    if (nthreads > nheads)
        nthreads = nheads;
    if (nthreads < 1)
        nthreads = 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int rc = 0;
    if (!jobs || !th) {
        rc = -1;
        goto done;
    }
    for (int i = 0; i < nthreads; ++i) {
        job_t j = {q, k, v, n, L, Hq, Hkv, d, block_tokens, heads, nheads,
                   i, nthreads, out != NULL, out, lse, head_mass, 0};
        jobs[i] = j;
    }
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, run_job, &jobs[i]) != 0)
            jobs[i].failed = 2;
    run_job(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) {
        if (jobs[i].failed == 2)
            run_job(&jobs[i]);     /* thread could not start: run it here */
        else
            pthread_join(th[i], NULL);
    }
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].failed == 1)
            rc = -1;
done:
    free(jobs);
    free(th);
    free(all);
    return rc;
}

int orc_decode_heads(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t n, int L, int Hq, int Hkv, int d, int block_tokens,
                     const int32_t *heads, int nheads, int nthreads,
                     double *out, double *lse, double *head_mass)
{
    elems_t ek = {k, NULL, NULL, NULL}, ev = {v, NULL, NULL, NULL};
    return decode_heads(q, ek, ev, n, L, Hq, Hkv, d, block_tokens, heads, nheads, nthreads,
                        out, lse, head_mass);
}

/*
 * Same, with K and V held as 8-bit codes [n][L][Hkv][d] whose values are
 * lut_k[code] and lut_v[code] (256 entries each).
 */
int orc_decode_heads_u8(const uint16_t *q, const uint8_t *k, const uint8_t *v,
                        const double *lut_k, const double *lut_v,
                        int64_t n, int L, int Hq, int Hkv, int d, int block_tokens,
                        const int32_t *heads, int nheads, int nthreads,
                        double *out, double *lse, double *head_mass)
{
    if (!lut_k || !lut_v)
        return -1;
    elems_t ek = {NULL, k, lut_k, NULL}, ev = {NULL, v, lut_v, NULL};
    return decode_heads(q, ek, ev, n, L, Hq, Hkv, d, block_tokens, heads, nheads, nthreads,
                        out, lse, head_mass);
}

/*
 * Same, with K and V as float32 values [n][L][Hkv][d].
 */
int orc_decode_heads_f32(const uint16_t *q, const float *k, const float *v,
                         int64_t n, int L, int Hq, int Hkv, int d, int block_tokens,
                         const int32_t *heads, int nheads, int nthreads,
                         double *out, double *lse, double *head_mass)
{
    if (!k || !v)
        return -1;
    elems_t ek = {NULL, NULL, NULL, k}, ev = {NULL, NULL, NULL, v};
    return decode_heads(q, ek, ev, n, L, Hq, Hkv, d, block_tokens, heads, nheads, nthreads,
                        out, lse, head_mass);
}

/*
 * Aggregate per-head block masses of one sequence into M(b):
 *   head_mass : [L][Hq][nb] (all heads, in order)
 *   mass      : [nb] out
 * Stream mass is the mean over the G query heads of a KV head, M the mean
 * of the L*Hkv stream masses, summed in (l, g) order.
 */
void orc_aggregate_mass(const double *head_mass, int64_t nb, int L, int Hq, int Hkv,
                        double *mass)
{
    const int G = Hq / Hkv;
    for (int64_t b = 0; b < nb; ++b) {
        double total = 0.0;
        for (int l = 0; l < L; ++l)
            for (int g = 0; g < Hkv; ++g) {
                double s = 0.0;
                for (int j = 0; j < G; ++j)
                    s += head_mass[((int64_t)l * Hq + g * G + j) * nb + b];
                total += s / (double)G;
            }
        mass[b] = total / (double)(L * Hkv);
    }
}
