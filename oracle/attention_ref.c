/*
 * Oracle for prefix-cached attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct causal attention on the CPU, accumulated in fp64.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code with the CUDA path: keys and values come in LOGICAL token order
 * (never through KV-pool slots), so it computes what a full recompute of the whole
 * prompt would compute.
 *
 * What it follows:
 *  - "Prompt Caching" (Ultralytics glossary), section "How prompt caching works":
 *    during prefill every layer computes a key and a value vector per prompt token;
 *    attention is causal, so a token's keys and values depend only on the tokens before
 *    it, and a cached copy of a shared prefix can replace recomputation.  A cache hit
 *    must give the next-token scores of the full computation up to floating-point
 *    rounding (same page, "Prompt caching and related terms", prompt engineering entry).
 *  - Scaled dot-product attention with a causal mask that includes the query token
 *    itself (the page's GPT-2 example computes the last position's scores over the
 *    whole prompt including that position).
 *
 * For one request, query row r sits at absolute position pos[r] and attends keys
 * 0..pos[r] (inclusive).  Query head h reads kv head h / (hq / hkv) (contiguous groups).
 *   s_j = scale * sum_d q[d] * k_j[d]
 *   m   = max_j s_j
 *   o   = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m)
 *   lse = m + log(sum_j exp(s_j - m))
 * Inputs are float32 (bf16 inputs are passed exactly widened); every product and sum is
 * in double precision; the output is rounded to float32, lse is returned in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
int oracle_attention_rows(int64_t n_rows, int32_t hq, int32_t hkv, int32_t d, int64_t ctx_len,
                          const float* q,        /* [n_rows, hq, d] */
                          const int64_t* pos,    /* [n_rows], 0 <= pos < ctx_len */
                          const float* k,        /* [ctx_len, hkv, d] logical order */
                          const float* v,        /* [ctx_len, hkv, d] logical order */
                          double scale,
                          float* out,            /* [n_rows, hq, d] */
                          double* lse,           /* [n_rows, hq] or NULL */
                          int32_t num_threads)   /* <= 0: the OpenMP default */
{
    if (n_rows < 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (pos[r] < 0 || pos[r] >= ctx_len) return -1;
    const int32_t group = hq / hkv;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
    const int64_t work = n_rows * (int64_t)hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; ++w) {
        const int64_t r = w / hq;
        const int32_t h = (int32_t)(w % hq);
        const int32_t g = h / group;
        const int64_t n_keys = pos[r] + 1;
        const float* qr = q + (r * hq + h) * (int64_t)d;
        double* s = (double*)malloc(sizeof(double) * (size_t)n_keys);
        double* acc = (double*)calloc((size_t)d, sizeof(double));
        if (!s || !acc) {
            free(s);
            free(acc);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            const float* kj = k + (j * hkv + g) * (int64_t)d;
            double dot = 0.0;
            for (int32_t x = 0; x < d; ++x) dot += (double)qr[x] * (double)kj[x];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            s[j] = exp(s[j] - m);
            den += s[j];
        }
        for (int64_t j = 0; j < n_keys; ++j) {
            const float* vj = v + (j * hkv + g) * (int64_t)d;
            for (int32_t x = 0; x < d; ++x) acc[x] += s[j] * (double)vj[x];
        }
        float* o = out + (r * hq + h) * (int64_t)d;
        for (int32_t x = 0; x < d; ++x) o[x] = (float)(acc[x] / den);
        if (lse) lse[r * hq + h] = m + log(den);
        free(s);
        free(acc);
    }
    return failed ? -2 : 0;
}

/* Number of threads an OpenMP parallel region would use (reported with CPU timings). */
int32_t oracle_max_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}
