/*
 * kvc_oracle.c -- plain, slow, fp64 CPU oracle for single-query decode
 * attention over a static KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (the pages' definitions, restated):
 *
 *   "10.3 -- KV cache implementation details", section 5 (the decode loop,
 *   step-by-step), attention bullet: the query is one row q_t per head, the
 *   keys and values are the whole cache, and the output is
 *       attn = softmax(q K^T / sqrt(d_head)) V .
 *
 *   "KV Cache Optimization: GQA Audit, In-Place Buffers, Persistent
 *   Prompts", section #2 (After): reads are sliced to the live length, so
 *   cache rows at or past it are never attended.  Here the live length of
 *   sequence b is valid_len[b].
 *
 *   Same page, section #1, and "10.3", section 4.2 (GQA): H_kv KV heads,
 *   each shared by g = H / H_kv query heads.  The pages do not say which
 *   query heads share a KV head; the reading taken is the contiguous one,
 *   query head h uses KV head h / g (the grouping a repeat-interleave of
 *   the KV heads produces).
 *
 * Evaluation: every stored element is widened exactly to double (bf16,
 * fp16 and fp32 are all exact in double; fp64 inputs -- the dequantised rows
 * of an int8 cache, code * scale, exact in double -- are taken as they are).  For each (b, h):
 *     s_j = (sum_d q[b,h,d] * K[b,k,j,d]) / sqrt(d_h)      for j < valid_b
 *     m   = max_j s_j
 *     w_j = exp(s_j - m)
 *     out[b,h,:] = (sum_j w_j V[b,k,j,:]) / (sum_j w_j)
 * Subtracting m before exp is the usual overflow-safe way to evaluate the
 * softmax; it cancels exactly in the ratio.
 *
 * Layouts (row-major, contiguous innermost dimension):
 *     q   [B, H, d_h]            out [B, H, d_h] (double)
 *     K,V [B, H_kv, ctx_stride, d_h]   -- "shape: [B, H_kv, max_context,
 *         head_size] per layer" ("KV-Cache Mechanics", AR Static KV-Cache).
 *
 * Parity status: pinned by the tests under tests/ (library attention in
 * fp64, closed forms, the cached == uncached invariant, GQA == MHA on
 * repeated heads, brute force on tiny inputs, and planted mutants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { KVO_BF16 = 0, KVO_FP32 = 1, KVO_FP16 = 2, KVO_FP64 = 3 };

enum {
    KVO_OK = 0,
    KVO_ERR_ARG = -1,      /* bad shape, dtype or pointer */
    KVO_ERR_LENGTH = -2,   /* a valid length outside [1, ctx_stride] */
    KVO_ERR_NOMEM = -3
};

/* bf16 is the top half of an IEEE binary32: shift it back into place. */
static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds subnormals, exponent 31 infinities and NaNs. */
static double fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

static double load_elem(const void *base, int64_t idx, int dtype)
{
    switch (dtype) {
    case KVO_BF16: return bf16_to_double(((const uint16_t *)base)[idx]);
    case KVO_FP16: return fp16_to_double(((const uint16_t *)base)[idx]);
    case KVO_FP64: return ((const double *)base)[idx];
    default:       return (double)((const float *)base)[idx];
    }
}

int kvo_abi_version(void) { return 1; }

int kvo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void kvo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Element conversion exposed for the tests' widening checks. */
double kvo_widen(const void *base, int64_t idx, int dtype)
{
    return load_elem(base, idx, dtype);
}

/*
 * Decode attention for one layer at one step: for every sequence b and query
 * head h, softmax(q K^T / sqrt(d_h)) V over cache rows [0, valid_len[b]).
 * Returns KVO_OK, or a negative code without touching out.
 */
int kvo_decode_attn(const void *q, const void *K, const void *V,
                    const int32_t *valid_len, int32_t B, int32_t H,
                    int32_t H_kv, int32_t d_h, int64_t ctx_stride,
                    int32_t dtype, double *out)
{
    if (!q || !K || !V || !valid_len || !out) return KVO_ERR_ARG;
    if (B < 1 || H < 1 || H_kv < 1 || d_h < 1 || ctx_stride < 1) return KVO_ERR_ARG;
    if (H % H_kv != 0) return KVO_ERR_ARG;
    if (dtype != KVO_BF16 && dtype != KVO_FP32 && dtype != KVO_FP16 && dtype != KVO_FP64) return KVO_ERR_ARG;
    for (int32_t b = 0; b < B; ++b)
        if (valid_len[b] < 1 || valid_len[b] > ctx_stride) return KVO_ERR_LENGTH;

    const int32_t g = H / H_kv;
    const double inv_sqrt_d = 1.0 / sqrt((double)d_h);
    int status = KVO_OK;

#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic)
#endif
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t h = 0; h < H; ++h) {
            const int32_t kv = h / g;
            const int64_t n = valid_len[b];
            const int64_t qrow = ((int64_t)b * H + h) * d_h;
            const int64_t kvrow0 = ((int64_t)b * H_kv + kv) * ctx_stride;
            double *w = (double *)malloc((size_t)n * sizeof(double));
            double *acc = (double *)calloc((size_t)d_h, sizeof(double));
            if (!w || !acc) {
                free(w);
                free(acc);
#ifdef _OPENMP
#pragma omp atomic write
#endif
                status = KVO_ERR_NOMEM;
                continue;
            }

            /* scores s_j = q . K_j / sqrt(d_h) */
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int32_t d = 0; d < d_h; ++d)
                    dot += load_elem(q, qrow + d, dtype) *
                           load_elem(K, (kvrow0 + j) * d_h + d, dtype);
                w[j] = dot * inv_sqrt_d;
                if (w[j] > m) m = w[j];
            }

            /* softmax weights and the weighted sum of value rows */
            double denom = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                w[j] = exp(w[j] - m);
                denom += w[j];
            }
            for (int64_t j = 0; j < n; ++j)
                for (int32_t d = 0; d < d_h; ++d)
                    acc[d] += w[j] * load_elem(V, (kvrow0 + j) * d_h + d, dtype);

            for (int32_t d = 0; d < d_h; ++d)
                out[qrow + d] = acc[d] / denom;
            free(w);
            free(acc);
        }
    }
    return status;
}
