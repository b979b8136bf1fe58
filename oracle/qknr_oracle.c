/*
 * qknr_oracle.c -- reference oracle for the fused, in-place, per-head
 * QK RMSNorm + rotary position embedding (RoPE).
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this file. The product path never calls
 * it; it shares no code, header or constant with the CUDA library.
 *
 * Source of the definitions: the web page "SGLang Diffusion fused operator
 * fused_inplace_qknorm_rope deep-dive" (m.lsln.cn/news/241376), cited below
 * as [deep-dive §n]:
 *   §2.1  QK RMSNorm: rms(x) = sqrt((1/head_dim) * sum_i x_i^2 + eps),
 *         out_i = x_i / rms(x) * w_i.
 *   §2.2  RoPE: cache row pos = [cos(pos*theta_0..theta_{r/2-1}) |
 *         sin(pos*theta_0..theta_{r/2-1})]; interleaved (GPT-J) pairs
 *         (2j, 2j+1), NeoX pairs (d, d+half) with half = rope_dim/2;
 *         only the first rope_dim dims rotate ("partial RoPE").
 *   §2.3  order: load, sum of squares, scale, x*scale*w, rotate the first
 *         rope_dim dims, write back in place.
 *   §3    tensor contract: q [T, n_qo, D], k [T, n_kv, D] (fp16/bf16,
 *         innermost stride 1), weights [D] in the q/k dtype, fp32 cache
 *         [any_len, rope_dim], positions [T] int32 or int64.
 *   §4.3  the mean is taken over head_dim (sum / kHeadDim), for every rope_dim.
 *   §4.4  the cos/sin index of a NeoX dim d is d mod (rope_dim/2).
 *
 * The fused op reaches exactly this plain definition (fusion changes memory
 * traffic only), so the oracle is the definition itself, evaluated in double
 * precision with no intermediate rounding. Outputs are returned unrounded
 * in double; the caller compares the GPU's rounded values against them.
 *
 * Readings where the page is silent or garbled (operators were stripped in
 * extraction): eps is added to the mean inside the square root; the weight
 * multiplies as w (no 1+w offset); normalisation and weighting happen before
 * the rotation; cos sits in the first half of a cache row and sin in the
 * second half, for both pairings.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Own copies of the tensor-contract codes (values fixed by the C ABI). */
#define ORC_BF16 0
#define ORC_FP16 1
#define ORC_POS_I64 0x100

#define ORC_OK 0
#define ORC_EINVAL 2
#define ORC_EUNSUP 3

/* bfloat16 is the upper half of an IEEE binary32 value: widening is exact. */
static double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_fp16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);            /* zero or subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(frac + 1024), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

double qknr_oracle_decode(int dtype, uint16_t bits)
{
    return (dtype & 0xff) == ORC_FP16 ? orc_fp16_to_double(bits) : orc_bf16_to_double(bits);
}

/*
 * One head [deep-dive §2.3]. x: D elements (stride 1) in the 16-bit dtype,
 * w: D weights, cos_row / sin_row: R/2 fp32 values each. out: D doubles.
 */
int qknr_oracle_head(const uint16_t *x, const uint16_t *w, const float *cos_row,
                     const float *sin_row, int head_dim, int rope_dim, int is_neox,
                     double eps, int dtype, double *out)
{
    int D = head_dim, R = rope_dim, i;
    double *n;
    double ss = 0.0, r;

    if (D <= 0 || R < 0 || R > D || (R % 2) != 0)
        return ORC_EINVAL;
    n = (double *)malloc(sizeof(double) * (size_t)D);
    if (!n)
        return ORC_EINVAL;

    /* step 1-2: widen to double (exact) and sum the squares over all D dims */
    for (i = 0; i < D; ++i) {
        double xi = qknr_oracle_decode(dtype, x[i]);
        n[i] = xi;
        ss += xi * xi;
    }
    /* step 3: inverse RMS, mean over head_dim, eps inside the root [§2.1, §4.3] */
    r = 1.0 / sqrt(ss / (double)D + eps);
    /* step 4: normalise and apply the per-channel weight */
    for (i = 0; i < D; ++i)
        n[i] = n[i] * r * qknr_oracle_decode(dtype, w[i]);

    /* step 5: rotate the first R dims [§2.2] */
    if (!is_neox) {
        /* interleaved (GPT-J): pair (2j, 2j+1) uses frequency j */
        for (i = 0; i < R / 2; ++i) {
            double c = (double)cos_row[i], s = (double)sin_row[i];
            double a = n[2 * i], b = n[2 * i + 1];
            out[2 * i] = a * c - b * s;
            out[2 * i + 1] = b * c + a * s;
        }
    } else {
        /* NeoX (LLaMA): pair (d, d + R/2) uses frequency d */
        int half = R / 2;
        for (i = 0; i < half; ++i) {
            double c = (double)cos_row[i], s = (double)sin_row[i];
            double a = n[i], b = n[i + half];
            out[i] = a * c - b * s;
            out[i + half] = b * c + a * s;
        }
    }
    /* step 6: dims past rope_dim keep the normalised values */
    for (i = R; i < D; ++i)
        out[i] = n[i];

    free(n);
    return ORC_OK;
}

/*
 * The whole op over every token and every head, first the n_qo query heads
 * with q_w, then the n_kv key heads with k_w [deep-dive §3, §4.2].
 *
 * q, k: base pointers of the 16-bit inputs; element (t, h, i) of q sits at
 *       q[t*q_stride + h*head_stride + i] (strides in elements), same for k.
 * q_out: dense [T, n_qo, D] doubles; k_out: dense [T, n_kv, D] doubles.
 * cache: fp32 [cache_len, R] row-major; positions: [T] int32, or int64 when
 *       dtype has ORC_POS_I64 set. A position outside [0, cache_len) is an
 *       error here (the op itself leaves it undefined).
 */
int qknr_oracle_apply(const uint16_t *q, const uint16_t *k, const uint16_t *q_w,
                      const uint16_t *k_w, const float *cache, int64_t cache_len,
                      const void *positions, int64_t num_tokens, int n_qo, int n_kv,
                      int head_dim, int rope_dim, int is_neox, int64_t q_stride,
                      int64_t k_stride, int64_t head_stride, float eps, int dtype,
                      double *q_out, double *k_out)
{
    int64_t t;
    int h, rc;
    int D = head_dim, R = rope_dim;
    if (num_tokens < 0 || n_qo < 0 || n_kv < 0 || D <= 0 || R <= 0 || R > D || (R % 2) != 0)
        return ORC_EINVAL;
    if ((dtype & 0xff) != ORC_BF16 && (dtype & 0xff) != ORC_FP16)
        return ORC_EUNSUP;

    for (t = 0; t < num_tokens; ++t) {
        int64_t pos = (dtype & ORC_POS_I64) ? ((const int64_t *)positions)[t]
                                            : (int64_t)((const int32_t *)positions)[t];
        const float *cos_row, *sin_row;
        if (pos < 0 || pos >= cache_len)
            return ORC_EINVAL;
        cos_row = cache + pos * R;
        sin_row = cos_row + R / 2;
        for (h = 0; h < n_qo; ++h) {
            rc = qknr_oracle_head(q + t * q_stride + (int64_t)h * head_stride, q_w, cos_row,
                                  sin_row, D, R, is_neox, (double)eps, dtype,
                                  q_out + (t * n_qo + h) * (int64_t)D);
            if (rc)
                return rc;
        }
        for (h = 0; h < n_kv; ++h) {
            rc = qknr_oracle_head(k + t * k_stride + (int64_t)h * head_stride, k_w, cos_row,
                                  sin_row, D, R, is_neox, (double)eps, dtype,
                                  k_out + (t * n_kv + h) * (int64_t)D);
            if (rc)
                return rc;
        }
    }
    return ORC_OK;
}
