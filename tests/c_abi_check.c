/*
 * A plain C consumer of the library's C ABI (include/qknr.h): no Python and no
 * torch between the caller and the kernels. For a few layouts it fills q, k,
 * weights, a cos|sin table and positions on the host, runs qknr_apply on device
 * copies, and compares every output element with the double-precision oracle
 * (oracle/qknr_oracle.c, test infrastructure) within 2^-7*|o| + 1e-5 (bf16).
 * It also checks the position-checked entry point's error report and that the
 * host-buffer entry point gives the same bits. Exit status 0 = all passed.
 *
 * Built and run by tests/test_c_abi.py.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "qknr.h"

/* the oracle's entry point (oracle/qknr_oracle.c) */
int qknr_oracle_apply(const uint16_t *q, const uint16_t *k, const uint16_t *q_w, const uint16_t *k_w,
                      const float *cache, int64_t cache_len, const void *positions, int64_t num_tokens,
                      int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox, int64_t q_stride,
                      int64_t k_stride, int64_t head_stride, float eps, int dtype, double *q_out,
                      double *k_out);

static int failures = 0;
#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            ++failures;                                   \
        }                                                 \
    } while (0)
#define CUDA(x)                                                                          \
    do {                                                                                 \
        cudaError_t e_ = (x);                                                            \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
            exit(2);                                                                     \
        }                                                                                \
    } while (0)

/* splitmix64: a counter-based generator for the test inputs */
static uint64_t next_u64(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static double next_unit(uint64_t *s) { return (double)(next_u64(s) >> 11) * (1.0 / 9007199254740992.0); }

/* float -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

typedef struct {
    int T, n_qo, n_kv, D, R, neox, pos64, head_pad, cache_len;
} Case;

static double run_case(const Case *c, uint64_t seed) {
    const int D = c->D, hs = c->D + c->head_pad;
    const int64_t qs = (int64_t)c->n_qo * hs, ks = (int64_t)c->n_kv * hs;
    const size_t qn = (size_t)c->T * qs, kn = (size_t)c->T * ks;
    uint16_t *q = calloc(qn, 2), *k = calloc(kn, 2), *w = malloc(2 * 2 * (size_t)D);
    float *cache = malloc(sizeof(float) * (size_t)c->cache_len * c->R);
    void *pos = malloc(8 * (size_t)c->T);
    double *oq = malloc(sizeof(double) * (size_t)c->T * c->n_qo * D);
    double *ok = malloc(sizeof(double) * (size_t)c->T * c->n_kv * D);
    uint64_t s = seed;
    for (size_t i = 0; i < qn; ++i) q[i] = to_bf16((float)(4.0 * next_unit(&s) - 2.0));
    for (size_t i = 0; i < kn; ++i) k[i] = to_bf16((float)(4.0 * next_unit(&s) - 2.0));
    for (int i = 0; i < 2 * D; ++i) w[i] = to_bf16((float)(0.8 + 0.4 * next_unit(&s)));
    for (int p = 0; p < c->cache_len; ++p)
        for (int j = 0; j < c->R / 2; ++j) {
            const double ang = p * pow(1e4, -2.0 * j / c->R);
            cache[(size_t)p * c->R + j] = (float)cos(ang);
            cache[(size_t)p * c->R + c->R / 2 + j] = (float)sin(ang);
        }
    for (int t = 0; t < c->T; ++t) {
        const int64_t p = (int64_t)(next_u64(&s) % (uint64_t)c->cache_len);
        if (c->pos64) ((int64_t *)pos)[t] = p;
        else ((int32_t *)pos)[t] = (int32_t)p;
    }
    const int dtype = QKNR_BF16 | (c->pos64 ? QKNR_POS_I64 : 0);
    const float eps = 1e-6f;
    CHECK(qknr_oracle_apply(q, k, w, w + D, cache, c->cache_len, pos, c->T, c->n_qo, c->n_kv, D, c->R, c->neox,
                            qs, ks, hs, eps, dtype, oq, ok) == 0, "oracle rejected the case");

    void *dq, *dk, *dw, *dpos;
    float *dcache;
    CUDA(cudaMalloc(&dq, qn * 2));
    CUDA(cudaMalloc(&dk, kn * 2));
    CUDA(cudaMalloc(&dw, 4 * (size_t)D));
    CUDA(cudaMalloc((void **)&dcache, sizeof(float) * (size_t)c->cache_len * c->R));
    CUDA(cudaMalloc(&dpos, 8 * (size_t)c->T));
    CUDA(cudaMemcpy(dq, q, qn * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dk, k, kn * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dw, w, 4 * (size_t)D, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dcache, cache, sizeof(float) * (size_t)c->cache_len * c->R, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dpos, pos, 8 * (size_t)c->T, cudaMemcpyHostToDevice));
    const char *dw8 = (const char *)dw;

    int rc = qknr_apply(dq, dk, dw8, dw8 + 2 * D, dcache, dpos, c->T, c->n_qo, c->n_kv, D, c->R, c->neox, qs, ks,
                        hs, eps, dtype, NULL);
    CHECK(rc == QKNR_OK, "qknr_apply returned %d: %s", rc, qknr_last_error());
    CUDA(cudaDeviceSynchronize());
    uint16_t *gq = malloc(qn * 2), *gk = malloc(kn * 2);
    CUDA(cudaMemcpy(gq, dq, qn * 2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gk, dk, kn * 2, cudaMemcpyDeviceToHost));

    double worst = 0.0;
    for (int t = 0; t < c->T; ++t)
        for (int side = 0; side < 2; ++side) {
            const int n = side ? c->n_kv : c->n_qo;
            const int64_t ts = side ? ks : qs;
            const uint16_t *g = side ? gk : gq, *x = side ? k : q;
            const double *o = side ? ok : oq;
            for (int h = 0; h < n; ++h)
                for (int i = 0; i < hs; ++i) {
                    const size_t at = (size_t)t * ts + (size_t)h * hs + i;
                    if (i >= D) { /* padding keeps its bits */
                        CHECK(g[at] == x[at], "padding changed at t=%d h=%d i=%d", t, h, i);
                        continue;
                    }
                    const double e = o[((size_t)t * n + h) * D + i];
                    const double v = fabs(from_bf16(g[at]) - e) / (ldexp(fabs(e), -7) + 1e-5);
                    if (v > worst) worst = v;
                }
        }
    CHECK(worst <= 1.0, "max error %.3f x tolerance", worst);

    /* the host-buffer entry point on pinned copies: the same bits */
    uint16_t *hq, *hk;
    void *hpos;
    CUDA(cudaHostAlloc((void **)&hq, qn * 2, cudaHostAllocDefault));
    CUDA(cudaHostAlloc((void **)&hk, kn * 2, cudaHostAllocDefault));
    CUDA(cudaHostAlloc(&hpos, 8 * (size_t)c->T, cudaHostAllocDefault));
    memcpy(hq, q, qn * 2);
    memcpy(hk, k, kn * 2);
    memcpy(hpos, pos, 8 * (size_t)c->T);
    rc = qknr_apply_host(hq, hk, dw8, dw8 + 2 * D, dcache, hpos, dq, dk, dpos, c->T, c->n_qo, c->n_kv, D, c->R,
                         c->neox, qs, ks, hs, eps, dtype, 0, QKNR_HOST_AUTO, NULL);
    CHECK(rc == QKNR_OK, "qknr_apply_host returned %d: %s", rc, qknr_last_error());
    CUDA(cudaDeviceSynchronize());
    CHECK(memcmp(hq, gq, qn * 2) == 0 && memcmp(hk, gk, kn * 2) == 0, "qknr_apply_host differs from qknr_apply");

    /* the checked entry point reports an out-of-range position and leaves that token */
    if (c->pos64) ((int64_t *)pos)[c->T / 2] = c->cache_len;
    else ((int32_t *)pos)[c->T / 2] = c->cache_len;
    CUDA(cudaMemcpy(dpos, pos, 8 * (size_t)c->T, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dq, q, qn * 2, cudaMemcpyHostToDevice));
    rc = qknr_apply_checked(dq, dk, dw8, dw8 + 2 * D, dcache, c->cache_len, dpos, c->T, c->n_qo, c->n_kv, D, c->R,
                            c->neox, qs, ks, hs, eps, dtype, NULL);
    CHECK(rc == QKNR_ERR_POSITION_OOB, "qknr_apply_checked returned %d, expected QKNR_ERR_POSITION_OOB", rc);
    CUDA(cudaMemcpy(gq, dq, qn * 2, cudaMemcpyDeviceToHost));
    CHECK(memcmp(gq + (size_t)(c->T / 2) * qs, q + (size_t)(c->T / 2) * qs, (size_t)qs * 2) == 0,
          "the token with a bad position was changed");

    cudaFreeHost(hq);
    cudaFreeHost(hk);
    cudaFreeHost(hpos);
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dw);
    cudaFree(dcache);
    cudaFree(dpos);
    free(q), free(k), free(w), free(cache), free(pos), free(oq), free(ok), free(gq), free(gk);
    return worst;
}

int main(void) {
    if (qknr_init(0) != QKNR_OK) {
        fprintf(stderr, "qknr_init: %s\n", qknr_last_error());
        return 2;
    }
    const Case cases[] = {
        {77, 6, 2, 128, 64, 1, 1, 0, 300},   /* GQA, partial NeoX, int64 positions */
        {33, 4, 4, 64, 64, 0, 0, 16, 100},   /* interleaved, padded heads, int32 positions */
        {129, 16, 4, 256, 128, 0, 0, 0, 500},/* head_dim 256, partial interleaved */
        {9, 3, 1, 96, 48, 1, 1, 8, 64},      /* head_dim 96, NeoX R = 48, padded */
    };
    for (size_t i = 0; i < sizeof(cases) / sizeof(cases[0]); ++i) {
        const double worst = run_case(&cases[i], 1234 + i);
        printf("case %zu: T=%d n_qo=%d n_kv=%d D=%d R=%d %s: max error %.3f of tolerance\n", i, cases[i].T,
               cases[i].n_qo, cases[i].n_kv, cases[i].D, cases[i].R, cases[i].neox ? "neox" : "interleaved", worst);
    }
    qknr_shutdown();
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("all passed\n");
    return 0;
}
