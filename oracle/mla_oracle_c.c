/*
 * Plain fp64 C restatement of the MLA paged decode step (CPU oracle).
 *
 * TEST INFRASTRUCTURE ONLY: built beside the NumPy oracle and loaded by the
 * tests (which check it against the NumPy oracle) and by the CPU-baseline
 * leg of the benchmark, which times it on the host cores.  The GPU library
 * never links or calls it, and it includes nothing of the GPU library.
 *
 * Definition followed (vLLM API page
 * vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, functions
 * m1c_inputs / attend / post; page
 * vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value, classes
 * MlaValue / MlaGate), for request r, row t of r, real head h:
 *   K_j   = e4m3fn(kv[pages[indptr[r]+j]]) * kv_scale
 *   s_j   = scale * <q[t,h,:576], K_j>
 *   lse   = ln sum_j exp(s_j);  latent = sum_j exp(s_j - lse) K_j[:512]
 *   out[t, h*128+v] = L_r > 0 ? (sum_c latent[c] W[h,v,c]) * sigmoid(g) : 0
 * Requests run in parallel (OpenMP, dynamic); everything else is loops.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D_QK 576
#define D_LAT 512
#define D_V 128

/* OCP FP8 E4M3 (bias 7, subnormals, S.1111.111 = NaN, no infinities). */
static double e4m3fn(uint8_t c) {
    int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

/* bfloat16 bits to double (exact: a bf16 is the top half of a binary32). */
static double bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int mla_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * q:      bf16 bits, row t head h at q[t*q_row_stride + h*576]
 * kv:     fp8 codes [pool, 576]; pages/indptr int32
 * w_uv:   bf16 bits [heads, 128, 512]; gate: bf16 bits [S, heads*128]
 * latent: [S, heads, 512]; lse: [S, heads]; out: [S, heads*128] (any may be NULL)
 * requests: the requests to compute (n_req of them), or NULL for all R.
 */
int mla_oracle_decode_step(const uint16_t *q, int64_t q_row_stride, const uint8_t *kv,
                           const int32_t *pages, const int32_t *indptr, int R, int qlen,
                           int heads, double scale, double kv_scale, const uint16_t *w_uv,
                           const uint16_t *gate, double *latent, double *lse, double *out,
                           const int32_t *requests, int n_req, int threads) {
    int n = requests ? n_req : R;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        int r = requests ? requests[i] : i;
        int64_t lo = indptr[r], L = (int64_t)indptr[r + 1] - indptr[r];
        double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D_QK);
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double qv[D_QK], lat[D_LAT];
        if (!K || !s) { failed = 1; free(K); free(s); continue; }
        for (int64_t j = 0; j < L; ++j)
            for (int d = 0; d < D_QK; ++d)
                K[j * D_QK + d] = e4m3fn(kv[(int64_t)pages[lo + j] * D_QK + d]) * kv_scale;
        for (int tq = 0; tq < qlen; ++tq) {
            int64_t t = (int64_t)r * qlen + tq;
            for (int h = 0; h < heads; ++h) {
                for (int d = 0; d < D_QK; ++d) qv[d] = bf16(q[t * q_row_stride + (int64_t)h * D_QK + d]);
                double mx = -INFINITY, sum = 0.0, l = -INFINITY;
                for (int64_t j = 0; j < L; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < D_QK; ++d) acc += qv[d] * K[j * D_QK + d];
                    s[j] = scale * acc;
                    if (s[j] > mx) mx = s[j];
                }
                for (int c = 0; c < D_LAT; ++c) lat[c] = 0.0;
                if (L > 0) {
                    for (int64_t j = 0; j < L; ++j) sum += exp(s[j] - mx);
                    l = mx + log(sum);
                    for (int64_t j = 0; j < L; ++j) {
                        double p = exp(s[j] - l);
                        for (int c = 0; c < D_LAT; ++c) lat[c] += p * K[j * D_QK + c];
                    }
                }
                if (latent) memcpy(latent + (t * heads + h) * D_LAT, lat, sizeof lat);
                if (lse) lse[t * heads + h] = l;
                if (out) {
                    for (int v = 0; v < D_V; ++v) {
                        double o = 0.0;
                        if (L > 0) {
                            double acc = 0.0;
                            const uint16_t *w = w_uv + ((int64_t)h * D_V + v) * D_LAT;
                            for (int c = 0; c < D_LAT; ++c) acc += lat[c] * bf16(w[c]);
                            double g = bf16(gate[t * (int64_t)heads * D_V + (int64_t)h * D_V + v]);
                            o = acc * (1.0 / (1.0 + exp(-g)));
                        }
                        out[t * (int64_t)heads * D_V + (int64_t)h * D_V + v] = o;
                    }
                }
            }
        }
        free(K);
        free(s);
    }
    return failed ? -1 : 0;
}
