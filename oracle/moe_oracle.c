/*
 * CPU oracle for the small-M MoE decode layer. TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * it; the CUDA library never links or calls it. Plain loops, no SIMD
 * intrinsics, no fast-math; built with -ffp-contract=off so that x86 and Arm
 * hosts give the same bits.
 *
 * Every function follows the definitions stated in moe_oracle.h; the
 * citations below name the page and section each step comes from.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e2m1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. Exponent
 * field 0 is subnormal: value = mantissa * 0.5. Otherwise value =
 * 2^(exp-1) * (1 + mantissa/2). This is the element format of MXFP4 named in
 * "3 ways to boost MoE inference on NVIDIA DGX Spark", Optimization 1. */
static double e2m1_magnitude(unsigned code) {
    unsigned e = (code >> 1) & 3u, m = code & 1u;
    if (e == 0) return 0.5 * (double)m;
    return ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
}

float oracle_mxfp4_value(uint8_t code, uint8_t scale) {
    if (scale == 255) return NAN; /* e8m0 NaN encoding */
    double mag = e2m1_magnitude(code & 7u);
    double v = ldexp(mag, (int)scale - 127);
    return (float)((code & 8u) ? -v : v);
}

int oracle_mxfp4_decode(const uint8_t* codes, const uint8_t* scales,
                        int64_t rows, int K, float* out) {
    if (!codes || !scales || !out || rows < 0 || K <= 0 || K % 32) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int c = 0; c < K; ++c) {
            uint8_t byte = codes[r * (K / 2) + c / 2];
            uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
            out[r * K + c] = oracle_mxfp4_value(code, scales[r * (K / 32) + c / 32]);
        }
    }
    return 0;
}

/* One weight element as fp32: bf16 row-major; MXFP4 codes + e8m0 scales
 * (one per 32 elements of a row); or FP8 e4m3 codes + fp32 scales (one per
 * 128 elements of a row, S then holds fp32 values). */
static float weight_at(const void* W, const uint8_t* S, int wfmt, int K,
                       int64_t row, int col) {
    if (wfmt == 0) return oracle_bf16_to_f32(((const uint16_t*)W)[row * K + col]);
    if (wfmt == 2) {
        const uint8_t code = ((const uint8_t*)W)[row * K + col];
        const float sc = ((const float*)S)[row * (K / 128) + col / 128];
        return (float)(oracle_fp8_e4m3_value(code) * (double)sc);
    }
    const uint8_t* q = (const uint8_t*)W;
    uint8_t byte = q[row * (K / 2) + col / 2];
    uint8_t code = (col & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
    return oracle_mxfp4_value(code, S[row * (K / 32) + col / 32]);
}

/* Router gate, softmax, top-k, renormalisation.
 * "Chasing the Batch-1 Floor", section "PDL: stacking the latency floors of
 * small kernels" (router chain: gate matvec, then top-k) and section "bf16
 * router gate and lm_head" (bf16 gate weight). Softmax over all experts and
 * renormalisation of the k selected probabilities is the plain reading of
 * "routes each token to eight of 512 routed experts" ("3 ways to boost MoE
 * inference", section "Model and baseline configuration"). */
int oracle_route_ex(const uint16_t* x, int M, int H, const uint16_t* Wg, int E,
                    int k, int scoring, const float* bias, float routed_scale,
                    int acc_double, float* logits, int32_t* idx, float* w) {
    if (!x || !Wg || !idx || !w || M < 0 || H <= 0 || E <= 0 || k <= 0 || k > E)
        return -1;
    if (scoring != 0 && scoring != 1) return -1;
    const double scale = routed_scale > 0.0f ? (double)routed_scale : 1.0;
    /* softmax without a bias ranks the logits themselves (the same order) */
    const int by_logit = scoring == 0 && !bias;
    double* l = (double*)malloc(sizeof(double) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* c = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!l || !p || !c || !taken) { free(l); free(p); free(c); free(taken); return -2; }
    for (int t = 0; t < M; ++t) {
        const uint16_t* xt = x + (int64_t)t * H;
        /* step 1: logits, accumulated in index order */
        for (int e = 0; e < E; ++e) {
            const uint16_t* we = Wg + (int64_t)e * H;
            if (acc_double) {
                double s = 0.0;
                for (int h = 0; h < H; ++h)
                    s += (double)oracle_bf16_to_f32(xt[h]) * (double)oracle_bf16_to_f32(we[h]);
                l[e] = s;
            } else {
                float s = 0.0f;
                for (int h = 0; h < H; ++h) {
                    float prod = oracle_bf16_to_f32(xt[h]) * oracle_bf16_to_f32(we[h]);
                    s = s + prod;
                }
                l[e] = (double)s;
            }
            if (logits) logits[(int64_t)t * E + e] = (float)l[e];
        }
        /* step 2: scores: softmax over all E (max-subtracted), or the
         * logistic function of each logit */
        if (scoring == 0) {
            double mx = l[0];
            for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
            if (acc_double) {
                double den = 0.0;
                for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); den += p[e]; }
                for (int e = 0; e < E; ++e) p[e] /= den;
            } else {
                float den = 0.0f;
                for (int e = 0; e < E; ++e) {
                    float pe = expf((float)l[e] - (float)mx);
                    p[e] = (double)pe;
                    den = den + pe;
                }
                for (int e = 0; e < E; ++e) p[e] = (double)((float)p[e] / den);
            }
        } else {
            for (int e = 0; e < E; ++e)
                p[e] = acc_double ? 1.0 / (1.0 + exp(-l[e]))
                                  : (double)(1.0f / (1.0f + expf(-(float)l[e])));
        }
        /* step 3: the k largest selection keys (logit; or score plus the
         * expert's bias), ties to the lower index */
        for (int e = 0; e < E; ++e) {
            const double b = bias ? (double)bias[e] : 0.0;
            c[e] = by_logit ? l[e] : acc_double ? p[e] + b : (double)((float)p[e] + (float)b);
        }
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || c[e] > c[best]) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
        }
        /* step 4: the selected (unbiased) scores renormalised to sum to one,
         * times the routed scaling factor */
        if (acc_double) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += p[idx[(int64_t)t * k + j]];
            for (int j = 0; j < k; ++j)
                w[(int64_t)t * k + j] = (float)(p[idx[(int64_t)t * k + j]] / s * scale);
        } else {
            float s = 0.0f;
            for (int j = 0; j < k; ++j) s = s + (float)p[idx[(int64_t)t * k + j]];
            for (int j = 0; j < k; ++j)
                w[(int64_t)t * k + j] = (float)p[idx[(int64_t)t * k + j]] / s * (float)scale;
        }
    }
    free(l); free(p); free(c); free(taken);
    return 0;
}

int oracle_route(const uint16_t* x, int M, int H, const uint16_t* Wg, int E,
                 int k, int acc_double, float* logits, int32_t* idx, float* w) {
    return oracle_route_ex(x, M, H, Wg, E, k, 0, NULL, 1.0f, acc_double, logits, idx, w);
}

/* One SwiGLU expert: g = W1 x, u = W3 x, h = silu(g) * u with
 * silu(g) = g / (1 + e^-g), computed in fp32 with no intermediate bf16
 * rounding; z = W2 h. "Chasing the Batch-1 Floor", section "Two fusions and a
 * retune" (silu(gate) * up in the up-GEMM epilogue, activation kept in float
 * before the multiply). */
int oracle_expert(const float* x, int H, int I, int wfmt,
                  const void* W1, const uint8_t* s1,
                  const void* W3, const uint8_t* s3,
                  const void* W2, const uint8_t* s2,
                  int acc_double, float* z) {
    if (!x || !W1 || !W3 || !W2 || !z || H <= 0 || I <= 0) return -1;
    if (wfmt == 1 && (!s1 || !s3 || !s2 || H % 32 || I % 32)) return -1;
    if (wfmt == 2 && (!s1 || !s3 || !s2 || H % 128 || I % 128)) return -1;
    if (wfmt != 0 && wfmt != 1 && wfmt != 2) return -1;
    double* hd = (double*)malloc(sizeof(double) * (size_t)I);
    if (!hd) return -2;
    for (int i = 0; i < I; ++i) {
        if (acc_double) {
            double g = 0.0, u = 0.0;
            for (int c = 0; c < H; ++c) {
                g += (double)weight_at(W1, s1, wfmt, H, i, c) * (double)x[c];
                u += (double)weight_at(W3, s3, wfmt, H, i, c) * (double)x[c];
            }
            hd[i] = g / (1.0 + exp(-g)) * u;
        } else {
            float g = 0.0f, u = 0.0f;
            for (int c = 0; c < H; ++c) {
                float pg = weight_at(W1, s1, wfmt, H, i, c) * x[c];
                float pu = weight_at(W3, s3, wfmt, H, i, c) * x[c];
                g = g + pg;
                u = u + pu;
            }
            float sg = g / (1.0f + expf(-g));
            hd[i] = (double)(sg * u);
        }
    }
    for (int o = 0; o < H; ++o) {
        if (acc_double) {
            double s = 0.0;
            for (int i = 0; i < I; ++i) s += (double)weight_at(W2, s2, wfmt, I, o, i) * hd[i];
            z[o] = (float)s;
        } else {
            float s = 0.0f;
            for (int i = 0; i < I; ++i) {
                float prod = weight_at(W2, s2, wfmt, I, o, i) * (float)hd[i];
                s = s + prod;
            }
            z[o] = s;
        }
    }
    free(hd);
    return 0;
}

/* Weighted combine of the selected experts plus the always-on shared expert,
 * summed in fp32 with no intermediate rounding ("Chasing the Batch-1 Floor",
 * section "PDL: stacking the latency floors of small kernels": fp32 sum with a
 * single final cast; "3 ways to boost MoE inference", section "Model and
 * baseline configuration": one shared expert). */
int oracle_ffn(const uint16_t* x, int M, int H, const int32_t* idx,
               const float* w, int k, int E, int I, int wfmt,
               const void* const* W1, const uint8_t* const* S1,
               const void* const* W3, const uint8_t* const* S3,
               const void* const* W2, const uint8_t* const* S2,
               int Is, const uint16_t* Ws1, const uint16_t* Ws3,
               const uint16_t* Ws2, int acc_double, float* y) {
    if (!x || !y || M < 0 || H <= 0 || k < 0 || E <= 0 || I <= 0 || Is < 0) return -1;
    if (k > 0 && (!idx || !w || !W1 || !W3 || !W2)) return -1;
    if (wfmt != 0 && k > 0 && (!S1 || !S3 || !S2)) return -1;
    if (Is > 0 && (!Ws1 || !Ws3 || !Ws2)) return -1;
    float* xt = (float*)malloc(sizeof(float) * (size_t)H);
    float* z = (float*)malloc(sizeof(float) * (size_t)H);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!xt || !z || !acc) { free(xt); free(z); free(acc); return -2; }
    int rc = 0;
    for (int t = 0; t < M && rc == 0; ++t) {
        for (int c = 0; c < H; ++c) xt[c] = oracle_bf16_to_f32(x[(int64_t)t * H + c]);
        for (int c = 0; c < H; ++c) acc[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = idx[(int64_t)t * k + j];
            if (e < 0 || e >= E || !W1[e] || !W3[e] || !W2[e]) { rc = -3; break; }
            const uint8_t *a = NULL, *b = NULL, *d = NULL;
            if (wfmt != 0) { a = S1[e]; b = S3[e]; d = S2[e]; }
            rc = oracle_expert(xt, H, I, wfmt, W1[e], a, W3[e], b, W2[e], d, acc_double, z);
            if (rc) break;
            float wj = w[(int64_t)t * k + j];
            for (int c = 0; c < H; ++c) {
                if (acc_double) acc[c] += (double)wj * (double)z[c];
                else acc[c] = (double)((float)acc[c] + wj * z[c]);
            }
        }
        if (rc == 0 && Is > 0) {
            rc = oracle_expert(xt, H, Is, 0, Ws1, NULL, Ws3, NULL, Ws2, NULL, acc_double, z);
            for (int c = 0; c < H && rc == 0; ++c) {
                if (acc_double) acc[c] += (double)z[c];
                else acc[c] = (double)((float)acc[c] + z[c]);
            }
        }
        for (int c = 0; c < H; ++c) y[(int64_t)t * H + c] = (float)acc[c];
    }
    free(xt); free(z); free(acc);
    return rc;
}

/* The same FFN with the work spread over host threads, for the timed CPU
 * baseline: the (token, selected expert) pairs and each token's shared expert
 * are independent oracle_expert calls, run by an OpenMP parallel loop
 * (nthreads threads, 0: all); their outputs are then combined exactly as
 * oracle_ffn combines them (same order, same arithmetic), so y is
 * bit-identical to oracle_ffn's. Without OpenMP the loop runs on one thread. */
int oracle_ffn_parallel(const uint16_t* x, int M, int H, const int32_t* idx,
                        const float* w, int k, int E, int I, int wfmt,
                        const void* const* W1, const uint8_t* const* S1,
                        const void* const* W3, const uint8_t* const* S3,
                        const void* const* W2, const uint8_t* const* S2,
                        int Is, const uint16_t* Ws1, const uint16_t* Ws3,
                        const uint16_t* Ws2, int acc_double, int nthreads, float* y) {
    if (!x || !y || M < 0 || H <= 0 || k < 0 || E <= 0 || I <= 0 || Is < 0) return -1;
    if (k > 0 && (!idx || !w || !W1 || !W3 || !W2)) return -1;
    if (wfmt != 0 && k > 0 && (!S1 || !S3 || !S2)) return -1;
    if (Is > 0 && (!Ws1 || !Ws3 || !Ws2)) return -1;
    const int per = k + (Is > 0 ? 1 : 0);
    const int ntask = M * per;
    float* xf = (float*)malloc(sizeof(float) * (size_t)M * H + 1);
    float* z = (float*)malloc(sizeof(float) * (size_t)ntask * H + 1);
    int* rcs = (int*)calloc((size_t)ntask + 1, sizeof(int));
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!xf || !z || !rcs || !acc) { free(xf); free(z); free(rcs); free(acc); return -2; }
    for (int64_t i = 0; i < (int64_t)M * H; ++i) xf[i] = oracle_bf16_to_f32(x[i]);
    int nt = nthreads;
#ifdef _OPENMP
    if (nt <= 0) nt = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int q = 0; q < ntask; ++q) {
        const int t = q / per, j = q % per;
        const float* xt = xf + (int64_t)t * H;
        float* zq = z + (int64_t)q * H;
        if (j < k) {
            const int e = idx[(int64_t)t * k + j];
            if (e < 0 || e >= E || !W1[e] || !W3[e] || !W2[e]) { rcs[q] = -3; continue; }
            const uint8_t *a = NULL, *b = NULL, *d = NULL;
            if (wfmt != 0) { a = S1[e]; b = S3[e]; d = S2[e]; }
            rcs[q] = oracle_expert(xt, H, I, wfmt, W1[e], a, W3[e], b, W2[e], d, acc_double, zq);
        } else {
            rcs[q] = oracle_expert(xt, H, Is, 0, Ws1, NULL, Ws3, NULL, Ws2, NULL, acc_double, zq);
        }
    }
    (void)nt;
    int rc = 0;
    for (int q = 0; q < ntask && rc == 0; ++q) rc = rcs[q];
    for (int t = 0; t < M && rc == 0; ++t) {
        for (int c = 0; c < H; ++c) acc[c] = 0.0;
        for (int j = 0; j < per; ++j) {
            const float* zq = z + ((int64_t)t * per + j) * H;
            const float wj = j < k ? w[(int64_t)t * k + j] : 1.0f;
            for (int c = 0; c < H; ++c) {
                if (j < k) {
                    if (acc_double) acc[c] += (double)wj * (double)zq[c];
                    else acc[c] = (double)((float)acc[c] + wj * zq[c]);
                } else {
                    if (acc_double) acc[c] += (double)zq[c];
                    else acc[c] = (double)((float)acc[c] + zq[c]);
                }
            }
        }
        for (int c = 0; c < H; ++c) y[(int64_t)t * H + c] = (float)acc[c];
    }
    free(xf); free(z); free(rcs); free(acc);
    return rc;
}

/* Threads an OpenMP parallel region may use here (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ FP8 */
/* OCP "OCP 8-bit Floating Point Specification (OFP8)", format E4M3. */
double oracle_fp8_e4m3_value(uint8_t code) {
    const int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

uint8_t oracle_fp8_e4m3_encode(float v) {
    if (isnan(v)) return 0x7f;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    /* non-negative finite codes 0x00..0x7e have increasing values: take the
       nearest, ties to the even code */
    int best = 0;
    double bd = a;
    for (int c = 1; c <= 0x7e; ++c) {
        const double d = fabs(oracle_fp8_e4m3_value((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return (uint8_t)(sign | best);
}

int oracle_fp8_quantize(const uint16_t* w, int64_t R, int K, int block,
                        uint8_t* codes, float* scales) {
    if (!w || !codes || !scales || R < 0 || K <= 0 || block <= 0 || K % block) return -1;
    const int nb = K / block;
    for (int64_t r = 0; r < R; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint16_t* src = w + r * K + (int64_t)b * block;
            float amax = 0.0f;
            for (int i = 0; i < block; ++i) {
                const float a = fabsf(oracle_bf16_to_f32(src[i]));
                if (a > amax) amax = a;
            }
            const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[r * nb + b] = sc;
            for (int i = 0; i < block; ++i)
                codes[r * K + (int64_t)b * block + i] = oracle_fp8_e4m3_encode(oracle_bf16_to_f32(src[i]) / sc);
        }
    return 0;
}

/* ------------------------------------------------------------------ lm_head */
/* "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative Decode on
   Blackwell", section "bf16 router gate and lm_head"; "3 ways to boost MoE
   inference on NVIDIA DGX Spark", "Optimization 2: Online FP8 LM head
   quantization" (FP8 weights of the output layer). */
int oracle_lm_head(const uint16_t* x, int M, int H, const void* W,
                   const float* scale, int V, int wfmt, int acc_double,
                   float* logits) {
    if (!x || !W || !logits || M < 0 || H <= 0 || V < 0) return -1;
    if (wfmt != 0 && wfmt != 2) return -1;
    if (wfmt == 2 && !scale) return -1;
    for (int t = 0; t < M; ++t)
        for (int v = 0; v < V; ++v) {
            double accd = 0.0;
            float accf = 0.0f;
            for (int h = 0; h < H; ++h) {
                const float xv = oracle_bf16_to_f32(x[(int64_t)t * H + h]);
                double wv;
                if (wfmt == 0)
                    wv = oracle_bf16_to_f32(((const uint16_t*)W)[(int64_t)v * H + h]);
                else
                    wv = oracle_fp8_e4m3_value(((const uint8_t*)W)[(int64_t)v * H + h]) * (double)scale[v];
                if (acc_double)
                    accd += (double)xv * wv;
                else
                    accf += xv * (float)wv;
            }
            logits[(int64_t)t * V + v] = acc_double ? (float)accd : accf;
        }
    return 0;
}

/* ------------------------------------------------------------------ RMSNorm */
/* Pre-MoE norm ("Chasing the Batch-1 Floor", "PDL: stacking the latency
   floors of small kernels": the router chain starts with the norm):
   x = h / sqrt(mean(h^2) + eps) * gamma, in float64, rounded once to bf16
   (nearest, ties to even). */
static uint16_t f64_to_bf16_rne(double v) {
    if (isnan(v)) return 0x7fc0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                        /* a = m 2^e, m in [0.5, 1) */
    const int sh = e - 1 < -126 ? 133 : 8 - e;  /* bf16 grid: 8 significant
                                                   bits, subnormals 2^-133 */
    const double r = ldexp(rint(ldexp(a, sh)), -sh);  /* ties to even */
    const float f = (float)r;            /* exact (or inf beyond the range) */
    uint32_t b;
    memcpy(&b, &f, 4);
    return (uint16_t)(sign | (b >> 16));
}

int oracle_rmsnorm(const uint16_t* h, int M, int H, const uint16_t* gamma, float eps, uint16_t* x) {
    if (!h || !gamma || !x || M < 0 || H <= 0) return -1;
    for (int t = 0; t < M; ++t) {
        double ss = 0.0;
        for (int i = 0; i < H; ++i) {
            const double v = oracle_bf16_to_f32(h[(int64_t)t * H + i]);
            ss += v * v;
        }
        const double r = 1.0 / sqrt(ss / H + (double)eps);
        for (int i = 0; i < H; ++i)
            x[(int64_t)t * H + i] = f64_to_bf16_rne((double)oracle_bf16_to_f32(h[(int64_t)t * H + i]) * r *
                                                    (double)oracle_bf16_to_f32(gamma[i]));
    }
    return 0;
}
