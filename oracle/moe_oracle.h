/*
 * CPU oracle for the small-M MoE decode layer (router, top-k routing, SwiGLU
 * experts, shared expert, weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this code: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header or table with the CUDA library.
 *
 * Source of the definition:
 *   "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative Decode on
 *   Blackwell" (lmsys.org), sections "The model", "PDL: stacking the latency
 *   floors of small kernels" and "Two fusions and a retune"; "3 ways to boost
 *   MoE inference on NVIDIA DGX Spark", section "Model and baseline
 *   configuration" (eight of 512 routed experts plus one shared expert per
 *   token, hidden 2560) and "Optimization 1" (MXFP4 expert weights).
 *
 * Precision: fp32 accumulation in index order (acc_double = 0), or fp64
 * throughout (acc_double = 1) for the oracle's own error bound.
 *
 * Layouts (row-major, nn.Linear [out, in]):
 *   x   bf16 [M, H]            Wg  bf16 [E, H]
 *   W1, W3 (per expert) bf16 [I, H]   W2 (per expert) bf16 [H, I]
 *   MXFP4 per expert: codes u8 [rows, K/2] (element 2j in the low nibble of
 *   byte j), scales u8 [rows, K/32] (e8m0, one per 32 consecutive elements of
 *   a row along the reduction dimension K).
 *   Ws1, Ws3 bf16 [Is, H]      Ws2 bf16 [H, Is]
 *
 * Return value: 0 on success, a negative number on a bad argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bf16 bit pattern -> float (exact). */
float oracle_bf16_to_f32(uint16_t b);

/* Value of one e2m1 code (low 4 bits of `code`) times 2^(scale-127).
 * scale == 255 is the e8m0 NaN encoding and returns NaN. */
float oracle_mxfp4_value(uint8_t code, uint8_t scale);

/* Decode `rows` MXFP4 rows of K elements to fp32 [rows, K]. */
int oracle_mxfp4_decode(const uint8_t* codes, const uint8_t* scales,
                        int64_t rows, int K, float* out);

/* Value of one FP8 e4m3 code (OCP 8-bit floating point, E4M3: sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent 0 encodes the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities; the
 * largest finite magnitude is 448). */
double oracle_fp8_e4m3_value(uint8_t code);

/* The e4m3 code nearest to v (ties to the code with an even mantissa),
 * saturating to +-448; NaN -> 0x7f; the sign of zero is kept. */
uint8_t oracle_fp8_e4m3_encode(float v);

/* Quantises bf16 rows [R, K] to e4m3 with one fp32 scale per block of
 * `block` consecutive elements of a row (K % block == 0): scale =
 * amax(block) / 448 in fp32 (1 for an all-zero block); code =
 * encode(w / scale), the quotient in fp32. scales is [R, K / block]. */
int oracle_fp8_quantize(const uint16_t* w, int64_t R, int K, int block,
                        uint8_t* codes, float* scales);

/* Output layer: logits[t, v] = sum_h x[t, h] * W[v, h] for M tokens and V
 * rows. wfmt 0: W bf16 [V, H]; wfmt 2: W e4m3 codes [V, H] whose value is
 * e4m3(code) * scale[v] (one fp32 scale per row). logits fp32 [M, V]. */
int oracle_lm_head(const uint16_t* x, int M, int H, const void* W,
                   const float* scale, int V, int wfmt, int acc_double,
                   float* logits);

/* Router: logits[t,e] = x[t,:] . Wg[e,:]; softmax over all E; the k largest
 * logits (ties: lower expert index first), in descending order; weights are
 * the selected probabilities renormalised to sum to one.
 * logits may be NULL. */
int oracle_route(const uint16_t* x, int M, int H, const uint16_t* Wg, int E,
                 int k, int acc_double, float* logits, int32_t* idx, float* w);

/* Pre-MoE RMSNorm of M tokens of the residual stream h (bf16 [M, H]):
 * x = h / sqrt(mean(h^2) + eps) * gamma, computed in float64 and rounded
 * once to bf16 (nearest, ties to even). */
int oracle_rmsnorm(const uint16_t* h, int M, int H, const uint16_t* gamma, float eps, uint16_t* x);

/* Router with a choice of scoring, a selection bias and a scaling factor
 * ("Chasing the Batch-1 Floor", "PDL: stacking the latency floors of small
 * kernels": a bias read by the top-k step). scoring 0: softmax over all E;
 * 1: the logistic function of each logit. The k experts with the largest
 * score + bias[e] are selected (bias may be NULL; with softmax and no bias
 * the logits themselves are ranked, the same order), ties to the lower
 * index, in descending order; their unbiased scores are renormalised to sum
 * to one and multiplied by routed_scale (a value <= 0 means 1). */
int oracle_route_ex(const uint16_t* x, int M, int H, const uint16_t* Wg, int E,
                    int k, int scoring, const float* bias, float routed_scale,
                    int acc_double, float* logits, int32_t* idx, float* w);

/* One SwiGLU expert on one token: z = W2 (silu(W1 x) * (W3 x)).
 * wfmt 0: W1/W3/W2 are bf16, s1/s3/s2 ignored. wfmt 1: MXFP4 codes + scales.
 * wfmt 2: FP8 e4m3 codes [rows, K] with fp32 scales [rows, K / 128] (the s
 * pointers then point at fp32 values).
 * x is fp32 [H]; z is fp32 [H]. */
int oracle_expert(const float* x, int H, int I, int wfmt,
                  const void* W1, const uint8_t* s1,
                  const void* W3, const uint8_t* s3,
                  const void* W2, const uint8_t* s2,
                  int acc_double, float* z);

/* Expert FFN with given routing: for each token t,
 *   y[t] = sum_j w[t,j] * expert_{idx[t,j]}(x[t]) + shared(x[t]).
 * W1/W3/W2 (and S1/S3/S2 for MXFP4) are arrays of E per-expert pointers; an
 * entry may be NULL when no token selects that expert. Is == 0 means no
 * shared expert. y is fp32 [M, H]. */
int oracle_ffn(const uint16_t* x, int M, int H, const int32_t* idx,
               const float* w, int k, int E, int I, int wfmt,
               const void* const* W1, const uint8_t* const* S1,
               const void* const* W3, const uint8_t* const* S3,
               const void* const* W2, const uint8_t* const* S2,
               int Is, const uint16_t* Ws1, const uint16_t* Ws3,
               const uint16_t* Ws2, int acc_double, float* y);

/* oracle_ffn computed by nthreads host threads (OpenMP over the (token,
 * selected expert) pairs and the shared expert; 0: all threads), combined in
 * oracle_ffn's order: y is bit-identical to oracle_ffn's. For the timed
 * all-core CPU baseline. */
int oracle_ffn_parallel(const uint16_t* x, int M, int H, const int32_t* idx,
                        const float* w, int k, int E, int I, int wfmt,
                        const void* const* W1, const uint8_t* const* S1,
                        const void* const* W3, const uint8_t* const* S3,
                        const void* const* W2, const uint8_t* const* S2,
                        int Is, const uint16_t* Ws1, const uint16_t* Ws3,
                        const uint16_t* Ws2, int acc_double, int nthreads, float* y);

/* Host threads available to oracle_ffn_parallel (1 without OpenMP). */
int oracle_threads(void);

#ifdef __cplusplus
}
#endif
#endif
