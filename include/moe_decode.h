/*
 * moe_decode.h - C ABI of the GB300 small-M MoE decode layer library
 * (libmoe_decode.so, sm_103a).
 *
 * The layer, for M = 1..16 tokens (batch-1 decode and speculative verify):
 *   logits = x Wg^T                      router gate matvec, bf16 weight
 *   p = softmax(logits) (or sigmoid(logits)); S = top-k(p + bias);
 *   w = routed_scale * p_S / sum p_S
 *   y_t = sum_j w_tj * E_{S_tj}(x_t) + E_shared(x_t)
 *   E(x) = W2 (silu(W1 x) * (W3 x)),   silu(g) = g / (1 + e^-g)
 * "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative Decode on
 * Blackwell" (lmsys.org): sections "The model" (512-expert MoE), "PDL:
 * stacking the latency floors of small kernels" (router chain norm -> gate
 * matvec -> top-k; MoE chain up-GEMM -> activation -> down-GEMM -> combine;
 * fp32 combine with one final cast), "Two fusions and a retune" (SwiGLU in
 * the up-GEMM epilogue), "bf16 router gate and lm_head"; "3 ways to boost MoE
 * inference on NVIDIA DGX Spark": "Model and baseline configuration" (8 of 512
 * routed experts plus one shared expert, hidden 2560) and "Optimization 1"
 * (MXFP4 expert weights).
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must be memory the GPU can address,
 *    owned by the caller, 16-byte aligned: normally HBM. The tokens x and
 *    the outputs y, idx_out, w_out may also be pinned host memory (on a
 *    coherent CPU-GPU link the kernel then reads and writes it directly,
 *    with no separate copy). The library allocates and frees nothing.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronise, except moe_read_status.
 *  - Return value: MOE_OK (0), or a negative MOE_E* code. A negative code
 *    from argument checking means nothing was launched. MOE_ECUDA means a
 *    CUDA call failed (cudaGetLastError is then cleared).
 *  - Conditions found on the device (an expert index out of range passed to
 *    moe_ffn, a bounded wait that ran out) do not fault: they are written to
 *    a status word inside the workspace; read it with moe_read_status.
 *  - A workspace (`ws`, `ws_bytes` >= moe_workspace_bytes(shape, M)) holds
 *    the router logits (each tagged with its call), the SwiGLU activations
 *    (for one-token bf16 layers also tagged with the call, with a 16-bit tag
 *    that repeats every 65,535 calls: calls of several shapes that share a
 *    workspace should be re-initialised at least that often), a call counter
 *    and the grid-barrier counters. Zero it once with moe_workspace_init
 *    before its first use; every call leaves it ready for the next. Calls
 *    that share a workspace must be ordered on one stream (or otherwise
 *    serialised).
 *
 * Layouts (row-major; nn.Linear [out, in], contiguous along the reduction
 * dimension):
 *   x      bf16 [M, H]           the (already normalised) layer input
 *   Wg     bf16 [E, H]
 *   w1, w3 bf16 [E, I, H]        gate and up projections of routed experts
 *   w2     bf16 [E, H, I]        down projections
 *   MXFP4 routed experts (wfmt = 1): w1, w3 u8 [E, I, H/2], s1, s3 u8
 *     [E, I, H/32]; w2 u8 [E, H, I/2], s2 u8 [E, H, I/32]. Codes are e2m1,
 *     element 2j in the low nibble of byte j; scales are e8m0 (2^(s-127)),
 *     one per 32 consecutive elements of a row.
 *   FP8 routed experts (wfmt = 2): w1, w3 u8 [E, I, H], s1, s3 fp32
 *     [E, I, H/128]; w2 u8 [E, H, I], s2 fp32 [E, H, I/128] (the s pointers
 *     of moe_weights then point at fp32 values). Codes are OCP e4m3; a weight
 *     is e4m3(code) * scale, one scale per 128 consecutive elements of a row
 *     ("Chasing the Batch-1 Floor", "Where the time goes now": FP8 block-128
 *     experts; a 128 x 128 tile scale repeats over its 128 rows).
 *   ws1, ws3 bf16 [Is, H]; ws2 bf16 [H, Is]   shared expert (always bf16)
 *   idx    int32 [M, k]  selected experts, by descending logit (ties: lower
 *                        index first)
 *   w      fp32  [M, k]  renormalised routing weights, same order
 *   y      bf16  [M, H]
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */
#define MOE_OK 0
#define MOE_EINVAL (-1)      /* null pointer or unknown flag/option */
#define MOE_ESHAPE (-2)      /* shape outside what the kernels support */
#define MOE_EM (-3)          /* M outside [1, 16] */
#define MOE_EWORKSPACE (-4)  /* workspace missing or smaller than required */
#define MOE_EALIGN (-5)      /* a pointer is not 16-byte aligned */
#define MOE_ECUDA (-6)       /* a CUDA runtime call failed */
#define MOE_ENODEVICE (-7)   /* no usable CUDA device */
#define MOE_ESCRATCH (-8)    /* moe_decode_layer_static_scratch: the shape
                                and M need more than
                                MOE_STATIC_SCRATCH_BYTES of scratch */
/* written by the device into the workspace status word */
#define MOE_EDEVICE_BAD_INDEX (-100) /* moe_ffn got an index outside [0, E);
                                        that (token, slot) was skipped */
#define MOE_ETIMEOUT (-101)          /* a bounded device wait ran out; the
                                        call's outputs are incomplete and the
                                        workspace must be re-initialised:
                                        until then every call on it refuses
                                        to run and reports MOE_ETIMEOUT */

/* flags of moe_decode_layer */
#define MOE_F_NO_PDL 1u                /* launch without programmatic
                                          dependent launch */
#define MOE_F_RESET_SCRATCH 2u         /* moe_decode_layer_static_scratch
                                          only: zero the static scratch
                                          before the launch */
#define MOE_F_DEBUG_FORCE_TIMEOUT 256u /* test hook: the routing step waits
                                          for router logits of a call that
                                          never comes, so the wait runs out
                                          and reports MOE_ETIMEOUT */

/* options of moe_set_option */
#define MOE_OPT_GRID_CTAS 1       /* CTAs of the persistent grid; 0 = one per
                                     SM (default). Values above the SM count
                                     are rejected. */
#define MOE_OPT_WAIT_TIMEOUT_NS 2 /* budget of each bounded device wait in
                                     ns (default 1e9) */
#define MOE_OPT_TRACE_BUFFER 3    /* diagnostic: device address of a uint64
                                     buffer of at least 16 x (grid CTAs)
                                     entries; each CTA writes the global timer
                                     (ns) at its phase boundaries into its 16
                                     entries. 0 (default) disables it. */

typedef struct moe_shape {
    int32_t hidden;       /* H: multiple of 256 (bf16) or 512 (MXFP4, FP8), <= 8192 */
    int32_t n_experts;    /* E: 1..1024 */
    int32_t top_k;        /* k: 1..min(16, E) */
    int32_t inter;        /* I: multiple of 64 (FP8: 128), at most 4096 */
    int32_t shared_inter; /* Is: 0 (no shared expert) or a multiple of 64, <= 4096 */
    int32_t wfmt;         /* routed expert weights: 0 = bf16, 1 = MXFP4, 2 = FP8 e4m3 */
    /* router configuration ("Chasing the Batch-1 Floor", "PDL: stacking the
     * latency floors of small kernels": the top-k step reads a selection
     * bias). Zero-initialised fields give the plain softmax router. */
    int32_t scoring;          /* 0: softmax over all E; 1: sigmoid of each logit */
    float routed_scale;       /* routing weights are multiplied by this (<= 0: 1) */
    const float* router_bias; /* NULL, or fp32 [E] (device) added to the scores
                                 to select the top k only; the weights use
                                 the unbiased scores, renormalised */
    /* layer input and output ("PDL: stacking the latency floors of small
     * kernels": the router chain starts with the norm; the residual add
     * closes the layer). Zero-initialised fields: x is taken as given. */
    const void* norm_weight;  /* NULL, or bf16 [H] (device, 16-byte aligned):
                                 the input is the residual stream h and the
                                 layer runs on x = bf16(h / sqrt(mean(h^2) +
                                 eps) * norm_weight) */
    float norm_eps;           /* RMSNorm epsilon (<= 0: 1e-6) */
    int32_t residual;         /* 1: y = input + MoE(x), added in fp32 before
                                 the single bf16 cast (moe_ffn and
                                 moe_decode_layer) */
} moe_shape;

typedef struct moe_weights {
    const void* w1;     /* routed gate projection  (device) */
    const void* w3;     /* routed up projection    (device) */
    const void* w2;     /* routed down projection  (device) */
    const uint8_t* s1;  /* MXFP4 (u8) or FP8 (fp32) scales of w1, w3, w2; NULL for bf16 */
    const uint8_t* s3;
    const uint8_t* s2;
    const void* ws1;    /* shared expert, bf16; NULL when Is == 0 */
    const void* ws3;
    const void* ws2;
    /* Optional copies of the down projections transposed: w2t bf16 [E, I, H]
     * (w2t[e, i, :] = w2[e, :, i]) and ws2t bf16 [Is, H] (NULL when Is == 0),
     * made once at weight load with moe_transpose_down. When both are given
     * (bf16 experts, H <= 5376), one-token moe_decode_layer calls split the down
     * projection along I: the CTA that computes rows i of an expert's SwiGLU
     * activation also streams rows i of w2t and keeps a partial output, and
     * one fixed-order sum of the partials closes the layer, so no grid
     * barrier separates the gate/up and down projections ("Chasing the
     * Batch-1 Floor", "Two fusions and a retune": expert weights re-laid
     * once at load time for the decode kernel). Other calls ignore them. */
    const void* w2t;
    const void* ws2t;
} moe_weights;

/* Bytes of workspace a call with this shape and M needs. 0 for a shape or M
 * the library rejects. At M = 1 this includes the split-K layer's partial
 * outputs (MOE_MAX_GRID x H fp32). */
#define MOE_MAX_GRID 256
size_t moe_workspace_bytes(const moe_shape* shape, int M);

/* Zeroes the whole workspace (device, ws_bytes) on `stream`; needed once
 * before the first call and after a call reported MOE_ETIMEOUT. */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Router alone: logits = x Wg^T in fp32, softmax, top-k, renormalised
 * weights. x bf16 [M,H], Wg bf16 [E,H] (device); idx int32 [M,k] and
 * w fp32 [M,k] (device) receive the routing. */
int moe_route(const void* x, int M, const void* Wg, const moe_shape* shape,
              int32_t* idx, float* w, void* ws, size_t ws_bytes, void* stream);

/* Expert FFN with the routing given: y = sum_j w[t,j] E_{idx[t,j]}(x_t)
 * + E_shared(x_t), gate/up + SwiGLU + down + combine; each touched expert's
 * weights are read from HBM once whatever M is. idx/w (device) as returned
 * by moe_route; an idx entry may repeat within a token (its weights then
 * add). An entry outside [0, E) is skipped and reported through the status
 * word. y bf16 [M,H] (device). */
int moe_ffn(const void* x, int M, const int32_t* idx, const float* w,
            const moe_weights* weights, const moe_shape* shape, void* y,
            void* ws, size_t ws_bytes, void* stream);

/* The whole layer in one persistent launch: router, top-k, gate/up +
 * SwiGLU, down + combine, shared expert. idx_out / w_out (device) may be
 * NULL. y bf16 [M,H] (device). flags: MOE_F_*. The result is deterministic:
 * every output element is accumulated in a fixed order, so it does not
 * depend on scheduling, PDL or the run. */
int moe_decode_layer(const void* x, int M, const void* Wg,
                     const moe_weights* weights, const moe_shape* shape,
                     int32_t* idx_out, float* w_out, void* y, void* ws,
                     size_t ws_bytes, uint32_t flags, void* stream);

/* Size of the library's static device scratch (512 KiB: a Ling-3.0-flash
 * shaped layer needs 255 KiB at M = 16). */
#define MOE_STATIC_SCRATCH_BYTES 524288u

/* moe_decode_layer without a caller workspace. The papers the library
 * follows have no counterpart of this entry point: it serves callers that
 * cannot hand over a workspace. The same kernel, launch configuration and
 * arithmetic as moe_decode_layer (so the same outputs, bit for bit), but the
 * workspace is a fixed array of MOE_STATIC_SCRATCH_BYTES in the library's
 * own device memory (one per device, created when the module loads). The
 * call allocates and frees nothing. Every call looks the array's device
 * address up again (cudaGetSymbolAddress, which allocates nothing); the
 * first call on a device, and the first after a device reset moved the
 * array, zeroes it on `stream`.
 *  - Returns MOE_ESCRATCH, before touching the device, when the shape and M
 *    need more than MOE_STATIC_SCRATCH_BYTES of workspace
 *    (moe_workspace_bytes > MOE_STATIC_SCRATCH_BYTES).
 *  - All calls on a device share the one scratch: they must be ordered on
 *    one stream (or otherwise serialised), also against other threads.
 *  - flags: MOE_F_NO_PDL, MOE_F_DEBUG_FORCE_TIMEOUT, MOE_F_RESET_SCRATCH
 *    (zeroes the scratch before the launch).
 *  - The transposed down projections (w2t, ws2t) are not used: one-token
 *    calls take the same path as moe_decode_layer without them.
 *  - Failure detection: the device status word lives in the scratch; read it
 *    with moe_static_scratch_status. After MOE_ETIMEOUT every later call
 *    refuses to run (it reports MOE_ETIMEOUT again and leaves its outputs
 *    unwritten) until one is made with MOE_F_RESET_SCRATCH.
 * Other arguments, layouts and errors as moe_decode_layer. */
int moe_decode_layer_static_scratch(const void* x, int M, const void* Wg,
                                    const moe_weights* weights,
                                    const moe_shape* shape, int32_t* idx_out,
                                    float* w_out, void* y, uint32_t flags,
                                    void* stream);

/* Synchronises `stream`, then copies the device status word of this
 * device's static scratch (moe_decode_layer_static_scratch) to *dev_status:
 * MOE_OK or a device code. Allocates nothing; not for the hot path. */
int moe_static_scratch_status(void* stream, int32_t* dev_status);

/* ------------------------------------------------------------ output layer
 * Output layer (lm_head) GEMV for M = 1..16 tokens: logits fp32 [M, V] =
 * x bf16 [M, H] . W^T. "Chasing the Batch-1 Floor: Ling-3.0-flash
 * Speculative Decode on Blackwell", "bf16 router gate and lm_head"; "3 ways
 * to boost MoE inference on NVIDIA DGX Spark", "Optimization 2: Online FP8
 * LM head quantization" (157,184 x 2,560 for the model).
 *  wfmt 0: W bf16 [V, H] (H a multiple of 8), w_scale unused (may be NULL).
 *  wfmt 2: W FP8 e4m3 codes [V, H] (H a multiple of 16) and w_scale fp32 [V],
 *          one scale per row: W[v, h] = e4m3(code) * w_scale[v] (see
 *          moe_fp8_quantize with block = H). Activations stay bf16.
 * H <= 8192. Every weight byte is read once per call. ws: a device buffer of
 * at least MOE_LM_HEAD_WORKSPACE_BYTES (status word; zero it once with
 * moe_workspace_init; moe_read_status reads it). flags: MOE_F_NO_PDL. One
 * launch; errors as for the layer calls. */
#define MOE_LM_HEAD_WORKSPACE_BYTES 1024u
int moe_lm_head(const void* x, int M, const void* W, const float* w_scale,
                int V, int H, int wfmt, float* logits, void* ws,
                size_t ws_bytes, uint32_t flags, void* stream);

/* FP8 e4m3 quantisation of bf16 rows [rows, K] with one fp32 scale per
 * block of `block` consecutive elements of a row (block a multiple of 32
 * dividing K): scale = amax(block) / 448 (1 for an all-zero block), code =
 * the e4m3 value nearest to w / scale (ties to even, saturating). codes u8
 * [rows, K], scales fp32 [rows, K / block] (all device). Not on the hot
 * path: it prepares weights for moe_lm_head. */
int moe_fp8_quantize(const void* w, int64_t rows, int K, int block,
                     uint8_t* codes, float* scales, void* stream);

/* Decodes e4m3 rows with the kernels' conversion: out fp32 [rows, K] =
 * e4m3(code) * scale[row, col / block] (all device). */
int moe_fp8_dequant(const uint8_t* codes, const float* scales, int64_t rows,
                    int K, int block, float* out, void* stream);

/* Transposed copy of down projections for the split-K one-token layer:
 * w2 bf16 [n, H, I] -> w2t bf16 [n, I, H] with w2t[e, i, h] = w2[e, h, i]
 * (n = E for the routed experts, n = 1 and I = Is for the shared expert).
 * Both device, not overlapping. Not on the hot path: run it once when the
 * weights are loaded. */
int moe_transpose_down(const void* w2, int64_t n, int H, int I, void* w2t,
                       void* stream);

/* Synchronises `stream`, then copies the device status word of `ws` to
 * *dev_status (MOE_OK or a device code above). Not for the hot path. */
int moe_read_status(const void* ws, void* stream, int32_t* dev_status);

/* Static description of a MOE_* code. */
const char* moe_status_str(int code);

/* Dequantises MXFP4 rows with the decode the kernels use: out fp32
 * [rows, K] = e2m1(code) * 2^(scale - 127). codes u8 [rows, K/2], scales
 * u8 [rows, K/32], out (all device); K a multiple of 32. */
int moe_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales,
                      int64_t rows, int K, float* out, void* stream);

/* Process-wide tuning and test options (MOE_OPT_*). Not thread-safe with
 * concurrent calls. */
int moe_set_option(int option, int64_t value);

/* Number of kernel launches the most recent launching call on this thread
 * made (1 for moe_decode_layer / moe_route / moe_ffn). */
int moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DECODE_H */
