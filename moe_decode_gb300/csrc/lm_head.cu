// Output layer (lm_head) for batch-1 decode and speculative verify:
// logits[t, v] = x_t . W[v] for M <= 16 tokens over a V x H weight matrix,
// bf16 or FP8 e4m3 with one scale per row, and the FP8 quantiser and decode
// that go with it.
//
// "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative Decode on
// Blackwell", section "bf16 router gate and lm_head" (the output GEMV is
// weight-bandwidth bound at batch 1); "3 ways to boost MoE inference on
// NVIDIA DGX Spark", "Optimization 2: Online FP8 LM head quantization" (the
// 157,184 x 2,560 vocabulary matrix stored in FP8 to halve its reads).
//
// A persistent kernel, one CTA per SM: CTA c owns the rows [cV/G, (c+1)V/G)
// and streams them once, in 32 KB bulk copies, through a ring of shared
// memory stages (one producer lane, full/empty mbarriers); each consumer
// warp takes whole rows against all M tokens. Every wait is bounded; a wait
// that runs out sets MOE_ETIMEOUT in the status word and the CTA stops.
#include "launch.h"
#include "layer_params.h"
#include "lm_params.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr uint32_t LSB = kStageBytes;

__device__ __forceinline__ bool lm_aborted(const volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ void lm_abort(const LmParams& p, volatile int* flag) {
    atomicCAS(reinterpret_cast<int*>(p.ctrl + kCtlStatus), 0, -101 /* MOE_ETIMEOUT */);
    *flag = 1;
}

__device__ __forceinline__ bool lm_wait(uint32_t bar, uint32_t parity, const LmParams& p, volatile int* flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (lm_aborted(flag)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            lm_abort(p, flag);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ float lm_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float lm_warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// acc[t] = row . x_t over H elements; this lane takes 16-byte weight vectors
// lane, lane + 32, ... (bf16: 8 elements, e4m3: 16 elements per vector).
template <int WT, int NT>
__device__ __forceinline__ void lm_dot(const uint4* __restrict__ row, const uint4* __restrict__ x0,
                                       const uint4* __restrict__ x1, int H, int lane, float (&acc)[NT]) {
    // partial sums p0..p3 (element e to p[e mod 4]) held as two (even, odd)
    // pairs, each element through the mixed-precision fma (16-bit operands,
    // fp32 addend, one rounding)
    float2 pa[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) pa[t][0] = pa[t][1] = make_float2(0.f, 0.f);
    if (WT == 0) {
        const int nvec = H / 8;
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) {
            const uint4 w = row[v];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 x = (t == 0 ? x0 : x1)[v];
                const uint32_t xx[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) fma_bf16x2(ww[e], xx[e], pa[t][e & 1].x, pa[t][e & 1].y);
            }
        }
    } else {
        // e4m3 codes as f16 pairs against the f16 tokens (held times 2^s_t,
        // vector pairs swizzled: vector 2v + b of a token row sits at
        // 2v + (b ^ ((v >> 2) & 1))), through the mixed-precision fma;
        // every product is exact
        const int nvec = H / 16;
#pragma unroll 2
        for (int v = lane; v < nvec; v += 32) {
            uint32_t w[8];
            e4m3x16_to_f16x2(row[v], w);
            const int sw = (v >> 2) & 1;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4* xt = t == 0 ? x0 : x1;
                const uint4 xa = xt[2 * v + sw], xb = xt[2 * v + (1 ^ sw)];
                const uint32_t xx[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    fma_f16x2(w[e], xx[e], pa[t][e & 1].x, pa[t][e & 1].y);
                    fma_f16x2(w[4 + e], xx[4 + e], pa[t][e & 1].x, pa[t][e & 1].y);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = (pa[t][0].x + pa[t][0].y) + (pa[t][1].x + pa[t][1].y);
}

// MMA (bf16 rows, M >= kLmMmaMinTokens): each stage's rows (at most eight,
// copied one per row at a pitch of their bytes + 16, so that ldmatrix reads
// of eight rows hit eight bank groups) go to one warp, round-robin, which
// computes them against all tokens on the tensor cores: the tokens (token
// rows H + 8 elements apart) are the 16-row operand of mma.sync m16n8k16,
// the rows the 8 columns, K = H with two accumulators.
template <int WT, bool MMA>
__global__ void __launch_bounds__(kLmThreads, 1) lm_head_kernel(const __grid_constant__ LmParams p) {
    constexpr int NCW = kLmConsumerWarps;
    constexpr int NCT = NCW * 32;
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bars = smem_u32(smem + p.off_bar);
    volatile int* flag = reinterpret_cast<volatile int*>(smem + p.off_bar + 2 * p.ns * 8);
    float* x_inv = reinterpret_cast<float*>(smem + p.off_bar + 128);  // FP8: 2^-s_t per token
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + p.off_x);
    if (tid == 0) {
        for (int i = 0; i < p.ns; ++i) {
            mbar_init(bars + i * 8, 1);
            mbar_init(bars + (p.ns + i) * 8, NCW);
        }
        *flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int c = (int)blockIdx.x;
    const int v0 = (int)((int64_t)c * p.V / p.G), v1 = (int)((int64_t)(c + 1) * p.V / p.G);
    const uint32_t rowbytes = (uint32_t)p.H * (WT == 0 ? 2u : 1u);
    const uint32_t pitch = MMA ? rowbytes + 16u : rowbytes;  // row pitch in a stage
    const int cap = MMA ? min(8, (int)(LSB / pitch)) : (int)(LSB / rowbytes);
    const int xpv = MMA ? p.H / 8 + 1 : p.H / 8;  // token row pitch in 16-byte vectors
    const uint32_t base = smem_u32(smem);

    if (warp == NCW) {
        if (lane == 0) {
            // the weights depend on no earlier launch: stream them at once
            const uint64_t pol = policy_evict_first();
            uint32_t n = 0, s = 0, ph = 0;
            bool ok = true;
            for (int r = v0; r < v1 && ok; r += cap, ++n) {
                const int nr = min(cap, v1 - r);
                if (n >= (uint32_t)p.ns) ok = lm_wait(bars + (p.ns + s) * 8, ph ^ 1u, p, flag);
                if (!ok) break;
                const uint32_t b = (uint32_t)nr * rowbytes;
                mbar_arrive_expect_tx(bars + s * 8, b);
                if (MMA) {
                    for (int j = 0; j < nr; ++j)
                        bulk_g2s(base + s * LSB + (uint32_t)j * pitch, p.W + (size_t)(r + j) * rowbytes, rowbytes,
                                 bars + s * 8, pol);
                } else {
                    bulk_g2s(base + s * LSB, p.W + (size_t)r * rowbytes, b, bars + s * 8, pol);
                }
                if (++s == (uint32_t)p.ns) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                const uint32_t lo = n > (uint32_t)p.ns ? n - p.ns : 0;
                for (uint32_t i = lo; i < n; ++i) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bars + (i % p.ns) * 8, (i / p.ns) & 1u))
                        if (global_timer_ns() - t0 > p.timeout_ns) break;
                }
            }
        }
    } else {
        pdl_wait();
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.x);
            uint4* dst = reinterpret_cast<uint4*>(xs);
            if (WT == 0) {
                const int nv = p.M * p.H / 8, nvt = p.H / 8;
                for (int i = tid; i < nv; i += NCT) dst[i + (i / nvt) * (xpv - nvt)] = __ldg(src + i);
            } else {
                // FP8 rows: tokens in f16 times 2^s_t, s_t chosen from the
                // token's largest magnitude (exact for bf16 values in f16's
                // normal range), one warp per token
                const int nvt = p.H / 8;
                for (int t = warp; t < p.M; t += NCW) {
                    float mx = 0.f;
                    for (int i = lane; i < nvt; i += 32) {
                        float f[8];
                        unpack8(__ldg(src + (size_t)t * nvt + i), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(f[e]));
                    }
                    mx = lm_warp_max(mx);
                    const int sh = f16_range_shift(mx);
                    const float sc = exp2i(sh);
                    for (int i = lane; i < nvt; i += 32) {
                        float f[8];
                        unpack8(__ldg(src + (size_t)t * nvt + i), f);
                        uint4 v;
                        v.x = f32x2_to_f16x2(f[0] * sc, f[1] * sc);
                        v.y = f32x2_to_f16x2(f[2] * sc, f[3] * sc);
                        v.z = f32x2_to_f16x2(f[4] * sc, f[5] * sc);
                        v.w = f32x2_to_f16x2(f[6] * sc, f[7] * sc);
                        dst[(size_t)t * nvt + (i ^ ((i >> 3) & 1))] = v;
                    }
                    if (lane == 0) x_inv[t] = exp2i(-sh);
                }
            }
        }
        named_bar_sync(1, NCT);
        uint32_t s = 0, ph = 0;
        int qm = 0;  // rows go round-robin over the warps: running row count mod NCW
        const int nvx = p.H / 8;
        for (int r = v0; r < v1; r += cap) {
            const int nr = min(cap, v1 - r);
            if (!lm_wait(bars + s * 8, ph, p, flag)) break;
            if (MMA) {
                // the stage goes to one warp (round-robin over the stages)
                if (warp == qm) {
                    const uint32_t sb = base + s * LSB;
                    const uint32_t baddr = sb + (uint32_t)min(lane & 7, nr - 1) * pitch + ((lane >> 3) & 1) * 16u;
                    const int qa = (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t arow =
                        smem_u32(xs) + (uint32_t)(qa < p.M ? qa : 0) * xpv * 16u + (uint32_t)(lane >> 4) * 16u;
                    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                    const int nks = p.H / 16;
                    int ks = 0;
#pragma unroll 4
                    for (; ks + 1 < nks; ks += 2) {
                        uint32_t a[4], b[2], a2[4], b2[2];
                        ldsm_x4(arow + (uint32_t)ks * 32u, a);
                        ldsm_x2(baddr + (uint32_t)ks * 32u, b);
                        ldsm_x4(arow + (uint32_t)ks * 32u + 32u, a2);
                        ldsm_x2(baddr + (uint32_t)ks * 32u + 32u, b2);
                        mma_bf16_16816(d0, a, b);
                        mma_bf16_16816(d1, a2, b2);
                    }
                    if (ks < nks) {
                        uint32_t a[4], b[2];
                        ldsm_x4(arow + (uint32_t)ks * 32u, a);
                        ldsm_x2(baddr + (uint32_t)ks * 32u, b);
                        mma_bf16_16816(d0, a, b);
                    }
                    // lane (g, t): tokens g and g + 8, rows 2t and 2t + 1
                    const int g = lane >> 2, t = lane & 3;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int q = g + 8 * half;
                        if (q >= p.M) continue;
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc)
                            if (2 * t + cc < nr)
                                p.logits[(size_t)q * p.V + r + 2 * t + cc] = d0[2 * half + cc] + d1[2 * half + cc];
                    }
                }
                qm = qm + 1 == NCW ? 0 : qm + 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + (p.ns + s) * 8);
                if (++s == (uint32_t)p.ns) {
                    s = 0;
                    ph ^= 1u;
                }
                continue;
            }
            const uint8_t* st = reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(base + s * LSB));
            const int j0 = warp >= qm ? warp - qm : warp - qm + NCW;  // first row of this warp
            qm = (qm + nr) % NCW;
            for (int j = j0; j < nr; j += NCW) {
                const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)j * rowbytes);
                const float sc = WT == 0 ? 1.f : __ldg(p.scale + r + j);
                int t = 0;
                for (; t + 2 <= p.M; t += 2) {
                    float acc[2];
                    const uint4* xa = reinterpret_cast<const uint4*>(xs) + (size_t)t * nvx;
                    lm_dot<WT, 2>(row, xa, xa + nvx, p.H, lane, acc);
                    acc[0] = lm_warp_sum(acc[0]);
                    acc[1] = lm_warp_sum(acc[1]);
                    if (WT != 0) acc[0] *= x_inv[t], acc[1] *= x_inv[t + 1];
                    if (lane == 0) {
                        p.logits[(size_t)t * p.V + r + j] = acc[0] * sc;
                        p.logits[(size_t)(t + 1) * p.V + r + j] = acc[1] * sc;
                    }
                }
                if (t < p.M) {
                    float acc[1];
                    const uint4* xa = reinterpret_cast<const uint4*>(xs) + (size_t)t * nvx;
                    lm_dot<WT, 1>(row, xa, xa, p.H, lane, acc);
                    acc[0] = lm_warp_sum(acc[0]);
                    if (WT != 0) acc[0] *= x_inv[t];
                    if (lane == 0) p.logits[(size_t)t * p.V + r + j] = acc[0] * sc;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + (p.ns + s) * 8);
            if (++s == (uint32_t)p.ns) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
}

// e4m3 quantisation of bf16 rows: one warp per (row, block); scale =
// amax / 448 in fp32 (1 for an all-zero block), code = nearest e4m3 to
// w / scale (ties to even, saturating), by the hardware conversion.
__global__ void fp8_quantize_kernel(const uint16_t* __restrict__ w, int64_t rows, int K, int block,
                                    uint8_t* __restrict__ codes, float* __restrict__ scales) {
    const int nb = K / block;
    const int64_t units = rows * nb;
    const int lane = threadIdx.x & 31;
    for (int64_t u = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; u < units;
         u += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t r = u / nb;
        const int b = (int)(u - r * nb);
        const uint16_t* src = w + r * K + (int64_t)b * block;
        float amax = 0.f;
        for (int i = lane; i < block; i += 32) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)src[i] << 16)));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        if (lane == 0) scales[u] = sc;
        uint8_t* dst = codes + r * K + (int64_t)b * block;
        for (int i = 2 * lane; i < block; i += 64) {
            const float a = __uint_as_float((uint32_t)src[i] << 16) / sc;
            const float bb = __uint_as_float((uint32_t)src[i + 1] << 16) / sc;
            uint16_t pr;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(bb), "f"(a));
            *reinterpret_cast<uint16_t*>(dst + i) = pr;
        }
    }
}

// e4m3 decode with the kernels' conversion: out = e4m3(code) * scale.
__global__ void fp8_dequant_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                                   int64_t rows, int K, int block, float* __restrict__ out) {
    const int64_t n = rows * (int64_t)K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / K;
        const int col = (int)(i - r * K);
        uint32_t lo, hi;
        e4m3x4_to_f16x2(codes[i], lo, hi);
        out[i] = f16x2_to_f32(lo).x * scales[r * (K / block) + col / block];
    }
}

}  // namespace

cudaError_t launch_lm_head(const LmParams& p, int wt, cudaStream_t stream, bool pdl) {
    void (*kern)(LmParams) = wt != 0                  ? lm_head_kernel<2, false>
                             : lm_uses_mma(p.M, p.H, wt) ? lm_head_kernel<0, true>
                                                         : lm_head_kernel<0, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G);
    cfg.blockDim = dim3(kLmThreads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_fp8_quantize(const uint16_t* w, int64_t rows, int K, int block, uint8_t* codes, float* scales,
                                cudaStream_t stream) {
    const int64_t units = rows * (K / block);
    if (units == 0) return cudaSuccess;
    int blocks = (int)((units * 32 + 255) / 256);
    if (blocks > 8192) blocks = 8192;
    fp8_quantize_kernel<<<blocks, 256, 0, stream>>>(w, rows, K, block, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_fp8_dequant(const uint8_t* codes, const float* scales, int64_t rows, int K, int block, float* out,
                               cudaStream_t stream) {
    const int64_t n = rows * (int64_t)K;
    if (n == 0) return cudaSuccess;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    fp8_dequant_kernel<<<blocks, 256, 0, stream>>>(codes, scales, rows, K, block, out);
    return cudaGetLastError();
}

}  // namespace moe
