// Inline-PTX helpers for sm_103a: mbarriers, bulk (TMA) copies, programmatic
// dependent launch, proxy fences, bounded waits, bf16 unpacking.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace moe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- bulk copies
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared bulk copy completing `bytes` of transaction count on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy view of global memory before
// its later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- sync
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Relaxed GPU-scope 32-bit load: a control word written by an earlier launch
// that has finished (the dependency wait makes its value visible). Unlike an
// acquire, it does not hold back the loads that follow it.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Relaxed GPU-scope 32-bit store and 4 x 32-bit load (each 32-bit element of
// the vector is single-copy atomic), and a relaxed reduction (an arrival
// count that nobody waits on at once).
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4u32(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void red_add_relaxed_gpu(unsigned* p, unsigned v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Release store / acquire load of a 32-bit word at CTA scope (a flag in
// shared memory that one warp publishes and another polls).
__device__ __forceinline__ void st_release_cta(int* p, int v) {
    asm volatile("st.release.cta.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Relaxed GPU-scope 64-bit store and paired 64-bit load. Each aligned
// 64-bit word is single-copy atomic: a reader sees it whole, old or new.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// The same eight values as four (even, odd) pairs, the operand shape of the
// paired fp32 FMA.
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
    return make_float2(bf16lo(w), bf16hi(w));
}
__device__ __forceinline__ void unpack8x2(const uint4 v, float2 (&f)[4]) {
    f[0] = bf16x2_to_f32x2(v.x);
    f[1] = bf16x2_to_f32x2(v.y);
    f[2] = bf16x2_to_f32x2(v.z);
    f[3] = bf16x2_to_f32x2(v.w);
}
// lo += w.lo * x.lo, hi += w.hi * x.hi for bf16 pairs w, x, in fp32 with
// one rounding each (the mixed-precision fma: bf16 operands, fp32 addend).
__device__ __forceinline__ void fma_bf16x2(uint32_t w, uint32_t x, float& lo, float& hi) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w), "r"(x));
}
// The same with f16 pairs (fma.rn.f32.f16).
__device__ __forceinline__ void fma_f16x2(uint32_t w, uint32_t x, float& lo, float& hi) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\tfma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w), "r"(x));
}
// d = a * b + c on both halves, each rounded once (fma.rn.f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

// ---------------------------------------------------------------- tensor cores
// ldmatrix: four (x4) or two (x2) 8 x 8 tiles of 16-bit elements from shared
// memory; lanes 8i..8i+7 give the row addresses (16 bytes each) of tile i.
// Thread l receives row l / 4, elements 2 (l % 4) and 2 (l % 4) + 1 of each
// tile, in register i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
// d += a . b for a 16 x 16 (row-major) bf16 tile a and a 16 x 8 (column-major)
// bf16 tile b, fp32 accumulate (mma.sync m16n8k16). Thread l holds d rows
// l / 4 (d[0], d[1]) and l / 4 + 8 (d[2], d[3]), columns 2 (l % 4) and
// 2 (l % 4) + 1.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---------------------------------------------------------------- MXFP4
// Eight e2m1 codes (one 32-bit word; element 2j in the low nibble of byte j)
// to four f16 pairs with the hardware conversion: w[j] holds elements 2j (low
// half) and 2j + 1 (high half). Every e2m1 value is exact in f16.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t v, uint32_t (&w)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "r"(v));
}

// ---------------------------------------------------------------- f16x2
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                        *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ float2 f16x2_to_f32(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
// (lo, hi) rounded to nearest into one f16 pair (lo in the low half).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// 2^e as an fp32 for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
// Power-of-two exponent s such that mx * 2^s lies in [128, 256) (mx > 0
// normal), clamped to [-100, 100]; 0 for mx == 0.
__device__ __forceinline__ int f16_range_shift(float mx) {
    if (!(mx > 0.f)) return 0;
    const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
    return max(-100, min(100, 7 - e));
}

// ---------------------------------------------------------------- FP8 e4m3
// Four e4m3 codes (one 32-bit word; element j in byte j) to two f16 pairs
// with the hardware conversion: lo holds elements 0, 1 and hi elements 2, 3
// (every e4m3 value is exact in f16).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(v));
}

// Sixteen e4m3 codes (one uint4) as eight f16 pairs: w[j] holds codes 2j
// (low half) and 2j + 1. Every e4m3 value is exact in f16.
__device__ __forceinline__ void e4m3x16_to_f16x2(const uint4 c, uint32_t (&w)[8]) {
    e4m3x4_to_f16x2(c.x, w[0], w[1]);
    e4m3x4_to_f16x2(c.y, w[2], w[3]);
    e4m3x4_to_f16x2(c.z, w[4], w[5]);
    e4m3x4_to_f16x2(c.w, w[6], w[7]);
}

// Sixteen e4m3 codes (one uint4) as eight fp32 (even, odd) pairs.
__device__ __forceinline__ void unpack16_e4m3x2(const uint4 c, float2 (&f)[8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t lo, hi;
        e4m3x4_to_f16x2(w[k], lo, hi);
        f[2 * k] = f16x2_to_f32(lo);
        f[2 * k + 1] = f16x2_to_f32(hi);
    }
}

// 2^(s-127) for an e8m0 byte s (s = 0 is the subnormal 2^-127; s = 255 NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
    if (s == 255u) return __uint_as_float(0x7fc00000u);
    return s ? __uint_as_float(s << 23) : __uint_as_float(1u << 22);
}

}  // namespace moe
