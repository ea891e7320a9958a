// Persistent fused small-M MoE decode layer for sm_103a.
//
// One CTA per SM. Each CTA runs one producer warp, whose elected lane streams
// weight tiles from HBM into a ring of shared-memory stages with bulk (TMA)
// copies completing on mbarriers, and eight consumer warps that compute from
// the ring. The layer runs in three phases separated by two bounded grid
// barriers:
//
//   phase 0  router gate matvec: CTA c owns router rows [cE/G, (c+1)E/G);
//            logits go to the workspace.              -> grid barrier 1
//            Every CTA then computes softmax / top-k / renormalisation for
//            all M tokens and builds the expert plan (distinct experts and
//            their token lists) in shared memory.
//   phase 1  gate/up + SwiGLU: the intermediate rows of the shared expert and
//            of every touched routed expert are split evenly over the CTAs;
//            h = silu(W1 x) * (W3 x) goes to the workspace in bf16.
//                                                       -> grid barrier 2
//   phase 2  down projection + weighted combine: CTA c owns output rows
//            [cH/G, (c+1)H/G) and accumulates, in a fixed order (shared
//            expert, then routed experts by ascending id, tokens ascending),
//            w * (W2 h) into fp32, then casts y to bf16 once.
//
// Every weight byte of a touched expert is read from HBM exactly once per
// call, whatever M is. The producer never waits on a grid barrier for weight
// tiles: it issues the shared expert's tiles before the router finishes, and
// the phase-2 weight tiles before barrier 2 completes (the activations part
// of those stages is fetched once the barrier has passed), so the barriers
// overlap the weight stream.
//
// Page references: "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative
// Decode on Blackwell", sections "PDL: stacking the latency floors of small
// kernels" (producer-independent loads before the dependency wait; fp32
// combine with a single final cast), "Two fusions and a retune" (SwiGLU fused
// into the up-GEMM; a single-launch, pair-axis token/expert grouping whose
// cost does not scale with the expert count) and "bf16 router gate and
// lm_head"; "3 ways to boost MoE inference on NVIDIA DGX Spark",
// "Optimization 1" (MXFP4 expert weights).
#pragma once
#include "layer_params.h"
#include "ptx.cuh"

namespace moe {

constexpr int NCW = kConsumerWarps;
constexpr int NCT = kConsumerThreads;
constexpr uint32_t SB = kStageBytes;
constexpr int TG = 4;  // tokens (pairs) per register group

// A unit of the ring: the tiles one stage holds.
struct Chunk {
    int kind;   // 0 router rows, 1 gate/up rows, 2 down rows
    int slot;   // -1 shared expert, else routed slot
    int r0, n;  // first row and row count
    int p0, np; // down: pair range within the slot
};

struct Ctx {
    const LayerParams& p;
    int c;  // CTA index
    const Plan* plan;
};

__device__ __forceinline__ int slot_expert(const Ctx& x, int s) { return x.plan->slot_e[s]; }

__device__ __forceinline__ int slot_npairs(const Ctx& x, int s) {
    return s < 0 ? x.p.M : x.plan->slot_p0[s + 1] - x.plan->slot_p0[s];
}

// ------------------------------------------------------------ chunk lists
// The producer and the consumers enumerate identical chunk sequences.

template <class F>
__device__ __forceinline__ void for_router_chunks(const Ctx& x, F&& f) {
    const LayerParams& p = x.p;
    int e0 = (int)((long long)x.c * p.E / p.G), e1 = (int)((long long)(x.c + 1) * p.E / p.G);
    int cap = (int)(SB / (uint32_t)(p.H * 2));
    for (int r = e0; r < e1; r += cap) f(Chunk{0, -1, r, min(cap, e1 - r), 0, 0});
}

template <int WFMT>
__device__ __forceinline__ int gateup_cap(const LayerParams& p, bool routed) {
    uint32_t pair = (WFMT == 1 && routed) ? (uint32_t)(2 * (p.H / 2 + p.H / 32)) : (uint32_t)(4 * p.H);
    return (int)(SB / pair);
}

template <int WFMT, class F>
__device__ __forceinline__ void for_shared_gateup_chunks(const Ctx& x, F&& f) {
    const LayerParams& p = x.p;
    if (p.Is <= 0) return;
    int i0 = (int)((long long)x.c * p.Is / p.G), i1 = (int)((long long)(x.c + 1) * p.Is / p.G);
    int cap = gateup_cap<WFMT>(p, false);
    for (int r = i0; r < i1; r += cap) f(Chunk{1, -1, r, min(cap, i1 - r), 0, 0});
}

template <int WFMT, class F>
__device__ __forceinline__ void for_routed_gateup_chunks(const Ctx& x, F&& f) {
    const LayerParams& p = x.p;
    long long R = (long long)x.plan->nslot * p.I;
    long long r = (long long)x.c * R / p.G, r1 = (long long)(x.c + 1) * R / p.G;
    int cap = gateup_cap<WFMT>(p, true);
    while (r < r1) {
        int s = (int)(r / p.I), i0 = (int)(r % p.I);
        int n = (int)min((long long)cap, min(r1 - r, (long long)(p.I - i0)));
        f(Chunk{1, s, i0, n, 0, 0});
        r += n;
    }
}

template <int WFMT>
__device__ __forceinline__ uint32_t down_rowbytes(const LayerParams& p, int slot) {
    if (slot < 0) return (uint32_t)p.Is * 2;
    return WFMT == 1 ? (uint32_t)(p.I / 2 + p.I / 32) : (uint32_t)p.I * 2;
}

template <int WFMT, class F>
__device__ __forceinline__ void for_down_chunks(const Ctx& x, F&& f) {
    const LayerParams& p = x.p;
    int h0 = (int)((long long)x.c * p.H / p.G), h1 = (int)((long long)(x.c + 1) * p.H / p.G);
    if (h1 <= h0) return;
    for (int s = (p.Is > 0 ? -1 : 0); s < x.plan->nslot; ++s) {
        int inter = s < 0 ? p.Is : p.I;
        uint32_t hrow = (uint32_t)inter * 2;
        uint32_t rowb = down_rowbytes<WFMT>(p, s);
        uint32_t reserve = (WFMT == 1 && s >= 0) ? 32u : 0u;
        int npairs = slot_npairs(x, s);
        int pg = max(1, min(npairs, (int)((SB / 2) / hrow)));
        for (int q0 = 0; q0 < npairs; q0 += pg) {
            int np = min(pg, npairs - q0);
            int cap = (int)((SB - (uint32_t)np * hrow - reserve) / rowb);
            for (int r = h0; r < h1; r += cap) f(Chunk{2, s, r, min(cap, h1 - r), q0, np});
        }
    }
}

// ------------------------------------------------------------ failure paths
__device__ __forceinline__ void raise_status(const LayerParams& p, int code) {
    atomicCAS(reinterpret_cast<int*>(p.ctrl + kCtlStatus), 0, code);
}

static __device__ __noinline__ void set_abort(const LayerParams& p, Plan* plan, int code) {
    raise_status(p, code);
    *reinterpret_cast<volatile int32_t*>(&plan->abort) = 1;
}

__device__ __forceinline__ bool aborted(const Plan* plan) {
    return *reinterpret_cast<const volatile int32_t*>(&plan->abort) != 0;
}

// Bounded mbarrier wait: false when the budget ran out or the CTA aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const LayerParams& p, Plan* plan) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (aborted(plan)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
            return false;
        }
    }
}

// Bounded wait until a grid-barrier counter reaches `target`.
__device__ __forceinline__ bool grid_wait(const unsigned* ctr, unsigned target, const LayerParams& p, Plan* plan) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(ctr) < target) {
        if (aborted(plan)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// ------------------------------------------------------------ producer
struct Ring {
    uint32_t base;  // shared address of stage 0
    uint32_t bars;  // full[ns] then empty[ns]
    int ns;
    uint32_t n;     // chunks issued / consumed so far
    __device__ __forceinline__ uint32_t stage(uint32_t i) const { return base + (i % ns) * SB; }
    __device__ __forceinline__ uint32_t full(uint32_t i) const { return bars + (i % ns) * 8; }
    __device__ __forceinline__ uint32_t empty(uint32_t i) const { return bars + (ns + i % ns) * 8; }
    __device__ __forceinline__ uint32_t parity(uint32_t i) const { return (i / ns) & 1u; }
};

struct Pending {
    uint32_t dst, bytes, bar;
    const void* src;
};

template <int WFMT>
struct Producer {
    const Ctx& x;
    Ring ring;
    Plan* plan;
    uint64_t pol_w;    // weights: evict first
    uint64_t pol_h;    // activations: keep
    bool b2_done;
    int npend;
    Pending pend[kMaxStages];
    uint32_t complete_upto;  // chunks whose copies were all issued

    __device__ bool poll_b2(bool block) {
        if (b2_done) return true;
        const unsigned* ctr = x.p.ctrl + kCtlBar2;
        bool ok = block ? grid_wait(ctr, (unsigned)x.p.G, x.p, plan) : (ld_acquire_gpu(ctr) >= (unsigned)x.p.G);
        if (!ok) return false;
        b2_done = true;
        fence_proxy_async_global();
        for (int i = 0; i < npend; ++i) bulk_g2s(pend[i].dst, pend[i].src, pend[i].bytes, pend[i].bar, pol_h);
        npend = 0;
        complete_upto = ring.n;
        return true;
    }

    // Waits for the stage of chunk ring.n to be free. In phase 2 it keeps
    // polling barrier 2 meanwhile, so that deferred activation copies go out
    // as soon as they may.
    __device__ bool acquire(bool phase2) {
        uint32_t i = ring.n;
        if (i < (uint32_t)ring.ns) return true;
        uint32_t bar = ring.empty(i), par = ring.parity(i) ^ 1u;
        if (mbar_try_wait(bar, par)) return true;
        uint64_t t0 = global_timer_ns();
        while (true) {
            if (mbar_try_wait(bar, par)) return true;
            if (aborted(plan)) return false;
            if (phase2) poll_b2(false);
            if (global_timer_ns() - t0 > x.p.timeout_ns) {
                set_abort(x.p, plan, -101);
                return false;
            }
        }
    }

    __device__ bool issue(const Chunk& ch) {
        const LayerParams& p = x.p;
        if (aborted(plan)) return false;
        if (!acquire(ch.kind == 2)) return false;
        uint32_t dst = ring.stage(ring.n), bar = ring.full(ring.n);
        if (ch.kind == 0) {
            uint32_t b = (uint32_t)ch.n * p.H * 2;
            mbar_arrive_expect_tx(bar, b);
            bulk_g2s(dst, p.Wg + (size_t)ch.r0 * p.H, b, bar, pol_w);
        } else if (ch.kind == 1) {
            if (ch.slot < 0 || WFMT == 0) {
                uint32_t b = (uint32_t)ch.n * p.H * 2;
                const uint8_t *a, *c;
                if (ch.slot < 0) {
                    a = reinterpret_cast<const uint8_t*>(p.ws1 + (size_t)ch.r0 * p.H);
                    c = reinterpret_cast<const uint8_t*>(p.ws3 + (size_t)ch.r0 * p.H);
                } else {
                    size_t off = ((size_t)slot_expert(x, ch.slot) * p.I + ch.r0) * p.H * 2;
                    a = p.w1 + off;
                    c = p.w3 + off;
                }
                mbar_arrive_expect_tx(bar, 2 * b);
                bulk_g2s(dst, a, b, bar, pol_w);
                bulk_g2s(dst + b, c, b, bar, pol_w);
            } else {
                uint32_t bc = (uint32_t)ch.n * (p.H / 2), bs = (uint32_t)ch.n * (p.H / 32);
                size_t row = (size_t)slot_expert(x, ch.slot) * p.I + ch.r0;
                mbar_arrive_expect_tx(bar, 2 * bc + 2 * bs);
                bulk_g2s(dst, p.w1 + row * (p.H / 2), bc, bar, pol_w);
                bulk_g2s(dst + bc, p.w3 + row * (p.H / 2), bc, bar, pol_w);
                bulk_g2s(dst + 2 * bc, p.s1 + row * (p.H / 32), bs, bar, pol_w);
                bulk_g2s(dst + 2 * bc + bs, p.s3 + row * (p.H / 32), bs, bar, pol_w);
            }
        } else {
            int inter = ch.slot < 0 ? p.Is : p.I;
            uint32_t hb = (uint32_t)ch.np * inter * 2;
            const void* hsrc;
            uint32_t wbytes;
            if (ch.slot < 0) {
                hsrc = p.hs + (size_t)ch.p0 * p.Is;
                wbytes = (uint32_t)ch.n * p.Is * 2;
                mbar_arrive_expect_tx(bar, hb + wbytes);
                bulk_g2s(dst + hb, p.ws2 + (size_t)ch.r0 * p.Is, wbytes, bar, pol_w);
            } else {
                hsrc = p.hr + (size_t)(x.plan->slot_p0[ch.slot] + ch.p0) * p.I;
                size_t row = (size_t)slot_expert(x, ch.slot) * p.H + ch.r0;
                if (WFMT == 0) {
                    wbytes = (uint32_t)ch.n * p.I * 2;
                    mbar_arrive_expect_tx(bar, hb + wbytes);
                    bulk_g2s(dst + hb, p.w2 + row * p.I * 2, wbytes, bar, pol_w);
                } else {
                    uint32_t bc = (uint32_t)ch.n * (p.I / 2);
                    size_t s0 = row * (p.I / 32), s1 = s0 + (size_t)ch.n * (p.I / 32);
                    size_t w0 = s0 & ~(size_t)15, w1 = (s1 + 15) & ~(size_t)15;
                    uint32_t bs = (uint32_t)(w1 - w0);
                    wbytes = bc + bs;
                    mbar_arrive_expect_tx(bar, hb + wbytes);
                    bulk_g2s(dst + hb, p.w2 + row * (p.I / 2), bc, bar, pol_w);
                    bulk_g2s(dst + hb + bc, p.s2 + w0, bs, bar, pol_w);
                }
            }
            if (b2_done) {
                bulk_g2s(dst, hsrc, hb, bar, pol_h);
            } else {
                pend[npend++] = Pending{dst, hb, bar, hsrc};
                ring.n++;
                return true;
            }
        }
        ring.n++;
        if (npend == 0) complete_upto = ring.n;
        return true;
    }

    // After an abort: wait (bounded) for every copy already issued, so that
    // no bulk copy is still writing this CTA's shared memory at exit.
    __device__ void drain() {
        // Deferred activation copies are issued regardless (their source is
        // valid workspace memory), so that every stage's barrier can complete.
        for (int i = 0; i < npend; ++i) bulk_g2s(pend[i].dst, pend[i].src, pend[i].bytes, pend[i].bar, pol_h);
        npend = 0;
        complete_upto = ring.n;
        uint32_t lo = complete_upto > (uint32_t)ring.ns ? complete_upto - ring.ns : 0;
        for (uint32_t i = lo; i < complete_upto; ++i) {
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(ring.full(i), ring.parity(i))) {
                if (global_timer_ns() - t0 > x.p.timeout_ns) break;
            }
        }
    }
};

// ------------------------------------------------------------ consumer math

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// acc[t] += row . xr[t] over nvec 16-byte vectors (bf16 x 8), lanes strided.
__device__ __forceinline__ void dot_bf16(const uint4* __restrict__ row, const uint4* const* xr, int cnt, int nvec,
                                         int lane, float (&acc)[TG]) {
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        float fw[8];
        unpack8(row[v], fw);
#pragma unroll
        for (int t = 0; t < TG; ++t) {
            if (t < cnt) {
                float fx[8];
                unpack8(xr[t][v], fx);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[t] = fmaf(fw[e], fx[e], acc[t]);
            }
        }
    }
}

// Gate and up rows against the same tokens.
__device__ __forceinline__ void dot2_bf16(const uint4* __restrict__ r1, const uint4* __restrict__ r3,
                                          const uint4* const* xr, int cnt, int nvec, int lane, float (&g)[TG],
                                          float (&u)[TG]) {
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        float f1[8], f3[8];
        unpack8(r1[v], f1);
        unpack8(r3[v], f3);
#pragma unroll
        for (int t = 0; t < TG; ++t) {
            if (t < cnt) {
                float fx[8];
                unpack8(xr[t][v], fx);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    g[t] = fmaf(f1[e], fx[e], g[t]);
                    u[t] = fmaf(f3[e], fx[e], u[t]);
                }
            }
        }
    }
}

// MXFP4 rows: 16-byte code blocks of 32 elements with one e8m0 scale each.
__device__ __forceinline__ void dot2_mxfp4(const uint4* __restrict__ c1, const uint8_t* __restrict__ s1,
                                           const uint4* __restrict__ c3, const uint8_t* __restrict__ s3,
                                           const uint4* const* xr, int cnt, int nblk, int lane, float (&g)[TG],
                                           float (&u)[TG]) {
    for (int b = lane; b < nblk; b += 32) {
        const uint4 q1 = c1[b], q3 = c3[b];
        float bg[TG], bu[TG];
#pragma unroll
        for (int t = 0; t < TG; ++t) bg[t] = bu[t] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t a = (&q1.x)[w], c = (&q3.x)[w];
            float d1[8], d3[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                d1[e] = e2m1_to_f32(a >> (4 * e));
                d3[e] = e2m1_to_f32(c >> (4 * e));
            }
#pragma unroll
            for (int t = 0; t < TG; ++t) {
                if (t < cnt) {
                    float fx[8];
                    unpack8(xr[t][b * 4 + w], fx);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        bg[t] = fmaf(d1[e], fx[e], bg[t]);
                        bu[t] = fmaf(d3[e], fx[e], bu[t]);
                    }
                }
            }
        }
        float sc1 = e8m0_to_f32(s1[b]), sc3 = e8m0_to_f32(s3[b]);
#pragma unroll
        for (int t = 0; t < TG; ++t) {
            g[t] = fmaf(bg[t], sc1, g[t]);
            u[t] = fmaf(bu[t], sc3, u[t]);
        }
    }
}

__device__ __forceinline__ void dot_mxfp4(const uint4* __restrict__ c, const uint8_t* __restrict__ s,
                                          const uint4* const* hr, int cnt, int nblk, int lane, float (&acc)[TG]) {
    for (int b = lane; b < nblk; b += 32) {
        const uint4 q = c[b];
        float ba[TG];
#pragma unroll
        for (int t = 0; t < TG; ++t) ba[t] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t a = (&q.x)[w];
            float d[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) d[e] = e2m1_to_f32(a >> (4 * e));
#pragma unroll
            for (int t = 0; t < TG; ++t) {
                if (t < cnt) {
                    float fx[8];
                    unpack8(hr[t][b * 4 + w], fx);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ba[t] = fmaf(d[e], fx[e], ba[t]);
                }
            }
        }
        float sc = e8m0_to_f32(s[b]);
#pragma unroll
        for (int t = 0; t < TG; ++t) acc[t] = fmaf(ba[t], sc, acc[t]);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ------------------------------------------------------------ consumer
template <int WFMT>
struct Consumer {
    const Ctx& x;
    Ring ring;
    Plan* plan;
    const uint16_t* xs;  // tokens in shared memory [M][H]
    float* yacc;         // [M][rpc]
    int warp, lane, tid;
    int q;               // running row counter (row ownership)

    __device__ bool wait_full() {
        return mbar_wait(ring.full(ring.n), ring.parity(ring.n), x.p, plan);
    }
    __device__ void release() {
        __syncwarp();
        if (lane == 0) mbar_arrive(ring.empty(ring.n));
        ring.n++;
    }
    __device__ const uint8_t* stage_ptr() const {
        return reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(ring.stage(ring.n)));
    }

    __device__ bool router(const Chunk& ch) {
        if (!wait_full()) return false;
        const LayerParams& p = x.p;
        const uint8_t* st = stage_ptr();
        const int nvec = p.H / 8;
        for (int j = 0; j < ch.n; ++j, ++q) {
            if (q % NCW != warp) continue;
            const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)j * p.H * 2);
            for (int t0 = 0; t0 < p.M; t0 += TG) {
                int cnt = min(TG, p.M - t0);
                const uint4* xr[TG];
#pragma unroll
                for (int t = 0; t < TG; ++t)
                    xr[t] = reinterpret_cast<const uint4*>(xs + (size_t)min(t0 + t, p.M - 1) * p.H);
                float acc[TG] = {0.f, 0.f, 0.f, 0.f};
                dot_bf16(row, xr, cnt, nvec, lane, acc);
#pragma unroll
                for (int t = 0; t < TG; ++t) acc[t] = warp_sum(acc[t]);
#pragma unroll
                for (int t = 0; t < TG; ++t)
                    if (t < cnt && lane == t) p.logits[(size_t)(t0 + t) * p.E + ch.r0 + j] = acc[t];
            }
        }
        release();
        return true;
    }

    __device__ bool gateup(const Chunk& ch) {
        if (!wait_full()) return false;
        const LayerParams& p = x.p;
        const uint8_t* st = stage_ptr();
        const bool shared = ch.slot < 0;
        const int inter = shared ? p.Is : p.I;
        const int npairs = slot_npairs(x, ch.slot);
        const int pbase = shared ? 0 : plan->slot_p0[ch.slot];
        uint16_t* hdst = shared ? p.hs : p.hr;
        for (int j = 0; j < ch.n; ++j, ++q) {
            if (q % NCW != warp) continue;
            const int i = ch.r0 + j;
            for (int q0 = 0; q0 < npairs; q0 += TG) {
                int cnt = min(TG, npairs - q0);
                const uint4* xr[TG];
#pragma unroll
                for (int t = 0; t < TG; ++t) {
                    int pp = min(q0 + t, npairs - 1);
                    int tok = shared ? pp : plan->pair_tok[pbase + pp];
                    xr[t] = reinterpret_cast<const uint4*>(xs + (size_t)tok * p.H);
                }
                float g[TG] = {0.f, 0.f, 0.f, 0.f}, u[TG] = {0.f, 0.f, 0.f, 0.f};
                if (WFMT == 0 || shared) {
                    const uint4* r1 = reinterpret_cast<const uint4*>(st + (size_t)j * p.H * 2);
                    const uint4* r3 = reinterpret_cast<const uint4*>(st + (size_t)(ch.n + j) * p.H * 2);
                    dot2_bf16(r1, r3, xr, cnt, p.H / 8, lane, g, u);
                } else {
                    const size_t cb = (size_t)p.H / 2, sbytes = (size_t)p.H / 32;
                    const uint4* c1 = reinterpret_cast<const uint4*>(st + j * cb);
                    const uint4* c3 = reinterpret_cast<const uint4*>(st + (ch.n + j) * cb);
                    const uint8_t* s1 = st + 2 * ch.n * cb + j * sbytes;
                    const uint8_t* s3 = st + 2 * ch.n * cb + (ch.n + j) * sbytes;
                    dot2_mxfp4(c1, s1, c3, s3, xr, cnt, p.H / 32, lane, g, u);
                }
#pragma unroll
                for (int t = 0; t < TG; ++t) {
                    g[t] = warp_sum(g[t]);
                    u[t] = warp_sum(u[t]);
                }
#pragma unroll
                for (int t = 0; t < TG; ++t)
                    if (t < cnt && lane == t)
                        hdst[(size_t)(pbase + q0 + t) * inter + i] = f32_to_bf16_bits(silu_mul(g[t], u[t]));
            }
        }
        release();
        return true;
    }

    __device__ bool down(const Chunk& ch, int h0) {
        if (!wait_full()) return false;
        const LayerParams& p = x.p;
        const uint8_t* st = stage_ptr();
        const bool shared = ch.slot < 0;
        const int inter = shared ? p.Is : p.I;
        const size_t hb = (size_t)ch.np * inter * 2;
        const int pbase = shared ? 0 : plan->slot_p0[ch.slot];
        size_t sofs = 0;
        if (WFMT == 1 && !shared) {
            size_t s0 = ((size_t)slot_expert(x, ch.slot) * p.H + ch.r0) * (p.I / 32);
            sofs = s0 - (s0 & ~(size_t)15);
        }
        for (int j = 0; j < ch.n; ++j) {
            const int r = ch.r0 + j;
            if ((r - h0) % NCW != warp) continue;
            for (int q0 = 0; q0 < ch.np; q0 += TG) {
                int cnt = min(TG, ch.np - q0);
                const uint4* hr[TG];
#pragma unroll
                for (int t = 0; t < TG; ++t)
                    hr[t] = reinterpret_cast<const uint4*>(st + (size_t)min(q0 + t, ch.np - 1) * inter * 2);
                float acc[TG] = {0.f, 0.f, 0.f, 0.f};
                if (WFMT == 0 || shared) {
                    const uint4* row = reinterpret_cast<const uint4*>(st + hb + (size_t)j * inter * 2);
                    dot_bf16(row, hr, cnt, inter / 8, lane, acc);
                } else {
                    const uint4* row = reinterpret_cast<const uint4*>(st + hb + (size_t)j * (p.I / 2));
                    const uint8_t* sc = st + hb + (size_t)ch.n * (p.I / 2) + sofs + (size_t)j * (p.I / 32);
                    dot_mxfp4(row, sc, hr, cnt, p.I / 32, lane, acc);
                }
#pragma unroll
                for (int t = 0; t < TG; ++t) acc[t] = warp_sum(acc[t]);
                if (lane == 0) {
#pragma unroll
                    for (int t = 0; t < TG; ++t) {
                        if (t < cnt) {
                            int pp = ch.p0 + q0 + t;
                            int tok = shared ? pp : plan->pair_tok[pbase + pp];
                            float wt = shared ? 1.0f : plan->pair_w[pbase + pp];
                            float* ya = yacc + (size_t)tok * p.rpc + (r - h0);
                            *ya = fmaf(wt, acc[t], *ya);
                        }
                    }
                }
            }
        }
        release();
        return true;
    }
};

// ------------------------------------------------------------ routing + plan

// Softmax, top-k (descending logit, ties to the lower index) and
// renormalisation for the tokens of this warp; writes plan->sel_e / sel_w.
static __device__ void topk_tokens(const LayerParams& p, Plan* plan, int warp, int lane) {
    for (int t = warp; t < p.M; t += NCW) {
        const float* lrow = p.logits + (size_t)t * p.E;
        float v[32];
        uint32_t taken = 0;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            int e = lane + 32 * j;
            if (e < p.E) {
                v[j] = __ldcg(lrow + e);
                mx = fmaxf(mx, v[j]);
            } else {
                v[j] = -INFINITY;
                taken |= 1u << j;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int sel[kMaxK];
        float selv[kMaxK];
#pragma unroll
        for (int jj = 0; jj < kMaxK; ++jj) {
            sel[jj] = 0;
            selv[jj] = 0.f;
            if (jj < p.k) {
                float bv = -INFINITY;
                int be = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (!((taken >> j) & 1u) && (v[j] > bv || be == 0x7fffffff)) {
                        bv = v[j];
                        be = lane + 32 * j;
                    }
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    if (ov > bv || (ov == bv && oe < be)) {
                        bv = ov;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                sel[jj] = be;
                selv[jj] = bv;
            }
        }
        float ex[kMaxK], den = 0.f;
#pragma unroll
        for (int jj = 0; jj < kMaxK; ++jj) {
            ex[jj] = 0.f;
            if (jj < p.k) {
                ex[jj] = expf(selv[jj] - mx);
                den += ex[jj];
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int jj = 0; jj < kMaxK; ++jj) {
                if (jj < p.k) {
                    plan->sel_e[t * p.k + jj] = sel[jj];
                    plan->sel_w[t * p.k + jj] = ex[jj] / den;
                }
            }
        }
    }
}


// Groups the M*k (token, expert) entries by expert with one pairwise pass per
// entry: rank = (#entries with a smaller expert id) + (#earlier entries with
// the same id). Nothing here scales with E. Entries whose expert id lies
// outside [0, E) (possible only when the routing is given) are dropped and
// reported.
static __device__ void build_plan(const LayerParams& p, Plan* plan, int tid, bool report) {
    const int N = p.M * p.k;
    const int BIG = 0x7fffffff;
    int e = BIG, less = 0;
    bool valid = false;
    if (tid < N) {
        e = plan->sel_e[tid];
        valid = e >= 0 && e < p.E;
        if (!valid) {
            if (report) raise_status(p, -100 /* MOE_EDEVICE_BAD_INDEX */);
            e = BIG;
        }
        int before = 0;
        for (int m = 0; m < N; ++m) {
            int em = plan->sel_e[m];
            if (!(em >= 0 && em < p.E)) em = BIG;
            less += em < e;
            before += (m < tid) && (em == e);
        }
        plan->rank[tid] = less + before;
        plan->first[tid] = (valid && before == 0) ? 1 : 0;
    }
    named_bar_sync(1, NCT);
    if (tid < N && valid) {
        int r = plan->rank[tid];
        plan->pair_tok[r] = (int16_t)(tid / p.k);
        plan->pair_w[r] = plan->sel_w[tid];
        if (plan->first[tid]) {
            int s = 0;
            for (int m = 0; m < N; ++m)
                if (plan->first[m] && plan->sel_e[m] < e) ++s;
            plan->slot_e[s] = (int16_t)e;
            plan->slot_p0[s] = (int16_t)less;
        }
    }
    if (tid == 0) {
        int u = 0, np = 0;
        for (int m = 0; m < N; ++m) {
            u += plan->first[m];
            int em = plan->sel_e[m];
            np += (em >= 0 && em < p.E);
        }
        plan->nslot = u;
        plan->npairs = np;
        plan->slot_p0[u] = (int16_t)np;
    }
    named_bar_sync(1, NCT);
}

// ------------------------------------------------------------ the kernel
template <int WFMT>
__global__ void __launch_bounds__(kThreads, 1) moe_layer_kernel(const __grid_constant__ LayerParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    // Early trigger: the next launch on the stream may start its prologue
    // (weight prefetch) as soon as SMs free up; it still waits for this grid
    // before reading anything this grid writes.
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Plan* plan = reinterpret_cast<Plan*>(smem + p.off_plan);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + p.off_x);
    float* yacc = reinterpret_cast<float*>(smem + p.off_yacc);
    const uint32_t bars = smem_u32(smem + p.off_bar);
    const uint32_t plan_bar = bars + 2u * p.ns * 8u;
    if (tid == 0) {
        for (int i = 0; i < p.ns; ++i) {
            mbar_init(bars + i * 8, 1);
            mbar_init(bars + (p.ns + i) * 8, NCW);
        }
        mbar_init(plan_bar, 1);
        plan->abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const Ctx cx{p, (int)blockIdx.x, plan};
    const Ring ring0{smem_u32(smem), bars, p.ns, 0};
    const bool has_route = (p.mode & kModeRoute) != 0, has_ffn = (p.mode & kModeFfn) != 0;

    if (warp == NCW) {
        // ---------------- producer (one elected lane)
        if (lane == 0) {
            Producer<WFMT> pr{cx, ring0, plan, policy_evict_first(), policy_evict_last(), false, 0, {}, 0};
            bool ok = true;
            auto issue = [&](const Chunk& c) {
                if (ok) ok = pr.issue(c);
            };
            // producer-independent tiles: router rows, shared expert gate/up
            if (has_route) for_router_chunks(cx, issue);
            if (has_ffn) for_shared_gateup_chunks<WFMT>(cx, issue);
            pdl_wait();
            if (ok && has_ffn) {
                ok = mbar_wait(plan_bar, 0, p, plan);
                if (ok) for_routed_gateup_chunks<WFMT>(cx, issue);
                if (ok) for_down_chunks<WFMT>(cx, issue);
                if (ok) ok = pr.poll_b2(true);
            }
            if (!ok || aborted(plan)) pr.drain();
        }
    } else {
        // ---------------- consumers
        Consumer<WFMT> cs{cx, ring0, plan, xs, yacc, warp, lane, tid, 0};
        pdl_wait();
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.x);
            uint4* dst = reinterpret_cast<uint4*>(xs);
            const int nv = p.M * p.H / 8;
            for (int i = tid; i < nv; i += NCT) dst[i] = __ldg(src + i);
            for (int i = tid; i < p.M * p.rpc; i += NCT) yacc[i] = 0.f;
            if (!has_route)
                for (int i = tid; i < p.M * p.k; i += NCT) {
                    plan->sel_e[i] = p.idx_in[i];
                    plan->sel_w[i] = p.w_in[i];
                }
        }
        named_bar_sync(1, NCT);
        bool ok = true;
        if (has_route) {
            for_router_chunks(cx, [&](const Chunk& c) {
                if (ok) ok = cs.router(c);
            });
            named_bar_sync(1, NCT);  // this CTA's logits are stored
            if (tid == 0 && !aborted(plan)) {
                __threadfence();
                atomicAdd(p.ctrl + kCtlBar1, 1u);
            }
        }
        cs.q = 0;
        // the shared expert needs no routing: compute it while barrier 1 fills
        if (has_ffn)
            for_shared_gateup_chunks<WFMT>(cx, [&](const Chunk& c) {
                if (ok) ok = cs.gateup(c);
            });
        if (has_route) {
            if (tid == 0 && !aborted(plan))
                grid_wait(p.ctrl + kCtlBar1, (unsigned)p.G + (p.force_timeout ? 1u : 0u), p, plan);
            named_bar_sync(1, NCT);
            if (!aborted(plan)) topk_tokens(p, plan, warp, lane);
            named_bar_sync(1, NCT);
            if (blockIdx.x == 0 && !aborted(plan)) {
                for (int i = tid; i < p.M * p.k; i += NCT) {
                    if (p.idx_out) p.idx_out[i] = plan->sel_e[i];
                    if (p.w_out) p.w_out[i] = plan->sel_w[i];
                }
            }
        }
        if (has_ffn) {
            build_plan(p, plan, tid, blockIdx.x == 0);
            if (tid == 0) mbar_arrive(plan_bar);
            for_routed_gateup_chunks<WFMT>(cx, [&](const Chunk& c) {
                if (ok && !aborted(plan)) ok = cs.gateup(c);
            });
            named_bar_sync(1, NCT);  // this CTA's activations are stored
            if (tid == 0 && !aborted(plan)) {
                __threadfence();
                atomicAdd(p.ctrl + kCtlBar2, 1u);
            }
            const int h0 = (int)((long long)blockIdx.x * p.H / p.G);
            const int h1 = (int)((long long)(blockIdx.x + 1) * p.H / p.G);
            for_down_chunks<WFMT>(cx, [&](const Chunk& c) {
                if (ok && !aborted(plan)) ok = cs.down(c, h0);
            });
            named_bar_sync(1, NCT);
            if (!aborted(plan)) {
                const int nr = h1 - h0;
                for (int i = tid; i < p.M * nr; i += NCT) {
                    int t = i / nr, r = i - t * nr;
                    p.y[(size_t)t * p.H + h0 + r] = f32_to_bf16_bits(yacc[(size_t)t * p.rpc + r]);
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0 && !aborted(plan)) {
        // Last CTA out re-arms the barrier counters for the next call.
        __threadfence();
        unsigned old = atomicAdd(p.ctrl + kCtlExit, 1u);
        if (old == (unsigned)p.G - 1u) {
            atomicExch(p.ctrl + kCtlBar1, 0u);
            atomicExch(p.ctrl + kCtlBar2, 0u);
            atomicExch(p.ctrl + kCtlExit, 0u);
        }
    }
}

}  // namespace moe
