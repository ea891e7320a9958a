// Persistent fused small-M MoE decode layer for sm_103a.
//
// One CTA per SM. Each CTA runs one producer warp, whose elected lane streams
// weight tiles from HBM into a ring of shared-memory stages with bulk (TMA)
// copies completing on mbarriers, and consumer warps (consumer_warps(WFMT))
// that compute from the ring. The layer runs in three phases, separated by a
// bounded wait on tagged data (the logits) and a bounded grid barrier:
//
//   phase 0  router gate matvec: CTA c owns router rows [cE/G, (c+1)E/G);
//            logits go to the workspace, each with this call's tag.
//            Every CTA then waits for all tagged logits, computes softmax /
//            top-k / renormalisation for all M tokens and builds the expert
//            plan (distinct experts and their token lists) in shared memory.
//   phase 1  gate/up + SwiGLU: the intermediate rows of the shared expert are
//            split evenly over the CTAs, those of the touched routed experts
//            are claimed chunk by chunk from a global counter;
//            h = silu(W1 x) * (W3 x) goes to the workspace in bf16.
//                                                       -> grid barrier 2
//            (one-token bf16 launches: no barrier; h goes out as tagged
//            words that ride with the down chunks' copies)
//   phase 2  down projection + weighted combine: CTA c owns output rows
//            [cH/G, (c+1)H/G); each (token, expert) pair's down result is
//            kept unweighted in shared memory, then y = shared expert +
//            sum of w * down over the token's pairs in ascending expert
//            order, in fp32, cast to bf16 once.
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

constexpr uint32_t SB = kStageBytes;

// Bank-conflict-free layout of the token rows (shared memory) and of the
// routed activation rows (workspace, copied row by row into the ring) for
// the MXFP4 and FP8 layers, whose dot products give each lane a whole
// block of consecutive 16-byte vectors (four for MXFP4, two for FP8), so
// that lanes are 64 or 32 bytes apart: vector v of a row is stored at
// v ^ ((v >> 3) & XM). The eight lanes of a quarter warp then hit eight
// different 16-byte bank groups both for block-wise reads and for plain
// one-vector-per-lane reads (router, shared expert). XM only flips bits of
// v inside an aligned group of four vectors, so a row of a multiple of four
// vectors maps onto itself. bf16 layers (XM = 0) keep the plain layout.
template <int WFMT>
constexpr int kXM = WFMT == 1 ? 3 : WFMT == 2 ? 1 : 0;
__device__ __forceinline__ int swz_vec(int v, int xm) { return v ^ ((v >> 3) & xm); }

// ------------------------------------------------------------ chunk lists
// The producer steps ChunkGen and writes each chunk's descriptor next to its
// stage; the consumers read the descriptors and run no generator. Phases: 0
// router rows, 1 shared-expert gate/up rows, 3 down rows (needs the plan);
// the routed gate/up rows (phase 2) are claimed dynamically instead
// (issue_routed_gateup). next() returns false at the end of each phase;
// begin(ph) starts a phase.
// PAD (the general bf16 kernel): a gate/up chunk for the tensor cores holds
// at most four row pairs, and each weight row sits in its stage at a pitch of
// its bytes + 16, so that the eight rows an ldmatrix reads fall into eight
// different 16-byte bank groups.
template <int WFMT, bool PAD = false>
__device__ __forceinline__ int gateup_cap(const LayerParams& p, bool routed) {
    // a routed row pair: codes plus scales (MXFP4 and FP8 both carry H / 32
    // scale bytes per row)
    uint32_t pair = !routed || WFMT == 0 ? (uint32_t)(4 * p.H + (PAD ? 32 : 0))
                    : (uint32_t)(2 * ((WFMT == 1 ? p.H / 2 : p.H) + p.H / 32));
    // a tensor-core chunk is one 8-column tile: at most four row pairs
    return PAD ? min(4, (int)(SB / pair)) : (int)(SB / pair);
}

// Bytes of one slot's segment of a packed MXFP4 / FP8 down chunk (kind 6):
// the pairs' bf16 activations, n rows of codes, and the rows' scales as
// copied from a 16-byte aligned window (at most 16 bytes more than they
// take). Every part is a multiple of 16 bytes.
template <int WFMT>
__device__ __forceinline__ uint32_t down_seg_bytes(const LayerParams& p, int npairs, int n) {
    constexpr int CD = WFMT == 1 ? 2 : 1;
    return (uint32_t)npairs * p.I * 2 + (uint32_t)n * (p.I / CD) + (((uint32_t)n * (p.I / 32) + 15u) & ~15u) + 16u;
}

template <int WFMT>
__device__ __forceinline__ uint32_t down_rowbytes(const LayerParams& p, int slot) {
    if (slot < 0) return (uint32_t)p.Is * 2;
    return WFMT == 0 ? (uint32_t)p.I * 2 : (uint32_t)((WFMT == 1 ? p.I / 2 : p.I) + p.I / 32);
}

// Tensor-core gate/up (the general bf16 kernel) for slots with at least this
// many tokens; below it the CUDA-core dots are faster.
constexpr int kMmaMinTokens = 4;
// Warps that split the K = H of one tensor-core chunk. A part's 512-byte
// partial goes into its own k-range of the chunk's rows (32 16-byte slots
// over as many rows as the range needs: any H of the API fits the stage).
constexpr int kMmaParts = 3;

template <int WFMT, bool PAD = false>
struct ChunkGen {
    int phase;
    int a, b, cap;                 // phases 0, 1: row cursor, end, rows per chunk
    int ds, nslot, q0, npairs, pg, np, rcap, h, h0, h1;  // phase 3

    __device__ __forceinline__ void begin(int ph, const LayerParams& p, const Plan* plan, int c) {
        phase = ph;
        const uint32_t G = (uint32_t)p.G, cc = (uint32_t)c;
        if (ph == 0) {
            a = (int)(cc * (uint32_t)p.E / G);
            b = (int)((cc + 1) * (uint32_t)p.E / G);
            cap = (int)(SB / (uint32_t)(p.H * 2));
        } else if (ph == 1) {
            a = (int)(cc * (uint32_t)p.Is / G);
            b = (int)((cc + 1) * (uint32_t)p.Is / G);
            cap = gateup_cap<WFMT, PAD>(p, false);
        } else {
            nslot = plan->nslot;
            h0 = (int)(cc * (uint32_t)p.H / G);
            h1 = (int)((cc + 1) * (uint32_t)p.H / G);
            ds = (p.Is > 0 ? -1 : 0) - 1;
            npairs = 0;
            q0 = 0;
            pg = 1;
            np = 0;
            rcap = 1;
            h = h1;  // forces the next slot on the first call
        }
    }

    __device__ __forceinline__ bool next(const LayerParams& p, const Plan* plan, Chunk& ch) {
        if (phase <= 1) {
            if (a >= b) return false;
            const int n = min(cap, b - a);
            ch = Chunk{phase == 0 ? 0 : 1, -1, a, n, 0, 0};
            a += n;
            return true;
        }
        // phase 3: slots (shared first), pair groups, row chunks
        if (h1 <= h0) return false;
        if (h >= h1) {
            q0 += pg;
            if (q0 >= npairs) {
                if (++ds >= nslot) return false;
                npairs = ds < 0 ? p.M : plan->slot_p0[ds + 1] - plan->slot_p0[ds];
                const uint32_t hrow = (uint32_t)(ds < 0 ? p.Is : p.I) * (!PAD && p.htag ? 4 : 2);
                pg = max(1, min(npairs, (int)((SB / 2) / hrow)));
                q0 = 0;
                if (WFMT != 0 && ds >= 0) {
                    // MXFP4 / FP8: the CTA's rows of one slot take a fraction
                    // of a stage; consecutive slots that fit whole share one
                    const int n = h1 - h0;
                    uint32_t tot = down_seg_bytes<WFMT>(p, npairs, n);
                    int k = 1;
                    if (npairs <= pg && tot <= SB) {
                        while (k < kMaxPack && ds + k < nslot) {
                            const int npk = plan->slot_p0[ds + k + 1] - plan->slot_p0[ds + k];
                            const uint32_t b = down_seg_bytes<WFMT>(p, npk, n);
                            if ((uint32_t)npk * hrow > SB / 2 || tot + b > SB) break;
                            tot += b;
                            ++k;
                        }
                    }
                    if (k > 1) {
                        ch = Chunk{6, ds, h0, n, 0, k};
                        ds += k - 1;
                        npairs = 0;  // the next call starts the slot after these
                        pg = 1;
                        h = h1;
                        return true;
                    }
                }
            }
            // chunk geometry of this (slot, pair group), computed once; tagged
            // activations take four bytes a value
            const uint32_t hrow = (uint32_t)(ds < 0 ? p.Is : p.I) * (!PAD && p.htag ? 4 : 2);
            const uint32_t reserve = (WFMT != 0 && ds >= 0) ? 32u : 0u;
            np = min(pg, npairs - q0);
            rcap = (int)((SB - (uint32_t)np * hrow - reserve) / down_rowbytes<WFMT>(p, ds));
            h = h0;
        }
        const int n = min(rcap, h1 - h);
        ch = Chunk{2, ds, h, n, q0, np};
        h += n;
        return true;
    }
};

// Optional phase trace: slot i of this CTA's 16-entry record gets the global
// timer (ns). Slots 0-7 are written by the consumer warps, 8-14 by the
// producer lane, 3 and 15 by the one-token top-k (all logits seen; k rounds
// done).
__device__ __forceinline__ void trace_mark(const LayerParams& p, int slot) {
    if (p.trace) p.trace[(size_t)blockIdx.x * 16 + slot] = global_timer_ns();
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
// The waiting warp suspends in the barrier probe (it issues nothing while
// suspended, leaving issue slots and the shared-memory pipe to the warps that
// compute) and resumes when the phase completes.
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

// ------------------------------------------------------------ call counters
// Grid barrier 2, the routed gate/up work counter and the entry counter of
// the call with this epoch (two sets, by parity).
__device__ __forceinline__ unsigned* ctl_bar2(const LayerParams& p, uint32_t epoch) {
    return p.ctrl + ((epoch & 1u) ? kCtlBar2Odd : kCtlBar2);
}
__device__ __forceinline__ unsigned* ctl_work(const LayerParams& p, uint32_t epoch) {
    return p.ctrl + ((epoch & 1u) ? kCtlWorkOdd : kCtlWork);
}
__device__ __forceinline__ unsigned* ctl_entry(const LayerParams& p, uint32_t epoch) {
    return p.ctrl + ((epoch & 1u) ? kCtlEntryOdd : kCtlEntry);
}

// Called by one CTA once every CTA of the call has read the epoch (all have
// arrived at a grid barrier, or counted themselves in, after reading it):
// zeroes the counter set of the next epoch (last used two calls ago, which
// has finished) and advances the epoch. The next call on the stream reads
// them only after this grid has finished.
__device__ __forceinline__ void advance_epoch(const LayerParams& p, uint32_t epoch) {
    const uint32_t n = epoch + 1u;
    atomicExch(ctl_bar2(p, n), 0u);
    atomicExch(ctl_work(p, n), 0u);
    atomicExch(ctl_entry(p, n), 0u);
    atomicExch(p.ctrl + kCtlEpoch, n);
}

// The 16-bit tag of a one-token call's activation words: 1 + epoch mod 65535
// (never 0, and never the previous call's).
__device__ __forceinline__ uint32_t htag16(const Plan* plan) { return plan->epoch % 0xffffu + 1u; }

// ------------------------------------------------------------ ring
// Stage cursor of the shared-memory ring, advanced chunk by chunk (no
// divisions). Chunk n lives in stage n % ns and is the (n / ns)-th use of it;
// ph is the parity of that use.
struct Ring {
    uint32_t base;  // shared address of stage 0
    uint32_t bars;  // full[ns], then empty[ns]
    uint32_t ns;
    uint32_t n, s, ph;
    __device__ __forceinline__ uint32_t stage() const { return base + s * SB; }
    __device__ __forceinline__ uint32_t full() const { return bars + s * 8; }
    __device__ __forceinline__ uint32_t empty() const { return bars + (ns + s) * 8; }
    __device__ __forceinline__ void advance() {
        ++n;
        if (++s == ns) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// ------------------------------------------------------------ producer
// One elected lane. Weight tiles of a chunk are issued as soon as its stage
// is free; the activation tiles of a down chunk are produced by all CTAs and
// may only be fetched after grid barrier 2, so until then they wait in a
// short list in shared memory (one-token bf16 launches copy tagged
// activations at once instead).
template <int WFMT, bool PAD = false>
struct Producer {
    const LayerParams& p;
    Plan* plan;
    Ring ring;
    uint64_t pol_w;  // weights: evict first
    uint64_t pol_h;  // activations: keep
    bool b2_done;
    uint32_t complete_upto;  // chunks whose copies were all issued
    uint32_t epoch;          // this call's epoch (from the plan, once it is published)

    __device__ __forceinline__ void flush_pending() {
        for (int i = 0; i < plan->npend; ++i)
            bulk_g2s(plan->pend_dst[i], plan->pend_src[i], plan->pend_bytes[i], plan->pend_bar[i], pol_h);
        plan->npend = 0;
        complete_upto = ring.n;
    }

    __device__ __forceinline__ bool poll_b2(bool block) {
        if (b2_done) return true;
        const unsigned* ctr = ctl_bar2(p, epoch);
        const bool ok = block ? grid_wait(ctr, (unsigned)p.G, p, plan) : (ld_acquire_gpu(ctr) >= (unsigned)p.G);
        if (!ok) return false;
        b2_done = true;
        if (blockIdx.x == 0) advance_epoch(p, epoch);
        fence_proxy_async_global();
        flush_pending();
        return true;
    }

    // Waits until the stage of the next chunk is free. In phase 2 it polls
    // without suspending, so that barrier 2 is seen as soon as it completes.
    __device__ __forceinline__ bool acquire(bool down) {
        if (ring.n < ring.ns) return true;
        const uint32_t bar = ring.empty(), par = ring.ph ^ 1u;
        if (mbar_test_wait(bar, par)) return true;
        const uint64_t t0 = global_timer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (down) {
                if (mbar_test_wait(bar, par)) return true;
                poll_b2(false);
                __nanosleep(32);
            } else if (mbar_try_wait(bar, par)) {
                return true;
            }
            if ((spin & 15u) == 0) {
                if (aborted(plan)) return false;
                if (global_timer_ns() - t0 > p.timeout_ns) {
                    set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
                    return false;
                }
            }
        }
    }

    // Ends a phase: a stage with a descriptor and no data. While activation
    // copies wait for barrier 2 (after the down chunks), the stage wait polls
    // the barrier: those stages are freed only once their copies are issued.
    __device__ __forceinline__ bool issue_end() {
        if (aborted(plan)) return false;
        if (!acquire(plan->npend > 0)) return false;
        plan->desc[ring.s] = Chunk{3, 0, 0, 0, 0, 0};
        mbar_arrive(ring.full());
        ring.advance();
        if (plan->npend == 0) complete_upto = ring.n;
        return true;
    }

    __device__ __forceinline__ bool issue(const Chunk& ch) {
        if (aborted(plan)) return false;
        // down chunks poll barrier 2 while they wait for a stage, unless the
        // activations come tagged (no barrier 2)
        if (!acquire((ch.kind == 2 || ch.kind == 6) && (PAD || !p.htag))) return false;
        plan->desc[ring.s] = ch;
        const uint32_t dst = ring.stage(), bar = ring.full();
        bool deferred = false;
        if (ch.kind == 0) {
            const uint32_t b = (uint32_t)ch.n * p.H * 2;
            mbar_arrive_expect_tx(bar, b);
            bulk_g2s(dst, p.Wg + (size_t)ch.r0 * p.H, b, bar, pol_w);
        } else if (ch.kind == 1) {
            if (ch.slot < 0 || WFMT == 0) {
                const uint32_t b = (uint32_t)ch.n * p.H * 2;
                const int np = ch.slot < 0 ? p.M : plan->slot_p0[ch.slot + 1] - plan->slot_p0[ch.slot];
                const bool mma = PAD && np >= kMmaMinTokens;
                if (mma) plan->desc[ring.s].kind = 5;
                const uint8_t *a, *c;
                if (ch.slot < 0) {
                    a = reinterpret_cast<const uint8_t*>(p.ws1 + (size_t)ch.r0 * p.H);
                    c = reinterpret_cast<const uint8_t*>(p.ws3 + (size_t)ch.r0 * p.H);
                } else {
                    const size_t off = ((size_t)plan->slot_e[ch.slot] * p.I + ch.r0) * p.H * 2;
                    a = p.w1 + off;
                    c = p.w3 + off;
                }
                mbar_arrive_expect_tx(bar, 2 * b);
                if (mma) {  // one copy per row, rows at a padded pitch
                    const uint32_t rb = (uint32_t)p.H * 2, pitch = rb + 16;
                    for (int j = 0; j < ch.n; ++j) {
                        bulk_g2s(dst + (uint32_t)j * pitch, a + (size_t)j * rb, rb, bar, pol_w);
                        bulk_g2s(dst + (uint32_t)(ch.n + j) * pitch, c + (size_t)j * rb, rb, bar, pol_w);
                    }
                } else {
                    bulk_g2s(dst, a, b, bar, pol_w);
                    bulk_g2s(dst + b, c, b, bar, pol_w);
                }
            } else {
                constexpr int CD = WFMT == 1 ? 2 : 1;  // elements per code byte
                const uint32_t bc = (uint32_t)ch.n * (p.H / CD), bs = (uint32_t)ch.n * (p.H / 32);
                const size_t row = (size_t)plan->slot_e[ch.slot] * p.I + ch.r0;
                mbar_arrive_expect_tx(bar, 2 * bc + 2 * bs);
                bulk_g2s(dst, p.w1 + row * (p.H / CD), bc, bar, pol_w);
                bulk_g2s(dst + bc, p.w3 + row * (p.H / CD), bc, bar, pol_w);
                bulk_g2s(dst + 2 * bc, p.s1 + row * (p.H / 32), bs, bar, pol_w);
                bulk_g2s(dst + 2 * bc + bs, p.s3 + row * (p.H / 32), bs, bar, pol_w);
            }
        } else if (WFMT == 0 && !PAD && p.htag) {
            // one token: the pair's tagged activations come with the weights
            const int inter = ch.slot < 0 ? p.Is : p.I;
            const uint32_t hb = (uint32_t)ch.np * inter * 4, rb = (uint32_t)inter * 2, wb = (uint32_t)ch.n * rb;
            const uint32_t* hsrc = p.htag + (ch.slot < 0 ? (size_t)ch.p0 * p.Is
                                                          : (size_t)p.Is + (size_t)(plan->slot_p0[ch.slot] + ch.p0) * p.I);
            const uint8_t* w = ch.slot < 0 ? reinterpret_cast<const uint8_t*>(p.ws2 + (size_t)ch.r0 * p.Is)
                                           : p.w2 + ((size_t)plan->slot_e[ch.slot] * p.H + ch.r0) * p.I * 2;
            mbar_arrive_expect_tx(bar, hb + wb);
            bulk_g2s(dst, hsrc, hb, bar, pol_h);
            bulk_g2s(dst + hb, w, wb, bar, pol_w);
        } else if (WFMT != 0 && ch.kind == 6) {
            // np routed slots, each segment laid out as a kind-2 chunk; the
            // activation copies wait for barrier 2 like any other
            constexpr int CD = WFMT == 1 ? 2 : 1;
            const uint32_t bc = (uint32_t)ch.n * (p.I / CD);
            uint32_t tot = 0;
            for (int k = 0; k < ch.np; ++k) {
                const int slot = ch.slot + k;
                const uint32_t hb = (uint32_t)(plan->slot_p0[slot + 1] - plan->slot_p0[slot]) * p.I * 2;
                const size_t s0 = ((size_t)plan->slot_e[slot] * p.H + ch.r0) * (p.I / 32);
                const size_t s1 = s0 + (size_t)ch.n * (p.I / 32);
                tot += hb + bc + (uint32_t)(((s1 + 15) & ~(size_t)15) - (s0 & ~(size_t)15));
            }
            mbar_arrive_expect_tx(bar, tot);
            uint32_t off = 0;
            for (int k = 0; k < ch.np; ++k) {
                const int slot = ch.slot + k;
                const int npairs = plan->slot_p0[slot + 1] - plan->slot_p0[slot];
                const uint32_t hb = (uint32_t)npairs * p.I * 2;
                const size_t row = (size_t)plan->slot_e[slot] * p.H + ch.r0;
                const size_t s0 = row * (p.I / 32), s1 = s0 + (size_t)ch.n * (p.I / 32);
                const size_t w0 = s0 & ~(size_t)15, w1 = (s1 + 15) & ~(size_t)15;
                bulk_g2s(dst + off + hb, p.w2 + row * (p.I / CD), bc, bar, pol_w);
                bulk_g2s(dst + off + hb + bc, p.s2 + w0, (uint32_t)(w1 - w0), bar, pol_w);
                const void* hsrc = p.hr + (size_t)plan->slot_p0[slot] * p.I;
                if (b2_done) {
                    bulk_g2s(dst + off, hsrc, hb, bar, pol_h);
                } else {
                    const int q = plan->npend++;
                    plan->pend_dst[q] = dst + off;
                    plan->pend_src[q] = hsrc;
                    plan->pend_bytes[q] = hb;
                    plan->pend_bar[q] = bar;
                    deferred = true;
                }
                off += down_seg_bytes<WFMT>(p, npairs, ch.n);
            }
        } else {
            const int inter = ch.slot < 0 ? p.Is : p.I;
            const uint32_t hb = (uint32_t)ch.np * inter * 2;
            const void* hsrc;
            if (ch.slot < 0 || WFMT == 0) {
                const uint8_t* w;
                if (ch.slot < 0) {
                    hsrc = p.hs + (size_t)ch.p0 * p.Is;
                    w = reinterpret_cast<const uint8_t*>(p.ws2 + (size_t)ch.r0 * p.Is);
                } else {
                    hsrc = p.hr + (size_t)(plan->slot_p0[ch.slot] + ch.p0) * p.I;
                    w = p.w2 + ((size_t)plan->slot_e[ch.slot] * p.H + ch.r0) * p.I * 2;
                }
                const uint32_t rb = (uint32_t)inter * 2, wb = (uint32_t)ch.n * rb;
                mbar_arrive_expect_tx(bar, hb + wb);
                bulk_g2s(dst + hb, w, wb, bar, pol_w);
            } else {
                hsrc = p.hr + (size_t)(plan->slot_p0[ch.slot] + ch.p0) * p.I;
                const size_t row = (size_t)plan->slot_e[ch.slot] * p.H + ch.r0;
                {
                    constexpr int CD = WFMT == 1 ? 2 : 1;
                    const uint32_t bc = (uint32_t)ch.n * (p.I / CD);
                    const size_t s0 = row * (p.I / 32), s1 = s0 + (size_t)ch.n * (p.I / 32);
                    const size_t w0 = s0 & ~(size_t)15, w1 = (s1 + 15) & ~(size_t)15;
                    const uint32_t bs = (uint32_t)(w1 - w0);
                    mbar_arrive_expect_tx(bar, hb + bc + bs);
                    bulk_g2s(dst + hb, p.w2 + row * (p.I / CD), bc, bar, pol_w);
                    bulk_g2s(dst + hb + bc, p.s2 + w0, bs, bar, pol_w);
                }
            }
            if (b2_done) {
                bulk_g2s(dst, hsrc, hb, bar, pol_h);
            } else {
                const int k = plan->npend++;
                plan->pend_dst[k] = dst;
                plan->pend_src[k] = hsrc;
                plan->pend_bytes[k] = hb;
                plan->pend_bar[k] = bar;
                deferred = true;
            }
        }
        ring.advance();
        if (!deferred && plan->npend == 0) complete_upto = ring.n;
        return true;
    }

    // After an abort: wait (bounded) for every copy already issued, so that
    // no bulk copy is still writing this CTA's shared memory at exit.
    // Deferred activation copies are issued regardless (their source is valid
    // workspace memory), so that every stage's barrier can complete.
    __device__ void drain() {
        flush_pending();
        const uint32_t n = complete_upto;
        const uint32_t lo = n > ring.ns ? n - ring.ns : 0;
        for (uint32_t i = lo; i < n; ++i) {
            const uint32_t bar = ring.bars + (i % ring.ns) * 8, par = (i / ring.ns) & 1u;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar, par)) {
                if (global_timer_ns() - t0 > p.timeout_ns) break;
            }
        }
    }
};

// ------------------------------------------------------------ consumer math
// Dot products over rows held in shared memory. Lanes stride the row's
// 16-byte vectors; each token keeps four independent partial sums so that the
// FMA dependency chains stay short and the loads of several vectors are in
// flight at once. bf16 x bf16 products go through the mixed-precision fma
// (fma.rn.f32.bf16: bf16 operands straight from the packed registers, fp32
// addend, one rounding), which needs no unpacking; with f16 tokens (MXFP4
// layers) the weights are unpacked to fp32 pairs and go through the paired
// fp32 FMA (fma.rn.f32x2). Either way each partial sum is rounded as a
// scalar fp32 fma would round it. Token groups are at most two wide (NT),
// which keeps all accumulators in registers.

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Warp sums of two values in one butterfly: at the first level each half of
// the warp keeps one of them, so lanes 0-15 end with sum(g) and lanes 16-31
// with sum(u). Every level pairs the same lanes as warp_sum, so each sum is
// bit-identical to warp_sum's.
__device__ __forceinline__ float warp_sum2(float g, float u, int lane) {
    const bool h16 = (lane & 16) != 0;
    float a = h16 ? u : g;
    a += __shfl_xor_sync(0xffffffffu, h16 ? g : u, 16);
#pragma unroll
    for (int o = 8; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return a;
}

// The same for four values: lanes 0-7 end with sum(g0), 8-15 with sum(u0),
// 16-23 with sum(g1), 24-31 with sum(u1).
__device__ __forceinline__ float warp_sum4(float g0, float u0, float g1, float u1, int lane) {
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    float kg = h16 ? g1 : g0, ku = h16 ? u1 : u0;
    kg += __shfl_xor_sync(0xffffffffu, h16 ? g0 : g1, 16);
    ku += __shfl_xor_sync(0xffffffffu, h16 ? u0 : u1, 16);
    float a = h8 ? ku : kg;
    a += __shfl_xor_sync(0xffffffffu, h8 ? kg : ku, 8);
#pragma unroll
    for (int o = 4; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return a;
}

// (p0 + p1) + (p2 + p3) of the four partial sums held as two pairs.
template <int NT>
__device__ __forceinline__ void sum4(const float2 (&pa)[NT][2], float (&acc)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = (pa[t][0].x + pa[t][0].y) + (pa[t][1].x + pa[t][1].y);
}

// Eight activations of one 16-byte vector as four fp32 pairs: bf16, or (XH)
// f16.
template <bool XH>
__device__ __forceinline__ void unpack8x2x(const uint4 v, float2 (&f)[4]) {
    if (XH) {
        f[0] = f16x2_to_f32(v.x);
        f[1] = f16x2_to_f32(v.y);
        f[2] = f16x2_to_f32(v.z);
        f[3] = f16x2_to_f32(v.w);
    } else {
        unpack8x2(v, f);
    }
}

// acc[t] = row . x_t (bf16 weights, bf16 or (XH) f16 activations, fp32
// accumulate) over nvec 16-byte vectors; this lane takes vectors lane,
// lane + STRIDE, ... Element e of a vector goes to partial sum e mod 4.
template <int NT, int STRIDE = 32, bool XH = false, int XM = 0>
__device__ __forceinline__ void dot_bf16(const uint4* __restrict__ row, const uint4* __restrict__ x0,
                                         const uint4* __restrict__ x1, int nvec, int lane, float (&acc)[NT]) {
    float2 pa[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) pa[t][0] = pa[t][1] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int v = lane; v < nvec; v += STRIDE) {
        if (!XH) {
            const uint4 w = row[v];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 x = (t == 0 ? x0 : x1)[swz_vec(v, XM)];
                const uint32_t xx[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) fma_bf16x2(ww[e], xx[e], pa[t][e & 1].x, pa[t][e & 1].y);
            }
            continue;
        }
        float2 fw[4];
        unpack8x2(row[v], fw);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float2 fx[4];
            unpack8x2x<XH>((t == 0 ? x0 : x1)[swz_vec(v, XM)], fx);
#pragma unroll
            for (int e = 0; e < 4; ++e) pa[t][e & 1] = ffma2(fw[e], fx[e], pa[t][e & 1]);
        }
    }
    sum4<NT>(pa, acc);
}

// Gate and up rows against the same tokens.
template <int NT, bool XH = false, int XM = 0>
__device__ __forceinline__ void dot2_bf16(const uint4* __restrict__ r1, const uint4* __restrict__ r3,
                                          const uint4* __restrict__ x0, const uint4* __restrict__ x1, int nvec,
                                          int lane, float (&g)[NT], float (&u)[NT]) {
    float2 pg[NT][2], pu[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) pg[t][0] = pg[t][1] = pu[t][0] = pu[t][1] = make_float2(0.f, 0.f);
#pragma unroll 5
    for (int v = lane; v < nvec; v += 32) {
        if (!XH) {
            const uint4 a = r1[v], b = r3[v];
            const uint32_t w1[4] = {a.x, a.y, a.z, a.w}, w3[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint4 x = (t == 0 ? x0 : x1)[swz_vec(v, XM)];
                const uint32_t xx[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    fma_bf16x2(w1[e], xx[e], pg[t][e & 1].x, pg[t][e & 1].y);
                    fma_bf16x2(w3[e], xx[e], pu[t][e & 1].x, pu[t][e & 1].y);
                }
            }
            continue;
        }
        float2 f1[4], f3[4];
        unpack8x2(r1[v], f1);
        unpack8x2(r3[v], f3);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float2 fx[4];
            unpack8x2x<XH>((t == 0 ? x0 : x1)[swz_vec(v, XM)], fx);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pg[t][e & 1] = ffma2(f1[e], fx[e], pg[t][e & 1]);
                pu[t][e & 1] = ffma2(f3[e], fx[e], pu[t][e & 1]);
            }
        }
    }
    sum4<NT>(pg, g);
    sum4<NT>(pu, u);
}

// Four rows (row0 + min(j, nrow - 1) * rstride, j < 4: rows past nrow repeat
// the last one and their results are dropped) against NT vectors at once:
// the four rows' loads and FMA chains are independent, so one warp keeps
// several rows in flight instead of finishing them one after another. Each
// row and token keeps two partial sums (even and odd elements).
template <int NT>
__device__ __forceinline__ void dot4_bf16(const uint4* __restrict__ row0, int rstride, int nrow,
                                          const uint4* __restrict__ h0, const uint4* __restrict__ h1, int nvec,
                                          int lane, float (&acc)[4][NT]) {
    const uint4* rows[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) rows[j] = row0 + min(j, nrow - 1) * rstride;
    float2 pa[4][NT];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) pa[j][t] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        uint32_t hh[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 h = (t == 0 ? h0 : h1)[v];
            hh[t][0] = h.x, hh[t][1] = h.y, hh[t][2] = h.z, hh[t][3] = h.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 w = rows[j][v];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) fma_bf16x2(ww[e], hh[t][e], pa[j][t].x, pa[j][t].y);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[j][t] = pa[j][t].x + pa[j][t].y;
}

// One token, tagged activations: dot4_bf16<1> with the activations held as
// 32-bit words, a 16-bit tag in the high half and the bf16 value in the low
// half (two 16-byte words per eight values). Returns false when any word
// this lane read carries another tag.
__device__ __forceinline__ bool dot4_bf16_tagged(const uint4* __restrict__ row0, int rstride, int nrow,
                                                 const uint4* __restrict__ ht, int nvec, int lane, uint32_t tag,
                                                 float (&acc)[4][1]) {
    const uint4* rows[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) rows[j] = row0 + min(j, nrow - 1) * rstride;
    float2 pa[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pa[j] = make_float2(0.f, 0.f);
    uint32_t bad = 0;
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        const uint4 a = ht[2 * v], b = ht[2 * v + 1];
        bad |= ((a.x >> 16) ^ tag) | ((a.y >> 16) ^ tag) | ((a.z >> 16) ^ tag) | ((a.w >> 16) ^ tag) |
               ((b.x >> 16) ^ tag) | ((b.y >> 16) ^ tag) | ((b.z >> 16) ^ tag) | ((b.w >> 16) ^ tag);
        const uint32_t hh[4] = {__byte_perm(a.x, a.y, 0x5410), __byte_perm(a.z, a.w, 0x5410),
                                __byte_perm(b.x, b.y, 0x5410), __byte_perm(b.z, b.w, 0x5410)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 w = rows[j][v];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) fma_bf16x2(ww[e], hh[e], pa[j].x, pa[j].y);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][0] = pa[j].x + pa[j].y;
    return bad == 0;
}

// ---- MXFP4 with f16 block sums. The codes of a 32-element block become
// f16 pairs by the hardware conversion; the activations are f16 scaled by a
// power of two so that their magnitude stays below 256. Every product of an
// e2m1 value (two significant bits) and such an activation (a bf16 value:
// eight significant bits) is exact in f16, and a 32-term block sum stays
// below 2^16; the block sum is accumulated in four f16 chains of eight
// terms, then converted to fp32, scaled by the block's e8m0 scale (and the
// activation's power of two) and accumulated in fp32.

// Block sum of 16 code pairs against 16 activation pairs (four uint4).
__device__ __forceinline__ float block_h(const uint32_t (&w)[16], const uint4 (&a)[4]) {
    uint32_t c0 = 0u, c1 = 0u, c2 = 0u, c3 = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        c0 = hfma2(w[4 * k + 0], a[k].x, c0);
        c1 = hfma2(w[4 * k + 1], a[k].y, c1);
        c2 = hfma2(w[4 * k + 2], a[k].z, c2);
        c3 = hfma2(w[4 * k + 3], a[k].w, c3);
    }
    const float2 f0 = f16x2_to_f32(c0), f1 = f16x2_to_f32(c1), f2 = f16x2_to_f32(c2), f3 = f16x2_to_f32(c3);
    return ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
}

__device__ __forceinline__ void decode_block(const uint4 q, uint32_t (&w)[16]) {
    uint32_t t[4];
    e2m1x8_to_f16x2(q.x, t);
    w[0] = t[0], w[1] = t[1], w[2] = t[2], w[3] = t[3];
    e2m1x8_to_f16x2(q.y, t);
    w[4] = t[0], w[5] = t[1], w[6] = t[2], w[7] = t[3];
    e2m1x8_to_f16x2(q.z, t);
    w[8] = t[0], w[9] = t[1], w[10] = t[2], w[11] = t[3];
    e2m1x8_to_f16x2(q.w, t);
    w[12] = t[0], w[13] = t[1], w[14] = t[2], w[15] = t[3];
}

// MXFP4 gate and up rows against tokens held in f16 times 2^s_t. The
// token's 2^-s_t (xi[t]) is folded into each block's e8m0 scale: a product
// of two powers of two is exact, so the result is what removing 2^s_t at the
// end would give, but an extreme block scale (up to 2^127) cannot overflow
// the sum of scaled tokens when the true sum is finite.
template <int NT>
__device__ __forceinline__ void dot2_mxh(const uint4* __restrict__ c1, const uint8_t* __restrict__ s1,
                                         const uint4* __restrict__ c3, const uint8_t* __restrict__ s3,
                                         const uint4* __restrict__ x0, const uint4* __restrict__ x1,
                                         const float (&xi)[NT], int nblk, int lane, float (&g)[NT],
                                         float (&u)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) g[t] = u[t] = 0.f;
#pragma unroll 2
    for (int b = lane; b < nblk; b += 32) {
        uint32_t w1[16], w3[16];
        decode_block(c1[b], w1);
        decode_block(c3[b], w3);
        const float sc1 = e8m0_to_f32(s1[b]), sc3 = e8m0_to_f32(s3[b]);
        const int r = (b >> 1) & 3;  // the block's swizzle (kXM<1>)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4* xb = (t == 0 ? x0 : x1) + 4 * b;
            const uint4 a[4] = {xb[r], xb[1 ^ r], xb[2 ^ r], xb[3 ^ r]};
            g[t] = fmaf(block_h(w1, a), sc1 * xi[t], g[t]);
            u[t] = fmaf(block_h(w3, a), sc3 * xi[t], u[t]);
        }
    }
}

// One bf16 activation block (32 values, four uint4 stored in the order
// k ^ r) as f16 times 2^s, s chosen from the block's own largest magnitude;
// returns 2^-s.
__device__ __forceinline__ float block_to_f16(const uint4* __restrict__ src, int r, uint4 (&a)[4]) {
    float f[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float t8[8];
        unpack8(src[k ^ r], t8);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[8 * k + e] = t8[e];
    }
    float mx = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(f[e]));
    const int sh = f16_range_shift(mx);
    const float sc = exp2i(sh);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a[k].x = f32x2_to_f16x2(f[8 * k + 0] * sc, f[8 * k + 1] * sc);
        a[k].y = f32x2_to_f16x2(f[8 * k + 2] * sc, f[8 * k + 3] * sc);
        a[k].z = f32x2_to_f16x2(f[8 * k + 4] * sc, f[8 * k + 5] * sc);
        a[k].w = f32x2_to_f16x2(f[8 * k + 6] * sc, f[8 * k + 7] * sc);
    }
    return exp2i(-sh);
}

// Four MXFP4 down rows (codes crow[j], scales srow[j]) against NT activation
// vectors (bf16, converted block by block).
template <int NT>
__device__ __forceinline__ void dot4_mxh(const uint8_t* const (&crow)[4], const uint8_t* const (&srow)[4],
                                         const uint4* __restrict__ h0, const uint4* __restrict__ h1, int nblk,
                                         int lane, float (&acc)[4][NT]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[j][t] = 0.f;
    for (int b = lane; b < nblk; b += 32) {
        uint4 a[NT][4];
        float inv[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) inv[t] = block_to_f16((t == 0 ? h0 : h1) + 4 * b, (b >> 1) & 3, a[t]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[16];
            decode_block(reinterpret_cast<const uint4*>(crow[j])[b], w);
            const float sw = e8m0_to_f32(srow[j][b]);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[j][t] = fmaf(block_h(w, a[t]) * inv[t], sw, acc[j][t]);
        }
    }
}

// dot4_mxh with the activation blocks already converted: lane b (< nblk,
// nblk <= 32) holds block b of each of the NT activations in a[t] (f16 times
// 2^s) and 2^-s in inv[t].
template <int NT>
__device__ __forceinline__ void dot4_mxh_pre(const uint8_t* const (&crow)[4], const uint8_t* const (&srow)[4],
                                             const uint4 (&a)[NT][4], const float (&inv)[NT], int nblk, int lane,
                                             float (&acc)[4][NT]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[j][t] = 0.f;
    if (lane < nblk) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[16];
            decode_block(reinterpret_cast<const uint4*>(crow[j])[lane], w);
            const float sw = e8m0_to_f32(srow[j][lane]);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[j][t] = block_h(w, a[t]) * inv[t] * sw;
        }
    }
}

// ---- FP8 e4m3 with one fp32 scale per 128 elements of a row: codes
// decoded to fp32 by the hardware conversion, products in fp32 through the
// paired FMA (even and odd partial sums of each 8-code half); each 16-code
// vector's partial sum is scaled by its block's scale.

// FP8 gate and up rows (codes c1, c3; scales s1, s3 per 128 elements)
// against bf16 tokens; this lane takes 16-element vectors lane, lane + 32, ...
template <int NT>
__device__ __forceinline__ void dot2_fp8(const uint4* __restrict__ c1, const float* __restrict__ s1,
                                         const uint4* __restrict__ c3, const float* __restrict__ s3,
                                         const uint4* __restrict__ x0, const uint4* __restrict__ x1, int nvec,
                                         int lane, float (&g)[NT], float (&u)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) g[t] = u[t] = 0.f;
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
        float2 f1[8], f3[8];
        unpack16_e4m3x2(c1[v], f1);
        unpack16_e4m3x2(c3[v], f3);
        const float sc1 = s1[v >> 3], sc3 = s3[v >> 3];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4* xt = t == 0 ? x0 : x1;
            const int r = (v >> 2) & 1;  // the vector pair's swizzle (kXM<2>)
            float2 fa[4], fb[4];
            unpack8x2(xt[2 * v + r], fa);
            unpack8x2(xt[2 * v + (1 ^ r)], fb);
            // (even, odd) partial sums of each half of the 16-code vector
            float2 pg[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            float2 pu[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pg[0] = ffma2(f1[e], fa[e], pg[0]);
                pg[1] = ffma2(f1[4 + e], fb[e], pg[1]);
                pu[0] = ffma2(f3[e], fa[e], pu[0]);
                pu[1] = ffma2(f3[4 + e], fb[e], pu[1]);
            }
            g[t] = fmaf((pg[0].x + pg[0].y) + (pg[1].x + pg[1].y), sc1, g[t]);
            u[t] = fmaf((pu[0].x + pu[0].y) + (pu[1].x + pu[1].y), sc3, u[t]);
        }
    }
}

// Four FP8 down rows (codes crow[j], scales srow[j], bytes of fp32) against
// NT bf16 activation vectors.
template <int NT>
__device__ __forceinline__ void dot4_fp8(const uint8_t* const (&crow)[4], const uint8_t* const (&srow)[4],
                                         const uint4* __restrict__ h0, const uint4* __restrict__ h1, int nvec,
                                         int lane, float (&acc)[4][NT]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[j][t] = 0.f;
    for (int v = lane; v < nvec; v += 32) {
        float2 fh[NT][8];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4* ht = t == 0 ? h0 : h1;
            const int r = (v >> 2) & 1;  // the vector pair's swizzle (kXM<2>)
            float2 a4[4], b4[4];
            unpack8x2(ht[2 * v + r], a4);
            unpack8x2(ht[2 * v + (1 ^ r)], b4);
#pragma unroll
            for (int e = 0; e < 4; ++e) fh[t][e] = a4[e], fh[t][4 + e] = b4[e];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 fw[8];
            unpack16_e4m3x2(reinterpret_cast<const uint4*>(crow[j])[v], fw);
            const float sc = reinterpret_cast<const float*>(srow[j])[v >> 3];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float2 q[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    q[0] = ffma2(fw[e], fh[t][e], q[0]);
                    q[1] = ffma2(fw[4 + e], fh[t][4 + e], q[1]);
                }
                acc[j][t] = fmaf((q[0].x + q[0].y) + (q[1].x + q[1].y), sc, acc[j][t]);
            }
        }
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ------------------------------------------------------------ consumer
// TWO: one-token MXFP4 launches, which hold the tokens twice, in f16 times
// 2^s_t (swizzled) for the routed experts and in plain bf16 for the router
// and the shared expert (the bf16 mixed-precision fma).
// MMA: the general bf16 kernel, whose gate/up rows of slots with at least
// kMmaMinTokens tokens run on the tensor cores (mma.sync m16n8k16, bf16 x
// bf16 -> fp32): the slot's tokens (up to 16) are the 16-row operand, eight
// weight rows the 8-column one. Token rows (p.xp elements apart: H + 8 for
// bf16 layers) and those weight rows (in a stage) sit at a pitch of their
// bytes + 16, so that every ldmatrix is free of bank conflicts.
template <int WFMT, bool TWO, bool MMA = false>
struct Consumer {
    static constexpr int NCW = consumer_warps(WFMT);
    const LayerParams& p;
    Plan* plan;
    Ring ring;
    const uint16_t* xs;  // tokens in shared memory [M][H]
    const uint16_t* xb;  // TWO: the same tokens in plain bf16
    float* ypair;        // down results per (pair, output row) [M + M*k][rpc]
    int warp, lane;
    int qm;              // rows go round-robin over the warps, continuing
                         // across chunks: the running row count mod NCW
    int h0;              // first output row of this CTA
    uint32_t redph;      // tensor-core chunks: parity bit of each stage's
                         // partial barrier

    __device__ __forceinline__ bool wait_full() { return mbar_wait(ring.full(), ring.ph, p, plan); }
    __device__ __forceinline__ void release() {
        __syncwarp();
        if (lane == 0) mbar_arrive(ring.empty());
        ring.advance();
    }
    // First row of a chunk of n rows that this warp owns (then every NCW-th
    // row); advances the running count past the chunk.
    __device__ __forceinline__ int claim_rows(int n) {
        const int j0 = warp >= qm ? warp - qm : warp - qm + NCW;
        qm = (qm + n) % NCW;
        return j0;
    }
    __device__ __forceinline__ const uint8_t* stage_ptr() const {
        return reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(ring.stage()));
    }
    __device__ __forceinline__ const uint4* xbrow(int tok) const {
        return reinterpret_cast<const uint4*>(xb + (size_t)tok * p.H);
    }
    __device__ __forceinline__ const uint4* xrow(int tok) const {
        return reinterpret_cast<const uint4*>(xs + (size_t)tok * p.xp);
    }

    // Router rows: logits[t][e] = Wg[e] . x_t, one warp per row.
    __device__ __forceinline__ void router(const Chunk& ch, const uint8_t* st) {
        const int nvec = p.H / 8;
        for (int j = claim_rows(ch.n); j < ch.n; j += NCW) {
            const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)j * p.H * 2);
            for (int t = 0; t < p.M; ++t) {
                float acc[1];
                if (TWO) {
                    const uint4* xt = xbrow(t);
                    dot_bf16<1>(row, xt, xt, nvec, lane, acc);
                } else {
                    const uint4* xt = xrow(t);
                    dot_bf16<1, 32, WFMT == 1, kXM<WFMT>>(row, xt, xt, nvec, lane, acc);
                }
                acc[0] = warp_sum(acc[0]);
                if (WFMT == 1 && !TWO) acc[0] *= plan->x_inv[t];
                // the logit and this call's tag in one 64-bit word: readers
                // need no barrier, they wait for the tag
                if (lane == 0)
                    st_relaxed_u64(p.logits + (size_t)t * p.Es + ch.r0 + j,
                                   ((unsigned long long)plan->tag << 32) | __float_as_uint(acc[0]));
            }
        }
    }

    template <int NT>
    __device__ __forceinline__ void gateup_group(const uint8_t* st, const Chunk& ch, int j, int t0tok, int t1tok,
                                                 bool shared, float (&g)[NT], float (&u)[NT]) const {
        if (WFMT == 0 || shared) {
            const uint4* r1 = reinterpret_cast<const uint4*>(st + (size_t)j * p.H * 2);
            const uint4* r3 = reinterpret_cast<const uint4*>(st + (size_t)(ch.n + j) * p.H * 2);
            if (TWO)
                dot2_bf16<NT>(r1, r3, xbrow(t0tok), xbrow(t1tok), p.H / 8, lane, g, u);
            else
                dot2_bf16<NT, WFMT == 1, kXM<WFMT>>(r1, r3, xrow(t0tok), xrow(t1tok), p.H / 8, lane, g, u);
        } else {
            const size_t cb = (size_t)p.H / (WFMT == 1 ? 2 : 1), sbytes = (size_t)p.H / 32;
            const uint4* c1 = reinterpret_cast<const uint4*>(st + j * cb);
            const uint4* c3 = reinterpret_cast<const uint4*>(st + (ch.n + j) * cb);
            const uint8_t* s1 = st + 2 * ch.n * cb + j * sbytes;
            const uint8_t* s3 = st + 2 * ch.n * cb + (ch.n + j) * sbytes;
            if (WFMT == 1) {
                float xi[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) xi[t] = plan->x_inv[t == 0 ? t0tok : t1tok];
                dot2_mxh<NT>(c1, s1, c3, s3, xrow(t0tok), xrow(t1tok), xi, p.H / 32, lane, g, u);
            }
            else
                dot2_fp8<NT>(c1, reinterpret_cast<const float*>(s1), c3, reinterpret_cast<const float*>(s3),
                             xrow(t0tok), xrow(t1tok), p.H / 16, lane, g, u);
        }
    }

    // Gate/up on the tensor cores (chunks of kind 5). The chunk's up to four
    // row pairs are the 8-column operand (column 2j gate row j, column 2j + 1
    // up row j), all tokens of the slot the 16-row one, and K = H is split
    // into kMmaParts parts handed to consecutive warps (continuing round-robin
    // from chunk to chunk); part q takes k-steps [q nks / P, (q + 1) nks / P)
    // of the nks = H / 16, with two accumulators. Parts 1.. write their 16 x 8
    // partial into the first two rows of their own k-range of the stage (bytes
    // no other warp reads) and arrive on the stage's partial barrier; the warp
    // of part 0 (the owner) waits for them, sums the parts in order, so that
    // each lane holds g and u of one row pair for two tokens, and stores h =
    // silu(g) * u in bf16. The owner's release of the stage comes after that
    // (its arrival completes the stage's empty barrier), so the partials stay
    // valid until it has read them.
    __device__ __forceinline__ bool gateup_mma(const Chunk& ch, const uint8_t* st) {
        constexpr int P = kMmaParts;
        const int part = claim_rows(P);
        const uint32_t rbar = ring.bars + (2u * ring.ns + 1u + ring.s) * 8u, rpar = (redph >> ring.s) & 1u;
        redph ^= 1u << ring.s;
        if (part >= P) return true;
        const int nks = p.H / 16;
        const uint32_t pitch = (uint32_t)p.H * 2 + 16, sbase = smem_u32(st);
        const int n = ch.n;
        const bool shared = ch.slot < 0;
        const int pbase = shared ? 0 : plan->slot_p0[ch.slot];
        const int npairs = shared ? p.M : plan->slot_p0[ch.slot + 1] - pbase;
        const int s0 = part * nks / P, s1 = (part + 1) * nks / P;
        const int nn = lane & 7, jr = (nn >> 1) < n ? nn >> 1 : 0;
        const uint32_t baddr = sbase + (uint32_t)((nn & 1) ? n + jr : jr) * pitch + ((lane >> 3) & 1) * 16u;
        const int qa = (lane & 7) + ((lane >> 3) & 1) * 8, khalf = lane >> 4;
        const int tq = qa < npairs ? qa : 0;
        const int tok = shared ? tq : plan->pair_tok[pbase + tq];
        const uint32_t arow = smem_u32(xs) + (uint32_t)tok * p.xp * 2 + (uint32_t)khalf * 16u;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        int ks = s0;
#pragma unroll 4
        for (; ks + 1 < s1; ks += 2) {
            uint32_t a[4], b[2], a2[4], b2[2];
            ldsm_x4(arow + (uint32_t)ks * 32u, a);
            ldsm_x2(baddr + (uint32_t)ks * 32u, b);
            ldsm_x4(arow + (uint32_t)ks * 32u + 32u, a2);
            ldsm_x2(baddr + (uint32_t)ks * 32u + 32u, b2);
            mma_bf16_16816(d0, a, b);
            mma_bf16_16816(d1, a2, b2);
        }
        if (ks < s1) {
            uint32_t a[4], b[2];
            ldsm_x4(arow + (uint32_t)ks * 32u, a);
            ldsm_x2(baddr + (uint32_t)ks * 32u, b);
            mma_bf16_16816(d0, a, b);
        }
        float acc[4] = {d0[0] + d1[0], d0[1] + d1[1], d0[2] + d1[2], d0[3] + d1[3]};
        // a part's 512-byte partial: lane l's 16 bytes in row l / per_row of
        // the stage, inside the part's own k-range
        auto slot_addr = [&](int q) {
            const int q0 = q * nks / P, per_row = ((q + 1) * nks / P - q0) * 2;
            return sbase + (uint32_t)(lane / per_row) * pitch + (uint32_t)q0 * 32u + (uint32_t)(lane % per_row) * 16u;
        };
        if (part > 0) {
            __syncwarp();  // every lane of this warp has read its k-range
            *reinterpret_cast<float4*>(__cvta_shared_to_generic(slot_addr(part))) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(rbar);
            return true;
        }
        if (!mbar_wait(rbar, rpar, p, plan)) return false;
#pragma unroll
        for (int q = 1; q < P; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(slot_addr(q)));
            acc[0] += v.x, acc[1] += v.y, acc[2] += v.z, acc[3] += v.w;
        }
        const int g = lane >> 2, t = lane & 3;
        if (t < n) {
            const int inter = shared ? p.Is : p.I;
            const int e = ch.r0 + t;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int q = g + 8 * half;
                if (q < npairs)
                    (shared ? p.hs : p.hr)[(size_t)(pbase + q) * inter + e] =
                        f32_to_bf16_bits(silu_mul(acc[2 * half], acc[2 * half + 1]));
            }
        }
        return true;
    }

    // Gate/up rows: one warp per row pair, all tokens of the slot; stores
    // h = silu(g) * u in bf16.
    __device__ __forceinline__ bool gateup(const Chunk& ch, const uint8_t* st) {
        if (MMA && ch.kind == 5) return gateup_mma(ch, st);
        const int j0 = claim_rows(ch.n);
        if (j0 >= ch.n) return true;
        const bool shared = ch.slot < 0;
        const int inter = shared ? p.Is : p.I;
        const int pbase = shared ? 0 : plan->slot_p0[ch.slot];
        const int npairs = shared ? p.M : plan->slot_p0[ch.slot + 1] - pbase;
        uint16_t* hdst = (shared ? p.hs : p.hr) + (size_t)pbase * inter;
        for (int j = j0; j < ch.n; j += NCW) {
            // column of this row in the activation rows (routed rows of
            // MXFP4 / FP8 layers are stored swizzled)
            const int e = ch.r0 + j;
            const int col = shared ? e : 8 * swz_vec(e >> 3, kXM<WFMT>) + (e & 7);
            int q0 = 0;
            for (; q0 + 2 <= npairs; q0 += 2) {
                const int ta = shared ? q0 : plan->pair_tok[pbase + q0];
                const int tb = shared ? q0 + 1 : plan->pair_tok[pbase + q0 + 1];
                float g[2], u[2];
                gateup_group<2>(st, ch, j, ta, tb, shared, g, u);
                // lanes 0 and 16 end with (g, u) of the pair's first and
                // second token
                float gs = warp_sum4(g[0], u[0], g[1], u[1], lane);
                float us = __shfl_down_sync(0xffffffffu, gs, 8);
                if ((lane & 15) == 0) {
                    // f16 tokens are held times 2^s_t (MXFP4); the routed
                    // MXFP4 dot removes it block by block
                    if (WFMT == 1 && shared && !TWO) {
                        const float xi = plan->x_inv[lane ? tb : ta];
                        gs *= xi, us *= xi;
                    }
                    hdst[(size_t)(q0 + (lane >> 4)) * inter + col] = f32_to_bf16_bits(silu_mul(gs, us));
                }
            }
            if (q0 < npairs) {
                const int ta = shared ? q0 : plan->pair_tok[pbase + q0];
                float g[1], u[1];
                gateup_group<1>(st, ch, j, ta, ta, shared, g, u);
                float gs = warp_sum2(g[0], u[0], lane);
                float us = __shfl_down_sync(0xffffffffu, gs, 16);
                if (lane == 0) {
                    if (WFMT == 1 && shared && !TWO) gs *= plan->x_inv[ta], us *= plan->x_inv[ta];
                    const uint32_t hv = f32_to_bf16_bits(silu_mul(gs, us));
                    if (WFMT == 0 && !MMA && p.htag)  // one token: the word carries the call's tag
                        st_relaxed_u32(p.htag + (shared ? 0 : p.Is + (size_t)(pbase + q0) * inter) + col,
                                       (htag16(plan) << 16) | hv);
                    else
                        hdst[(size_t)q0 * inter + col] = (uint16_t)hv;
                }
            }
        }
        return true;
    }

    // One-token bf16 layers: polls (bounded) the tagged activations of a down
    // chunk's pair where the CTAs store them until every tag is this call's,
    // all of a lane's loads issued before any is examined, and writes them
    // over the stage's copy (other warps may do the same: they write the same
    // words). False when the wait ran out or the CTA aborted.
    __device__ __noinline__ bool refresh_tagged_h(const Chunk& ch, const uint8_t* st) {
        const uint32_t tag = htag16(plan);
        const int inter = ch.slot < 0 ? p.Is : p.I;
        const uint32_t* src = p.htag + (ch.slot < 0 ? (size_t)ch.p0 * p.Is
                                                    : (size_t)p.Is + (size_t)(plan->slot_p0[ch.slot] + ch.p0) * p.I);
        uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(st));
        const int nv = inter / 4;  // 16-byte vectors
        for (int v0 = 0; v0 < nv; v0 += 8 * 32) {
            const uint64_t t0 = global_timer_ns();
            while (true) {
                uint4 w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int v = v0 + lane + 32 * j;
                    w[j] = make_uint4(tag << 16, tag << 16, tag << 16, tag << 16);
                    if (v < nv) w[j] = ld_relaxed_v4u32(src + 4 * v);
                }
                bool cur = true;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    cur &= (w[j].x >> 16) == tag && (w[j].y >> 16) == tag && (w[j].z >> 16) == tag &&
                           (w[j].w >> 16) == tag;
                if (__all_sync(0xffffffffu, cur)) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int v = v0 + lane + 32 * j;
                        if (v < nv) dst[v] = w[j];
                    }
                    break;
                }
                const bool stop = aborted(plan) || global_timer_ns() - t0 > p.timeout_ns;
                if (__any_sync(0xffffffffu, stop)) {
                    if (lane == 0 && !aborted(plan)) set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
                    return false;
                }
                __nanosleep(64);
            }
        }
        // the stage is next written by a bulk copy
        fence_proxy_async_shared();
        __syncwarp();
        return true;
    }

    // Down projection. A down chunk (one slot, a pair group, a block of
    // output rows) is split into parts of four consecutive rows; parts go
    // round-robin over the warps, continuing from chunk to chunk, so that the
    // chunks resident together are worked on by all warps at once. Each
    // (pair, row) result is written exactly once, unweighted, into ypair; the
    // weighted combine runs after the last chunk, in pair order.
    // MXFP4 routed down rows (I <= 1024: at most one 32-value block per
    // lane): one warp takes the whole segment, converts each pair's
    // activation block once (block_to_f16) and runs every four-row part of
    // the segment against it, instead of one part per warp each converting
    // the activations again (a third of the instructions of the part).
    __device__ __forceinline__ void down_seg_mx(const Chunk& ch, const uint8_t* st, int nparts) {
        if (claim_rows(1) != 0) return;
        const int gbase = p.M + plan->slot_p0[ch.slot] + ch.p0;
        const size_t s0 = ((size_t)plan->slot_e[ch.slot] * p.H + ch.r0) * (p.I / 32);
        const size_t sofs = s0 - (s0 & ~(size_t)15);
        const size_t hbytes = (size_t)ch.np * p.I * 2;
        const uint8_t* codes = st + hbytes;
        const uint8_t* scls = st + hbytes + (size_t)ch.n * (p.I / 2) + sofs;
        const int nblk = p.I / 32;
        const int bl = lane < nblk ? lane : 0;  // lanes past the blocks convert block 0 and add nothing
        int q0 = 0;
        for (; q0 + 2 <= ch.np; q0 += 2) {
            uint4 a[2][4];
            float inv[2];
#pragma unroll
            for (int t = 0; t < 2; ++t)
                inv[t] = block_to_f16(reinterpret_cast<const uint4*>(st + (size_t)(q0 + t) * p.I * 2) + 4 * bl,
                                      (bl >> 1) & 3, a[t]);
            for (int part = 0; part < nparts; ++part) {
                const int r = ch.r0 + 4 * part, nrow = min(4, ch.r0 + ch.n - r);
                const uint8_t* crow[4];
                const uint8_t* srow[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * part + min(jj, nrow - 1);
                    crow[jj] = codes + (size_t)j * (p.I / 2);
                    srow[jj] = scls + (size_t)j * nblk;
                }
                float acc[4][2];
                dot4_mxh_pre<2>(crow, srow, a, inv, nblk, lane, acc);
                reduce_store<2>(acc, nrow, ypair + (size_t)(gbase + q0) * p.rpc + (r - h0));
            }
        }
        if (q0 < ch.np) {
            uint4 a[1][4];
            float inv[1];
            inv[0] = block_to_f16(reinterpret_cast<const uint4*>(st + (size_t)q0 * p.I * 2) + 4 * bl, (bl >> 1) & 3,
                                  a[0]);
            for (int part = 0; part < nparts; ++part) {
                const int r = ch.r0 + 4 * part, nrow = min(4, ch.r0 + ch.n - r);
                const uint8_t* crow[4];
                const uint8_t* srow[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * part + min(jj, nrow - 1);
                    crow[jj] = codes + (size_t)j * (p.I / 2);
                    srow[jj] = scls + (size_t)j * nblk;
                }
                float acc[4][1];
                dot4_mxh_pre<1>(crow, srow, a, inv, nblk, lane, acc);
                reduce_store<1>(acc, nrow, ypair + (size_t)(gbase + q0) * p.rpc + (r - h0));
            }
        }
    }

    __device__ __forceinline__ void down(const Chunk& ch, const uint8_t* st) {
        if (WFMT != 0 && ch.kind == 6) {
            // packed routed slots: each segment as a kind-2 chunk (its parts
            // continue the round-robin over the warps)
            uint32_t off = 0;
            for (int k = 0; k < ch.np; ++k) {
                const int slot = ch.slot + k;
                const int npairs = plan->slot_p0[slot + 1] - plan->slot_p0[slot];
                down_seg(Chunk{2, slot, ch.r0, ch.n, 0, npairs}, st + off);
                off += down_seg_bytes<WFMT>(p, npairs, ch.n);
            }
            return;
        }
        down_seg(ch, st);
    }

    __device__ __forceinline__ void down_seg(const Chunk& ch, const uint8_t* st) {
        const int nparts = (ch.n + 3) >> 2;
        if (WFMT == 1 && ch.slot >= 0 && p.I <= 1024 && !(!MMA && p.htag)) {
            down_seg_mx(ch, st, nparts);
            return;
        }
        const int part0 = claim_rows(nparts);
        if (part0 >= nparts) return;
        const bool shared = ch.slot < 0;
        const int gbase = (shared ? 0 : p.M + plan->slot_p0[ch.slot]) + ch.p0;  // pair index of q0 = 0
        size_t sofs = 0;
        if (WFMT != 0 && !shared) {
            const size_t s0 = ((size_t)plan->slot_e[ch.slot] * p.H + ch.r0) * (p.I / 32);
            sofs = s0 - (s0 & ~(size_t)15);
        }
        const int inter = shared ? p.Is : p.I;
        if (WFMT == 0 && !MMA && p.htag) {
            // one token (one pair a chunk), tagged activations in the stage
            const uint4* ht = reinterpret_cast<const uint4*>(st);
            const int rstride = inter / 8;
            const uint32_t tag = htag16(plan);
            for (int part = part0; part < nparts; part += NCW) {
                const int r = ch.r0 + 4 * part;
                const int nrow = min(4, ch.r0 + ch.n - r);
                const uint4* row0 = reinterpret_cast<const uint4*>(st + (size_t)inter * 4 + (size_t)(r - ch.r0) * inter * 2);
                float acc[4][1];
                for (int attempt = 0;; ++attempt) {
                    const bool cur = dot4_bf16_tagged(row0, rstride, nrow, ht, rstride, lane, tag, acc);
                    if (__all_sync(0xffffffffu, cur)) break;
                    // the stage's copy came before every CTA had stored this
                    // pair: read it again where the CTAs store it
                    if (attempt > 0) {  // cannot happen: the refreshed words are all current
                        set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
                        return;
                    }
                    if (!refresh_tagged_h(ch, st)) return;
                }
                reduce_store<1>(acc, nrow, ypair + (size_t)gbase * p.rpc + (r - h0));
            }
            return;
        }
        for (int part = part0; part < nparts; part += NCW) {
            const int r = ch.r0 + 4 * part;
            const int nrow = min(4, ch.r0 + ch.n - r);
            float* out = ypair + (size_t)gbase * p.rpc + (r - h0);
            if (WFMT == 0 || shared) {
                const size_t hb = (size_t)ch.np * inter * 2;
                const int rstride = inter / 8;  // uint4 per row
                const uint4* row0 = reinterpret_cast<const uint4*>(st + hb + (size_t)(r - ch.r0) * inter * 2);
                int q0 = 0;
                for (; q0 + 2 <= ch.np; q0 += 2) {
                    float acc[4][2];
                    const uint4* ha = reinterpret_cast<const uint4*>(st + (size_t)q0 * inter * 2);
                    if (nrow > 1) {
                        dot4_bf16<2>(row0, rstride, nrow, ha, ha + rstride, rstride, lane, acc);
                    } else {
                        float a1[2];
                        dot_bf16<2>(row0, ha, ha + rstride, rstride, lane, a1);
                        acc[0][0] = a1[0];
                        acc[0][1] = a1[1];
                    }
                    reduce_store<2>(acc, nrow, out + (size_t)q0 * p.rpc);
                }
                if (q0 < ch.np) {
                    float acc[4][1];
                    const uint4* ha = reinterpret_cast<const uint4*>(st + (size_t)q0 * inter * 2);
                    if (nrow > 1) {
                        dot4_bf16<1>(row0, rstride, nrow, ha, ha, rstride, lane, acc);
                    } else {
                        float a1[1];
                        dot_bf16<1>(row0, ha, ha, rstride, lane, a1);
                        acc[0][0] = a1[0];
                    }
                    reduce_store<1>(acc, nrow, out + (size_t)q0 * p.rpc);
                }
                continue;
            }
            // MXFP4 / FP8 routed rows (rows past the part's end repeat its
            // last row; their results are dropped)
            constexpr int CD = WFMT == 1 ? 2 : 1;
            const size_t hbytes = (size_t)ch.np * p.I * 2;
            const uint8_t* codes = st + hbytes;
            const uint8_t* scls = st + hbytes + (size_t)ch.n * (p.I / CD) + sofs;
            const int nblk = p.I / 32;
            const uint8_t* crow[4];
            const uint8_t* srow[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = r - ch.r0 + min(jj, nrow - 1);
                crow[jj] = codes + (size_t)j * (p.I / CD);
                srow[jj] = scls + (size_t)j * nblk;
            }
            int q0 = 0;
            for (; q0 + 2 <= ch.np; q0 += 2) {
                float acc[4][2];
                const uint4* ha = reinterpret_cast<const uint4*>(st + (size_t)q0 * p.I * 2);
                if (WFMT == 1)
                    dot4_mxh<2>(crow, srow, ha, ha + p.I / 8, nblk, lane, acc);
                else
                    dot4_fp8<2>(crow, srow, ha, ha + p.I / 8, p.I / 16, lane, acc);
                reduce_store<2>(acc, nrow, out + (size_t)q0 * p.rpc);
            }
            if (q0 < ch.np) {
                float acc[4][1];
                const uint4* ha = reinterpret_cast<const uint4*>(st + (size_t)q0 * p.I * 2);
                if (WFMT == 1)
                    dot4_mxh<1>(crow, srow, ha, ha, nblk, lane, acc);
                else
                    dot4_fp8<1>(crow, srow, ha, ha, p.I / 16, lane, acc);
                reduce_store<1>(acc, nrow, out + (size_t)q0 * p.rpc);
            }
        }
    }

    // Warp sums of a four-row group's lane partials, four rows per
    // butterfly (row jj ends in lanes 8 jj .. 8 jj + 7); lane 8 jj stores
    // row jj, if jj < nrow, for each of the NT pairs (pair stride rpc).
    template <int NT>
    __device__ __forceinline__ void reduce_store(float (&acc)[4][NT], int nrow, float* out) const {
        const int jj = lane >> 3;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float a = warp_sum4(acc[0][t], acc[1][t], acc[2][t], acc[3][t], lane);
            if ((lane & 7) == 0 && jj < nrow) out[(size_t)t * p.rpc + jj] = a;
        }
    }

    // Consumes the chunks of one phase, up to its end marker: waits for each
    // stage, reads its descriptor, computes this warp's share, frees it.
    __device__ __forceinline__ bool consume_phase() {
        while (true) {
            if (!wait_full()) return false;
            const Chunk ch = plan->desc[ring.s];
            if (ch.kind == 3) {
                release();
                return true;
            }
            const uint8_t* st = stage_ptr();
            if (ch.kind == 0)
                router(ch, st);
            else if (ch.kind == 1 || ch.kind == 5) {
                if (!gateup(ch, st)) return false;
            } else {
                down(ch, st);
            }
            release();
        }
    }
};

// ------------------------------------------------------------ routing + plan

// Order-preserving map of an fp32 value to a u32 key (larger value ->
// larger key), and back; hardware warp reductions on u32 then rank logits.
__device__ __forceinline__ uint32_t f32_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Scores, top-k and routing weights for one token, by one warp. The logits
// come from every CTA as 64-bit words (logit, tag): the warp reads them with
// relaxed loads until every tag is this call's (a bounded wait; no grid
// barrier). Lane l holds experts 64j + 2l and 64j + 2l + 1 (EPL of them).
//  - Plain softmax router (no bias): the logits themselves are ranked (the
//    same order as the probabilities); w_j = exp(l_j - max) / sum over the
//    selected of exp(l - max) (the full softmax denominator cancels).
//  - Otherwise the scores s (softmax over all E, or the sigmoid of each
//    logit) plus the expert's bias are ranked, and w_j = s_j / sum over the
//    selected of s.
// Ties go to the lower expert index; the weights are multiplied by the
// routed scaling factor. Each of the k rounds takes the warp maximum of the
// ranking keys with one hardware reduction and the lowest expert index
// among the lanes holding it with a second; the winning lane drops the entry
// and rescans. The code stays small on purpose: it runs once per launch, so
// its instructions are fetched cold. Returns false when the wait ran out
// (the CTA is then aborted).
// PUBNUM (split-K one-token layer): each published slot also carries its
// unnormalised weight (exp(l_j - l_max), or the score s_j), and the final
// factor routed_scale / sum is published once all k rounds are done.
template <int EPL, bool VAR, bool PUBNUM = false>
__device__ __noinline__ bool topk_warp(const unsigned long long* __restrict__ lrow, const int E, const int k,
                                       int lane, uint32_t tag, const LayerParams& p, Plan* plan,
                                       const float* __restrict__ bias, int32_t* __restrict__ sel_e,
                                       float* __restrict__ sel_w, bool publish) {
    float lg[EPL];
    uint64_t t0 = 0;
    for (int spin = 0;; ++spin) {
        // all of a lane's loads are issued before any of their words is
        // examined, so that one poll costs one round trip, not EPL / 2
        unsigned long long wa[EPL / 2], wb[EPL / 2];
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j) {
            const int e = 64 * j + 2 * lane;
            wa[j] = wb[j] = 0ull;
            if (e < E) ld_relaxed_v2u64(lrow + e, wa[j], wb[j]);
        }
        bool ok = true;
#pragma unroll
        for (int j = 0; j < EPL / 2; ++j) {
            const int e = 64 * j + 2 * lane;
            lg[2 * j] = lg[2 * j + 1] = -INFINITY;
            if (e < E) {
                ok &= (uint32_t)(wa[j] >> 32) == tag;
                lg[2 * j] = __uint_as_float((uint32_t)wa[j]);
                if (e + 1 < E) {
                    ok &= (uint32_t)(wb[j] >> 32) == tag;
                    lg[2 * j + 1] = __uint_as_float((uint32_t)wb[j]);
                }
            }
        }
        if (__all_sync(0xffffffffu, ok)) {
            if (publish && lane == 0) trace_mark(p, 3);  // every tag of this call seen
            break;
        }
        if (spin == 0) t0 = global_timer_ns();
        if (aborted(plan)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            if (lane == 0) set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
            __syncwarp();
            return false;
        }
        __nanosleep(64);
    }
    auto idx_of = [lane](int j) { return (uint32_t)(64 * (j >> 1) + 2 * lane + (j & 1)); };
    // VAR: unbiased scores and biased ranking keys; else the logits themselves
    constexpr bool by_logit = !VAR;
    float sc[EPL];
    uint32_t key[EPL];
    if (by_logit) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) sc[j] = lg[j];
    } else if (p.scoring == 0) {
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < EPL; ++j) mx = fmaxf(mx, lg[j]);
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            sc[j] = (uint32_t)idx_of(j) < (uint32_t)E ? expf(lg[j] - mx) : 0.f;
            den += sc[j];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
#pragma unroll
        for (int j = 0; j < EPL; ++j) sc[j] = sc[j] / den;
    } else {
#pragma unroll
        for (int j = 0; j < EPL; ++j) sc[j] = 1.0f / (1.0f + expf(-lg[j]));
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const uint32_t e = idx_of(j);
        float kv = sc[j];
        if (!by_logit && bias && e < (uint32_t)E) kv += bias[e];
        // -0 and +0 rank as equal (ties go to the lower index)
        key[j] = e < (uint32_t)E ? f32_key(kv == 0.f ? 0.f : kv) : 0u;
    }
    uint32_t bk = 0u, bi = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        if (key[j] > bk) {
            bk = key[j];
            bi = idx_of(j);
        }
    float mine = 0.f, first = 0.f;
    for (int jj = 0; jj < k; ++jj) {
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t we = __reduce_min_sync(0xffffffffu, bk == wk ? bi : 0xffffffffu);
        float ws = 0.f;
        if (lane == 0) {
            sel_e[jj] = (int32_t)we;
            if (publish && !PUBNUM) {  // slot jj is the jj-th selected expert: its tiles may stream now
                plan->slot_e[jj] = (int16_t)we;
                st_release_cta(&plan->known, jj + 1);
            }
        }
        if (we == bi) {  // this lane won: take its score, drop the entry, find the next best
            bk = 0u;
            bi = 0xffffffffu;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                if (idx_of(j) == we) {
                    ws = sc[j];
                    key[j] = 0u;
                }
                if (key[j] > bk) {
                    bk = key[j];
                    bi = idx_of(j);
                }
            }
        }
        if (by_logit)
            ws = key_f32(wk);  // the winning key is the logit itself
        else
            ws = __shfl_sync(0xffffffffu, ws, (int)((we & 63u) >> 1));  // from the winning lane
        if (jj == 0) first = ws;
        if (lane == jj) mine = ws;
        if (PUBNUM && publish && lane == 0) {  // the slot and its unnormalised weight
            plan->slot_e[jj] = (int16_t)we;
            plan->slot_num[jj] = by_logit ? expf(ws - first) : ws;
            st_release_cta(&plan->known, jj + 1);
        }
    }
    if (publish && lane == 0) trace_mark(p, 15);  // k rounds done
    const float num = lane < k ? (by_logit ? expf(mine - first) : mine) : 0.f;
    float den = num;
#pragma unroll
    for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane < k) sel_w[lane] = num / den * p.routed_scale;
    if (PUBNUM && publish && lane == 0) plan->wscale = p.routed_scale / den;
    return true;
}

static __device__ __forceinline__ void topk_tokens(const LayerParams& p, Plan* plan, const float* bias, int warp,
                                                   int lane, int nwarps, bool publish) {
    // the debug hook waits for a tag that never comes
    const uint32_t tag = plan->tag + (p.force_timeout ? 1u : 0u);
    for (int t = warp; t < p.M; t += nwarps) {
        const unsigned long long* lrow = p.logits + (size_t)t * p.Es;
        int32_t* se = plan->sel_e + t * p.k;
        float* sw = plan->sel_w + t * p.k;
        const bool var = p.scoring != 0 || p.bias != nullptr;
        bool ok;
        const bool pub = publish && t == 0;
        if (p.E <= 512)
            ok = var ? topk_warp<16, true>(lrow, p.E, p.k, lane, tag, p, plan, bias, se, sw, pub)
                     : topk_warp<16, false>(lrow, p.E, p.k, lane, tag, p, plan, bias, se, sw, pub);
        else
            ok = var ? topk_warp<32, true>(lrow, p.E, p.k, lane, tag, p, plan, bias, se, sw, pub)
                     : topk_warp<32, false>(lrow, p.E, p.k, lane, tag, p, plan, bias, se, sw, pub);
        if (!ok) return;
    }
}

// Groups the M*k (token, expert) entries by expert with one pairwise pass per
// entry: rank = (#entries with a smaller expert id) + (#earlier entries with
// the same id). Nothing here scales with E. Entries whose expert id lies
// outside [0, E) (possible only when the routing is given) are dropped and
// reported.
static __device__ void build_plan(const LayerParams& p, Plan* plan, int tid, int nct, bool report) {
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
    named_bar_sync(1, nct);
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
    named_bar_sync(1, nct);
}

// Tokens into shared memory, one warp per token, for the cases that need
// arithmetic. With a norm weight g the input is the residual stream h and the
// token is x = bf16(h / rms * g), rms = sqrt(mean(h^2) + eps). MXFP4 layers
// hold the tokens in f16 times 2^s_t (x_inv[t] = 2^-s_t), s_t chosen from
// the token's largest magnitude (exact for bf16 values in f16's normal
// range). Token row t starts xpv vectors after row t - 1. Not inlined: it
// runs once per launch and keeps the kernel's other code compact; its
// arguments are plain values.
template <int WFMT, bool TWO>
__device__ __noinline__ void load_tokens(const uint4* __restrict__ src, const uint4* __restrict__ gam, int M, int H,
                                         int xpv, float eps, uint4* __restrict__ dst, uint4* __restrict__ dstb,
                                         float* __restrict__ x_inv, int warp, int lane, int nwarps) {
    const int nvt = H / 8;
    for (int t = warp; t < M; t += nwarps) {
        const uint4* ht = src + (size_t)t * nvt;
        float r = 1.f;
        if (gam) {
            float ss = 0.f;
            for (int i = lane; i < nvt; i += 32) {
                float f[8];
                unpack8(__ldg(ht + i), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
            ss = warp_sum(ss);
            r = 1.0f / sqrtf(ss / (float)H + eps);
        }
        auto token_vec = [&](int i, float (&f)[8]) {
            unpack8(__ldg(ht + i), f);
            if (gam) {
                float g[8];
                unpack8(__ldg(gam + i), g);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = bf16lo(f32_to_bf16_bits(f[e] * r * g[e]));
            }
        };
        if (WFMT != 1) {
            for (int i = lane; i < nvt; i += 32) {
                float f[8];
                token_vec(i, f);
                uint4 v;
                v.x = f32_to_bf16_bits(f[0]) | ((uint32_t)f32_to_bf16_bits(f[1]) << 16);
                v.y = f32_to_bf16_bits(f[2]) | ((uint32_t)f32_to_bf16_bits(f[3]) << 16);
                v.z = f32_to_bf16_bits(f[4]) | ((uint32_t)f32_to_bf16_bits(f[5]) << 16);
                v.w = f32_to_bf16_bits(f[6]) | ((uint32_t)f32_to_bf16_bits(f[7]) << 16);
                dst[(size_t)t * xpv + swz_vec(i, kXM<WFMT>)] = v;
            }
            continue;
        }
        float mx = 0.f;
        for (int i = lane; i < nvt; i += 32) {
            float f[8];
            token_vec(i, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(f[e]));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int sh = f16_range_shift(mx);
        const float sc = exp2i(sh);
        for (int i = lane; i < nvt; i += 32) {
            float f[8];
            token_vec(i, f);
            uint4 v;
            v.x = f32x2_to_f16x2(f[0] * sc, f[1] * sc);
            v.y = f32x2_to_f16x2(f[2] * sc, f[3] * sc);
            v.z = f32x2_to_f16x2(f[4] * sc, f[5] * sc);
            v.w = f32x2_to_f16x2(f[6] * sc, f[7] * sc);
            dst[(size_t)t * xpv + swz_vec(i, kXM<WFMT>)] = v;
            if (TWO) {  // the plain bf16 copy (the values are bf16 already)
                uint4 b;
                b.x = f32_to_bf16_bits(f[0]) | ((uint32_t)f32_to_bf16_bits(f[1]) << 16);
                b.y = f32_to_bf16_bits(f[2]) | ((uint32_t)f32_to_bf16_bits(f[3]) << 16);
                b.z = f32_to_bf16_bits(f[4]) | ((uint32_t)f32_to_bf16_bits(f[5]) << 16);
                b.w = f32_to_bf16_bits(f[6]) | ((uint32_t)f32_to_bf16_bits(f[7]) << 16);
                dstb[(size_t)t * nvt + i] = b;
            }
        }
        if (lane == 0) x_inv[t] = exp2i(-sh);
    }
}

// Routed gate/up rows, scheduled dynamically: the rows of all slots form one
// list of chunks (slot by slot, cap row pairs each), and every CTA's
// producer claims the next chunk from a global counter, so that CTAs that
// run ahead take more. Two claims are kept in flight to hide the atomic's
// latency. Which CTA computes a row does not change its result.
// With one token (incremental plan) the slots are the selected experts in
// selection order, published one top-k round at a time: a claim waits
// (bounded) until its slot is known, so the first expert's tiles stream
// while the top-k is still ranking the others.
template <int WFMT>
__device__ __forceinline__ bool wait_known(const LayerParams& p, Plan* plan, int n) {
    if (ld_acquire_cta(&plan->known) >= n) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        __nanosleep(32);
        if (ld_acquire_cta(&plan->known) >= n) return true;
        if ((spin & 15u) == 0) {
            if (aborted(plan)) return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
                return false;
            }
        }
    }
}

template <int WFMT, bool PAD>
__device__ __forceinline__ bool issue_routed_gateup(Producer<WFMT, PAD>& pr, const LayerParams& p, Plan* plan,
                                                    bool incremental) {
    const uint32_t cap = (uint32_t)gateup_cap<WFMT, PAD>(p, true), I = (uint32_t)p.I;
    const uint32_t cps = (I + cap - 1) / cap;  // chunks per slot
    if (incremental && !wait_known<WFMT>(p, plan, 1)) return false;
    // the plan (or the first slot) is published after the consumers stored
    // the call's epoch
    pr.epoch = plan->epoch;
    const uint32_t U = (uint32_t)plan->nslot * cps;
    unsigned* wc = ctl_work(p, pr.epoch);
    // Each claim takes two consecutive chunks, and the next claim is in
    // flight while a chunk is issued: half the atomics on the one counter
    // that every CTA hits (with one chunk per claim the counter's queue held
    // the stream back: bf16 M = 1 24.4 -> 23.9 us; four per claim leave a
    // longer tail).
    constexpr uint32_t kPer = 2;
    uint32_t a = atomicAdd(wc, 1u), b = atomicAdd(wc, 1u);
    bool ok = true;
    while (ok && kPer * a < U) {
        uint32_t nxt = 0;
        for (uint32_t h = 0; h < kPer; ++h) {
            const uint32_t u = kPer * a + h;
            if (h == 0) nxt = atomicAdd(wc, 1u);
            if (u >= U) break;
            const uint32_t slot = u / cps, r0 = (u - slot * cps) * cap;
            if (incremental && !wait_known<WFMT>(p, plan, (int)slot + 1)) return false;
            const Chunk c{1, (int)slot, (int)r0, (int)min(cap, I - r0), 0, 0};
            ok = pr.issue(c);
            if (!ok) break;
        }
        a = b;
        b = nxt;
    }
    // the down tiles that follow need every slot's expert
    if (ok && incremental) ok = wait_known<WFMT>(p, plan, plan->nslot);
    return ok;
}

// ------------------------------------------------------------ the kernel
// IO: the input is normalised in the kernel and/or the residual is added
// (compiled only into the launches that ask for it). ONE: a one-token layer
// launch (route + FFN, M = 1), whose plan is built incrementally; a separate
// instantiation, so that the general kernel's code stays as it is.
template <int WFMT, bool IO, bool ONE>
__global__ void __launch_bounds__(block_threads(WFMT), 1) moe_layer_kernel(const __grid_constant__ LayerParams p) {
    constexpr int NCW = consumer_warps(WFMT);
    constexpr int NCT = NCW * 32;
    // one-token bf16 launches: tagged activations instead of grid barrier 2
    const bool tagged = ONE && WFMT == 0 && p.htag != nullptr;
    // bf16 experts with more than a one-token plan: the tensor-core path
    constexpr bool MMA = WFMT == 0 && !ONE;
    extern __shared__ __align__(1024) uint8_t smem[];
    // Early trigger: the next launch on the stream may start its prologue
    // (weight prefetch) as soon as SMs free up; it still waits for this grid
    // before reading anything this grid writes.
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = (int)blockIdx.x;
    Plan* plan = reinterpret_cast<Plan*>(smem + p.off_plan);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + p.off_x);
    float* ypair = reinterpret_cast<float*>(smem + p.off_yacc);
    const uint32_t bars = smem_u32(smem + p.off_bar);
    const uint32_t plan_bar = bars + 2u * p.ns * 8u;
    if (tid == 0) {
        for (int i = 0; i < p.ns; ++i) {
            mbar_init(bars + i * 8, 1);
            mbar_init(bars + (p.ns + i) * 8, NCW);
        }
        mbar_init(plan_bar, 1);
        if (MMA)  // per-stage barriers of the tensor-core chunks' partials
            for (int i = 0; i < p.ns; ++i) mbar_init(plan_bar + 8u + i * 8u, kMmaParts - 1);
        plan->abort = 0;
        plan->npend = 0;
        plan->known = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) trace_mark(p, 0);

    const Ring ring0{smem_u32(smem), bars, (uint32_t)p.ns, 0u, 0u, 0u};
    const bool has_route = (p.mode & kModeRoute) != 0, has_ffn = (p.mode & kModeFfn) != 0;
    // One token: the plan is built incrementally, one slot per top-k round
    constexpr bool incremental = ONE;
    ChunkGen<WFMT, MMA> gen;
    Chunk ch;

    if (warp == NCW) {
        // ---------------- producer (one elected lane)
        if (lane == 0) {
            trace_mark(p, 8);
            Producer<WFMT, MMA> pr{p, plan, ring0, policy_evict_first(), policy_evict_last(), false, 0u, 0u};
            bool ok = true;
            // producer-independent tiles: router rows, shared-expert gate/up
            // rows; an end marker closes each phase of the consumers
            if (has_route) {
                for (gen.begin(0, p, plan, cta); ok && gen.next(p, plan, ch);) ok = pr.issue(ch);
                if (ok) ok = pr.issue_end();
            }
            if (has_ffn)
                for (gen.begin(1, p, plan, cta); ok && gen.next(p, plan, ch);) ok = pr.issue(ch);
            trace_mark(p, 9);
            pdl_wait();
            if (ok && has_ffn) {
                if (!incremental) ok = mbar_wait(plan_bar, 0, p, plan);
                trace_mark(p, 10);
                if (ok) ok = issue_routed_gateup(pr, p, plan, incremental);
                if (ok) ok = pr.issue_end();
                trace_mark(p, 11);
                if (ok)
                    for (gen.begin(3, p, plan, cta); ok && gen.next(p, plan, ch);) ok = pr.issue(ch);
                if (ok) ok = pr.issue_end();
                trace_mark(p, 12);
                if (!tagged) {
                    if (ok) ok = pr.poll_b2(true);
                } else if (ok && cta == 0) {
                    // no barrier 2: every CTA counted itself in once it had
                    // read the epoch (long done by now)
                    if ((ok = grid_wait(ctl_entry(p, pr.epoch), (unsigned)p.G, p, plan))) advance_epoch(p, pr.epoch);
                }
                trace_mark(p, 13);
            }
            if (!ok || aborted(plan)) pr.drain();
            trace_mark(p, 14);
        }
    } else {
        // ---------------- consumers
        const int h0 = (int)((uint32_t)cta * (uint32_t)p.H / (uint32_t)p.G);
        const int h1 = (int)((uint32_t)(cta + 1) * (uint32_t)p.H / (uint32_t)p.G);
        constexpr bool TWO = ONE && WFMT == 1;
        Consumer<WFMT, TWO, MMA> cs{p, plan, ring0, xs, reinterpret_cast<const uint16_t*>(smem + p.off_xb), ypair,
                                    warp, lane, 0, h0, 0u};
        const float* bias_s = p.bias ? reinterpret_cast<const float*>(smem + p.off_bias) : nullptr;
        // The router's selection bias is a model parameter, not an output of
        // the previous launch: it is staged before the dependency wait.
        if (p.bias)
            for (int i = tid; i < p.E; i += NCT) const_cast<float*>(bias_s)[i] = __ldg(p.bias + i);
        pdl_wait();
        // The call's epoch and the status word, read by the last consumer
        // warp (which loads no token vectors at M = 1), both loads in flight
        // together and alongside the token loads.
        const bool ctl_thread = tid == NCT - 32;
        uint32_t ctl_epoch = 0, ctl_status = 0;
        if (ctl_thread) {
            ctl_epoch = ld_relaxed_gpu(p.ctrl + kCtlEpoch);
            ctl_status = ld_relaxed_gpu(p.ctrl + kCtlStatus);
        }
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.x);
            uint4* dst = reinterpret_cast<uint4*>(xs);
            const int nv = p.M * p.H / 8;
            if (IO) {
                load_tokens<WFMT, TWO>(src, reinterpret_cast<const uint4*>(p.gamma), p.M, p.H, p.xp / 8, p.eps, dst,
                                       reinterpret_cast<uint4*>(smem + p.off_xb), plan->x_inv, warp, lane, NCW);
            } else if (WFMT == 0 && p.xp != p.H) {
                const int nvt = p.H / 8, xpv = p.xp / 8;
                for (int i = tid; i < nv; i += NCT) {
                    const int t = i / nvt;
                    dst[i + t * (xpv - nvt)] = __ldg(src + i);
                }
            } else if (WFMT == 0) {
                for (int i = tid; i < nv; i += NCT) dst[i] = __ldg(src + i);
            } else if (WFMT == 2) {
                const int nvt = p.H / 8;
                for (int i = tid; i < nv; i += NCT) {
                    const int v = i % nvt;
                    dst[i - v + swz_vec(v, kXM<WFMT>)] = __ldg(src + i);
                }
            } else {
                // MXFP4 layers hold the tokens in f16 times 2^s_t, s_t chosen
                // from the token's largest magnitude (exact for bf16 values
                // in f16's normal range); one-token launches also keep the
                // plain bf16 copy
                if (TWO) {
                    uint4* dstb = reinterpret_cast<uint4*>(smem + p.off_xb);
                    for (int i = tid; i < nv; i += NCT) dstb[i] = __ldg(src + i);
                }
                const int nvt = p.H / 8;
                for (int t = warp; t < p.M; t += NCW) {
                    float mx = 0.f;
                    for (int i = lane; i < nvt; i += 32) {
                        float f[8];
                        unpack8(__ldg(src + (size_t)t * nvt + i), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(f[e]));
                    }
#pragma unroll
                    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
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
                        dst[(size_t)t * nvt + swz_vec(i, kXM<WFMT>)] = v;
                    }
                    if (lane == 0) plan->x_inv[t] = exp2i(-sh);
                }
            }
            if (!has_route)
                for (int i = tid; i < p.M * p.k; i += NCT) {
                    plan->sel_e[i] = p.idx_in[i];
                    plan->sel_w[i] = p.w_in[i];
                }
        }
        if (ctl_thread) {
            plan->epoch = ctl_epoch;
            plan->tag = ctl_epoch % 0xffffffffu + 1u;
            // a call that ran out of time left the control words stale: every
            // later call on this workspace refuses to run until it is zeroed
            if ((int)ctl_status == -101 /* MOE_ETIMEOUT */) set_abort(p, plan, -101);
            if (tagged) red_add_relaxed_gpu(ctl_entry(p, ctl_epoch), 1u);
        }
        named_bar_sync(1, NCT);
        if (tid == 0) trace_mark(p, 1);
        bool ok = true;
        if (has_route && incremental) {
            ok = cs.consume_phase();
            if (tid == 0) trace_mark(p, 2);
            // One token: the k selected experts are distinct, and slot s is
            // the s-th one selected (one pair each). Warp 0 ranks the token
            // and publishes each slot as its round completes; the producer
            // starts streaming that expert's gate/up tiles at once. The
            // other warps go straight on to the ring. The combine still
            // sums the pairs in ascending expert order (plan->order).
            if (warp == 0) {
                for (int i = lane; i <= p.k; i += 32) plan->slot_p0[i] = (int16_t)i;
                for (int i = lane; i < p.k; i += 32) plan->pair_tok[i] = 0;
                if (lane == 0) {
                    plan->nslot = p.k;
                    plan->npairs = p.k;
                }
                __syncwarp();
                if (!aborted(plan)) topk_tokens(p, plan, bias_s, warp, lane, 1, true);
                if (tid == 0) trace_mark(p, 4);
                __syncwarp();
                if (lane < p.k && !aborted(plan)) {
                    const int e = plan->sel_e[lane];
                    plan->pair_w[lane] = plan->sel_w[lane];
                    int rk = 0;
                    for (int j = 0; j < p.k; ++j) rk += plan->sel_e[j] < e;
                    plan->order[rk] = (int16_t)lane;
                    if (cta == 0) {
                        if (p.idx_out) p.idx_out[lane] = e;
                        if (p.w_out) p.w_out[lane] = plan->sel_w[lane];
                    }
                }
                if (tid == 0) trace_mark(p, 5);
            }
        } else if (has_route) {
            ok = cs.consume_phase();
            if (tid == 0) trace_mark(p, 2);
            // no grid barrier: each token's warp waits for the tagged logits
            if (!aborted(plan)) topk_tokens(p, plan, bias_s, warp, lane, NCW, false);
            if (tid == 0) trace_mark(p, 4);
            named_bar_sync(1, NCT);
            if (cta == 0 && !aborted(plan)) {
                for (int i = tid; i < p.M * p.k; i += NCT) {
                    if (p.idx_out) p.idx_out[i] = plan->sel_e[i];
                    if (p.w_out) p.w_out[i] = plan->sel_w[i];
                }
            }
        }
        if (has_ffn) {
            if (!incremental) {
                build_plan(p, plan, tid, NCT, cta == 0);
                if (tid == 0) {
                    mbar_arrive(plan_bar);
                    trace_mark(p, 5);
                }
            }
            // the shared expert's tiles were fetched before routing finished;
            // computing them now overlaps the first routed tiles' latency
            // one token: the first row goes to warp 1, so that the top-k warp
            // (warp 0, busy ranking) owns none of the shared expert's rows
            // and their stages free up without waiting for it
            cs.qm = incremental ? 1 : 0;
            if (ok) ok = cs.consume_phase();  // shared, then routed gate/up
            named_bar_sync(1, NCT);  // this CTA's activations are stored
            if (tid == 0) trace_mark(p, 6);
            if (tid == 0 && !aborted(plan) && !tagged) {
                __threadfence();
                atomicAdd(ctl_bar2(p, plan->epoch), 1u);
            }
            if (ok) ok = cs.consume_phase();  // down
            named_bar_sync(1, NCT);
            if (tid == 0) trace_mark(p, 7);
            if (!aborted(plan)) {
                const int nr = h1 - h0;
                // y[t][r] = shared(t)[r] + sum over routed pairs of token t, in
                // ascending expert order, of w * down(pair)[r]
                const int npr = plan->npairs;
                for (int i = tid; i < p.M * nr; i += NCT) {
                    const int t = i / nr, r = i - t * nr;
                    float v = p.Is > 0 ? ypair[(size_t)t * p.rpc + r] : 0.f;
                    if (incremental) {  // one token: its k pairs, in the published order
                        for (int qq = 0; qq < npr; ++qq) {
                            const int q = plan->order[qq];
                            v = fmaf(plan->pair_w[q], ypair[(size_t)(1 + q) * p.rpc + r], v);
                        }
                    } else {  // pairs are grouped by ascending expert
                        for (int q = 0; q < npr; ++q)
                            if (plan->pair_tok[q] == t)
                                v = fmaf(plan->pair_w[q], ypair[(size_t)(p.M + q) * p.rpc + r], v);
                    }
                    if (IO && p.residual) v += bf16lo(p.x[(size_t)t * p.H + h0 + r]);  // the layer's input
                    p.y[(size_t)t * p.H + h0 + r] = f32_to_bf16_bits(v);
                }
            }
        }
    }
    if (!has_ffn) {
        // A routing-only call has no grid barrier: the last CTA out advances
        // the epoch (the next call's logit tag).
        __syncthreads();
        if (tid == 0 && !aborted(plan)) {
            __threadfence();
            const unsigned old = atomicAdd(p.ctrl + kCtlExit, 1u);
            if (old == (unsigned)p.G - 1u) {
                atomicExch(p.ctrl + kCtlExit, 0u);
                advance_epoch(p, plan->epoch);
            }
        }
    }
}

}  // namespace moe
