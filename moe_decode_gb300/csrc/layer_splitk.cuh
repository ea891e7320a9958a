// One-token fused MoE layer with a split-K down projection (bf16 experts).
//
// With one token the down projection needs no token grouping, so it can be
// split along the intermediate dimension instead of the output dimension:
// the CTA that computes h[i] = silu(W1[i] x) * (W3[i] x) for a few rows i of
// an expert also streams the matching rows of the expert's transposed down
// projection W2^T [I, H] (one contiguous H-row per i) and accumulates
// w * h[i] * W2^T[i, :] into its own partial output. Gate, up and down rows
// of the same i travel together in one ring stage (a unit of up to two rows),
// so no grid barrier separates the gate/up and down phases and no activation
// crosses CTAs. The layer closes with one fixed-order reduction of the
// per-CTA partials, each CTA summing the output rows it owns.
//
// Work split: every CTA takes, from each expert (the shared one first, then
// the routed ones in selection order), one block of rows [b R / G,
// (b + 1) R / G) with block b = (cta + slot) mod G. Rotating the block by one
// CTA per slot spreads the blocks that hold one row more, so every CTA streams
// the same bytes to within one row per expert set. The shared expert's units
// do not depend on the routing and stream while the router runs; a routed
// slot's units stream as soon as the top-k has published that slot.
//
// Warp roles: warp 0 waits for the router logits, ranks the token and
// publishes each slot (expert, unnormalised weight) as its round completes;
// warps 1..kUnitWarps compute the router rows and then the units in
// lock-step (one barrier per unit between the gate/up dots, which are split
// over all of them, and the down rows); the last warp's elected lane issues
// the bulk copies.
//
// Page references: "Chasing the Batch-1 Floor: Ling-3.0-flash Speculative
// Decode on Blackwell", sections "PDL: stacking the latency floors of small
// kernels" (producer-independent loads before the dependency wait, fp32
// combine with one final cast) and "Two fusions and a retune" (SwiGLU fused
// where gate and up are produced; a load-time interleave of the expert
// weights, here a load-time transpose of the down projection).
#pragma once
#include "layer_kernel.cuh"

namespace moe {

constexpr int kUnitWarps = 10;                 // warps 1..10 compute units
constexpr int kUnitThreads = kUnitWarps * 32;

// Rows [r0, r1) of a slot with R rows taken by CTA c (slot position j).
__device__ __forceinline__ void splitk_rows(int c, int j, int R, int G, int& r0, int& r1) {
    const uint32_t b = (uint32_t)((c + j) % G);
    r0 = (int)(b * (uint32_t)R / (uint32_t)G);
    r1 = (int)((b + 1) * (uint32_t)R / (uint32_t)G);
}

// Rows per unit: a unit's gate, up and transposed down rows (6 H bytes per
// row) fill at most one ring stage; at most two. The host launches this
// kernel only when one row fits (H <= 5461).
__device__ __forceinline__ int splitk_unit_rows(int H) { return min(2, (int)(SB / (6u * (uint32_t)H))); }

// Bulk copies of one unit: n <= 2 rows, row q being row rq of slot sq (-1:
// the shared expert). Stage layout: the n gate rows, the n up rows, the n
// transposed down rows, each H bf16.
__device__ __forceinline__ bool issue_unit(Producer<0>& pr, const LayerParams& p, Plan* plan, int n, int s0, int r0,
                                           int s1, int r1) {
    if (aborted(plan)) return false;
    if (3u * (uint32_t)n * (uint32_t)p.H * 2u > SB) {  // never issued: the host checks H
        set_abort(p, plan, -101 /* MOE_ETIMEOUT */);
        return false;
    }
    if (!pr.acquire(false)) return false;
    plan->desc[pr.ring.s] = Chunk{4, s0, r0, n, s1, r1};
    const uint32_t dst = pr.ring.stage(), bar = pr.ring.full(), rb = (uint32_t)p.H * 2;
    mbar_arrive_expect_tx(bar, 3u * (uint32_t)n * rb);
    for (int q = 0; q < n; ++q) {
        const int s = q == 0 ? s0 : s1, r = q == 0 ? r0 : r1;
        const uint16_t *a, *b, *c;
        if (s < 0) {
            a = p.ws1 + (size_t)r * p.H;
            b = p.ws3 + (size_t)r * p.H;
            c = p.ws2t + (size_t)r * p.H;
        } else {
            const size_t row = (size_t)plan->slot_e[s] * p.I + r;
            a = reinterpret_cast<const uint16_t*>(p.w1) + row * p.H;
            b = reinterpret_cast<const uint16_t*>(p.w3) + row * p.H;
            c = p.w2t + row * p.H;
        }
        bulk_g2s(dst + (uint32_t)q * rb, a, rb, bar, pr.pol_w);
        bulk_g2s(dst + (uint32_t)(n + q) * rb, b, rb, bar, pr.pol_w);
        bulk_g2s(dst + (uint32_t)(2 * n + q) * rb, c, rb, bar, pr.pol_w);
    }
    pr.ring.advance();
    pr.complete_upto = pr.ring.n;
    return true;
}

// The producer's unit schedule: the shared expert's rows of this CTA, then
// (after the dependency wait) the routed rows slot by slot, each slot once the
// top-k has published it; routed rows are packed two to a unit across slot
// boundaries.
__device__ __forceinline__ bool issue_units(Producer<0>& pr, const LayerParams& p, Plan* plan, int cta,
                                            bool shared_part) {
    const int jb = p.Is > 0 ? 1 : 0;
    if (shared_part) {
        if (!jb) return true;
        int r0, r1;
        splitk_rows(cta, 0, p.Is, p.G, r0, r1);
        const int ur = splitk_unit_rows(p.H);
        for (int r = r0; r < r1; r += ur)
            if (!issue_unit(pr, p, plan, min(ur, r1 - r), -1, r, -1, r + 1)) return false;
        return true;
    }
    const bool two = splitk_unit_rows(p.H) > 1;
    int ps = -1, pr_row = 0;  // a routed row waiting for its unit's second row
    for (int s = 0; s < p.k; ++s) {
        if (!wait_known<0>(p, plan, s + 1)) return false;
        int r0, r1;
        splitk_rows(cta, s + jb, p.I, p.G, r0, r1);
        for (int r = r0; r < r1; ++r) {
            if (!two) {
                if (!issue_unit(pr, p, plan, 1, s, r, s, r)) return false;
            } else if (ps < 0) {
                ps = s;
                pr_row = r;
            } else {
                if (!issue_unit(pr, p, plan, 2, ps, pr_row, s, r)) return false;
                ps = -1;
            }
        }
    }
    if (ps >= 0 && !issue_unit(pr, p, plan, 1, ps, pr_row, ps, pr_row)) return false;
    return true;
}

// acc[i][e] += h0 * W2^T[row 0][8 v + e] + h1 * W2^T[row 1][8 v + e] for this
// thread's output vectors v = ut + i * kUnitThreads (a unit of n rows; the
// transposed down rows follow the gate and up rows in the stage).
template <int VPT>
__device__ __forceinline__ void down_rows(const uint4* __restrict__ st, int n, int nvec, int ut, float h0, float h1,
                                          float (&acc)[VPT][8]) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = ut + i * kUnitThreads;
        if (v >= nvec) break;
        float f[8];
        unpack8(st[(size_t)(2 * n) * nvec + v], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(h0, f[e], acc[i][e]);
        if (n > 1) {
            unpack8(st[(size_t)(2 * n + 1) * nvec + v], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(h1, f[e], acc[i][e]);
        }
    }
}

// VPT: output vectors (8 values) per unit thread, H <= 8 * kUnitThreads * VPT.
template <bool IO, int VPT>
__global__ void __launch_bounds__(block_threads(0), 1) moe_layer_splitk_kernel(const __grid_constant__ LayerParams p) {
    constexpr int NCW = consumer_warps(0);  // warps 0..NCW-1: routing warp + unit warps
    constexpr int NCT = NCW * 32;
    static_assert(NCW == kUnitWarps + 1, "one routing warp and the unit warps");
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = (int)blockIdx.x;
    Plan* plan = reinterpret_cast<Plan*>(smem + p.off_plan);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + p.off_x);
    float* red = reinterpret_cast<float*>(smem + p.off_yacc);  // [2][kUnitWarps][4], then [NCT] reduce scratch
    const uint32_t bars = smem_u32(smem + p.off_bar);
    if (tid == 0) {
        for (int i = 0; i < p.ns; ++i) {
            mbar_init(bars + i * 8, 1);
            mbar_init(bars + (p.ns + i) * 8, kUnitWarps);
        }
        mbar_init(bars + 2u * p.ns * 8u, kUnitWarps);  // per-unit cross-warp sums
        plan->abort = 0;
        plan->npend = 0;
        plan->known = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) trace_mark(p, 0);
    const Ring ring0{smem_u32(smem), bars, (uint32_t)p.ns, 0u, 0u, 0u};
    const int nvec = p.H / 8;

    if (warp == NCW) {
        // ---------------- producer
        if (lane == 0) {
            trace_mark(p, 8);
            Producer<0> pr{p, plan, ring0, policy_evict_first(), policy_evict_last(), false, 0u};
            ChunkGen<0> gen;
            Chunk ch;
            bool ok = true;
            for (gen.begin(0, p, plan, cta); ok && gen.next(p, plan, ch);) ok = pr.issue(ch);
            if (ok) ok = pr.issue_end();
            if (ok) ok = issue_units(pr, p, plan, cta, true);
            trace_mark(p, 9);
            pdl_wait();
            if (ok) ok = issue_units(pr, p, plan, cta, false);
            if (ok) ok = pr.issue_end();
            trace_mark(p, 12);
            if (!ok || aborted(plan)) pr.drain();
            trace_mark(p, 14);
        }
    } else {
        const float* bias_s = p.bias ? reinterpret_cast<const float*>(smem + p.off_bias) : nullptr;
        if (p.bias)
            for (int i = tid; i < p.E; i += NCT) const_cast<float*>(bias_s)[i] = __ldg(p.bias + i);
        pdl_wait();
        // epoch and status: the last consumer warp, both loads in flight
        // together and alongside the token loads
        const bool ctl_thread = tid == NCT - 32;
        uint32_t ctl_epoch = 0, ctl_status = 0;
        if (ctl_thread) {
            ctl_epoch = ld_relaxed_gpu(p.ctrl + kCtlEpoch);
            ctl_status = ld_relaxed_gpu(p.ctrl + kCtlStatus);
        }
        if (IO) {
            load_tokens<0, false>(reinterpret_cast<const uint4*>(p.x), reinterpret_cast<const uint4*>(p.gamma), 1,
                                  p.H, p.H / 8, p.eps, reinterpret_cast<uint4*>(xs), nullptr, plan->x_inv, warp, lane,
                                  NCW);
        } else {
            for (int i = tid; i < nvec; i += NCT) reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
        }
        if (ctl_thread) {
            plan->epoch = ctl_epoch;
            plan->tag = ctl_epoch % 0xffffffffu + 1u;
            if ((int)ctl_status == -101 /* MOE_ETIMEOUT */) set_abort(p, plan, -101);
        }
        named_bar_sync(1, NCT);
        if (tid == 0) trace_mark(p, 1);
        const int h0 = (int)((uint32_t)cta * (uint32_t)p.H / (uint32_t)p.G);
        const int h1 = (int)((uint32_t)(cta + 1) * (uint32_t)p.H / (uint32_t)p.G);

        // this thread's output accumulators (unit warps): shared expert and
        // routed experts (the latter with unnormalised routing weights)
        float ysh[VPT][8], yrt[VPT][8];
        bool ok = true;
        if (warp == 0) {
            // ---------------- routing warp
            if (!aborted(plan)) {
                const unsigned long long* lrow = p.logits;
                const uint32_t tag = plan->tag + (p.force_timeout ? 1u : 0u);
                const bool var = p.scoring != 0 || p.bias != nullptr;
                if (p.E <= 512)
                    var ? topk_warp<16, true, true>(lrow, p.E, p.k, lane, tag, p, plan, bias_s, plan->sel_e,
                                                    plan->sel_w, true)
                        : topk_warp<16, false, true>(lrow, p.E, p.k, lane, tag, p, plan, bias_s, plan->sel_e,
                                                     plan->sel_w, true);
                else
                    var ? topk_warp<32, true, true>(lrow, p.E, p.k, lane, tag, p, plan, bias_s, plan->sel_e,
                                                    plan->sel_w, true)
                        : topk_warp<32, false, true>(lrow, p.E, p.k, lane, tag, p, plan, bias_s, plan->sel_e,
                                                     plan->sel_w, true);
            }
            if (tid == 0) trace_mark(p, 4);
            __syncwarp();
            if (cta == 0 && lane < p.k && !aborted(plan)) {
                if (p.idx_out) p.idx_out[lane] = plan->sel_e[lane];
                if (p.w_out) p.w_out[lane] = plan->sel_w[lane];
            }
        } else {
            // ---------------- unit warps
            const int ut = tid - 32, uw = warp - 1;
            Ring ring = ring0;
            // router rows: one warp per row
            int qm = 0;
            while (ok) {
                if (!mbar_wait(ring.full(), ring.ph, p, plan)) {
                    ok = false;
                    break;
                }
                const Chunk ch = plan->desc[ring.s];
                if (ch.kind == 0) {
                    const uint8_t* st = reinterpret_cast<const uint8_t*>(__cvta_shared_to_generic(ring.stage()));
                    int j = uw >= qm ? uw - qm : uw - qm + kUnitWarps;
                    qm = (qm + ch.n) % kUnitWarps;
                    for (; j < ch.n; j += kUnitWarps) {
                        float acc[1];
                        const uint4* xt = reinterpret_cast<const uint4*>(xs);
                        dot_bf16<1>(reinterpret_cast<const uint4*>(st + (size_t)j * p.H * 2), xt, xt, nvec, lane,
                                    acc);
                        acc[0] = warp_sum(acc[0]);
                        if (lane == 0)
                            st_relaxed_u64(p.logits + ch.r0 + j,
                                           ((unsigned long long)plan->tag << 32) | __float_as_uint(acc[0]));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ring.empty());
                ring.advance();
                if (ch.kind == 3) break;
            }
            if (tid == 32) trace_mark(p, 2);
            uint4 xv[VPT];
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int v = ut + i * kUnitThreads;
                xv[i] = v < nvec ? reinterpret_cast<const uint4*>(xs)[v] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int e = 0; e < 8; ++e) ysh[i][e] = yrt[i][e] = 0.f;
            }
            // the unit warps exchange their gate/up partial sums through a
            // double-buffered array and an mbarrier (bounded wait: a warp that
            // gives up never leaves the others waiting)
            const uint32_t ubar = bars + 2u * p.ns * 8u;
            uint32_t uph = 0;
            while (ok) {
                if (!mbar_wait(ring.full(), ring.ph, p, plan)) {
                    ok = false;
                    break;
                }
                const Chunk ch = plan->desc[ring.s];
                if (ch.kind == 3) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ring.empty());
                    ring.advance();
                    break;
                }
                const uint4* st = reinterpret_cast<const uint4*>(__cvta_shared_to_generic(ring.stage()));
                const int n = ch.n;
                // gate and up dots of the unit's rows over this thread's vectors
                float g[2] = {0.f, 0.f}, u[2] = {0.f, 0.f};
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    const int v = ut + i * kUnitThreads;
                    if (v >= nvec) break;
                    const uint32_t xx[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        if (q >= n) break;
                        const uint4 a = st[(size_t)q * nvec + v], b = st[(size_t)(n + q) * nvec + v];
                        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
                        float gl = 0.f, gh = 0.f, ul = 0.f, uh = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            fma_bf16x2(wa[e], xx[e], gl, gh);
                            fma_bf16x2(wb[e], xx[e], ul, uh);
                        }
                        g[q] += gl + gh;
                        u[q] += ul + uh;
                    }
                }
                // lanes 0-7: g0, 8-15: u0, 16-23: g1, 24-31: u1
                const float wsum = warp_sum4(g[0], u[0], g[1], u[1], lane);
                float* rb = red + (uph & 1u) * (kUnitWarps * 4);
                if ((lane & 7) == 0) rb[uw * 4 + (lane >> 3)] = wsum;
                __syncwarp();
                if (lane == 0) mbar_arrive(ubar);
                if (!mbar_wait(ubar, uph & 1u, p, plan)) {
                    ok = false;
                    break;
                }
                ++uph;
                float r = 0.f;
                if (lane < 4)
                    for (int w = 0; w < kUnitWarps; ++w) r += rb[w * 4 + lane];
                const float g0 = __shfl_sync(0xffffffffu, r, 0), u0 = __shfl_sync(0xffffffffu, r, 1);
                const float g1 = __shfl_sync(0xffffffffu, r, 2), u1 = __shfl_sync(0xffffffffu, r, 3);
                const bool shared = ch.slot < 0;
                // routed rows carry their slot's unnormalised weight; the
                // common factor routed_scale / sum is applied at the end
                const float w0 = shared ? 1.f : plan->slot_num[ch.slot];
                const float w1 = shared ? 1.f : plan->slot_num[ch.p0];
                const float hv0 = silu_mul(g0, u0) * w0;
                const float hv1 = n > 1 ? silu_mul(g1, u1) * w1 : 0.f;
                // down rows: y[v] += h0 W2^T[row0][v] + h1 W2^T[row1][v]
                if (shared)
                    down_rows<VPT>(st, n, nvec, ut, hv0, hv1, ysh);
                else
                    down_rows<VPT>(st, n, nvec, ut, hv0, hv1, yrt);
                __syncwarp();
                if (lane == 0) mbar_arrive(ring.empty());
                ring.advance();
            }
            if (tid == 32) trace_mark(p, 6);
        }
        // ---------------- all consumer warps
        // the routing warp has published its final factor: the unit threads
        // write the CTA's partial output
        named_bar_sync(1, NCT);
        if (warp > 0 && ok && !aborted(plan)) {
            const int ut = tid - 32;
            const float wsc = plan->wscale;
            float* dst = p.ypart + (size_t)cta * p.H;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int v = ut + i * kUnitThreads;
                if (v >= nvec) break;
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = fmaf(yrt[i][e], wsc, ysh[i][e]);
                reinterpret_cast<float4*>(dst)[2 * v] = make_float4(o[0], o[1], o[2], o[3]);
                reinterpret_cast<float4*>(dst)[2 * v + 1] = make_float4(o[4], o[5], o[6], o[7]);
            }
        }
        // grid-wide: every CTA's partial is written
        named_bar_sync(1, NCT);
        if (tid == 0) trace_mark(p, 5);
        if (tid == 0 && !aborted(plan)) {
            __threadfence();
            atomicAdd(ctl_bar2(p, plan->epoch), 1u);
            if (grid_wait(ctl_bar2(p, plan->epoch), (unsigned)p.G, p, plan) && cta == 0)
                advance_epoch(p, plan->epoch);
        }
        named_bar_sync(1, NCT);
        {
            // output rows [h0, h1): row r is the sum over the G partials in
            // CTA order, split into NQ consecutive groups summed separately,
            // then the groups in order. Every thread passes the same
            // barriers whether or not the CTA aborted.
            const bool go = !aborted(plan);
            float* tmp = red + 2 * kUnitWarps * 4;
            const int nr = h1 - h0;
            const int NQ = nr > 0 ? max(1, min(p.G, NCT / nr)) : 1;
            if (go) {
                for (int i = tid; i < nr * NQ; i += NCT) {
                    const int r = i % nr, q = i / nr;
                    const int c0 = q * p.G / NQ, c1 = (q + 1) * p.G / NQ;
                    // eight independent loads in flight at a time, summed in order
                    const float* src = p.ypart + h0 + r;
                    float v = 0.f;
                    for (int cb = c0; cb < c1; cb += 8) {
                        float t[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) t[j] = cb + j < c1 ? __ldcg(src + (size_t)(cb + j) * p.H) : 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (cb + j < c1) v += t[j];
                    }
                    if (NQ > 1) {
                        tmp[i] = v;
                    } else {
                        if (IO && p.residual) v += bf16lo(p.x[h0 + r]);
                        p.y[h0 + r] = f32_to_bf16_bits(v);
                    }
                }
            }
            if (NQ > 1) {
                named_bar_sync(1, NCT);
                if (go)
                    for (int r = tid; r < nr; r += NCT) {
                        float v = 0.f;
                        for (int q = 0; q < NQ; ++q) v += tmp[q * nr + r];
                        if (IO && p.residual) v += bf16lo(p.x[h0 + r]);
                        p.y[h0 + r] = f32_to_bf16_bits(v);
                    }
            }
        }
        if (tid == 0) trace_mark(p, 7);
    }
}

}  // namespace moe
