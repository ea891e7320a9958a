// Launch parameters shared by the host launcher and the persistent layer
// kernel. Plain C++ (no CUDA types), included by both sides.
#pragma once
#include <cstdint>

namespace moe {

// Consumer warps per CTA for each routed-weight format; one producer warp
// comes on top. The total (12 warps) spreads evenly over the SM's four
// schedulers and keeps the per-thread register budget at 168.
constexpr int consumer_warps(int) { return 11; }
constexpr int block_threads(int wfmt) { return (consumer_warps(wfmt) + 1) * 32; }
constexpr uint32_t kStageBytes = 32768;               // one ring stage
constexpr int kMaxStages = 6;
constexpr int kMaxPack = 4;  // routed slots' down rows in one MXFP4 / FP8 chunk
constexpr int kMaxM = 16;
constexpr int kMaxK = 16;
constexpr int kMaxE = 1024;
constexpr int kMaxEntries = kMaxM * kMaxK;
constexpr int kMaxGrid = 256;  // CTAs of a split-K layer launch (workspace sizing)

// workspace control block (uint32 words, 128 bytes apart but for the two
// entry counters): status, launch epoch, the exit counter of routing-only
// calls, and per epoch parity a set of grid barrier 2, routed gate/up work
// counter and entry counter. A call with an FFN uses the set of its epoch's
// parity; once every CTA has read the epoch (all have passed grid barrier 2,
// or all have counted themselves in), one CTA zeroes the other set and
// advances the epoch, so that the next call on the workspace finds its
// counters at zero and no CTA does any atomics at exit.
constexpr int kCtlStatus = 0;
constexpr int kCtlEpoch = 32;
constexpr int kCtlBar2 = 64;
constexpr int kCtlExit = 96;
constexpr int kCtlWork = 128;  // next routed gate/up chunk to claim
constexpr int kCtlBar2Odd = 160;
constexpr int kCtlWorkOdd = 192;
constexpr int kCtlEntry = 224;     // CTAs that have read the epoch
constexpr int kCtlEntryOdd = 240;  // (never in use at the same time as 224)
constexpr uint32_t kCtlBytes = 1024;

enum : int { kModeRoute = 1, kModeFfn = 2, kModeLayer = 3 };

struct LayerParams {
    const uint16_t* x;     // [M, H] bf16
    const uint16_t* Wg;    // [E, H] bf16
    const uint8_t* w1;     // routed weights (bf16 or MXFP4 codes), bytes
    const uint8_t* w3;
    const uint8_t* w2;
    const uint8_t* s1;     // MXFP4 scales
    const uint8_t* s3;
    const uint8_t* s2;
    const uint16_t* ws1;   // shared expert, bf16
    const uint16_t* ws3;
    const uint16_t* ws2;
    const uint16_t* w2t;   // optional down projections transposed, bf16 [E, I, H]
    const uint16_t* ws2t;  // and the shared expert's, [Is, H] (split-K layer)
    float* ypart;          // split-K layer: per-CTA partial outputs [G, H] fp32
    const int32_t* idx_in; // FFN mode routing
    const float* w_in;
    int32_t* idx_out;      // may be null
    float* w_out;
    uint16_t* y;           // [M, H] bf16
    unsigned* ctrl;        // workspace control block
    // router logits [M, Es]: 64-bit words, the fp32 logit in the low half and
    // the call's tag in the high half (Es = E rounded up to even)
    unsigned long long* logits;
    int Es;
    uint16_t* hs;          // shared-expert activations [M, Is] bf16
    uint16_t* hr;          // routed activations [M*k, I] bf16, grouped by expert
    // one-token bf16 layers: the activations of the shared expert and of the
    // k routed pairs as 32-bit words, a 16-bit tag of the call in the high
    // half and the bf16 value in the low half, [Is + k*I]; null otherwise.
    // A down chunk's copy brings its pair's words along with the weights, with
    // no grid barrier; the consumers check the tags and re-read any pair
    // whose copy came too early.
    uint32_t* htag;
    const uint16_t* gamma; // RMSNorm weight [H] bf16, or null (x taken as given)
    float eps;             // RMSNorm epsilon
    int residual;          // 1: y += input
    const float* bias;     // router selection bias [E], may be null
    float routed_scale;    // routing-weight factor (1 for none)
    int scoring;           // 0 softmax, 1 sigmoid
    int M, H, E, k, I, Is;
    int xp;                // elements from one token row to the next in shared
                           // memory (bf16 layers: H + 8, so that tensor-core
                           // loads of eight token rows hit eight bank groups)
    int mode;
    int G;                 // CTAs in the grid
    int ns;                // ring stages
    int rpc;               // rows of y owned per CTA, upper bound (ceil(H/G))
    int force_timeout;
    unsigned long long timeout_ns;
    unsigned long long* trace;  // optional [G][16] phase timestamps (ns), may be null
    // shared-memory offsets: barriers, plan, tokens, a second copy of the
    // tokens in plain bf16 (one-token MXFP4 launches; otherwise the same
    // buffer), per-pair down results
    // router selection bias staged from p.bias (only when p.bias is set)
    uint32_t off_bar, off_plan, off_x, off_xb, off_yacc, off_bias, smem_bytes;
};

// A unit of the ring: the tiles one stage holds. kind 0 router rows, 1
// gate/up rows, 2 down rows, 3 end of a phase (no data), 4 a split-K unit
// (gate, up and transposed down rows), 5 gate/up rows laid out for the
// tensor cores (rows at a padded pitch), 6 the down rows of np consecutive
// routed slots (MXFP4 / FP8), each slot a segment laid out as a kind-2 chunk
// with all its pairs and the CTA's rows [r0, r0 + n).
struct Chunk {
    int32_t kind;
    int32_t slot;    // -1 shared expert, else routed slot
    int32_t r0, n;   // first row and row count
    int32_t p0, np;  // down: pair range within the slot
};

// Expert plan, rebuilt by every CTA after routing.
struct Plan {
    // the chunk each ring stage holds, written by the producer before it
    // issues the stage's copies and read by the consumers after the stage's
    // full barrier
    Chunk desc[kMaxStages];
    int32_t sel_e[kMaxEntries];   // routing, token-major [M][k]
    float sel_w[kMaxEntries];
    int32_t rank[kMaxEntries];
    int32_t first[kMaxEntries];
    int16_t pair_tok[kMaxEntries];  // routed (token, weight) pairs grouped by expert
    float pair_w[kMaxEntries];
    int16_t slot_e[kMaxEntries];    // distinct routed experts (ascending; at
                                    // M = 1 in selection order)
    int16_t slot_p0[kMaxEntries + 1];
    int16_t order[kMaxK];           // M = 1: its pairs by ascending expert (combine order)
    int32_t known;                  // M = 1: slots whose expert is known so far
    float slot_num[kMaxK];          // split-K layer: unnormalised routing weight of
                                    // each slot, published with the slot
    float wscale;                   // split-K layer: routed_scale / sum of slot_num
    float x_inv[kMaxM];             // MXFP4 layers: tokens are held in f16 times
                                    // 2^s_t; x_inv[t] = 2^-s_t
    int32_t nslot;
    int32_t npairs;
    uint32_t tag;                   // this call's tag: 1 + epoch mod (2^32 - 1)
    int32_t abort;
    uint32_t epoch;                 // this call's launch epoch
    // Activation copies of down chunks issued before grid barrier 2
    // (producer only): destination, barrier, bytes, source.
    uint32_t pend_dst[kMaxStages * kMaxPack], pend_bar[kMaxStages * kMaxPack], pend_bytes[kMaxStages * kMaxPack];
    const void* pend_src[kMaxStages * kMaxPack];
    int32_t npend;
};


}  // namespace moe
