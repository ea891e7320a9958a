// Launch parameters of the output-layer (lm_head) kernel. Plain C++, shared
// by the host launcher and the kernel.
#pragma once
#include <cstdint>

namespace moe {

constexpr int kLmConsumerWarps = 11;
constexpr int kLmThreads = (kLmConsumerWarps + 1) * 32;
// bf16 rows against at least this many tokens run on the tensor cores (K in
// steps of 16: H a multiple of 16)
constexpr int kLmMmaMinTokens = 3;
inline bool lm_uses_mma(int M, int H, int wt) { return wt == 0 && M >= kLmMmaMinTokens && H % 16 == 0; }

struct LmParams {
    const uint16_t* x;     // [M, H] bf16
    const uint8_t* W;      // [V, H] bf16 or e4m3 codes, bytes
    const float* scale;    // e4m3: [V] per-row scale
    float* logits;         // [M, V]
    unsigned* ctrl;        // status word (workspace control block)
    int M, H, V;
    int G;                 // CTAs
    int ns;                // ring stages
    unsigned long long timeout_ns;
    uint32_t off_bar, off_x, smem_bytes;
};

}  // namespace moe
