// C ABI of the small-M MoE decode layer library: argument checking,
// workspace layout, launch configuration. Declarations and the contract of
// every entry point are in include/moe_decode.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "moe_decode.h"
#include "launch.h"
#include "layer_params.h"

// Scratch of moe_decode_layer_static_scratch (a fixed array per device,
// created with the module).
static __device__ __align__(256) uint8_t g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

namespace {

using moe::LayerParams;

struct Options {
    int grid_ctas = 0;
    long long timeout_ns = 1000000000LL;
    unsigned long long* trace = nullptr;
};
Options g_opt;
thread_local int g_last_launches = 0;

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
    bool coop = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ENODEVICE;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.sms == 0) {
        int coop = 0;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
            cudaGetLastError();
            d.sms = 0;
            return MOE_ENODEVICE;
        }
        d.coop = coop != 0;
    }
    *out = d;
    return MOE_OK;
}

void* g_scratch_ptr[kMaxDevices];

// Device address of this device's static scratch. cudaGetSymbolAddress is
// called on every call (it allocates nothing): after a device reset the
// module is loaded again and the array may sit elsewhere. The first call on a
// device, and the first after the address changed, zeroes the array on `st`.
int static_scratch(void** out, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ENODEVICE;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_scratch_ptr[dev] != ptr) {
        if (cudaMemsetAsync(ptr, 0, MOE_STATIC_SCRATCH_BYTES, st) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ECUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = ptr;
    return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape limits of the kernels (see moe_decode.h).
int check_shape(const moe_shape* s, int M) {
    if (!s) return MOE_EINVAL;
    if (M < 1 || M > moe::kMaxM) return MOE_EM;
    const int H = s->hidden, E = s->n_experts, k = s->top_k, I = s->inter, Is = s->shared_inter;
    if (s->wfmt != 0 && s->wfmt != 1 && s->wfmt != 2) return MOE_ESHAPE;
    if (H <= 0 || H % (s->wfmt == 0 ? 256 : 512) != 0 || H > 8192) return MOE_ESHAPE;
    if (E < 1 || E > moe::kMaxE) return MOE_ESHAPE;
    if (k < 1 || k > moe::kMaxK || k > E) return MOE_ESHAPE;
    if (I <= 0 || I % (s->wfmt == 2 ? 128 : 64) != 0 || I > 4096) return MOE_ESHAPE;
    if (Is < 0 || Is % 64 != 0 || Is > 4096) return MOE_ESHAPE;
    if (s->scoring != 0 && s->scoring != 1) return MOE_ESHAPE;
    if (s->router_bias && (reinterpret_cast<uintptr_t>(s->router_bias) & 3u)) return MOE_EALIGN;
    if (s->residual != 0 && s->residual != 1) return MOE_ESHAPE;
    if (s->norm_weight && !aligned16(s->norm_weight)) return MOE_EALIGN;
    return MOE_OK;
}

struct WsLayout {
    size_t logits, hs, hr, ypart, htag, total;
};

// splitk: the one-token split-K layer's per-CTA partial outputs follow
WsLayout ws_layout(const moe_shape* s, int M, bool splitk) {
    WsLayout w;
    size_t off = moe::kCtlBytes;
    w.logits = off;
    off = align_up(off + (size_t)M * ((s->n_experts + 1) & ~1) * 8, 256);
    w.hs = off;
    off = align_up(off + (size_t)M * s->shared_inter * 2, 256);
    w.hr = off;
    off = align_up(off + (size_t)M * s->top_k * s->inter * 2, 256);
    w.ypart = off;
    if (splitk) off = align_up(off + (size_t)MOE_MAX_GRID * s->hidden * 4, 256);
    // one-token bf16 layers: the tagged activations of the shared expert and
    // the k routed pairs
    w.htag = off;
    if (M == 1 && s->wfmt == 0) off = align_up(off + (size_t)(s->shared_inter + s->top_k * s->inter) * 4, 256);
    w.total = off;
    return w;
}

// The split-K one-token layer: bf16 experts with both transposed down
// projections given, H <= 5461.
bool use_splitk(const moe_shape* s, int M, int mode, const moe_weights* W) {
    // one unit row (gate, up and transposed down rows: 6 H bytes) must fit a
    // ring stage
    return M == 1 && mode == moe::kModeLayer && s->wfmt == 0 && W && W->w2t &&
           (s->shared_inter == 0 || W->ws2t) && 6u * (uint32_t)s->hidden <= moe::kStageBytes;
}

// Grid, ring depth and shared-memory carve-up of one call.
int configure(const moe_shape* s, int M, int mode, void* ws, size_t ws_bytes, LayerParams& p, DeviceInfo& dev,
              bool splitk = false) {
    int rc = device_info(&dev);
    if (rc) return rc;
    if (!ws) return MOE_EWORKSPACE;
    if (!aligned16(ws)) return MOE_EALIGN;
    WsLayout wl = ws_layout(s, M, splitk);
    if (ws_bytes < wl.total) return MOE_EWORKSPACE;
    int G = g_opt.grid_ctas > 0 ? g_opt.grid_ctas : dev.sms;
    if (G > dev.sms || (splitk && G > MOE_MAX_GRID)) return MOE_EINVAL;
    p.M = M;
    p.H = s->hidden;
    p.E = s->n_experts;
    p.k = s->top_k;
    p.I = s->inter;
    p.Is = s->shared_inter;
    p.mode = mode;
    p.G = G;
    p.rpc = (p.H + G - 1) / G;
    p.scoring = s->scoring;
    p.routed_scale = s->routed_scale > 0.f ? s->routed_scale : 1.f;
    p.bias = s->router_bias;
    p.gamma = static_cast<const uint16_t*>(s->norm_weight);
    p.eps = s->norm_eps > 0.f ? s->norm_eps : 1e-6f;
    p.residual = s->residual;
    p.timeout_ns = (unsigned long long)g_opt.timeout_ns;
    p.trace = g_opt.trace;
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.ctrl = reinterpret_cast<unsigned*>(base);
    p.logits = reinterpret_cast<unsigned long long*>(base + wl.logits);
    p.Es = (s->n_experts + 1) & ~1;
    p.hs = reinterpret_cast<uint16_t*>(base + wl.hs);
    p.hr = reinterpret_cast<uint16_t*>(base + wl.hr);
    p.ypart = splitk ? reinterpret_cast<float*>(base + wl.ypart) : nullptr;
    // one-token bf16 layers (not split-K): tagged activations, no barrier 2
    p.htag = (M == 1 && mode == moe::kModeLayer && s->wfmt == 0 && !splitk)
                 ? reinterpret_cast<uint32_t*>(base + wl.htag)
                 : nullptr;

    const size_t other_plan = align_up(sizeof(moe::Plan), 128);
    // one-token MXFP4 layers keep two copies of the tokens: f16 for the
    // routed experts, bf16 for the router and the shared expert
    const bool two = s->wfmt == 1 && M == 1 && mode == moe::kModeLayer;
    p.xp = s->wfmt == 0 ? p.H + 8 : p.H;
    const size_t x_one = align_up((size_t)M * p.xp * 2, 128);
    const size_t x_bytes = x_one * (two ? 2 : 1);
    // down-projection results per (pair, output row): [M + M*k][rpc]; the
    // split-K layer keeps its cross-warp sums there instead
    size_t y_bytes = align_up((size_t)(M + M * s->top_k) * p.rpc * 4, 128);
    if (splitk) y_bytes = std::max(y_bytes, align_up((size_t)(2 * 10 * 4 + 12 * 32) * 4, 128));
    // mbarriers: full and empty per stage, the plan, per-stage partials
    const size_t bar_bytes = 256;
    // the router's selection bias, staged before the dependency wait
    const size_t bias_bytes = s->router_bias ? align_up((size_t)s->n_experts * 4, 128) : 0;
    size_t fixed = other_plan + x_bytes + y_bytes + bar_bytes + bias_bytes;
    if ((size_t)dev.smem_optin <= fixed) return MOE_ESHAPE;
    int ns = (int)(((size_t)dev.smem_optin - fixed) / moe::kStageBytes);
    if (ns > moe::kMaxStages) ns = moe::kMaxStages;
    if (ns < 2) return MOE_ESHAPE;
    p.ns = ns;
    size_t off = (size_t)ns * moe::kStageBytes;
    p.off_bar = (uint32_t)off;
    off += bar_bytes;
    p.off_plan = (uint32_t)off;
    off += other_plan;
    p.off_x = (uint32_t)off;
    p.off_xb = (uint32_t)(off + (two ? x_one : 0));
    off += x_bytes;
    p.off_yacc = (uint32_t)off;
    off += y_bytes;
    p.off_bias = (uint32_t)off;
    off += bias_bytes;
    p.smem_bytes = (uint32_t)off;
    return MOE_OK;
}

int launch(const LayerParams& p, int wfmt, cudaStream_t st, bool pdl, DeviceInfo& dev) {
    bool coop = dev.coop;
    cudaError_t err = p.ypart     ? moe::launch_layer_splitk(p, st, pdl, coop)
                      : wfmt == 1 ? moe::launch_layer_mxfp4(p, st, pdl, coop)
                      : wfmt == 2 ? moe::launch_layer_fp8(p, st, pdl, coop)
                                  : moe::launch_layer_bf16(p, st, pdl, coop);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = 1;
    return MOE_OK;
}

bool weights_ok(const moe_weights* W, const moe_shape* s) {
    if (!W || !W->w1 || !W->w3 || !W->w2) return false;
    if (s->wfmt != 0 && (!W->s1 || !W->s3 || !W->s2)) return false;
    if (s->shared_inter > 0 && (!W->ws1 || !W->ws3 || !W->ws2)) return false;
    return true;
}

bool weights_aligned(const moe_weights* W, const moe_shape* s) {
    bool ok = aligned16(W->w1) && aligned16(W->w3) && aligned16(W->w2) && aligned16(W->w2t) && aligned16(W->ws2t);
    if (s->wfmt != 0) ok = ok && aligned16(W->s1) && aligned16(W->s3) && aligned16(W->s2);
    if (s->shared_inter > 0) ok = ok && aligned16(W->ws1) && aligned16(W->ws3) && aligned16(W->ws2);
    return ok;
}

void set_weights(LayerParams& p, const moe_weights* W) {
    p.w1 = static_cast<const uint8_t*>(W->w1);
    p.w3 = static_cast<const uint8_t*>(W->w3);
    p.w2 = static_cast<const uint8_t*>(W->w2);
    p.s1 = W->s1;
    p.s3 = W->s3;
    p.s2 = W->s2;
    p.ws1 = static_cast<const uint16_t*>(W->ws1);
    p.ws3 = static_cast<const uint16_t*>(W->ws3);
    p.ws2 = static_cast<const uint16_t*>(W->ws2);
    p.w2t = static_cast<const uint16_t*>(W->w2t);
    p.ws2t = static_cast<const uint16_t*>(W->ws2t);
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_shape* shape, int M) {
    if (check_shape(shape, M) != MOE_OK) return 0;
    return ws_layout(shape, M, M == 1).total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws) return MOE_EINVAL;
    if (ws_bytes < moe::kCtlBytes) return MOE_EWORKSPACE;
    if (cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    return MOE_OK;
}

int moe_route(const void* x, int M, const void* Wg, const moe_shape* shape, int32_t* idx, float* w, void* ws,
              size_t ws_bytes, void* stream) {
    g_last_launches = 0;
    int rc = check_shape(shape, M);
    if (rc) return rc;
    if (!x || !Wg || !idx || !w) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(Wg)) return MOE_EALIGN;
    LayerParams p = {};
    DeviceInfo dev;
    rc = configure(shape, M, moe::kModeRoute, ws, ws_bytes, p, dev);
    if (rc) return rc;
    p.x = static_cast<const uint16_t*>(x);
    p.Wg = static_cast<const uint16_t*>(Wg);
    p.idx_out = idx;
    p.w_out = w;
    return launch(p, shape->wfmt, static_cast<cudaStream_t>(stream), true, dev);
}

int moe_ffn(const void* x, int M, const int32_t* idx, const float* w, const moe_weights* weights,
            const moe_shape* shape, void* y, void* ws, size_t ws_bytes, void* stream) {
    g_last_launches = 0;
    int rc = check_shape(shape, M);
    if (rc) return rc;
    if (!x || !idx || !w || !y || !weights_ok(weights, shape)) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(y) || !weights_aligned(weights, shape)) return MOE_EALIGN;
    LayerParams p = {};
    DeviceInfo dev;
    rc = configure(shape, M, moe::kModeFfn, ws, ws_bytes, p, dev);
    if (rc) return rc;
    p.x = static_cast<const uint16_t*>(x);
    p.idx_in = idx;
    p.w_in = w;
    p.y = static_cast<uint16_t*>(y);
    set_weights(p, weights);
    return launch(p, shape->wfmt, static_cast<cudaStream_t>(stream), true, dev);
}

int moe_decode_layer(const void* x, int M, const void* Wg, const moe_weights* weights, const moe_shape* shape,
                     int32_t* idx_out, float* w_out, void* y, void* ws, size_t ws_bytes, uint32_t flags,
                     void* stream) {
    g_last_launches = 0;
    int rc = check_shape(shape, M);
    if (rc) return rc;
    if (flags & ~(MOE_F_NO_PDL | MOE_F_DEBUG_FORCE_TIMEOUT)) return MOE_EINVAL;
    if (!x || !Wg || !y || !weights_ok(weights, shape)) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(y) || !weights_aligned(weights, shape)) return MOE_EALIGN;
    LayerParams p = {};
    DeviceInfo dev;
    rc = configure(shape, M, moe::kModeLayer, ws, ws_bytes, p, dev, use_splitk(shape, M, moe::kModeLayer, weights));
    if (rc) return rc;
    p.x = static_cast<const uint16_t*>(x);
    p.Wg = static_cast<const uint16_t*>(Wg);
    p.idx_out = idx_out;
    p.w_out = w_out;
    p.y = static_cast<uint16_t*>(y);
    p.force_timeout = (flags & MOE_F_DEBUG_FORCE_TIMEOUT) ? 1 : 0;
    set_weights(p, weights);
    return launch(p, shape->wfmt, static_cast<cudaStream_t>(stream), (flags & MOE_F_NO_PDL) == 0, dev);
}

int moe_decode_layer_static_scratch(const void* x, int M, const void* Wg, const moe_weights* weights,
                                    const moe_shape* shape, int32_t* idx_out, float* w_out, void* y,
                                    uint32_t flags, void* stream) {
    g_last_launches = 0;
    int rc = check_shape(shape, M);
    if (rc) return rc;
    if (flags & ~(MOE_F_NO_PDL | MOE_F_RESET_SCRATCH | MOE_F_DEBUG_FORCE_TIMEOUT)) return MOE_EINVAL;
    if (ws_layout(shape, M, false).total > MOE_STATIC_SCRATCH_BYTES) return MOE_ESCRATCH;
    if (!x || !Wg || !y || !weights_ok(weights, shape)) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(y) || !weights_aligned(weights, shape)) return MOE_EALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    rc = static_scratch(&ws, st);
    if (rc) return rc;
    if ((flags & MOE_F_RESET_SCRATCH) && cudaMemsetAsync(ws, 0, MOE_STATIC_SCRATCH_BYTES, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    LayerParams p = {};
    DeviceInfo dev;
    rc = configure(shape, M, moe::kModeLayer, ws, MOE_STATIC_SCRATCH_BYTES, p, dev);
    if (rc) return rc;
    p.x = static_cast<const uint16_t*>(x);
    p.Wg = static_cast<const uint16_t*>(Wg);
    p.idx_out = idx_out;
    p.w_out = w_out;
    p.y = static_cast<uint16_t*>(y);
    p.force_timeout = (flags & MOE_F_DEBUG_FORCE_TIMEOUT) ? 1 : 0;
    set_weights(p, weights);
    p.w2t = p.ws2t = nullptr;  // not used here (the classic path)
    return launch(p, shape->wfmt, st, (flags & MOE_F_NO_PDL) == 0, dev);
}

int moe_static_scratch_status(void* stream, int32_t* dev_status) {
    if (!dev_status) return MOE_EINVAL;
    void* ws = nullptr;
    const int rc = static_scratch(&ws, static_cast<cudaStream_t>(stream));
    if (rc) return rc;
    return moe_read_status(ws, stream, dev_status);
}

int moe_lm_head(const void* x, int M, const void* W, const float* w_scale, int V, int H, int wfmt, float* logits,
                void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
    g_last_launches = 0;
    if (M < 1 || M > moe::kMaxM) return MOE_EM;
    if (wfmt != 0 && wfmt != 2) return MOE_ESHAPE;
    if (V < 1 || H <= 0 || H > 8192 || H % (wfmt == 0 ? 8 : 16) != 0) return MOE_ESHAPE;
    if (flags & ~MOE_F_NO_PDL) return MOE_EINVAL;
    if (!x || !W || !logits || (wfmt == 2 && !w_scale)) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(W)) return MOE_EALIGN;
    if (!ws) return MOE_EWORKSPACE;
    if (!aligned16(ws)) return MOE_EALIGN;
    if (ws_bytes < MOE_LM_HEAD_WORKSPACE_BYTES) return MOE_EWORKSPACE;
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc) return rc;
    moe::LmParams p = {};
    p.x = static_cast<const uint16_t*>(x);
    p.W = static_cast<const uint8_t*>(W);
    p.scale = w_scale;
    p.logits = logits;
    p.ctrl = static_cast<unsigned*>(ws);
    p.M = M;
    p.H = H;
    p.V = V;
    p.G = g_opt.grid_ctas > 0 ? g_opt.grid_ctas : dev.sms;
    if (p.G > dev.sms) return MOE_EINVAL;
    p.timeout_ns = (unsigned long long)g_opt.timeout_ns;
    // barriers and the abort flag in the first 128 bytes, per-token scales
    // (FP8 rows) in the next 128
    // token rows: bf16 launches on the tensor cores keep them H + 8 elements apart
    const size_t xrow = (size_t)H * 2 + (moe::lm_uses_mma(M, H, wfmt) ? 16 : 0);
    const size_t bar_bytes = 256, x_bytes = align_up((size_t)M * xrow, 128);
    if ((size_t)dev.smem_optin <= bar_bytes + x_bytes) return MOE_ESHAPE;
    int ns = (int)(((size_t)dev.smem_optin - bar_bytes - x_bytes) / moe::kStageBytes);
    if (ns > moe::kMaxStages) ns = moe::kMaxStages;
    if (ns < 2) return MOE_ESHAPE;
    p.ns = ns;
    p.off_bar = (uint32_t)(ns * moe::kStageBytes);
    p.off_x = p.off_bar + (uint32_t)bar_bytes;
    p.smem_bytes = p.off_x + (uint32_t)x_bytes;
    if (moe::launch_lm_head(p, wfmt, static_cast<cudaStream_t>(stream), (flags & MOE_F_NO_PDL) == 0) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = 1;
    return MOE_OK;
}

int moe_fp8_quantize(const void* w, int64_t rows, int K, int block, uint8_t* codes, float* scales, void* stream) {
    g_last_launches = 0;
    if (!w || !codes || !scales) return MOE_EINVAL;
    if (rows < 0 || K <= 0 || block <= 0 || block % 32 != 0 || K % block != 0) return MOE_ESHAPE;
    if (moe::launch_fp8_quantize(static_cast<const uint16_t*>(w), rows, K, block, codes, scales,
                                 static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = rows > 0 ? 1 : 0;
    return MOE_OK;
}

int moe_fp8_dequant(const uint8_t* codes, const float* scales, int64_t rows, int K, int block, float* out,
                    void* stream) {
    g_last_launches = 0;
    if (!codes || !scales || !out) return MOE_EINVAL;
    if (rows < 0 || K <= 0 || block <= 0 || K % block != 0) return MOE_ESHAPE;
    if (moe::launch_fp8_dequant(codes, scales, rows, K, block, out, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = rows > 0 ? 1 : 0;
    return MOE_OK;
}

int moe_transpose_down(const void* w2, int64_t n, int H, int I, void* w2t, void* stream) {
    g_last_launches = 0;
    if (!w2 || !w2t) return MOE_EINVAL;
    if (n < 0 || H <= 0 || I <= 0) return MOE_ESHAPE;
    if (moe::launch_transpose_bf16(static_cast<const uint16_t*>(w2), n, H, I, static_cast<uint16_t*>(w2t),
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = n > 0 ? 1 : 0;
    return MOE_OK;
}

int moe_read_status(const void* ws, void* stream, int32_t* dev_status) {
    if (!ws || !dev_status) return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, static_cast<const uint8_t*>(ws) + moe::kCtlStatus * 4, sizeof v, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    *dev_status = v;
    return MOE_OK;
}

const char* moe_status_str(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_EINVAL: return "invalid argument (null pointer, flag or option)";
        case MOE_ESHAPE: return "shape not supported by the kernels";
        case MOE_EM: return "M outside [1, 16]";
        case MOE_EWORKSPACE: return "workspace missing or too small";
        case MOE_EALIGN: return "pointer not 16-byte aligned";
        case MOE_ECUDA: return "CUDA runtime error";
        case MOE_ENODEVICE: return "no usable CUDA device";
        case MOE_ESCRATCH: return "shape and M need more than the static scratch (MOE_STATIC_SCRATCH_BYTES = 512 KiB)";
        case MOE_EDEVICE_BAD_INDEX: return "device: expert index out of range (entry skipped)";
        case MOE_ETIMEOUT: return "device: bounded wait ran out (outputs incomplete; re-initialise the workspace)";
        default: return "unknown status";
    }
}

int moe_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, float* out, void* stream) {
    g_last_launches = 0;
    if (!codes || !scales || !out) return MOE_EINVAL;
    if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_ESHAPE;
    if (moe::launch_mxfp4_dequant(codes, scales, rows, K, out, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    g_last_launches = rows > 0 ? 1 : 0;
    return MOE_OK;
}

int moe_set_option(int option, int64_t value) {
    switch (option) {
        case MOE_OPT_GRID_CTAS:
            if (value < 0 || value > 65535) return MOE_EINVAL;
            g_opt.grid_ctas = (int)value;
            return MOE_OK;
        case MOE_OPT_WAIT_TIMEOUT_NS:
            if (value <= 0) return MOE_EINVAL;
            g_opt.timeout_ns = value;
            return MOE_OK;
        case MOE_OPT_TRACE_BUFFER:
            if (value < 0 || (value & 7)) return MOE_EINVAL;
            g_opt.trace = reinterpret_cast<unsigned long long*>(value);
            return MOE_OK;
        default: return MOE_EINVAL;
    }
}

int moe_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
