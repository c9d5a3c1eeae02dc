// rf_moe.cu -- device top-k router and the routed MoE SwiGLU FFN.
//
// neurostream, "How it works" 2: the router runs first and names the experts
// this token needs; only those are read.  "The idea": expert e owns rows
// [e*out, (e+1)*out) of each stacked (n_expert, out, in) tensor and is walked
// in row windows of block_rows rows like any other projection.  The routing
// result stays on the device: the GEMV launches resolve expert ids from it,
// so there is no host synchronisation between routing and the projections.
#include <cfloat>
#include <cstring>
#include <mutex>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kRouterThreads = 1024;
constexpr int kMaxTopK = kMaxTerms;

// One CTA: k rounds of a block-wide argmax (largest logit, lowest index on
// ties; a NaN logit counts as -inf), then a softmax over the k selected
// logits.
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const float *__restrict__ logits,
                                                                int n_expert, int top_k,
                                                                int32_t *__restrict__ idx,
                                                                float *__restrict__ w)
{
    __shared__ float s_val[32];
    __shared__ int s_idx[32];
    __shared__ int s_sel[kMaxTopK];
    __shared__ float s_logit[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_warps = blockDim.x >> 5;
    const float lg = tid < n_expert ? logits[tid] : -FLT_MAX;
    const float v0 = lg != lg ? -INFINITY : lg;   // a NaN logit counts as -inf
    bool taken = tid >= n_expert;
    for (int k = 0; k < top_k; ++k) {
        float v = taken ? -INFINITY : v0;
        int i = taken ? 0x7fffffff : tid;
        // (v, i) beats (v2, i2) if v > v2, or v == v2 and i < i2.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
            if (v2 > v || (v2 == v && i2 < i)) {
                v = v2;
                i = i2;
            }
        }
        if (lane == 0) {
            s_val[warp] = v;
            s_idx[warp] = i;
        }
        __syncthreads();
        if (warp == 0) {
            v = lane < n_warps ? s_val[lane] : -INFINITY;
            i = lane < n_warps ? s_idx[lane] : 0x7fffffff;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
                const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
                if (v2 > v || (v2 == v && i2 < i)) {
                    v = v2;
                    i = i2;
                }
            }
            if (lane == 0) {
                s_sel[k] = i;
                s_logit[k] = v;
            }
        }
        __syncthreads();
        if (tid == s_sel[k]) taken = true;
    }
    if (tid == 0) {
        const float m = s_logit[0];
        float e[kMaxTopK];
        float sum = 0.f;
        for (int k = 0; k < top_k; ++k) {
            e[k] = expf(s_logit[k] - m);
            sum += e[k];
        }
        for (int k = 0; k < top_k; ++k) {
            idx[k] = s_sel[k];
            w[k] = e[k] / sum;
        }
    }
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Scratch for rf_moe_ffn_noalloc: routing result (two 256-byte slots) and up
// to RF_MOE_STATIC_MAX_H activations, laid out like an rf_moe_ffn workspace.
constexpr size_t kStaticScratchBytes =
    512 + sizeof(float) * (size_t)RF_MOE_STATIC_MAX_H + xrec_bytes(RF_MOE_STATIC_MAX_H);
static __device__ __align__(256) unsigned char g_moe_scratch[kStaticScratchBytes];

// Device address of g_moe_scratch per device.  In host code the symbol is
// only a stand-in; its device address comes from cudaGetSymbolAddress with
// the device current.
std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

rf_status static_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_moe_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return RF_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return RF_OK;
}

}  // namespace

rf_status launch_router(const float *logits, int n_expert, int top_k, int32_t *idx, float *w,
                        cudaStream_t stream)
{
    if (!logits || !idx || !w) return RF_ERR_INVALID_ARG;
    if (n_expert < 1 || n_expert > kRouterThreads || top_k < 1 || top_k > kMaxTopK ||
        top_k > n_expert)
        return RF_ERR_INVALID_ARG;
    const int threads = ((n_expert + 31) / 32) * 32;
    router_kernel<<<1, threads, 0, stream>>>(logits, n_expert, top_k, idx, w);
    return last_cuda_error();
}

}  // namespace rf

using namespace rf;

extern "C" {

rf_status rf_moe_route(const float *logits, int n_expert, int top_k, int32_t *idx, float *w,
                       void *stream)
{
    return launch_router(logits, n_expert, top_k, idx, w, static_cast<cudaStream_t>(stream));
}

size_t rf_moe_workspace_bytes(int top_k, int64_t n_ff, int64_t n_embd, int64_t block_rows)
{
    (void)n_embd;
    (void)block_rows;
    if (top_k < 1 || top_k > kMaxTopK || n_ff <= 0) return 0;
    if (n_ff % 32 != 0) return 0;
    return align256(sizeof(int32_t) * kMaxTopK) + align256(sizeof(float) * kMaxTopK) +
           align256(sizeof(float) * (size_t)top_k * (size_t)n_ff) +
           xrec_bytes((int64_t)top_k * n_ff);
}

}  // extern "C"

namespace {

// Biased experts with the clamped SwiGLU (rf_moe_ffn_biased); all zero /
// off for the plain routed FFN.
struct ExpertBias {
    const float *gate = nullptr, *up = nullptr, *down = nullptr;
    bool clamp = false;
    float alpha = 0.f, limit = 0.f;
};

// The routed FFN; host = the stacked tensors are page-locked, device-mapped
// host memory read in place (gate, up, down are their device aliases).
rf_status moe_ffn(int fmt, const float *router_logits, int n_expert, int top_k, const void *gate,
                  const void *up, const void *down, int64_t n_ff, int64_t n_embd,
                  int64_t block_rows, const float *x, float *y, void *workspace, void *stream,
                  bool host, const ExpertBias &eb = ExpertBias())
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!router_logits || !gate || !up || !down || !x || !y || !workspace)
        return RF_ERR_INVALID_ARG;
    if (n_expert < 1 || n_expert > kRouterThreads || top_k < 1 || top_k > kMaxTopK ||
        top_k > n_expert)
        return RF_ERR_INVALID_ARG;
    if (n_ff <= 0 || n_embd <= 0 || n_ff % block_elems_of(fmt) != 0 ||
        n_embd % block_elems_of(fmt) != 0 || block_rows < 0)
        return RF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RF_ERR_MISALIGNED;
    for (const void *p : {gate, up, down})
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return RF_ERR_MISALIGNED;
    if ((int64_t)n_expert * n_ff > 0x7fffffffLL || (int64_t)n_expert * n_embd > 0x7fffffffLL)
        return RF_ERR_TOO_LARGE;
    if (const rf_status c = check_in_dim(fmt, n_embd, 1)) return c;
    if (const rf_status c = check_in_dim(fmt, n_ff, top_k)) return c;

    const int64_t br_ff = block_rows == 0 ? n_ff : block_rows;
    const int64_t br_embd = block_rows == 0 ? n_embd : block_rows;
    const int64_t win_ff = (n_ff + br_ff - 1) / br_ff;
    const int64_t win_embd = (n_embd + br_embd - 1) / br_embd;
    if (top_k * win_ff > 4 * kMaxJobs || win_embd > 4 * kMaxJobs) return RF_ERR_TOO_LARGE;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *idx = reinterpret_cast<int32_t *>(ws);
    float *wts = reinterpret_cast<float *>(ws + align256(sizeof(int32_t) * kMaxTopK));
    float *h = reinterpret_cast<float *>(ws + align256(sizeof(int32_t) * kMaxTopK) +
                                         align256(sizeof(float) * kMaxTopK));
    // Digits of h, written by the gate/up launch and read by the down launch.
    void *hdig = ws + align256(sizeof(int32_t) * kMaxTopK) + align256(sizeof(float) * kMaxTopK) +
                 align256(sizeof(float) * (size_t)top_k * (size_t)n_ff);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Routing happens inside both launches (every CTA ranks the logits
    // itself), so no launch waits for a separate router and the down
    // launch's weight copies can start while gate/up still runs.  The first
    // launch also stores the routing result in the workspace.
    rf_status st = RF_OK;

    // Gate/up: one job per (selected expert k, row window j); the SwiGLU
    // epilogue writes h_k[window].
    static thread_local Job jobs[4 * kMaxJobs];
    int nj = 0;
    for (int k = 0; k < top_k; ++k) {
        for (int64_t j = 0; j < win_ff; ++j) {
            Job &J = jobs[nj++];
            std::memset(&J, 0, sizeof(J));
            const int64_t r0 = j * br_ff;
            J.term[0] = Term{static_cast<const uint8_t *>(gate), 0, k, 0, 0, eb.gate};
            J.term[1] = Term{static_cast<const uint8_t *>(up), 0, k, 0, 0, eb.up};
            J.y = h + (int64_t)k * n_ff + r0;
            J.row0 = r0;
            J.expert_rows = n_ff;
            J.expert_count = n_expert;
            J.n_rows = (int32_t)(r0 + br_ff < n_ff ? br_ff : n_ff - r0);
            J.n_terms = 2;
            J.combine = kCombineSwiGLU;
            if (eb.clamp) {
                J.act = kActClampSwiGLU;
                J.alpha = eb.alpha;
                J.limit = eb.limit;
            }
        }
    }
    LaunchDesc d1;
    d1.fmt = fmt;
    d1.in_dim = n_embd;
    d1.jobs = jobs;
    d1.n_jobs = nj;
    d1.x[0] = x;
    d1.n_x = 1;
    d1.any_expert = true;
    d1.host_weights = host;
    d1.pdl = false;
    d1.route_logits = router_logits;
    d1.route_n = n_expert;
    d1.route_k = top_k;
    d1.route_idx_out = idx;
    d1.route_w_out = wts;
    d1.xr_out = hdig;
    d1.xr_y_base = h;
    st = launch_rowwin(d1, s);
    if (st != RF_OK) return st;

    // Down: one job per output row window with one term per selected expert;
    // y = sum_k w_k * down_k . h_k in selection order.
    nj = 0;
    for (int64_t j = 0; j < win_embd; ++j) {
        Job &J = jobs[nj++];
        std::memset(&J, 0, sizeof(J));
        const int64_t r0 = j * br_embd;
        for (int k = 0; k < top_k; ++k)
            J.term[k] = Term{static_cast<const uint8_t *>(down), k, k, 0, 0, eb.down};
        J.y = y + r0;
        J.row0 = r0;
        J.expert_rows = n_embd;
        J.expert_count = n_expert;
        J.n_rows = (int32_t)(r0 + br_embd < n_embd ? br_embd : n_embd - r0);
        J.n_terms = top_k;
        J.combine = kCombineRouted;
    }
    LaunchDesc d2;
    d2.fmt = fmt;
    d2.in_dim = n_ff;
    d2.jobs = jobs;
    d2.n_jobs = nj;
    for (int k = 0; k < top_k; ++k) d2.x[k] = h + (int64_t)k * n_ff;
    d2.n_x = top_k;
    d2.any_expert = true;
    d2.host_weights = host;
    d2.pdl = true;
    d2.route_logits = router_logits;
    d2.route_n = n_expert;
    d2.route_k = top_k;
    d2.xr_in = hdig;
    return launch_rowwin(d2, s);
}

// Device alias of a page-locked, mapped host pointer, or nullptr.
const void *mapped_alias(const void *host)
{
    cudaPointerAttributes attr;
    if (!host || cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

}  // namespace

extern "C" {

rf_status rf_moe_ffn(int fmt, const float *router_logits, int n_expert, int top_k,
                     const void *gate, const void *up, const void *down, int64_t n_ff,
                     int64_t n_embd, int64_t block_rows, const float *x, float *y,
                     void *workspace, void *stream)
{
    return moe_ffn(fmt, router_logits, n_expert, top_k, gate, up, down, n_ff, n_embd, block_rows,
                   x, y, workspace, stream, false);
}

rf_status rf_moe_ffn_host(int fmt, const float *router_logits, int n_expert, int top_k,
                          const void *host_gate, const void *host_up, const void *host_down,
                          int64_t n_ff, int64_t n_embd, int64_t block_rows, const float *x,
                          float *y, void *workspace, void *stream)
{
    if (!host_gate || !host_up || !host_down) return RF_ERR_INVALID_ARG;
    const void *g = mapped_alias(host_gate), *u = mapped_alias(host_up), *d = mapped_alias(host_down);
    if (!g || !u || !d) return RF_ERR_NOT_PINNED;
    return moe_ffn(fmt, router_logits, n_expert, top_k, g, u, d, n_ff, n_embd, block_rows, x, y,
                   workspace, stream, true);
}

rf_status rf_moe_ffn_biased(int fmt, const float *router_logits, int n_expert, int top_k,
                            const void *gate, const void *up, const void *down,
                            const float *gate_bias, const float *up_bias, const float *down_bias,
                            float alpha, float limit, int64_t n_ff, int64_t n_embd,
                            int64_t block_rows, const float *x, float *y, void *workspace,
                            void *stream)
{
    if (!(alpha == alpha) || alpha == INFINITY || alpha == -INFINITY || !(limit > 0.f))
        return RF_ERR_INVALID_ARG;   // NaN or infinite alpha; limit NaN or not positive
    for (const float *b : {gate_bias, up_bias, down_bias})
        if ((reinterpret_cast<uintptr_t>(b) & 3u) != 0) return RF_ERR_MISALIGNED;
    ExpertBias eb;
    eb.gate = gate_bias;
    eb.up = up_bias;
    eb.down = down_bias;
    eb.clamp = true;
    eb.alpha = alpha;
    eb.limit = limit;
    return moe_ffn(fmt, router_logits, n_expert, top_k, gate, up, down, n_ff, n_embd, block_rows,
                   x, y, workspace, stream, false, eb);
}

rf_status rf_moe_ffn_noalloc(int fmt, const float *router_logits, int n_expert, int top_k,
                             const void *gate, const void *up, const void *down, int64_t n_ff,
                             int64_t n_embd, int64_t block_rows, const float *x, float *y,
                             void *stream)
{
    if (top_k < 1 || top_k > kMaxTopK || n_ff <= 0) return RF_ERR_INVALID_ARG;
    if ((int64_t)top_k * n_ff > RF_MOE_STATIC_MAX_H) return RF_ERR_TOO_LARGE;
    if (rf_moe_workspace_bytes(top_k, n_ff, n_embd, block_rows) > kStaticScratchBytes)
        return RF_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if (const rf_status st = static_scratch(&scratch)) return st;
    return rf_moe_ffn(fmt, router_logits, n_expert, top_k, gate, up, down, n_ff, n_embd,
                      block_rows, x, y, scratch, stream);
}

}  // extern "C"
