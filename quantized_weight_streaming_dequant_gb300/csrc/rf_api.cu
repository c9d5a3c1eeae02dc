// rf_api.cu -- C ABI entry points: sizes, status, dequantize, GEMV, batched
// windows, elementwise activations and the two-phase dense SwiGLU FFN.
#include <cuda_fp16.h>

#include <algorithm>

#include <cstring>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

// ---------------------------------------------------------------- dequantize
// One thread per block: decode 32 weights to fp32.  Every value d*q,
// d*(q-8) and e2m1*2^(E-127) is exactly representable, so any correct
// multiply is bit-exact (RAMforge, "Milestone 5 - Native Quantized Tensor
// Support" for Q4_0/Q8_0; OCP MX E2M1/E8M0 for MXFP4).
__device__ __forceinline__ float e2m1_value(uint32_t c)
{
    // magnitude by code bits e1 e0 m: 0, .5, 1, 1.5, 2, 3, 4, 6
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = e == 0 ? 0.5f * (float)m
                             : __uint_as_float((uint32_t)(126 + e) << 23) * (1.0f + 0.5f * (float)m);
    return (c & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e8m0_value(uint32_t E)
{
    // 2^(E-127); E = 0 is the subnormal 2^-127; E = 255 is NaN in the format.
    if (E == 255u) return __uint_as_float(0x7fc00000u);
    return E == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(E << 23);
}

// Weight e of one block, exactly as the format defines it (one rounding to
// fp32 where the value is not exact; the same operations as the oracle).
template <int FMT>
__device__ __forceinline__ float block_elem(const uint8_t *p, int e)
{
    if constexpr (FMT == RF_Q6_K) {
        // Weight e = 128n + 32k + l: q = low | high << 4 from ql byte
        // 64n + 32(k&1) + l (low nibble for k < 2, high for k >= 2) and the
        // bit pair 2k of qh byte 128 + 32n + l; w = d * scale[e/16] * (q-32).
        // d * scale is exact in fp32 (11 x 8 significant bits) and so is its
        // product with q - 32 (6 more), so the result is exact.
        const float d = __half2float(__ushort_as_half((unsigned short)(p[208] | (p[209] << 8))));
        const int n = e >> 7, k = (e >> 5) & 3, l = e & 31;
        const int lb = p[64 * n + 32 * (k & 1) + l];
        const int low = k < 2 ? (lb & 15) : (lb >> 4);
        const int high = (p[128 + 32 * n + l] >> (2 * k)) & 3;
        return (d * (float)(int8_t)p[192 + (e >> 4)]) * (float)((low | (high << 4)) - 32);
    } else if constexpr (FMT == RF_Q4_K) {
        // d*sc and dmin*m are exact in fp32 (11-bit times 6-bit significands)
        // and so is d*sc*q, so one fused multiply-add rounds the exact value
        // once.
        const float d = __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(p[2] | (p[3] << 8))));
        const uint8_t *sc = p + 4, *qs = p + 16;
        const int j = e >> 5, l = e & 31;
        int sv, m;
        if (j < 4) {
            sv = sc[j] & 63;
            m = sc[j + 4] & 63;
        } else {
            sv = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
            m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
        }
        const uint8_t q = qs[32 * (j >> 1) + l];
        const int v = (j & 1) ? (q >> 4) : (q & 15);
        return fmaf(d * (float)sv, (float)v, -(dmin * (float)m));
    } else if constexpr (FMT == RF_Q8_0) {
        const float d = __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
        return d * (float)(int8_t)p[2 + e];
    } else if constexpr (FMT == RF_Q4_0) {
        const float d = __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
        const int q = e < 16 ? (p[2 + e] & 15) : (p[2 + e - 16] >> 4);
        return d * (float)(q - 8);
    } else {
        const uint32_t c = e < 16 ? (p[1 + e] & 15u) : (uint32_t)(p[1 + e - 16] >> 4);
        return e2m1_value(c) * e8m0_value(p[0]);
    }
}

// Thread t writes outputs 4t .. 4t+3 (always within one block: blocks hold a
// multiple of 4 weights), so a warp's stores are 512 contiguous bytes.
template <int FMT>
__global__ void dequant_kernel(const uint8_t *__restrict__ W, int64_t n_blocks,
                               float *__restrict__ out, bool vec)
{
    constexpr int BE = FMT == RF_Q4_K || FMT == RF_Q6_K ? 256 : 32;
    constexpr int BB = FMT == RF_Q8_0 ? 34 : FMT == RF_Q4_0 ? 18 : FMT == RF_MXFP4 ? 17
                                                            : FMT == RF_Q4_K ? 144 : 210;
    const int64_t quads = n_blocks * (BE / 4);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < quads;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = t / (BE / 4);
        const int e0 = (int)(t % (BE / 4)) * 4;
        const uint8_t *p = W + BB * b;
        const float v0 = block_elem<FMT>(p, e0), v1 = block_elem<FMT>(p, e0 + 1);
        const float v2 = block_elem<FMT>(p, e0 + 2), v3 = block_elem<FMT>(p, e0 + 3);
        float *o = out + 4 * t;
        if (vec) {
            *reinterpret_cast<float4 *>(o) = make_float4(v0, v1, v2, v3);
        } else {
            o[0] = v0;
            o[1] = v1;
            o[2] = v2;
            o[3] = v3;
        }
    }
}

// -------------------------------------------------------------- activations
__global__ void swiglu_kernel(const float *__restrict__ g, const float *__restrict__ u,
                              float *__restrict__ h, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float z = g[i];
        h[i] = z / (1.f + expf(-z)) * u[i];
    }
}

__global__ void gelu_kernel(const float *__restrict__ z, float *__restrict__ h, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = z[i];
        h[i] = 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
    }
}

int elementwise_grid(int64_t n)
{
    const int64_t want = (n + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace
}  // namespace rf

using namespace rf;

extern "C" {

const char *rf_status_str(int status)
{
    switch (status) {
    case RF_OK: return "RF_OK";
    case RF_ERR_INVALID_ARG: return "RF_ERR_INVALID_ARG";
    case RF_ERR_UNSUPPORTED_FMT: return "RF_ERR_UNSUPPORTED_FMT";
    case RF_ERR_NOT_PINNED: return "RF_ERR_NOT_PINNED";
    case RF_ERR_ARENA_TOO_SMALL: return "RF_ERR_ARENA_TOO_SMALL";
    case RF_ERR_CUDA: return "RF_ERR_CUDA";
    case RF_ERR_TIMEOUT: return "RF_ERR_TIMEOUT";
    case RF_ERR_OOM: return "RF_ERR_OOM";
    case RF_ERR_MISALIGNED: return "RF_ERR_MISALIGNED";
    case RF_ERR_TOO_LARGE: return "RF_ERR_TOO_LARGE";
    default: return "RF_ERR_UNKNOWN";
    }
}

int rf_version(void) { return 100; }

size_t rf_block_bytes(int fmt) { return block_bytes_of(fmt); }

size_t rf_row_bytes(int fmt, int64_t in_dim)
{
    if (!fmt_ok(fmt) || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0) return 0;
    return (size_t)(in_dim / block_elems_of(fmt)) * block_bytes_of(fmt);
}

int64_t rf_max_in_dim(int fmt, int n_x) { return max_in_dim(fmt, n_x); }

rf_status rf_dequantize(int fmt, const void *W, int64_t n_blocks, float *out, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (n_blocks < 0 || (n_blocks > 0 && (!W || !out))) return RF_ERR_INVALID_ARG;
    if (n_blocks == 0) return RF_OK;
    const int threads = 256;
    const int64_t quads = n_blocks * (block_elems_of(fmt) / 4);
    if (quads / (block_elems_of(fmt) / 4) != n_blocks) return RF_ERR_TOO_LARGE;
    const int grid = (int)std::min<int64_t>((quads + threads - 1) / threads, (int64_t)num_sms() * 8);
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t *w = static_cast<const uint8_t *>(W);
    switch (fmt) {
    case RF_Q4_0: dequant_kernel<RF_Q4_0><<<grid, threads, 0, s>>>(w, n_blocks, out, vec); break;
    case RF_Q8_0: dequant_kernel<RF_Q8_0><<<grid, threads, 0, s>>>(w, n_blocks, out, vec); break;
    case RF_Q4_K: dequant_kernel<RF_Q4_K><<<grid, threads, 0, s>>>(w, n_blocks, out, vec); break;
    case RF_Q6_K: dequant_kernel<RF_Q6_K><<<grid, threads, 0, s>>>(w, n_blocks, out, vec); break;
    default: dequant_kernel<RF_MXFP4><<<grid, threads, 0, s>>>(w, n_blocks, out, vec); break;
    }
    return last_cuda_error();
}

rf_status rf_gemv(int fmt, const void *W, int64_t row_start, int64_t row_end, int64_t in_dim,
                  const float *x, float *y, void *stream)
{
    return rf_gemv_ex(fmt, W, row_start, row_end, in_dim, x, y, 0u, stream);
}

rf_status rf_gemv_ex(int fmt, const void *W, int64_t row_start, int64_t row_end, int64_t in_dim,
                     const float *x, float *y, unsigned flags, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!W || !x || !y || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || row_start < 0 ||
        row_end < row_start)
        return RF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (row_end - row_start > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
    if (row_end == row_start) return RF_OK;
    if (const rf_status c = check_in_dim(fmt, in_dim, 1)) return c;
    Job J;
    std::memset(&J, 0, sizeof(J));
    J.term[0] = Term{static_cast<const uint8_t *>(W), 0, -1, 0, 0};
    J.y = y;
    J.row0 = row_start;
    J.n_rows = (int32_t)(row_end - row_start);
    J.n_terms = 1;
    J.combine = kCombineSum;
    LaunchDesc d;
    d.fmt = fmt;
    d.in_dim = in_dim;
    d.jobs = &J;
    d.n_jobs = 1;
    d.x[0] = x;
    d.n_x = 1;
    d.pdl = (flags & RF_CHAIN) != 0;
    return launch_rowwin(d, static_cast<cudaStream_t>(stream));
}

rf_status rf_gemv_multi(int fmt, const void *W, int64_t row_start, int64_t row_end, int64_t in_dim,
                        int n_tok, const float *X, int64_t ldx, float *Y, int64_t ldy,
                        unsigned flags, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!W || !X || !Y || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || row_start < 0 ||
        row_end < row_start || n_tok < 1 || ldx < in_dim || ldy < row_end - row_start)
        return RF_ERR_INVALID_ARG;
    if (n_tok > kMaxTerms || n_tok > kMaxX) return RF_ERR_TOO_LARGE;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (row_end - row_start > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
    if (row_end == row_start) return RF_OK;
    if (const rf_status c = check_in_dim(fmt, in_dim, n_tok)) return c;
    // One job whose terms are the same matrix against each token's
    // activations; each term's dot goes to its own output row.
    Job J;
    std::memset(&J, 0, sizeof(J));
    for (int t = 0; t < n_tok; ++t) J.term[t] = Term{static_cast<const uint8_t *>(W), t, -1, 0, 0};
    J.y = Y;
    J.y_stride = ldy;
    J.row0 = row_start;
    J.n_rows = (int32_t)(row_end - row_start);
    J.n_terms = n_tok;
    J.combine = kCombineEach;
    LaunchDesc d;
    d.fmt = fmt;
    d.in_dim = in_dim;
    d.jobs = &J;
    d.n_jobs = 1;
    for (int t = 0; t < n_tok; ++t) d.x[t] = X + (int64_t)t * ldx;
    d.n_x = n_tok;
    d.pdl = (flags & RF_CHAIN) != 0;
    return launch_rowwin(d, static_cast<cudaStream_t>(stream));
}

rf_status rf_gemv_host(int fmt, const void *host_W, int64_t row_start, int64_t row_end,
                       int64_t in_dim, const float *x, float *y, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!host_W || !x || !y || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || row_start < 0 ||
        row_end < row_start)
        return RF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(host_W) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (row_end - row_start > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_W) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_NOT_PINNED;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return RF_ERR_NOT_PINNED;
    if (row_end == row_start) return RF_OK;
    if (const rf_status c = check_in_dim(fmt, in_dim, 1)) return c;
    Job J;
    std::memset(&J, 0, sizeof(J));
    J.term[0] = Term{static_cast<const uint8_t *>(attr.devicePointer), 0, -1, 0, 0};
    J.y = y;
    J.row0 = row_start;
    J.n_rows = (int32_t)(row_end - row_start);
    J.n_terms = 1;
    J.combine = kCombineSum;
    LaunchDesc d;
    d.fmt = fmt;
    d.in_dim = in_dim;
    d.jobs = &J;
    d.n_jobs = 1;
    d.x[0] = x;
    d.n_x = 1;
    d.host_weights = true;
    return launch_rowwin(d, static_cast<cudaStream_t>(stream));
}

rf_status rf_gemv_batch(int fmt, int64_t in_dim, int n_windows, const rf_window *windows,
                        void *stream)
{
    return rf_gemv_batch_ex(fmt, in_dim, n_windows, windows, 0u, stream);
}

rf_status rf_gemv_batch_ex(int fmt, int64_t in_dim, int n_windows, const rf_window *windows,
                           unsigned flags, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || n_windows < 0 || (n_windows > 0 && !windows))
        return RF_ERR_INVALID_ARG;
    if (n_windows > kMaxJobs) return RF_ERR_TOO_LARGE;
    Job jobs[kMaxJobs];
    LaunchDesc d;
    d.fmt = fmt;
    d.in_dim = in_dim;
    int n_x = 0;
    for (int i = 0; i < n_windows; ++i) {
        const rf_window &w = windows[i];
        if (!w.W || !w.x || !w.y || w.row_start < 0 || w.row_end < w.row_start)
            return RF_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(w.W) & 15u) != 0) return RF_ERR_MISALIGNED;
        if (w.row_end - w.row_start > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
        int slot = -1;
        for (int s = 0; s < n_x; ++s)
            if (d.x[s] == w.x) slot = s;
        if (slot < 0) {
            if (n_x == kMaxX) return RF_ERR_TOO_LARGE;
            d.x[n_x] = w.x;
            slot = n_x++;
        }
        std::memset(&jobs[i], 0, sizeof(Job));
        jobs[i].term[0] = Term{static_cast<const uint8_t *>(w.W), slot, -1, 0, 0};
        jobs[i].y = w.y;
        jobs[i].row0 = w.row_start;
        jobs[i].n_rows = (int32_t)(w.row_end - w.row_start);
        jobs[i].n_terms = 1;
        jobs[i].combine = kCombineSum;
    }
    if (n_windows == 0) return RF_OK;
    if (const rf_status c = check_in_dim(fmt, in_dim, n_x)) return c;
    d.jobs = jobs;
    d.n_jobs = n_windows;
    d.n_x = n_x;
    d.pdl = (flags & RF_CHAIN) != 0;
    return launch_rowwin(d, static_cast<cudaStream_t>(stream));
}

rf_status rf_swiglu(const float *g, const float *u, float *h, int64_t n, void *stream)
{
    if (n < 0 || (n > 0 && (!g || !u || !h))) return RF_ERR_INVALID_ARG;
    if (n == 0) return RF_OK;
    swiglu_kernel<<<elementwise_grid(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(g, u, h, n);
    return last_cuda_error();
}

rf_status rf_gelu(const float *z, float *h, int64_t n, void *stream)
{
    if (n < 0 || (n > 0 && (!z || !h))) return RF_ERR_INVALID_ARG;
    if (n == 0) return RF_OK;
    gelu_kernel<<<elementwise_grid(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(z, h, n);
    return last_cuda_error();
}

rf_status rf_ffn_swiglu(int fmt, const void *gate, const void *up, const void *down,
                        int64_t n_ff, int64_t n_embd, const float *x, float *y, float *h,
                        void *stream)
{
    return rf_ffn_swiglu_ex(fmt, gate, up, down, n_ff, n_embd, x, y, h, 0u, stream);
}

rf_status rf_ffn_swiglu_ex(int fmt, const void *gate, const void *up, const void *down,
                           int64_t n_ff, int64_t n_embd, const float *x, float *y, float *h,
                           unsigned flags, void *stream)
{
    return rf_ffn_swiglu_ws(fmt, gate, up, down, n_ff, n_embd, x, y, h, nullptr, flags, stream);
}

size_t rf_ffn_workspace_bytes(int64_t n_ff)
{
    return n_ff > 0 && n_ff % 32 == 0 ? xrec_bytes(n_ff) : 0;
}

rf_status rf_ffn_swiglu_ws(int fmt, const void *gate, const void *up, const void *down,
                           int64_t n_ff, int64_t n_embd, const float *x, float *y, float *h,
                           void *workspace, unsigned flags, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!gate || !up || !down || !x || !y || !h || n_ff <= 0 || n_embd <= 0 ||
        n_ff % block_elems_of(fmt) != 0 || n_embd % block_elems_of(fmt) != 0)
        return RF_ERR_INVALID_ARG;
    if (n_ff > 0x7fffffffLL || n_embd > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
    for (const void *p : {gate, up, down})
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return RF_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (const rf_status c = check_in_dim(fmt, n_embd, 1)) return c;
    if (const rf_status c = check_in_dim(fmt, n_ff, 1)) return c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Phase 1: walk gate and up by neuron; SwiGLU in the epilogue.
    Job J;
    std::memset(&J, 0, sizeof(J));
    J.term[0] = Term{static_cast<const uint8_t *>(gate), 0, -1, 0, 0};
    J.term[1] = Term{static_cast<const uint8_t *>(up), 0, -1, 0, 0};
    J.y = h;
    J.n_rows = (int32_t)n_ff;
    J.n_terms = 2;
    J.combine = kCombineSwiGLU;
    LaunchDesc d1;
    d1.fmt = fmt;
    d1.in_dim = n_embd;
    d1.jobs = &J;
    d1.n_jobs = 1;
    d1.x[0] = x;
    d1.n_x = 1;
    d1.pdl = (flags & RF_CHAIN) != 0;
    d1.xr_out = workspace;   // with a workspace, phase 1 also writes h's digits
    d1.xr_y_base = h;
    rf_status st = launch_rowwin(d1, s);
    if (st != RF_OK) return st;
    // Phase 2: walk down by output dimension (programmatic dependent launch:
    // its weight copies overlap the tail of phase 1).
    Job K;
    std::memset(&K, 0, sizeof(K));
    K.term[0] = Term{static_cast<const uint8_t *>(down), 0, -1, 0, 0};
    K.y = y;
    K.n_rows = (int32_t)n_embd;
    K.n_terms = 1;
    K.combine = kCombineSum;
    LaunchDesc d2;
    d2.fmt = fmt;
    d2.in_dim = n_ff;
    d2.jobs = &K;
    d2.n_jobs = 1;
    d2.x[0] = h;
    d2.n_x = 1;
    d2.pdl = true;
    d2.xr_in = workspace;    // ... which phase 2 copies instead of building
    return launch_rowwin(d2, s);
}

rf_status rf_device_status(void)
{
    const rf_status a = read_and_clear_device_status();
    if (a == RF_ERR_CUDA) return a;
    const rf_status b = read_and_clear_gemm_status();
    return a != RF_OK ? a : b;
}

rf_status rf_debug_arm_wait_fault(uint32_t limit_us) { return arm_wait_fault(limit_us); }

}  // extern "C"
