// rf_gemv.cu -- the fused row-window dequant-GEMV kernel for sm_103a.
//
// What it computes (neurostream, "How it works" 4-5; RAMforge, "Milestone 6",
// matrix layout): for every row r of a window, y[r] = sum_i w[r,i] * x[i],
// multiplying straight from the raw quantized block bytes.  Batch-1 GEMV is
// bound by HBM bandwidth, not by a dense contraction, so no tensor cores are
// used; the design targets the per-byte instruction budget instead.
//
// Design (GB300):
//   * Lane-per-row.  A warp owns 32 consecutive rows; every lane walks its own
//     row, so every lane needs the same activation block at the same time and
//     the activation reads are shared-memory broadcasts.
//   * K split over the 8 warps of a CTA.  Warp w walks blocks
//     [G*floor(w*nG/8), G*floor((w+1)*nG/8)) of each of the 32 rows (G = the
//     format's alignment group, nG = ceil(nb/G)); the CTA sums the 8 warp
//     partials of a row in warp order.  The split depends only on (format,
//     in_dim), so a row's result is the same in every window and every launch.
//   * Weights move global -> shared through rings of `stages` slots guarded
//     by mbarriers, in one of three modes chosen per launch from the row
//     bytes: rows that are 16-byte aligned go as 2-D tensor copies (32 rows x
//     one group of blocks per warp chunk) issued by a ninth, producer warp;
//     misaligned rows whose 32-row group fits a stage go as one 1-D bulk copy
//     per (group, term) into a CTA-wide ring; other rows, and weights in mapped
//     host memory, go as 16-byte cp.async per lane, rounded out to 16-byte
//     boundaries.  Slot sizes and ring depths are launch parameters.
//   * Integer dot products.  Each 32-element activation block is turned once
//     per CTA into a fixed-point integer X = rint(x * 2^s) with |X| < 2^15
//     (s from the block maximum) split into two byte planes.  The block dot
//     sum_j q_j X_j is then exact dp4a chains over the raw quant bytes (Q8_0
//     bytes are used as they are; Q4_0 nibbles are masked in place, the high
//     ones scaled by 16; MXFP4 codes go through two byte-permute lookups
//     whose sum is 128 + 2*e2m1), and one fp32 FMA per block applies
//     d * 2^-s.  Q4_0's "-8" and the MXFP4 offset are per-block constants
//     (-8 and -128 times sum_j X_j).
//     Error: |x_j - X_j*2^-s| <= 2^-15 * max|x_block|, so by Cauchy-Schwarz
//     the activation rounding moves y_r by at most sqrt(32)*2^-15*||W_r||*||x||
//     (< 1.8e-4 * ||W_r||*||x||), inside the parity tolerance 1e-3*||W_r||*||x||.
//   * Rows whose byte length is not a multiple of 16 but whose 32-row group
//     fits a shared-memory stage are staged whole: one 1-D bulk copy per
//     (group, term) holds the group's rows back to back (the rows of a window
//     are contiguous in memory), all 8 warps read their K parts from it, and
//     the last warp to finish with a stage issues the copy that refills it.
//   * Persistent CTAs each take a contiguous range of 32-row groups across all
//     jobs of the launch.
//   * Programmatic dependent launch: weight copies for the first chunks are
//     issued before griddepcontrol.wait, so they overlap the previous kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {

namespace {

// Device status word (see rf_device_status).
__device__ int g_device_status = 0;

constexpr int kNW = 8;             // consumer warps of the staged and per-lane kernels
constexpr int kThreads = kNW * 32;
constexpr int kRows = 32;          // rows per group (one per lane)
// The canonical reduction of a row: its blocks fall into kParts consecutive K
// parts; each part is accumulated in block order in fp32 by one lane, and the
// row's dot is the sum of the parts' partials in part order.  Every kernel
// mode computes exactly these partials, whichever warp owns which part.
constexpr int kParts = 16;

// Fixed-point digits of one 32-element activation block.
struct __align__(16) XRec {
    uint32_t p0[8];   // byte 0 of X (unsigned), 4 elements per word
    uint32_t p1[8];   // byte 1 of X (signed: X >> 8)
    int32_t corr;     // per-format multiple of sum_j X_j (see xrec_corr);
                      // Q6_K: sum of X_j over elements 0..15
    float scale;      // 2^-s
    int32_t pad[2];   // Q6_K: pad[0] = sum of X_j over elements 16..31
};
static_assert(sizeof(XRec) == 80, "XRec layout");

template <int FMT>
struct FmtT;
template <>
struct FmtT<RF_Q4_0> {
    static constexpr int BS = 18, HDR = 2, QW = 4, G = 8, RPB = 1;
};
template <>
struct FmtT<RF_Q8_0> {
    static constexpr int BS = 34, HDR = 2, QW = 8, G = 8, RPB = 1;
};
template <>
struct FmtT<RF_MXFP4> {
    static constexpr int BS = 17, HDR = 1, QW = 4, G = 16, RPB = 1;
};
// Q4_K: a "block" is the 256-weight super-block (144 B, always 16-byte
// aligned); it has RPB = 8 activation digit records, one per sub-block.
template <>
struct FmtT<RF_Q4_K> {
    static constexpr int BS = 144, G = 1, RPB = 8;
};
// Q6_K: the 256-weight super-block is 210 B (never a whole number of 16-byte
// units, so its rows are always staged whole or copied per lane); one scale
// per 16 weights, so its digit records carry both 16-element sums.
template <>
struct FmtT<RF_Q6_K> {
    static constexpr int BS = 210, G = 1, RPB = 8;
};

constexpr int kMaxMaps = 16;   // distinct weight tensors per launch (tensor-map path)
// Shared ints: group counters (3) and the CTA's failure flag (at 3),
// flat-mode stage counters (up to 4, at 4) and copies issued per stage (up to
// 4, at 8), the launch's own routing: expert ids (8, at 16) and weights (8
// floats, at 24), and the producer-mode queue of upcoming groups (8, at 32).
constexpr int kCntInts = 40;
constexpr int kGroupQ = 8;
// Group tickets of launches scheduled dynamically (producer mode): a launch
// takes slot (launch sequence number mod kSchedSlots), its CTAs take groups
// past their first from it with atomicAdd, and the CTA that draws the last
// ticket puts it back to zero.  Slots are reused only kSchedSlots launches
// later, so launches that may overlap never share one.
constexpr int kSchedSlots = 1024;
__device__ unsigned int g_sched[kSchedSlots];
// CTAs of a dynamically scheduled launch that have finished drawing tickets;
// the last one puts both words of its slot back to zero, so the slot is
// clean for its next launch even when a failure stopped the draws early.
__device__ unsigned int g_sched_done[kSchedSlots];

// Kernel parameters.  Two sizes: launches with at most 4 windows and 4 weight
// tensors (nearly all of them) pass about 1.6 KB instead of 18 KB per launch.
template <int NJ, int NM>
struct KParamsT {
    CUtensorMap maps[NM];   // 2-D views [rows][row bytes] of 16-byte aligned rows
    Job jobs[NJ];
    const float *x[kMaxX];
    const int32_t *expert_idx;
    int32_t n_jobs, n_x, nb, total_groups;
    int32_t stages, kc, slot, prefetch_early, max_terms, n_maps;
    const float *route_logits;   // non-null: route inside the launch (see LaunchDesc)
    int32_t *route_idx_out;
    float *route_w_out;
    XRec *xr_out;                // activation digits out / in (see LaunchDesc)
    const float *xr_y_base;
    const XRec *xr_in;
    int32_t route_n, route_k;
    int32_t sched_slot;          // >= 0: dynamic group scheduling (producer mode)
    int32_t chained;             // launched behind a previous grid (dependency wait)
    unsigned long long wait_limit_ns;   // limit of every bounded wait
    int32_t fault_withhold;      // test hook: CTA 0 withholds warp 0's first copy
    int32_t row_bulk;            // per-lane mode over device memory: one bulk copy per row
};
using KParamsSmall = KParamsT<4, 4>;
using KParamsLarge = KParamsT<kMaxJobs, kMaxMaps>;

// Element of the 32-block packed into byte `byte` of plane word `word`, in the
// order the format's decoder produces quant bytes.
template <int FMT>
__device__ __forceinline__ int elem_of(int word, int byte)
{
    if constexpr (FMT == RF_MXFP4) {
        // Decoder order per code word k: (4k, 4k+16, 4k+1, 4k+17) then
        // (4k+2, 4k+18, 4k+3, 4k+19).
        return 4 * (word >> 1) + 2 * (word & 1) + (byte >> 1) + 16 * (byte & 1);
    } else {
        return 4 * word + byte;
    }
}

// 2^k as a float for k in [-149, 127].
__device__ __forceinline__ float exp2i(int k)
{
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23)
                     : __uint_as_float(1u << (k + 149));
}

// The record's per-block integer correction, from sum_j X_j: Q4_0's "-8"
// (-8 * sum), the offset of the MXFP4 lookup (-128 * sum), and Q4_K's sum
// itself (its min term); Q8_0 needs none.
template <int FMT>
__device__ __forceinline__ int32_t xrec_corr(int sum)
{
    if constexpr (FMT == RF_Q4_0) return -8 * sum;
    else if constexpr (FMT == RF_MXFP4) return -128 * sum;
    else if constexpr (FMT == RF_Q4_K) return sum;
    else return 0;
}

// Fixed-point digits of one 32-element activation block, computed by a quad
// of consecutive lanes: lane `part` of the quad owns plane words 2*part and
// 2*part+1 (8 elements).  xrec_load fetches the lane's 8 elements (in plane
// byte order); xrec_build turns them into digits.  All 32 lanes of the warp
// must call xrec_build (shuffles); inactive lanes only take part in them.
template <int FMT>
__device__ __forceinline__ void xrec_load(const float *xb, int part, bool active, float (&v)[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
    if (!active) return;
    if ((reinterpret_cast<uintptr_t>(xb) & 15u) == 0) {
        if constexpr (FMT == RF_MXFP4) {
            const float4 a = reinterpret_cast<const float4 *>(xb)[part];       // 4k..4k+3
            const float4 b = reinterpret_cast<const float4 *>(xb)[4 + part];   // 16+4k..
            v[0] = a.x; v[1] = b.x; v[2] = a.y; v[3] = b.y;
            v[4] = a.z; v[5] = b.z; v[6] = a.w; v[7] = b.w;
        } else {
            const float4 a = reinterpret_cast<const float4 *>(xb)[2 * part];
            const float4 b = reinterpret_cast<const float4 *>(xb)[2 * part + 1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = xb[elem_of<FMT>(2 * part + (i >> 2), i & 3)];
    }
}
template <int FMT>
__device__ __forceinline__ void xrec_build(const float (&v)[8], int part, bool active, XRec *out)
{
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    // m < 2^e with e from the exponent field (zero/subnormal m: e = -125).
    const int biased = (int)(__float_as_uint(m) >> 23);
    const int e = biased == 0 ? -125 : biased - 126;
    const int s = 15 - e;   // |x * 2^s| < 2^15; s in [-114, 140]
    const float f1 = exp2i(min(s, 127)), f2 = exp2i(max(s - 127, 0));
    int X[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // round to nearest even through the 1.5*2^23 magic constant
        const float t = (v[i] * f1) * f2 + 12582912.0f;
        const int q = (int)(__float_as_uint(t) - 0x4b400000u);
        X[i] = max(-32767, min(32767, q));
        sum += X[i];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    const int half_sum = sum;   // parts 0, 1: elements 0..15; parts 2, 3: 16..31
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (!active) return;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const uint32_t a = (uint32_t)X[4 * hh], b = (uint32_t)X[4 * hh + 1];
        const uint32_t c = (uint32_t)X[4 * hh + 2], d = (uint32_t)X[4 * hh + 3];
        out->p0[2 * part + hh] = prmt(prmt(a, b, 0x0040u), prmt(c, d, 0x0040u), 0x5410u);
        out->p1[2 * part + hh] = prmt(prmt(a, b, 0x0051u), prmt(c, d, 0x0051u), 0x5410u);
    }
    if (part == 0) {
        out->corr = FMT == RF_Q6_K ? half_sum : xrec_corr<FMT>(sum);
        out->scale = exp2i(-s);
        if (FMT != RF_Q6_K) out->pad[0] = 0;
        out->pad[1] = 0;
    } else if (FMT == RF_Q6_K && part == 2) {
        out->pad[0] = half_sum;
    }
}

// Digits of one 32-element block held one element per lane (lane j = element
// j), written to *out: the same record xrec_build makes from those values.
// All 32 lanes must call it.
template <int FMT>
__device__ __forceinline__ void xrec_emit(float v, XRec *out)
{
    const int lane = threadIdx.x & 31;
    float m = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int biased = (int)(__float_as_uint(m) >> 23);
    const int e = biased == 0 ? -125 : biased - 126;
    const int s = 15 - e;
    const float f1 = exp2i(min(s, 127)), f2 = exp2i(max(s - 127, 0));
    const float t = (v * f1) * f2 + 12582912.0f;
    const int X = max(-32767, min(32767, (int)(__float_as_uint(t) - 0x4b400000u)));
    int hs = X;   // sum over this lane's 16-element half, then over all 32
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) hs += __shfl_xor_sync(0xffffffffu, hs, o);
    const int sum = hs + __shfl_xor_sync(0xffffffffu, hs, 16);
    const int h0 = __shfl_sync(0xffffffffu, hs, 0), h1 = __shfl_sync(0xffffffffu, hs, 16);
    // Lane L < 16 assembles plane L >> 3, word L & 7.
    const int w = lane & 7;
    const uint32_t a = (uint32_t)__shfl_sync(0xffffffffu, X, elem_of<FMT>(w, 0));
    const uint32_t b = (uint32_t)__shfl_sync(0xffffffffu, X, elem_of<FMT>(w, 1));
    const uint32_t c = (uint32_t)__shfl_sync(0xffffffffu, X, elem_of<FMT>(w, 2));
    const uint32_t d = (uint32_t)__shfl_sync(0xffffffffu, X, elem_of<FMT>(w, 3));
    const uint32_t sel = lane < 8 ? 0x0040u : 0x0051u;
    const uint32_t word = prmt(prmt(a, b, sel), prmt(c, d, sel), 0x5410u);
    uint32_t *o32 = reinterpret_cast<uint32_t *>(out);
    if (lane < 16)
        o32[lane] = word;
    else if (lane == 16)
        o32[16] = (uint32_t)(FMT == RF_Q6_K ? h0 : xrec_corr<FMT>(sum));
    else if (lane == 17)
        o32[17] = __float_as_uint(exp2i(-s));
    else if (lane < 20)
        o32[lane] = (FMT == RF_Q6_K && lane == 18) ? (uint32_t)h1 : 0u;
}

// One Q4_K super-block held as 36 words (d and dmin, 3 words of packed 6-bit
// scales and mins, 32 quant words) against its 8 digit records: sub-block j
// contributes (d*sc_j * sum_l q_l X_l - dmin*m_j * sum_l X_l) * 2^-s_j.  Quant
// word 4+8i+k holds weights 4k..4k+3 of sub-block 2i in its low nibbles and of
// sub-block 2i+1 in its high nibbles; the high ones stay in place (16*q) and
// the exact sums are divided by 16.
__device__ __forceinline__ float q4k_superblock(const uint32_t *v, const XRec *xr, float acc)
{
    const float d = __half2float(__ushort_as_half((unsigned short)(v[0] & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(v[0] >> 16)));
    const uint32_t s0 = v[1], s1 = v[2], s2 = v[3];
    const uint32_t scA = s0 & 0x3f3f3f3fu;                                       // sc 0..3
    const uint32_t mA = s1 & 0x3f3f3f3fu;                                        // m 0..3
    const uint32_t scB = (s2 & 0x0f0f0f0fu) | ((s0 >> 2) & 0x30303030u);         // sc 4..7
    const uint32_t mB = ((s2 >> 4) & 0x0f0f0f0fu) | ((s1 >> 2) & 0x30303030u);  // m 4..7
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int sh = 8 * (j & 3);
        const float sc = (float)(((j < 4 ? scA : scB) >> sh) & 0xffu);
        const float m = (float)(((j < 4 ? mA : mB) >> sh) & 0xffu);
        const XRec &x = xr[j];
        const uint4 *P0 = reinterpret_cast<const uint4 *>(x.p0);
        const uint4 *P1 = reinterpret_cast<const uint4 *>(x.p1);
        const uint4 a0 = P0[0], a1 = P0[1], b0 = P1[0], b1 = P1[1];
        const uint32_t p0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t p1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t *q = v + 4 + 8 * (j >> 1);
        const uint32_t mask = (j & 1) ? 0xf0f0f0f0u : 0x0f0f0f0fu;
        int t0 = 0, t1 = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t n = q[k] & mask;
            t0 = dp4a_uu(n, p0[k], t0);
            t1 = dp4a_us(n, p1[k], t1);
        }
        const int idot = (j & 1) ? (t1 >> 4) * 256 + (t0 >> 4) : t1 * 256 + t0;
        const float t = fmaf((float)idot, d * sc, -((float)x.corr * (dmin * m)));
        acc = fmaf(t, x.scale, acc);
    }
    return acc;
}

// One Q6_K super-block starting `o` bytes (o even) into a 4-byte aligned
// buffer, against its 8 digit records.  Record j = 4n + k (half n, quarter
// k) covers weights 128n + 32k + l, l < 32: quant q = low | high << 4 with
// low the low (k < 2) or high (k >= 2) nibble of ql byte 64n + 32(k&1) + l
// and high the bit pair 2k of qh byte 32n + l; weight = d * sc * (q - 32)
// with one signed scale per 16 weights.  Per 16 weights the exact integer
// sum_l (q_l - 32) X_l (|.| < 2^24) becomes a float, times its scale, and
// the record's pair times d * 2^-s joins the fp32 accumulator.  Reads one
// word past the block (the buffers leave room for it); the bytes it
// brings in are masked off.
__device__ __forceinline__ float q6k_superblock(const uint8_t *buf, int o, const XRec *xr,
                                                float acc)
{
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(buf + (o & ~3));
    const int sh = 8 * (o & 3);
    auto word = [&](int i) { return __funnelshift_r(wp[i], wp[i + 1], sh); };
    const uint32_t sw[4] = {word(48), word(49), word(50), word(51)};   // 16 scale bytes
    const float d = __half2float(__ushort_as_half((unsigned short)(word(52) & 0xffffu)));
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        uint32_t ql[16], qh[8];
#pragma unroll
        for (int i = 0; i < 16; ++i) ql[i] = word(16 * n + i);
#pragma unroll
        for (int i = 0; i < 8; ++i) qh[i] = word(32 + 8 * n + i);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const XRec &x = xr[4 * n + k];
            const uint4 *P0 = reinterpret_cast<const uint4 *>(x.p0);
            const uint4 *P1 = reinterpret_cast<const uint4 *>(x.p1);
            const uint4 a0 = P0[0], a1 = P0[1], b0 = P1[0], b1 = P1[1];
            const uint32_t p0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t p1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            int lo0 = 0, lo1 = 0, hi0 = 0, hi1 = 0;   // sub-blocks of weights 0..15, 16..31
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w = ql[8 * (k & 1) + i];
                const uint32_t low = (k < 2 ? w : (w >> 4)) & 0x0f0f0f0fu;
                const uint32_t high = ((qh[i] >> (2 * k)) & 0x03030303u) << 4;
                const uint32_t q = low | high;
                if (i < 4) {
                    lo0 = dp4a_uu(q, p0[i], lo0);
                    lo1 = dp4a_us(q, p1[i], lo1);
                } else {
                    hi0 = dp4a_uu(q, p0[i], hi0);
                    hi1 = dp4a_us(q, p1[i], hi1);
                }
            }
            const int dot_a = lo1 * 256 + lo0 - 32 * x.corr;
            const int dot_b = hi1 * 256 + hi0 - 32 * x.pad[0];
            const uint32_t sc = sw[2 * n + (k >> 1)] >> (16 * (k & 1));
            const float sc_a = (float)(int8_t)(sc & 0xffu), sc_b = (float)(int8_t)((sc >> 8) & 0xffu);
            const float t = fmaf((float)dot_b, sc_b, (float)dot_a * sc_a);
            acc = fmaf(t, d * x.scale, acc);
        }
    }
    return acc;
}

// Integer dot of one block's quant words with the block's digit planes;
// returns sum_j q_j X_j as a float.
template <int FMT>
__device__ __forceinline__ float block_idot(const uint32_t (&q)[FmtT<FMT>::QW], const XRec &r)
{
    const uint4 *P0 = reinterpret_cast<const uint4 *>(r.p0);
    const uint4 *P1 = reinterpret_cast<const uint4 *>(r.p1);
    const uint4 a0 = P0[0], a1 = P0[1], b0 = P1[0], b1 = P1[1];
    const uint32_t p0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t p1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    if constexpr (FMT == RF_Q4_0) {
        // Low nibbles are elements 4k..4k+3, high nibbles 16+4k..; the high
        // ones stay in place (16*q), and the exact sums are divided by 16.
        int l0 = 0, l1 = 0, h0 = 0, h1 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = q[k] & 0x0f0f0f0fu;
            const uint32_t hi = q[k] & 0xf0f0f0f0u;
            l0 = dp4a_uu(lo, p0[k], l0);
            l1 = dp4a_us(lo, p1[k], l1);
            h0 = dp4a_uu(hi, p0[k + 4], h0);
            h1 = dp4a_us(hi, p1[k + 4], h1);
        }
        return (float)((l1 + (h1 >> 4)) * 256 + l0 + (h0 >> 4) + r.corr);
    } else if constexpr (FMT == RF_Q8_0) {
        int a = 0, b = 0, c = 0, d = 0;
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            a = dp4a_su(q[k], p0[k], a);
            b = dp4a_ss(q[k], p1[k], b);
            c = dp4a_su(q[k + 1], p0[k + 1], c);
            d = dp4a_ss(q[k + 1], p1[k + 1], d);
        }
        return (float)((b + d) * 256 + a + c);
    } else {
        // MXFP4: each code c = (s, i) stands for v = +-u_i with u_i = 2*e2m1
        // in {0,1,2,3,4,6,8,12}.  Two byte-permute lookups give, per byte,
        // P = 2*u_i when s = 0 and 0 when s = 1 (the selector's top bit is
        // the sign bit, which replicates the table byte's clear top bit), and
        // M = 128 - u_i (the magnitude bits alone).  P + M = 128 + v lies in
        // [116, 140], so one 32-bit add forms all four bytes without carries;
        // the record's corr holds -128 * sum_j X_j and removes the offset.
        constexpr uint32_t kTwoLo = 0x06040200u, kTwoHi = 0x18100c08u;
        constexpr uint32_t kOffLo = 0x7d7e7f80u, kOffHi = 0x74787a7cu;
        int a = 0, b = 0, c = 0, d = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t v = q[k];
            const uint32_t m = v & 0x77777777u;
            const uint32_t vh = v >> 16, mh = m >> 16;
            const uint32_t wa = prmt(kTwoLo, kTwoHi, v) + prmt(kOffLo, kOffHi, m);
            const uint32_t wb = prmt(kTwoLo, kTwoHi, vh) + prmt(kOffLo, kOffHi, mh);
            a = dp4a_uu(wa, p0[2 * k], a);
            b = dp4a_us(wa, p1[2 * k], b);
            c = dp4a_uu(wb, p0[2 * k + 1], c);
            d = dp4a_us(wb, p1[2 * k + 1], d);
        }
        return (float)((b + d) * 256 + a + c + r.corr);
    }
}

// Block scale (times the activation block's 2^-s) from the header bits.
template <int FMT>
__device__ __forceinline__ float block_scale(uint32_t hdr, float xscale)
{
    if constexpr (FMT == RF_MXFP4) {
        // The lookup holds 2*e2m1, so the scale is 2^(E-128).
        const uint32_t E = hdr & 0xffu;
        const uint32_t bits = E >= 2u ? (E - 1u) << 23 : (0x00200000u << E);
        return __uint_as_float(bits) * xscale;
    } else {
        return __half2float(__ushort_as_half((unsigned short)(hdr & 0xffffu))) * xscale;
    }
}

__device__ __forceinline__ uint32_t word_at(const uint32_t *v, int byte)
{
    const int w = byte >> 2, sh = byte & 3;
    return sh ? __funnelshift_r(v[w], v[w + 1], 8 * sh) : v[w];
}

// One group of G blocks (a multiple of 16 bytes) held in registers.
template <int FMT>
struct GroupRegs {
    static constexpr int NV = FmtT<FMT>::G * FmtT<FMT>::BS / 16;
    uint32_t v[4 * NV + 1];
};

template <int FMT>
__device__ __forceinline__ void load_group(const uint8_t *src, GroupRegs<FMT> &r)
{
#pragma unroll
    for (int i = 0; i < GroupRegs<FMT>::NV; ++i) {
        const uint4 t = reinterpret_cast<const uint4 *>(src)[i];
        r.v[4 * i] = t.x;
        r.v[4 * i + 1] = t.y;
        r.v[4 * i + 2] = t.z;
        r.v[4 * i + 3] = t.w;
    }
    r.v[4 * GroupRegs<FMT>::NV] = 0;
}

template <int FMT>
__device__ __forceinline__ float compute_group(const GroupRegs<FMT> &r, const XRec *xr, float acc)
{
    using F = FmtT<FMT>;
    if constexpr (FMT == RF_Q4_K) {
        return q4k_superblock(r.v, xr, acc);
    } else {
#pragma unroll
        for (int b = 0; b < F::G; ++b) {
            const int o = b * F::BS;
            const uint32_t hdr = word_at(r.v, o);
            uint32_t q[F::QW];
#pragma unroll
            for (int k = 0; k < F::QW; ++k) q[k] = word_at(r.v, o + F::HDR + 4 * k);
            const XRec &x = xr[b];
            acc = fmaf(block_idot<FMT>(q, x), block_scale<FMT>(hdr, x.scale), acc);
        }
        return acc;
    }
}

// Blocks [B0, B1) of a group held in registers (words of the group past
// those blocks need not be loaded yet).
template <int FMT, int B0, int B1>
__device__ __forceinline__ float compute_blocks(const GroupRegs<FMT> &r, const XRec *xr, float acc)
{
    using F = FmtT<FMT>;
#pragma unroll
    for (int b = B0; b < B1; ++b) {
        const int o = b * F::BS;
        const uint32_t hdr = word_at(r.v, o);
        uint32_t q[F::QW];
#pragma unroll
        for (int k = 0; k < F::QW; ++k) q[k] = word_at(r.v, o + F::HDR + 4 * k);
        const XRec &x = xr[b];
        acc = fmaf(block_idot<FMT>(q, x), block_scale<FMT>(hdr, x.scale), acc);
    }
    return acc;
}

// 16-byte words [I0, I1) of a group from shared memory into registers.
template <int FMT, int I0, int I1>
__device__ __forceinline__ void load_group_part(const uint8_t *src, GroupRegs<FMT> &r)
{
#pragma unroll
    for (int i = I0; i < I1; ++i) {
        const uint4 t = reinterpret_cast<const uint4 *>(src)[i];
        r.v[4 * i] = t.x;
        r.v[4 * i + 1] = t.y;
        r.v[4 * i + 2] = t.z;
        r.v[4 * i + 3] = t.w;
    }
}

// Aligned chunk: `kn` blocks (a multiple of G) at a 16-byte aligned address.
template <int FMT>
__device__ __forceinline__ float chunk_aligned(const uint8_t *src, int kn, const XRec *xr,
                                               float acc)
{
    using F = FmtT<FMT>;
    for (int g0 = 0; g0 < kn; g0 += F::G) {
        GroupRegs<FMT> r;
        load_group<FMT>(src + g0 * F::BS, r);
        acc = compute_group<FMT>(r, xr + g0 * F::RPB, acc);
    }
    return acc;
}

// Any alignment: `kn` blocks starting `phi` bytes into a 16-byte aligned slot.
template <int FMT>
__device__ __forceinline__ float chunk_generic(const uint8_t *slot, int phi, int kn,
                                               const XRec *xr, float acc)
{
    using F = FmtT<FMT>;
    if constexpr (FMT == RF_Q6_K) {
        for (int b = 0; b < kn; ++b) acc = q6k_superblock(slot, phi + b * F::BS, xr + b * F::RPB, acc);
        return acc;
    } else if constexpr (FMT == RF_Q4_K) {
        // Super-blocks at any 4-byte phase (rows of 144-byte blocks are always
        // 16-byte aligned, so this only serves unaligned slots).
        for (int b = 0; b < kn; ++b) {
            const int o = phi + b * F::BS;
            const uint32_t *wp = reinterpret_cast<const uint32_t *>(slot + (o & ~3));
            const int sh = 8 * (o & 3);
            uint32_t w[36];
#pragma unroll
            for (int k = 0; k < 36; ++k) w[k] = __funnelshift_r(wp[k], wp[k + 1], sh);
            acc = q4k_superblock(w, xr + b * F::RPB, acc);
        }
        return acc;
    } else {
        for (int b = 0; b < kn; ++b) {
            const int o = phi + b * F::BS;
            uint32_t hdr;
            if constexpr (FMT == RF_MXFP4)
                hdr = slot[o];
            else
                hdr = *reinterpret_cast<const uint16_t *>(slot + o);   // o is even
            const int qa = o + F::HDR;
            const uint32_t *wp = reinterpret_cast<const uint32_t *>(slot + (qa & ~3));
            const int sh = 8 * (qa & 3);
            uint32_t w[F::QW + 1];
#pragma unroll
            for (int k = 0; k <= F::QW; ++k) w[k] = wp[k];
            uint32_t q[F::QW];
#pragma unroll
            for (int k = 0; k < F::QW; ++k) q[k] = __funnelshift_r(w[k], w[k + 1], sh);
            const XRec &r = xr[b];
            acc = fmaf(block_idot<FMT>(q, r), block_scale<FMT>(hdr, r.scale), acc);
        }
        return acc;
    }
}

// Walks the (group, term, chunk) items of one warp in order.
struct Cursor {
    int g, j, t, c;
    bool valid;
};

__device__ __forceinline__ int groups_of(const Job &J) { return (J.n_rows + kRows - 1) / kRows; }

__device__ __forceinline__ void cursor_fix_job(const Job *jobs, int n_jobs, Cursor &cu)
{
    while (cu.j < n_jobs && cu.g >= jobs[cu.j].group_begin + groups_of(jobs[cu.j])) ++cu.j;
}

__device__ __forceinline__ void cursor_advance(const Job *jobs, int n_jobs, Cursor &cu,
                                               int n_chunks, int g_hi)
{
    if (++cu.c < n_chunks) return;
    cu.c = 0;
    if (++cu.t < jobs[cu.j].n_terms) return;
    cu.t = 0;
    if (++cu.g >= g_hi) {
        cu.valid = false;
        return;
    }
    cursor_fix_job(jobs, n_jobs, cu);
}

__device__ __forceinline__ const uint8_t *term_matrix(const int32_t *expert_idx, const Job &J,
                                                      int t, int64_t row_bytes)
{
    const Term &T = J.term[t];
    const uint8_t *W = T.W;
    if (T.expert_slot >= 0) W += (int64_t)expert_idx[T.expert_slot] * J.expert_rows * row_bytes;
    return W;
}

// Order-preserving unsigned key of a float that is not NaN (-0 and +0 equal).
__device__ __forceinline__ uint32_t route_key(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of n logits by one warp (ties to the lower index; the same order as
// the standalone router) and the softmax over the k selected, into idx/w.
// A NaN logit counts as -inf.  Lane L holds experts L + 32*m, m < NM (slots
// past n hold -inf with an index above every real one, so they are never
// chosen while k <= n).  Each round takes the warp's largest key and then the
// lowest index holding it with two warp reductions; only the winning lane
// rescans its own NM slots.  The rounds are a rolled loop: the routing runs
// once per launch from a cold instruction cache, so short code matters more
// than instruction count.
template <int NM>
__device__ __forceinline__ void route_warp_n(const float *__restrict__ logits, int n, int k,
                                             int32_t *idx, float *w)
{
    const int lane = threadIdx.x & 31;
    float lv[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
        const int e = lane + 32 * m;
        const float v = e < n ? logits[e] : -INFINITY;
        lv[m] = v != v ? -INFINITY : v;
    }
    uint32_t taken = 0;
    float bv = -INFINITY;   // this lane's first largest untaken slot
    int bm = -1;
    auto local_best = [&] {
        bv = -INFINITY;
        bm = -1;
#pragma unroll
        for (int m = 0; m < NM; ++m)
            if (!((taken >> m) & 1u) && (bm < 0 || lv[m] > bv)) {
                bv = lv[m];
                bm = m;
            }
    };
    local_best();
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        const uint32_t key = bm < 0 ? 0u : route_key(bv);
        const uint32_t top = __reduce_max_sync(0xffffffffu, key);
        const uint32_t win = __reduce_min_sync(
            0xffffffffu, (bm >= 0 && key == top) ? (uint32_t)(lane + 32 * bm) : 0xffffffffu);
        if ((int)(win & 31u) == lane) {
            idx[r] = (int32_t)win;
            w[r] = bv;
            taken |= 1u << bm;
            local_best();
        }
    }
    __syncwarp();
    if (lane == 0) {
        const float m = w[0];
        float sum = 0.f;
#pragma unroll 1
        for (int r = 0; r < k; ++r) {
            const float e = expf(w[r] - m);
            w[r] = e;
            sum += e;
        }
#pragma unroll 1
        for (int r = 0; r < k; ++r) w[r] = w[r] / sum;
    }
}

__device__ __forceinline__ void route_warp(const float *__restrict__ logits, int n, int k,
                                           int32_t *idx, float *w)
{
    if (n <= 128)
        route_warp_n<4>(logits, n, k, idx, w);
    else
        route_warp_n<32>(logits, n, k, idx, w);
}

// Modes: kModeTensorWS -- rows are 16-byte aligned; each chunk of a warp (32
// rows x one group of blocks) is one 2-D tensor copy issued by a ninth,
// producer warp (lane w feeds warp w's ring, waiting on the ring's "slot
// released" barriers), so the eight consumer warps only wait, decode and
// accumulate.  kModeFlat -- one 1-D bulk copy per (group, term) into a
// CTA-wide ring.  kModePerLane -- any alignment (and mapped host memory);
// the warp copies its rows' chunks with 16-byte cp.async.
constexpr int kModePerLane = 0, kModeFlat = 2, kModeTensorWS = 3;

// Consumer warps of a CTA: producer mode with the 4-bit formats runs 16, one
// K part each, so a 32-row group streams through all of them at once; every
// other kernel runs 8, each owning two adjacent parts (the 272-byte chunks of
// Q8_0 and MXFP4 need more registers than 16 warps leave).
template <int FMT, int MODE>
__host__ __device__ constexpr int nwc_of()
{
    return (MODE == kModeTensorWS && (FMT == RF_Q4_0 || FMT == RF_Q4_K)) ? 16 : kNW;
}
int nwc_host(int fmt, int mode)
{
    return (mode == kModeTensorWS && (fmt == RF_Q4_0 || fmt == RF_Q4_K)) ? 16 : kNW;
}

template <int FMT, int MODE>
constexpr int threads_of() { return 32 * nwc_of<FMT, MODE>() + (MODE == kModeTensorWS ? 32 : 0); }

// Minimum CTAs per SM the register budget is sized for: producer mode runs
// one CTA per SM (its ring takes most of the shared memory).
template <int FMT, int MODE>
constexpr int min_ctas()
{
    return MODE == kModeTensorWS ? 1 : 2;
}

template <int FMT, int MODE, class KP>
__global__ void __launch_bounds__(threads_of<FMT, MODE>(), min_ctas<FMT, MODE>())
    rowwin_kernel(const __grid_constant__ KP p)
{
    using F = FmtT<FMT>;
    constexpr bool WS = MODE == kModeTensorWS;
    constexpr bool FLAT = MODE == kModeFlat;
    constexpr int NWC = nwc_of<FMT, MODE>();   // consumer warps
    constexpr int PPW = kParts / NWC;          // K parts per consumer warp (1 or 2)
    extern __shared__ __align__(128) uint8_t smem[];

    const int nb = p.nb;
    const int ST = p.stages;
    const int KC = p.kc;
    const int SLOT = p.slot;
    const int NT = p.max_terms;
    const int64_t RB = (int64_t)nb * F::BS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    XRec *xrec = reinterpret_cast<XRec *>(smem);
    const int nrx = nb * F::RPB;   // digit records per activation vector
    size_t off = ((size_t)p.n_x * nrx * sizeof(XRec) + 127) & ~(size_t)127;
    uint8_t *slots = smem + off;
    off += FLAT ? (size_t)ST * SLOT : (size_t)NWC * ST * kRows * SLOT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + off);   // slot filled
    off += (size_t)(FLAT ? ST : NWC * ST) * sizeof(uint64_t);
    uint64_t *ebars = reinterpret_cast<uint64_t *>(smem + off);  // producer mode: slot released
    if constexpr (WS) off += (size_t)NWC * ST * sizeof(uint64_t);
    float *red = reinterpret_cast<float *>(smem + off);   // [2][NT][kParts][32]
    off += (size_t)2 * NT * kParts * 32 * sizeof(float);
    int *cnt = reinterpret_cast<int *>(smem + off);       // arrivals per parity, then groups done
    int *emp = cnt + 4;                                   // flat mode: readers done per stage
    volatile int *fl_fail = cnt + 3;                      // a wait of this CTA gave up
    int *fl_issued = cnt + 8;                             // flat mode: copies issued per stage
    volatile int *gq = cnt + 32;                          // producer mode: upcoming groups
    off += kCntInts * sizeof(int);
    Job *jobs = reinterpret_cast<Job *>(smem + off);      // this launch's jobs, read once
    const int n_jobs = p.n_jobs;
    const unsigned long long limit = p.wait_limit_ns;
    // A wait that gives up (or finds the device status already set) ends the
    // warp's work: every lane of the warp takes the same decision.
    auto wait_all_lanes = [&](uint64_t *bar, uint32_t par) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, par, &g_device_status, limit));
    };

    const int G_total = p.total_groups;
    // Static ranges: every CTA `base` groups, the first `extra` CTAs one
    // more (with two CTAs per SM the extras then land on distinct SMs).
    const int g_base = G_total / (int)gridDim.x, g_extra = G_total - g_base * (int)gridDim.x;
    const int g_lo = (int)blockIdx.x * g_base + min((int)blockIdx.x, g_extra);
    const int g_hi = g_lo + g_base + ((int)blockIdx.x < g_extra ? 1 : 0);

    // This warp's K parts, in blocks: part q is blocks
    // [GS*floor(q*nG/kParts), GS*floor((q+1)*nG/kParts)).  Split granularity:
    // the format's 16-byte group when rows are 16-byte aligned (tensor copies
    // need it), single blocks otherwise.  Either way it depends only on
    // (format, in_dim).  A warp with two parts keeps two accumulators and
    // switches at kb_mid.
    const int GS = RB % 16 == 0 ? F::G : 1;
    const int nG = (nb + GS - 1) / GS;
    auto part_lo = [&](int q) { return min(nb, GS * (q * nG / kParts)); };
    const int kb_lo = part_lo(warp * PPW);
    const int kb_mid = part_lo(warp * PPW + (PPW - 1));
    const int kb_hi = part_lo((warp + 1) * PPW);
    const int n_chunks = (kb_hi - kb_lo + KC - 1) / KC;
    // Items a cursor walks per (group, term): this warp's chunks, or one
    // CTA-wide stage in flat mode.
    const int cur_chunks = FLAT ? 1 : n_chunks;

    if constexpr (FLAT) {
        if ((int)threadIdx.x < ST) mbar_init(&bars[threadIdx.x], 1);
    } else if constexpr (WS) {
        if (warp < NWC && lane < ST) {
            mbar_init(&bars[warp * ST + lane], 1);
            mbar_init(&ebars[warp * ST + lane], 1);
        }
    } else {
        if (lane < ST) mbar_init(&bars[warp * ST + lane], p.row_bulk ? 1 : 32);
    }
    if (threadIdx.x < kCntInts) cnt[threadIdx.x] = 0;
    if constexpr (WS) {
        if ((int)threadIdx.x < p.n_maps)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.maps[threadIdx.x]))
                         : "memory");
    }
    // Routing inside the launch.  A launch that waits on a previous grid, or
    // whose activations come as digits, ranks its logits first thing (warp 0,
    // while the other warps copy the job table) so that its weight copies can
    // start early.  A launch with nothing to wait for ranks them later, while
    // warps 1.. build the activation digits (route_late, below).
    int32_t *s_eidx = cnt + 16;
    float *s_ew = reinterpret_cast<float *>(cnt + 24);
    const bool route_late = !WS && p.route_logits && !p.chained && !p.xr_in;
    const bool route_now = p.route_logits && !route_late;
    if (route_now && warp == 0) route_warp(p.route_logits, p.route_n, p.route_k, s_eidx, s_ew);
    {   // copy the job table out of parameter space in one parallel pass
        const int words = n_jobs * (int)(sizeof(Job) / 4);
        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.jobs);
        uint32_t *dst = reinterpret_cast<uint32_t *>(jobs);
        const int skip = route_now ? 32 : 0;
        if ((int)threadIdx.x >= skip)
            for (int i = (int)threadIdx.x - skip; i < words; i += (int)blockDim.x - skip)
                dst[i] = src[i];
    }
    fence_barrier_init();
    __syncthreads();
    const int32_t *eidx = p.route_logits ? s_eidx : p.expert_idx;
    auto write_route = [&] {
        if (blockIdx.x == 0 && (int)threadIdx.x < p.route_k && p.route_idx_out) {
            p.route_idx_out[threadIdx.x] = s_eidx[threadIdx.x];
            p.route_w_out[threadIdx.x] = s_ew[threadIdx.x];
        }
    };
    if (route_now) write_route();

    uint8_t *my_slots = slots + (size_t)warp * ST * kRows * SLOT;
    uint64_t *my_bars = bars + warp * ST;

    Cursor ic{g_lo, 0, 0, 0, g_lo < g_hi && cur_chunks > 0};
    if (ic.valid) cursor_fix_job(jobs, n_jobs, ic);
    int is = 0;   // stage of the next copy
    uint32_t iph = 0;                  // its phase parity
    uint32_t armed = 0, armed_ph = 0;  // row-bulk copies not yet seen landed, and their parity
    bool lane_withhold = p.fault_withhold && p.row_bulk && blockIdx.x == 0 && warp == 0;

    // Per-lane mode: row r's chunk, rounded out to 16-byte boundaries, goes
    // to row r's slot.  Device memory: lane r issues one 1-D bulk copy of its
    // row's chunk (the copy engine takes 32 requests per chunk; 16-byte
    // cp.async of every piece made the warp wait on hundreds of outstanding
    // requests per chunk), lane 0 arming the stage with the chunk's total
    // bytes.  Mapped host memory: the warp copies one row at a time, lane i
    // taking its i-th 16 bytes, so each copy instruction reads contiguous
    // bytes of the link.
    auto issue = [&](const Cursor &cu) {
        uint64_t *bar = &my_bars[is];
        uint8_t *dst = my_slots + (size_t)is * kRows * SLOT;
        if (lane_withhold) {   // test hook: this stage is never armed and never fills
            lane_withhold = false;
            if (++is == ST) {
                is = 0;
                iph ^= 1u;
            }
            return;
        }
        if (p.row_bulk) {
            armed |= 1u << is;
            armed_ph = (armed_ph & ~(1u << is)) | (iph << is);
        }
        if (++is == ST) {
            is = 0;
            iph ^= 1u;
        }
        const Job &J = jobs[cu.j];
        const int64_t rel0 = (int64_t)(cu.g - J.group_begin) * kRows;
        const int nr = (int)min((int64_t)kRows, (int64_t)J.n_rows - rel0);
        const uint8_t *W = term_matrix(eidx, J, cu.t, RB);
        const int kb = kb_lo + cu.c * KC;
        const int kn = min(KC, kb_hi - kb);
        uintptr_t s = reinterpret_cast<uintptr_t>(W + (J.row0 + rel0) * RB + (int64_t)kb * F::BS);
        if (p.row_bulk) {
            uintptr_t a = 0;
            uint32_t bytes = 0;
            if (lane < nr) {
                const uintptr_t sl = s + (uintptr_t)lane * (uintptr_t)RB;
                a = sl & ~(uintptr_t)15;
                bytes = (uint32_t)(((sl + (uintptr_t)kn * F::BS + 15) & ~(uintptr_t)15) - a);
            }
            const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
            if (lane == 0) mbar_arrive_expect_tx(bar, total);
            __syncwarp();
            if (bytes)
                bulk_g2s(dst + (size_t)lane * SLOT, reinterpret_cast<const void *>(a), bytes, bar);
            return;
        }
        for (int r = 0; r < nr; ++r, s += (uintptr_t)RB) {
            const uintptr_t a = s & ~(uintptr_t)15;
            const int n16 = (int)(((s + (uintptr_t)kn * F::BS + 15) & ~(uintptr_t)15) - a) >> 4;
            for (int i = lane; i < n16; i += 32)
                cp_async16(dst + (size_t)r * SLOT + 16 * i,
                           reinterpret_cast<const void *>(a + 16 * (uintptr_t)i));
        }
        cp_async_arrive(bar);
    };

    // Flat mode: the rows of (group, term) of cursor `cu`, back to back, into
    // CTA stage `st` (one thread).  The copy starts at the 16-byte boundary at
    // or before the group and ends at the one at or after it.
    auto issue_flat = [&](const Cursor &cu, int st) {
        const Job &J = jobs[cu.j];
        const int64_t rel = (int64_t)(cu.g - J.group_begin) * kRows;
        const int64_t nr = min((int64_t)kRows, (int64_t)J.n_rows - rel);
        const uintptr_t src =
            reinterpret_cast<uintptr_t>(term_matrix(eidx, J, cu.t, RB) + (J.row0 + rel) * RB);
        const uintptr_t a = src & ~(uintptr_t)15;
        const uintptr_t e = (src + (uintptr_t)(nr * RB) + 15) & ~(uintptr_t)15;
        ++fl_issued[st];
        mbar_arrive_expect_tx(&bars[st], (uint32_t)(e - a));
        bulk_g2s(slots + (size_t)st * SLOT, reinterpret_cast<const void *>(a), (uint32_t)(e - a),
                 &bars[st]);
    };
    // Next copy at priming time: this warp's chunk, or (one thread) a stage.
    auto prime = [&](int st) {
        if constexpr (FLAT) {
            if (threadIdx.x == 0) issue_flat(ic, st);
        } else {
            issue(ic);
        }
        cursor_advance(jobs, n_jobs, ic, cur_chunks, g_hi);
    };

    // Weights never depend on the previous kernel: when this launch may
    // overlap it (programmatic dependent launch), fill every stage before
    // waiting (unless the rows come from a routing result the previous
    // kernel writes).  A CTA that becomes resident while the previous kernel
    // runs then holds its first chunks by the time the activations exist.
    int primed = 0;
    if constexpr (WS) {
        if (warp == NWC) {
            // Producer.  Groups come from the static range [g_lo, g_hi) or,
            // scheduled dynamically, the CTA's own first group (blockIdx.x)
            // and then tickets (the next one drawn a group ahead).  For each
            // group, lane w copies warp w's chunks, refilling each slot as
            // soon as warp w has released it; a warp with no chunks gets one
            // empty arrival per group instead.  The group index goes to the
            // shared queue before its first arrival; a negative index ends it.
            if (!p.prefetch_early) pdl_wait();   // rows may depend on a previous grid
            const bool dyn = p.sched_slot >= 0;
            const int total = p.total_groups;
            auto draw = [&]() -> int {
                int t = 0;
                if (lane == 0) t = (int)atomicAdd(&g_sched[p.sched_slot], 1u);
                t = __shfl_sync(0xffffffffu, t, 0);
                const int ng = (int)gridDim.x + t;
                return ng < total ? ng : -1;
            };
            const int w = lane & (NWC - 1);
            const int kbl = part_lo(w * PPW);
            const int kbh = part_lo((w + 1) * PPW);
            const int nch = lane < NWC ? (kbh - kbl + KC - 1) / KC : 0;
            int max_nch = nch;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) max_nch = max(max_nch, __shfl_xor_sync(0xffffffffu, max_nch, o));
            uint8_t *wslots = slots + (size_t)w * ST * kRows * SLOT;
            int st = 0;
            uint32_t ph = 0;
            // Slots of warp w whose latest use carries a copy, and the phase
            // parity it was armed at: drained before the CTA exits.
            uint32_t armed = 0, armed_ph = 0;
            bool failed = false;
            bool withhold = p.fault_withhold && blockIdx.x == 0 && lane == 0;
            auto acquire = [&]() -> bool {   // next slot of warp w, once warp w released it
                return mbar_wait_bounded(&ebars[w * ST + st], ph ^ 1u, &g_device_status, limit);
            };
            auto advance = [&] {
                if (++st == ST) {
                    st = 0;
                    ph ^= 1u;
                }
            };
            int g = dyn ? (int)blockIdx.x : (g_lo < g_hi ? g_lo : -1);
            int gnext = g < 0 ? -1 : (dyn ? draw() : (g + 1 < g_hi ? g + 1 : -1));
            int jj = 0;
            for (int gi = 0;; ++gi) {
                if (lane == 0) gq[gi & (kGroupQ - 1)] = g;
                __syncwarp();
                if (g < 0) {
                    if (lane < NWC && acquire()) {
                        mbar_arrive(&bars[w * ST + st]);
                        armed &= ~(1u << st);
                    }
                    break;
                }
                while (jj < n_jobs && g >= jobs[jj].group_begin + groups_of(jobs[jj])) ++jj;
                const Job &J = jobs[jj];
                if (lane < NWC && nch == 0) {
                    if (acquire()) {
                        mbar_arrive(&bars[w * ST + st]);
                        armed &= ~(1u << st);
                        advance();
                    } else {
                        failed = true;
                    }
                }
                for (int t = 0; t < J.n_terms; ++t) {
                    const Term &T = J.term[t];
                    int64_t y = J.row0 + (int64_t)(g - J.group_begin) * kRows;
                    if (T.expert_slot >= 0) y += (int64_t)eidx[T.expert_slot] * J.expert_rows;
                    for (int c = 0; c < max_nch; ++c) {
                        if (c < nch && !failed) {
                            if (!acquire()) {
                                failed = true;
                                continue;
                            }
                            if (withhold) {   // test hook: this stage never fills
                                withhold = false;
                                armed &= ~(1u << st);
                                advance();
                                continue;
                            }
                            const int x = (kbl + c * KC) * F::BS / 2;   // uint16 units
                            mbar_arrive_expect_tx(&bars[w * ST + st], (uint32_t)(kRows * SLOT));
                            tma_2d_g2s(wslots + (size_t)st * kRows * SLOT, &p.maps[T.tmap], x,
                                       (int)y, &bars[w * ST + st]);
                            armed |= 1u << st;
                            armed_ph = (armed_ph & ~(1u << st)) | (ph << st);
                            advance();
                        }
                    }
                }
                // After a failure no further copy is issued; the consumer
                // warps find their next stages empty and leave.
                if (__any_sync(0xffffffffu, failed)) break;
                g = gnext;
                gnext = g < 0 ? -1 : (dyn ? draw() : (g + 1 < g_hi ? g + 1 : -1));
            }
            // Every issued copy lands before the CTA may exit (on the normal
            // path its consumer has already seen it: each check passes at once).
            if (lane < NWC)
                for (int i = 0; i < ST; ++i)
                    if ((armed >> i) & 1u) mbar_drain(&bars[w * ST + i], (armed_ph >> i) & 1u);
            if (dyn && lane == 0) {
                __threadfence();   // this CTA's draws come before its count
                if (atomicAdd(&g_sched_done[p.sched_slot], 1u) == gridDim.x - 1) {
                    g_sched[p.sched_slot] = 0;
                    g_sched_done[p.sched_slot] = 0;
                }
            }
            return;
        }
    } else if (p.prefetch_early) {
        for (; primed < ST && ic.valid; ++primed) prime(primed);
    }
    // A chained launch brings the activations it will read into L2 while the
    // previous grid drains (L2 is the coherence point, so lines that grid
    // still writes stay current): each consumer warp its own K range in
    // producer mode, else the whole vectors spread over the CTA.  Activations
    // the weight stream has evicted then cost an L2 hit after the wait
    // instead of a DRAM round trip.
    if (p.chained && !p.xr_in) {
        const int lo = WS ? kb_lo * F::RPB * 32 : 0;
        const int hi = WS ? kb_hi * F::RPB * 32 : nrx * 32;
        const int t0 = WS ? lane : (int)threadIdx.x;
        const int nt = WS ? 32 : kThreads;
        for (int sl = 0; sl < p.n_x; ++sl)
            for (int e = lo + 32 * t0; e < hi; e += 32 * nt)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.x[sl] + e));
    }
    pdl_launch_dependents();
    pdl_wait();

    // Activation digits, copied when the launch that produced the activations
    // also wrote their digits, otherwise built by four lanes per 32-element
    // block.  Producer mode: every consumer warp reads only the records of its
    // own K part, so it prepares just those and starts at once (no CTA-wide
    // barrier).  Other modes: all records once per CTA, the first kXPre
    // passes' loads issued before the remaining weight copies so they do not
    // queue behind them.
    if constexpr (WS) {
        const int rlo = kb_lo * F::RPB, nrw = (kb_hi - kb_lo) * F::RPB;
        const int total = p.n_x * nrw;   // records this warp prepares
        if (total > 0 && p.xr_in) {
            constexpr int kV = (int)(sizeof(XRec) / 16);
            constexpr int kU = 8;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.xr_in);
            uint4 *dst = reinterpret_cast<uint4 *>(xrec);
            const int n16 = total * kV;
            for (int base = 0; base < n16; base += kU * 32) {
                uint4 t[kU];
                int at[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = base + u * 32 + lane;
                    at[u] = 0;
                    if (i < n16) {
                        const int r = i / kV, h = i - kV * r;
                        const int sl = p.n_x == 1 ? 0 : r / nrw, k = r - sl * nrw;
                        at[u] = (sl * nrx + rlo + k) * kV + h;
                        t[u] = src[at[u]];
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (base + u * 32 + lane < n16) dst[at[u]] = t[u];
            }
        } else if (total > 0) {
            constexpr int kXPre = 4;
            const int passes = (total + 7) / 8;
            auto pass_src = [&](int ps, bool &active, int &rec) -> const float * {
                const int r = ps * 8 + (lane >> 2);
                active = r < total;
                const int rr = active ? r : 0;
                const int sl = p.n_x == 1 ? 0 : rr / nrw, k = rr - sl * nrw;
                rec = sl * nrx + rlo + k;
                return p.x[sl] + 32 * (int64_t)(rlo + k);
            };
            for (int ps0 = 0; ps0 < passes; ps0 += kXPre) {
                float v[kXPre][8];
                bool act[kXPre];
                int rec[kXPre];
#pragma unroll
                for (int u = 0; u < kXPre; ++u) {
                    act[u] = false;
                    rec[u] = 0;
                    if (ps0 + u < passes) {
                        const float *xb = pass_src(ps0 + u, act[u], rec[u]);
                        xrec_load<FMT>(xb, lane & 3, act[u], v[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < kXPre; ++u)
                    if (ps0 + u < passes) xrec_build<FMT>(v[u], lane & 3, act[u], &xrec[rec[u]]);
            }
        }
        __syncwarp();
    } else {
        if (p.xr_in) {
            const int n16 = p.n_x * nrx * (int)(sizeof(XRec) / 16);
            const uint4 *src = reinterpret_cast<const uint4 *>(p.xr_in);
            uint4 *dst = reinterpret_cast<uint4 *>(xrec);
            constexpr int kU = 8;
            for (int base = 0; base < n16; base += kU * kThreads) {
                uint4 t[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = base + u * kThreads + (int)threadIdx.x;
                    if (i < n16) t[u] = src[i];
                }
                if (base == 0)
                    for (int s = primed; s < ST && ic.valid; ++s) prime(s);
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = base + u * kThreads + (int)threadIdx.x;
                    if (i < n16) dst[i] = t[u];
                }
            }
        } else if (route_late && warp == 0) {
            // Warp 0 ranks the logits while warps 1.. build the digits.  In
            // flat mode (one thread issues every copy) it then starts the first
            // stages at once; otherwise the copies start after the barrier.
            route_warp(p.route_logits, p.route_n, p.route_k, s_eidx, s_ew);
            if constexpr (FLAT) {
                __syncwarp();
                for (; primed < ST && ic.valid; ++primed) prime(primed);
            }
        } else {
            constexpr int kXPre = 8;
            const int xt = route_late ? (int)threadIdx.x - 32 : (int)threadIdx.x;
            const int xn = route_late ? kThreads - 32 : kThreads;
            const int n_rec = p.n_x * nrx;
            const int passes = (4 * n_rec + xn - 1) / xn;
            auto pass_src = [&](int ps, bool &active, int &rec) -> const float * {
                const int idx = ps * xn + xt;
                active = idx < 4 * n_rec;
                rec = active ? idx >> 2 : 0;
                const int sl = p.n_x == 1 ? 0 : rec / nrx, b = rec - sl * nrx;
                return p.x[sl] + 32 * (int64_t)b;
            };
            float v[kXPre][8];
            bool act[kXPre];
            int rec[kXPre];
#pragma unroll
            for (int ps = 0; ps < kXPre; ++ps) {
                act[ps] = false;
                rec[ps] = 0;
                if (ps < passes) {
                    const float *xb = pass_src(ps, act[ps], rec[ps]);
                    xrec_load<FMT>(xb, xt & 3, act[ps], v[ps]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[ps][i] = 0.f;
                }
            }
            if (!route_late)
                for (int s = primed; s < ST && ic.valid; ++s) prime(s);
#pragma unroll
            for (int ps = 0; ps < kXPre; ++ps)
                if (ps < passes) xrec_build<FMT>(v[ps], xt & 3, act[ps], &xrec[rec[ps]]);
            for (int ps = kXPre; ps < passes; ++ps) {
                bool a = false;
                int rc = 0;
                const float *xb = pass_src(ps, a, rc);
                float w[8];
                xrec_load<FMT>(xb, xt & 3, a, w);
                xrec_build<FMT>(w, xt & 3, a, &xrec[rc]);
            }
        }
        __syncthreads();
        if (route_late) {
            write_route();
            if constexpr (FLAT) {
                // Every thread keeps its own cursor: bring the other warps'
                // to where warp 0's priming left its own.
                if (warp != 0)
                    for (; primed < ST && ic.valid; ++primed) cursor_advance(jobs, n_jobs, ic, 1, g_hi);
            } else {
                for (int s = primed; s < ST && ic.valid; ++s) prime(s);
            }
        }
    }

    int cs = 0;          // stage of the next chunk to consume
    uint32_t cph = 0;    // its mbarrier phase parity
    int j = 0;
    bool failed = false;
    for (int gi = 0, g = g_lo;; ++gi, ++g) {
        if constexpr (WS) {
            // The producer names the group before the arrival that fills (or,
            // for a warp without chunks, only signals) this warp's next slot.
            if (!wait_all_lanes(&my_bars[cs], cph)) break;
            g = gq[gi & (kGroupQ - 1)];
            if (g < 0) break;
            if (n_chunks == 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&ebars[warp * ST + cs]);
                if (++cs == ST) {
                    cs = 0;
                    cph ^= 1u;
                }
            }
        } else if (g >= g_hi) {
            break;
        }
        while (j < n_jobs && g >= jobs[j].group_begin + groups_of(jobs[j])) ++j;
        const Job &J = jobs[j];
        const int n_terms = J.n_terms;
        const bool aligned = WS || J.aligned;
        const int64_t rowrel = (int64_t)(g - J.group_begin) * kRows + lane;
        const bool row_ok = rowrel < J.n_rows;
        const int par = gi & 1;
        float *red_g = red + (size_t)par * NT * kParts * 32;
        // The partial buffer of this parity was last used by group gi-2; wait
        // until that group has been combined.
        if (gi >= 2) {
            volatile int *done = cnt + 2;
            bool ok = true;
            if (*done < gi - 1) {
                const unsigned long long t0 = globaltimer_ns();
                for (uint32_t it = 0; *done < gi - 1; ++it) {
                    if ((it & 63u) != 63u) continue;
                    if (*reinterpret_cast<volatile int *>(&g_device_status) != 0) {
                        ok = false;
                        break;
                    }
                    if (globaltimer_ns() - t0 > limit) {
                        record_status(&g_device_status, RF_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if constexpr (FLAT) *fl_fail = 1;
                break;
            }
            __threadfence_block();
        }
        for (int t = 0; t < n_terms; ++t) {
            float acc = 0.f, acc1 = 0.f;   // parts warp*PPW and warp*PPW + 1
            uintptr_t row_src = 0;
            if (!FLAT && !aligned && row_ok)
                row_src = reinterpret_cast<uintptr_t>(term_matrix(eidx, J, t, RB) +
                                                      (J.row0 + rowrel) * RB);
            const XRec *xr_row = xrec + (size_t)J.term[t].xslot * nrx;
            if constexpr (FLAT) {
                // Every warp waits for the stage (so none runs ahead of the
                // ring), reads its K part of its lane's row, then counts
                // itself out; the last one refills the stage.
                const int st = cs;
                if (!wait_all_lanes(&bars[st], cph)) {
                    *fl_fail = 1;
                    failed = true;
                    break;
                }
                if (row_ok && kb_hi > kb_lo) {
                    const uintptr_t src = reinterpret_cast<uintptr_t>(
                        term_matrix(eidx, J, t, RB) + (J.row0 + rowrel - lane) * RB);
                    const uintptr_t rp = reinterpret_cast<uintptr_t>(slots + (size_t)st * SLOT) +
                                         (src & 15) + (uintptr_t)((int64_t)lane * RB) +
                                         (uintptr_t)kb_lo * F::BS;
                    const uintptr_t rp1 = rp + (uintptr_t)(kb_mid - kb_lo) * F::BS;
                    acc = chunk_generic<FMT>(reinterpret_cast<const uint8_t *>(rp & ~(uintptr_t)3),
                                             (int)(rp & 3), kb_mid - kb_lo,
                                             xr_row + kb_lo * F::RPB, acc);
                    acc1 = chunk_generic<FMT>(reinterpret_cast<const uint8_t *>(rp1 & ~(uintptr_t)3),
                                              (int)(rp1 & 3), kb_hi - kb_mid,
                                              xr_row + kb_mid * F::RPB, acc1);
                }
                if (++cs == ST) {
                    cs = 0;
                    cph ^= 1u;
                }
                __syncwarp();
                if (lane == 0 && atomicAdd(&emp[st], 1) == NWC - 1) {
                    emp[st] = 0;
                    if (ic.valid && *fl_fail == 0) issue_flat(ic, st);
                }
                if (ic.valid) cursor_advance(jobs, n_jobs, ic, 1, g_hi);
            }
            for (int c = 0; c < (FLAT ? 0 : n_chunks); ++c) {
                const int cur = cs;
                if (!wait_all_lanes(&my_bars[cur], cph)) {
                    failed = true;
                    break;
                }
                armed &= ~(1u << cur);
                const uint8_t *slot = my_slots + ((size_t)cur * kRows + lane) * SLOT;
                if (++cs == ST) {
                    cs = 0;
                    cph ^= 1u;
                }
                const int kb = kb_lo + c * KC;
                const int kn = min(KC, kb_hi - kb);
                if constexpr (WS) {
                    // A chunk is exactly one G-group, which never straddles a
                    // part boundary: it joins the accumulator of its part.
                    float &a = (PPW == 1 || kb < kb_mid) ? acc : acc1;
                    if constexpr (FMT == RF_MXFP4) {
                        // 16 blocks of 17 bytes: the first 8 come from the
                        // first 9 16-byte words; decode them before loading
                        // the rest, so that fewer words are live at once.
                        GroupRegs<FMT> r;
                        load_group_part<FMT, 0, 9>(slot, r);
                        a = compute_blocks<FMT, 0, 8>(r, xr_row + kb * F::RPB, a);
                        load_group_part<FMT, 9, 17>(slot, r);
                        r.v[68] = 0;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ebars[warp * ST + cur]);
                        a = compute_blocks<FMT, 8, 16>(r, xr_row + kb * F::RPB, a);
                    } else {
                        // Copy the chunk to registers, hand the slot straight
                        // back to the producer, then compute.
                        GroupRegs<FMT> r;
                        load_group<FMT>(slot, r);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ebars[warp * ST + cur]);
                        a = compute_group<FMT>(r, xr_row + kb * F::RPB, a);
                    }
                    continue;
                }
                // Blocks [kb, kb + n0) belong to this warp's first part, the
                // rest of the chunk to its second.
                const int n0 = max(0, min(kn, kb_mid - kb));
                if constexpr (FMT == RF_Q6_K) {
                    const int phi = (int)((row_src + (uintptr_t)kb * F::BS) & 15);
                    if (n0 > 0) acc = chunk_generic<FMT>(slot, phi, n0, xr_row + kb * F::RPB, acc);
                    if (n0 < kn)
                        acc1 = chunk_generic<FMT>(slot, phi + n0 * F::BS, kn - n0,
                                                  xr_row + (kb + n0) * F::RPB, acc1);
                } else if (aligned) {
                    // chunks are G-groups and parts start on G-group bounds
                    if (n0 > 0) acc = chunk_aligned<FMT>(slot, kn, xr_row + kb * F::RPB, acc);
                    else acc1 = chunk_aligned<FMT>(slot, kn, xr_row + kb * F::RPB, acc1);
                } else {
                    const int phi = (int)((row_src + (uintptr_t)kb * F::BS) & 15);
                    if (n0 > 0) acc = chunk_generic<FMT>(slot, phi, n0, xr_row + kb * F::RPB, acc);
                    if (n0 < kn)
                        acc1 = chunk_generic<FMT>(slot, phi + n0 * F::BS, kn - n0,
                                                  xr_row + (kb + n0) * F::RPB, acc1);
                }
                __syncwarp();
                if (ic.valid) {
                    issue(ic);
                    cursor_advance(jobs, n_jobs, ic, n_chunks, g_hi);
                }
            }
            if (failed) break;
            red_g[((size_t)t * kParts + warp * PPW) * 32 + lane] = acc;
            if constexpr (PPW == 2) red_g[((size_t)t * kParts + warp * PPW + 1) * 32 + lane] = acc1;
        }
        if (failed) break;
        // The last warp to finish this group sums the partials in part order.
        __syncwarp();
        __threadfence_block();
        int arrived = 0;
        if (lane == 0) arrived = atomicAdd(&cnt[par], 1);
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == NWC - 1) {
            __threadfence_block();
            float yacc = 0.f, gate = 0.f;
            for (int t = 0; t < n_terms; ++t) {
                const float *rt = red_g + (size_t)t * kParts * 32 + lane;
                float dot = rt[0];
#pragma unroll
                for (int q = 1; q < kParts; ++q) dot += rt[q * 32];
                const Term &T = J.term[t];
                if (T.bias && row_ok) {   // biased projection: the row's bias joins its dot
                    int64_t bi = J.row0 + rowrel;
                    if (T.expert_slot >= 0) bi += (int64_t)eidx[T.expert_slot] * J.expert_rows;
                    dot += T.bias[bi];
                }
                if (J.combine == kCombineEach) {
                    if (row_ok) J.y[t * J.y_stride + rowrel] = dot;
                    continue;
                }
                if (J.combine == kCombineSwiGLU) {
                    if (t == 0) {
                        gate = dot;
                    } else if (J.act == kActClampSwiGLU) {
                        const float g = fminf(gate, J.limit);
                        const float u = fminf(fmaxf(dot, -J.limit), J.limit);
                        yacc = g / (1.f + expf(-J.alpha * g)) * (u + 1.f);
                    } else {
                        yacc = gate / (1.f + expf(-gate)) * dot;
                    }
                } else if (J.combine == kCombineRouted) {
                    yacc = fmaf(s_ew[J.term[t].expert_slot], dot, yacc);
                } else if (J.weights) {
                    yacc = fmaf(J.weights[t], dot, yacc);
                } else {
                    yacc = t == 0 ? dot : yacc + dot;
                }
            }
            float out = yacc;
            if (J.act == kActGelu) out = 0.5f * out * (1.f + erff(out * 0.70710678118654752f));
            if (row_ok && J.combine != kCombineEach) J.y[rowrel] = out;
            if (p.xr_out)
                xrec_emit<FMT>(row_ok ? out : 0.f,
                               p.xr_out + ((J.y - p.xr_y_base) + (rowrel - lane)) / kRows);
            __syncwarp();
            if (lane == 0) {
                cnt[par] = 0;
                __threadfence_block();
                atomicAdd(&cnt[2], 1);
            }
        }
    }
    // Nothing this CTA issued may still be writing its shared memory when it
    // exits: after a failure, wait for the bulk copies of every stage (each
    // lands whatever else failed); cp.async copies are this thread's own.
    if constexpr (FLAT) {
        __syncthreads();
        if (threadIdx.x == 0 && *fl_fail)
            for (int i = 0; i < ST; ++i)
                if (fl_issued[i] > 0) mbar_drain(&bars[i], (uint32_t)(fl_issued[i] - 1) & 1u);
    } else if constexpr (!WS) {
        cp_async_wait_all();
        // Row-bulk copies issued into stages this warp never consumed land
        // before the CTA exits.
        if (lane == 0)
            for (int st = 0; st < ST; ++st)
                if (armed & (1u << st)) mbar_drain(&my_bars[st], (armed_ph >> st) & 1u);
    }
}

struct DevInfo {
    int max_smem_block = 0;   // opt-in maximum per CTA
    int max_smem_sm = 0;
    int reserved_per_block = 0;
    int sms = 1;
};
DevInfo g_dev[64];
std::once_flag g_dev_once[64];

const DevInfo &dev_info(int dev)
{
    std::call_once(g_dev_once[dev & 63], [dev] {
        DevInfo &d = g_dev[dev & 63];
        cudaDeviceGetAttribute(&d.max_smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&d.max_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&d.reserved_per_block, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        if (d.sms < 1) d.sms = 1;
    });
    return g_dev[dev & 63];
}

int fmt_group(int fmt) { return fmt == RF_MXFP4 ? 16 : (fmt == RF_Q4_K || fmt == RF_Q6_K ? 1 : 8); }

// Chunk of `kc` blocks and its slot size.  Aligned rows copy exactly KC*BS
// bytes; others need up to 15 bytes of rounding on either side.  Slots are an
// odd number of 16-byte units so the 32 lanes' 16-byte loads spread over all
// banks.
struct ChunkGeom {
    int kc, slot;
};
ChunkGeom chunk_geom(int fmt, bool aligned)
{
    const int bs = (int)block_bytes_of(fmt);
    if (aligned) {
        // A dense [32][kc*bs] tensor box; kc*bs = 144 or 272 bytes, an odd
        // number of 16-byte units.
        const int kc = fmt_group(fmt);
        return {kc, kc * bs};
    }
    const int kc = fmt == RF_Q4_K || fmt == RF_Q6_K ? 1 : 8;
    int n = (kc * bs + 30 + 15) / 16 * 16;
    if ((n / 16) % 2 == 0) n += 16;
    return {kc, n};
}

// Flat mode: a stage holds one 32-row group back to back, plus the 16-byte
// rounding at both ends and a word of overrun for the last row's decode.
int flat_slot(int64_t row_bytes) { return (int)((kRows * row_bytes + 32 + 127) / 128 * 128); }

// nrx: activation digit records per x (in_dim / 32); nwc: consumer warps.
size_t smem_bytes(int n_x, int nrx, int stages, int slot, int max_terms, int n_jobs,
                  bool flat = false, bool ws = false, int nwc = kNW)
{
    return (((size_t)n_x * nrx * sizeof(XRec) + 127) & ~(size_t)127) +
           (flat ? (size_t)stages * slot : (size_t)nwc * stages * kRows * slot) +
           (size_t)(flat ? stages : nwc * stages * (ws ? 2 : 1)) * sizeof(uint64_t) +
           (size_t)2 * max_terms * kParts * 32 * sizeof(float) + kCntInts * sizeof(int) +
           (size_t)n_jobs * sizeof(Job);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        cudaGetLastError();
    });
    return fn;
}

// 2-D view of `rows` rows of `rb` bytes at `base` as uint16 elements; boxes of
// 32 rows x `chunk` bytes.
bool encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t rb, int chunk)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(rb / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)rb};
    const cuuint32_t box[2] = {(cuuint32_t)(chunk / 2), (cuuint32_t)kRows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int MODE, class KP>
rf_status launch_fmt(const KP &p, int grid, size_t smem, bool pdl, cudaStream_t stream, int dev)
{
    static std::once_flag attr_once[64];
    const int maxs = dev_info(dev).max_smem_block;
    static bool attr_ok[64];
    std::call_once(attr_once[dev & 63], [maxs, dev] {
        attr_ok[dev & 63] = cudaFuncSetAttribute(rowwin_kernel<FMT, MODE, KP>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 maxs) == cudaSuccess;
        cudaGetLastError();
    });
    if (!attr_ok[dev & 63]) return RF_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads_of<FMT, MODE>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, rowwin_kernel<FMT, MODE, KP>, p) != cudaSuccess) return RF_ERR_CUDA;
    return RF_OK;
}

template <int MODE, class KP>
rf_status launch_mode(int fmt, const KP &p, int grid, size_t smem, bool pdl, cudaStream_t stream,
                      int dev)
{
    switch (fmt) {
    case RF_Q4_0: return launch_fmt<RF_Q4_0, MODE>(p, grid, smem, pdl, stream, dev);
    case RF_Q8_0: return launch_fmt<RF_Q8_0, MODE>(p, grid, smem, pdl, stream, dev);
    case RF_Q4_K: return launch_fmt<RF_Q4_K, MODE>(p, grid, smem, pdl, stream, dev);
    case RF_Q6_K:   // 210-byte super-blocks never take tensor copies
        if constexpr (MODE == kModeTensorWS) return RF_ERR_INVALID_ARG;
        else return launch_fmt<RF_Q6_K, MODE>(p, grid, smem, pdl, stream, dev);
    default: return launch_fmt<RF_MXFP4, MODE>(p, grid, smem, pdl, stream, dev);
    }
}

template <class KP>
rf_status launch_any(int fmt, int mode, const KP &p, int grid, size_t smem, bool pdl,
                     cudaStream_t stream, int dev)
{
    if (mode == kModeTensorWS)
        return launch_mode<kModeTensorWS>(fmt, p, grid, smem, pdl, stream, dev);
    if (mode == kModeFlat) return launch_mode<kModeFlat>(fmt, p, grid, smem, pdl, stream, dev);
    return launch_mode<kModePerLane>(fmt, p, grid, smem, pdl, stream, dev);
}

// Tensor maps of recent weight tensors (host-side encoding is not free and
// the same tensors recur every token).
struct MapKey {
    const void *base;
    int64_t rows, rb;
    int chunk, dev;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && rows == o.rows && rb == o.rb && chunk == o.chunk && dev == o.dev;
    }
};
std::atomic<uint32_t> g_sched_seq{0};
// One-shot test fault for the next producer-mode launch (0 = none): the wait
// limit in nanoseconds that launch runs with.
std::atomic<unsigned long long> g_fault_limit_ns{0};

constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_next = 0;

bool cached_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t rb, int chunk, int dev)
{
    const MapKey k{base, rows, rb, chunk, dev};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (int i = 0; i < kMapCache; ++i)
            if (g_map_key[i] == k) {
                *m = g_map_val[i];
                return true;
            }
    }
    if (!encode_rows_map(m, base, rows, rb, chunk)) return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_map_key[g_map_next] = k;
    g_map_val[g_map_next] = *m;
    g_map_next = (g_map_next + 1) % kMapCache;
    return true;
}

}  // namespace

bool encode_u16_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long take_wait_fault() { return g_fault_limit_ns.exchange(0); }

rf_status arm_wait_fault(uint32_t limit_us)
{
    if (limit_us > 2000000u) return RF_ERR_INVALID_ARG;
    g_fault_limit_ns.store((unsigned long long)limit_us * 1000ull);
    return RF_OK;
}

rf_status read_and_clear_device_status()
{
    if (cudaDeviceSynchronize() != cudaSuccess) return RF_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
            return RF_ERR_CUDA;
    }
    return static_cast<rf_status>(v);
}

bool fmt_ok(int fmt)
{
    return fmt == RF_Q4_0 || fmt == RF_Q8_0 || fmt == RF_MXFP4 || fmt == RF_Q4_K ||
           fmt == RF_Q6_K;
}

size_t block_bytes_of(int fmt)
{
    switch (fmt) {
    case RF_Q4_0: return 18;
    case RF_Q8_0: return 34;
    case RF_MXFP4: return 17;
    case RF_Q4_K: return 144;
    case RF_Q6_K: return 210;
    default: return 0;
    }
}

rf_status last_cuda_error() { return cudaGetLastError() == cudaSuccess ? RF_OK : RF_ERR_CUDA; }

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return dev_info(dev).sms;
}

int64_t max_in_dim(int fmt, int n_x)
{
    if (!fmt_ok(fmt) || n_x < 1 || n_x > kMaxX) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const size_t maxs = (size_t)dev_info(dev).max_smem_block;
    const int slot = std::max(chunk_geom(fmt, true).slot, chunk_geom(fmt, false).slot);
    const size_t fixed = smem_bytes(n_x, 0, 1, slot, kMaxTerms, kMaxJobs);
    if (maxs <= fixed) return 0;
    const int64_t elems = (int64_t)((maxs - fixed) / ((size_t)n_x * sizeof(XRec))) * 32;
    return elems / block_elems_of(fmt) * block_elems_of(fmt);
}

rf_status check_in_dim(int fmt, int64_t in_dim, int n_x)
{
    const int64_t m = max_in_dim(fmt, n_x);
    if (m == 0) return RF_ERR_CUDA;
    return in_dim > m ? RF_ERR_TOO_LARGE : RF_OK;
}

namespace {

// B starts where A ends, with identical terms and epilogue.
bool continues(const Job &A, const Job &B)
{
    if (A.n_terms != B.n_terms || A.combine != B.combine || A.act != B.act ||
        A.weights != B.weights || A.expert_rows != B.expert_rows ||
        A.expert_count != B.expert_count || A.y_stride != B.y_stride ||
        A.alpha != B.alpha || A.limit != B.limit)
        return false;
    if (B.row0 != A.row0 + A.n_rows || B.y != A.y + A.n_rows) return false;
    if ((int64_t)A.n_rows + B.n_rows > 0x7fffffffLL) return false;
    for (int t = 0; t < A.n_terms; ++t)
        if (A.term[t].W != B.term[t].W || A.term[t].xslot != B.term[t].xslot ||
            A.term[t].expert_slot != B.term[t].expert_slot || A.term[t].bias != B.term[t].bias)
            return false;
    return true;
}

}  // namespace

static rf_status launch_merged(const LaunchDesc &d, int nb, int64_t RB, cudaStream_t stream);

rf_status launch_rowwin(const LaunchDesc &d, cudaStream_t stream)
{
    if (!fmt_ok(d.fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (d.in_dim <= 0 || d.in_dim % block_elems_of(d.fmt) != 0) return RF_ERR_INVALID_ARG;
    if (d.n_jobs < 0 || d.n_x < 1 || d.n_x > kMaxX) return RF_ERR_INVALID_ARG;
    if (d.n_jobs > 0 && !d.jobs) return RF_ERR_INVALID_ARG;
    for (int s = 0; s < d.n_x; ++s)
        if (!d.x[s]) return RF_ERR_INVALID_ARG;
    if (d.any_expert && !d.expert_idx && !d.route_logits) return RF_ERR_INVALID_ARG;
    if (d.xr_out) {
        if (!d.xr_y_base || (reinterpret_cast<uintptr_t>(d.xr_out) & 15u) != 0)
            return RF_ERR_INVALID_ARG;
        for (int i = 0; i < d.n_jobs; ++i)
            if ((d.jobs[i].y - d.xr_y_base) % kRows != 0 || d.jobs[i].n_rows % kRows != 0 ||
                d.jobs[i].y < d.xr_y_base)
                return RF_ERR_INVALID_ARG;
    }
    if (d.xr_in && (reinterpret_cast<uintptr_t>(d.xr_in) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (d.route_logits && (d.route_n < 1 || d.route_n > 1024 || d.route_k < 1 ||
                           d.route_k > kMaxTerms || d.route_k > d.route_n))
        return RF_ERR_INVALID_ARG;
    const int64_t nb64 = d.in_dim / block_elems_of(d.fmt);
    if (nb64 > (1 << 24)) return RF_ERR_TOO_LARGE;
    const int nb = (int)nb64;
    const int64_t RB = nb64 * (int64_t)block_bytes_of(d.fmt);

    // Validate every job before enqueueing anything.
    for (int i = 0; i < d.n_jobs; ++i) {
        const Job &J = d.jobs[i];
        if (J.n_rows < 0 || J.row0 < 0 || J.n_terms < 1 || J.n_terms > kMaxTerms)
            return RF_ERR_INVALID_ARG;
        if (J.n_rows > 0 && !J.y) return RF_ERR_INVALID_ARG;
        if (J.combine == kCombineSwiGLU && J.n_terms != 2) return RF_ERR_INVALID_ARG;
        if (J.combine == kCombineEach &&
            (d.xr_out || (J.n_terms > 1 && J.y_stride < (int64_t)J.n_rows)))
            return RF_ERR_INVALID_ARG;
        for (int t = 0; t < J.n_terms; ++t) {
            const Term &T = J.term[t];
            if (!T.W) return RF_ERR_INVALID_ARG;
            if ((reinterpret_cast<uintptr_t>(T.W) & 15u) != 0) return RF_ERR_MISALIGNED;
            if (T.xslot < 0 || T.xslot >= d.n_x) return RF_ERR_INVALID_ARG;
            if (T.expert_slot >= kMaxTerms) return RF_ERR_INVALID_ARG;
            if (T.expert_slot >= 0 && ((!d.expert_idx && !d.route_logits) || J.expert_rows <= 0))
                return RF_ERR_INVALID_ARG;
            if (T.expert_slot >= 0 && d.route_logits && T.expert_slot >= d.route_k)
                return RF_ERR_INVALID_ARG;
        }
    }
    // Windows that continue one another (same matrices, activations and
    // epilogue; the next rows of the matrix written to the next outputs) are
    // one window to the kernel.  Every output row's arithmetic is unchanged.
    static thread_local std::vector<Job> merged;
    merged.clear();
    for (int i = 0; i < d.n_jobs; ++i) {
        const Job &J = d.jobs[i];
        if (J.n_rows == 0) continue;
        if (!merged.empty() && continues(merged.back(), J)) {
            merged.back().n_rows += J.n_rows;
            continue;
        }
        merged.push_back(J);
    }
    LaunchDesc dm = d;
    dm.jobs = merged.data();
    dm.n_jobs = (int)merged.size();
    return launch_merged(dm, nb, RB, stream);
}

static rf_status launch_merged(const LaunchDesc &d, int nb, int64_t RB, cudaStream_t stream)
{
    const int nrx = (int)(d.in_dim / 32);   // activation digit records per x
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    const DevInfo &di = dev_info(dev);
    if (di.max_smem_block == 0) return RF_ERR_CUDA;

    // Rows are 16-byte aligned when the row bytes are (weights are 16-byte
    // aligned): then chunks are copied exactly.  Q6_K's 210-byte super-blocks
    // never fill whole 16-byte units, so its rows take the other modes.
    const bool aligned = RB % 16 == 0 && d.fmt != RF_Q6_K;
    ChunkGeom geo = chunk_geom(d.fmt, aligned);
    int max_terms = 1;
    for (int i = 0; i < d.n_jobs; ++i) max_terms = std::max(max_terms, (int)d.jobs[i].n_terms);
    const int nj_max = std::min(d.n_jobs, kMaxJobs);
    const size_t per2 = (size_t)di.max_smem_sm / 2 - (size_t)di.reserved_per_block;
    // Mapped host memory is read with per-lane 16-byte copies (plain loads of
    // the link), never with tensor or bulk copies.
    int mode = aligned && !d.host_weights ? kModeTensorWS : kModePerLane;
    int ctas_per_sm = 0, stages = 0;
    // Misaligned rows: stage whole 32-row groups when two of them fit (two
    // CTAs per SM if possible).
    if (!aligned && !d.host_weights) {
        const int fs = flat_slot(RB);
        for (int st = 3; st >= 2 && !ctas_per_sm; --st)
            if (smem_bytes(d.n_x, nrx, st, fs, max_terms, nj_max, true) <= per2) {
                ctas_per_sm = 2;
                stages = st;
            }
        // One CTA per SM: Q6_K's super-block decode costs so much per byte
        // that the CTA-wide stage (refilled only when all 8 warps are done
        // with it) leaves the copy engine idle; its rows take per-lane
        // bulk copies instead, where every warp pipelines its own chunks
        // (the 4096/11008 Q6_K layer: 2.11 vs 1.73 TB/s).
        for (int st = 4; st >= 2 && !ctas_per_sm && d.fmt != RF_Q6_K; --st)
            if (smem_bytes(d.n_x, nrx, st, fs, max_terms, nj_max, true) <=
                (size_t)di.max_smem_block) {
                ctas_per_sm = 1;
                stages = st;
            }
        if (ctas_per_sm) {
            mode = kModeFlat;
            geo = {1, fs};
        }
    }
    // Otherwise per-warp rings.  Producer mode runs one CTA per SM.  With 16
    // consumer warps (Q4_0, Q4_K) it takes the deepest ring that fits; with 8
    // (Q8_0, MXFP4) likewise when the launch has at most four 32-row groups
    // per SM (fewer, deeper CTAs stream such launches faster), else at most 4
    // stages.  When not even one stage fits beside the activation digits,
    // the rows take per-lane copies instead.  Per-lane mode prefers two CTAs
    // per SM with at least 2 stages, else one CTA with up to 4.
    int64_t all_groups = 0;
    for (int i = 0; i < d.n_jobs; ++i) all_groups += (d.jobs[i].n_rows + kRows - 1) / kRows;
    if (mode == kModeTensorWS) {
        const int nwc = nwc_host(d.fmt, mode);
        const bool deep = nwc == 16 || all_groups <= 4 * (int64_t)di.sms;
        for (int st = deep ? 6 : 4; st >= 1 && !ctas_per_sm; --st)
            if (smem_bytes(d.n_x, nrx, st, geo.slot, max_terms, nj_max, false, true, nwc) <=
                (size_t)di.max_smem_block) {
                ctas_per_sm = 1;
                stages = st;
            }
        if (!ctas_per_sm) mode = kModePerLane;
    }
    const bool ws = mode == kModeTensorWS;
    for (int st = 4; st >= 2 && !ctas_per_sm && mode == kModePerLane; --st)
        if (smem_bytes(d.n_x, nrx, st, geo.slot, max_terms, nj_max) <= per2) {
            ctas_per_sm = 2;
            stages = st;
        }
    for (int st = 4; st >= 1 && !ctas_per_sm; --st)
        if (smem_bytes(d.n_x, nrx, st, geo.slot, max_terms, nj_max) <=
            (size_t)di.max_smem_block) {
            ctas_per_sm = 1;
            stages = st;
        }
    if (!ctas_per_sm) return RF_ERR_TOO_LARGE;
    const size_t smem = smem_bytes(d.n_x, nrx, stages, geo.slot, max_terms, nj_max,
                                   mode == kModeFlat, ws, nwc_host(d.fmt, mode));

    // Launch in batches of kMaxJobs windows.
    for (int base = 0; base < d.n_jobs; base += kMaxJobs) {
        const int nj = std::min(kMaxJobs, d.n_jobs - base);
        static thread_local Job jobs[kMaxJobs];
        int total = 0;
        for (int i = 0; i < nj; ++i) {
            jobs[i] = d.jobs[base + i];
            jobs[i].group_begin = total;
            jobs[i].aligned = aligned ? 1 : 0;
            total += (jobs[i].n_rows + kRows - 1) / kRows;
        }
        if (total == 0) continue;
        // One tensor map per distinct weight base, covering every row the
        // batch's jobs can touch.
        const void *bases[kMaxMaps];
        int64_t extent[kMaxMaps];
        int n_maps = 0;
        if (mode == kModeTensorWS) {
            for (int i = 0; i < nj; ++i) {
                Job &J = jobs[i];
                for (int t = 0; t < J.n_terms; ++t) {
                    Term &T = J.term[t];
                    const int64_t need = T.expert_slot >= 0 ? J.expert_count * J.expert_rows
                                                            : J.row0 + J.n_rows;
                    int m = 0;
                    while (m < n_maps && bases[m] != T.W) ++m;
                    if (m == n_maps) {
                        if (n_maps == kMaxMaps) return RF_ERR_TOO_LARGE;
                        bases[m] = T.W;
                        extent[m] = 0;
                        ++n_maps;
                    }
                    extent[m] = std::max(extent[m], need);
                    T.tmap = m;
                }
            }
            for (int m = 0; m < n_maps; ++m)
                if (extent[m] > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
        }
        // Producer mode: one group per CTA to start with, the rest drawn as
        // CTAs finish (no tail from an uneven split of groups over SMs).
        // Other modes: the same number of groups (or one fewer) on every CTA.
        const int max_grid = ctas_per_sm * di.sms;
        const int per_cta = (total + max_grid - 1) / max_grid;
        const int grid = (mode == kModeTensorWS || (mode == kModeFlat && ctas_per_sm == 2))
                             ? std::min(total, max_grid)
                             : (total + per_cta - 1) / per_cta;
        const int sched_slot =
            mode == kModeTensorWS && total > grid
                ? (int)(g_sched_seq.fetch_add(1, std::memory_order_relaxed) % kSchedSlots)
                : -1;

        auto fill = [&](auto &p) -> rf_status {
            std::memcpy(p.jobs, jobs, sizeof(Job) * nj);
            for (int m = 0; m < n_maps; ++m)
                if (!cached_rows_map(&p.maps[m], bases[m], extent[m], RB, geo.slot, dev))
                    return RF_ERR_CUDA;
            for (int s2 = 0; s2 < kMaxX; ++s2) p.x[s2] = s2 < d.n_x ? d.x[s2] : nullptr;
            p.expert_idx = d.expert_idx;
            p.n_jobs = nj;
            p.n_x = d.n_x;
            p.nb = nb;
            p.total_groups = total;
            p.stages = stages;
            p.kc = geo.kc;
            p.slot = geo.slot;
            // Weights may be fetched before the previous grid finishes unless
            // their rows come from a routing result that grid writes.
            p.prefetch_early = (d.pdl && (!d.any_expert || d.route_logits)) ? 1 : 0;
            p.chained = d.pdl ? 1 : 0;
            p.route_logits = d.route_logits;
            p.route_idx_out = d.route_idx_out;
            p.route_w_out = d.route_w_out;
            p.route_n = d.route_n;
            p.route_k = d.route_k;
            p.xr_out = static_cast<XRec *>(d.xr_out);
            p.xr_y_base = d.xr_y_base;
            p.xr_in = static_cast<const XRec *>(d.xr_in);
            p.sched_slot = sched_slot;
            p.max_terms = max_terms;
            p.n_maps = n_maps;
            p.wait_limit_ns = kWaitLimitNs;
            p.fault_withhold = 0;
            p.row_bulk = (mode == kModePerLane && !d.host_weights) ? 1 : 0;
            if ((mode == kModeTensorWS || p.row_bulk) &&
                g_fault_limit_ns.load(std::memory_order_relaxed)) {
                const unsigned long long lim = g_fault_limit_ns.exchange(0);
                if (lim) {
                    p.wait_limit_ns = lim;
                    p.fault_withhold = 1;
                }
            }
            return RF_OK;
        };
        rf_status st;
        if (nj <= 4 && n_maps <= 4) {
            KParamsSmall p;
            if ((st = fill(p)) != RF_OK) return st;
            st = launch_any(d.fmt, mode, p, grid, smem, d.pdl, stream, dev);
        } else {
            static thread_local KParamsLarge p;   // about 18 KB: keep it off the stack
            if ((st = fill(p)) != RF_OK) return st;
            st = launch_any(d.fmt, mode, p, grid, smem, d.pdl, stream, dev);
        }
        if (st != RF_OK) return st;
    }
    return RF_OK;
}

}  // namespace rf
