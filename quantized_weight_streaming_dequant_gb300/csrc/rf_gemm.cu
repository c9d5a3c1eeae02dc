// rf_gemm.cu -- prefill dequant-GEMM on the fifth-generation tensor cores.
//
// What it computes (neurostream, "What the numbers taught us": a prompt or
// an image prefills through one pass over the weights for the whole chunk of
// tokens): Y[t][r - row_start] = sum_i w[r,i] * X[t][i] for every row r of a
// window and every token t of the chunk.  Unlike batch-1 decode this is a
// dense contraction (2 * n_tok flops per weight), so it runs on tcgen05.mma.
//
// gemm_tc_kernel:
//   * A pre-pass rounds X to fp16 once, into the operand layout of the MMA
//     (tiles of N tokens x 64 inputs, K-major core matrices), in a caller
//     workspace; the same launch zeroes the outputs of tiles split in K.
//   * A CTA owns 128 rows x N tokens (N = 64, 128 or 256) and accumulates
//     the whole of K (or half of it, for a tile of a last partial wave) in
//     tensor memory (N fp32 columns per MMA issuer).
//   * Rows whose byte length is a multiple of 16: one thread streams the
//     raw quantized bytes of its 128 rows, a chunk of 8 or 16 blocks (one
//     Q4_K super-block) at a time, with 2-D tensor copies into a ring.
//     Other rows (a tensor map cannot describe them): each decoder thread
//     reads its row's raw bytes itself with aligned 4-byte loads, the next
//     slice's while it decodes the current one.
//   * One thread streams the fp16 activation tiles with 1-D bulk copies.
//   * Twelve decoder warps turn each 64-input slice of the raw rows into
//     fp16 weights w = d * q (one rounding; MXFP4 values are exact; Q4_K's
//     d*sc*q - dmin*m is rounded to fp32 first) in the core-matrix layout;
//     three groups of four warps take the slices round-robin.
//   * One thread issues four tcgen05.mma (M=128, N, K=16) per slice and
//     commits them to the slice's "empty" barrier (two threads, on alternate
//     slices and separate accumulators, where the ring allows); the last
//     commits release the epilogue, which reads the accumulators out of
//     tensor memory.
//   Error: w and x each carry one fp16 rounding (relative 2^-11, absolute
//   2^-25 below the normal range), accumulation is fp32.
//
// Every wait is bounded; after a failure every role stops, copies and MMAs
// already issued are waited for, and tensor memory is freed on every path.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

__device__ int g_gemm_status = 0;   // bounded-wait failures (read by rf_device_status)

constexpr int kGM = 128;       // rows per CTA (MMA M)

// Shared-memory matrix descriptor of a K-major tile without swizzle: start
// address, leading-dimension byte offset 128 (the next core matrix along K),
// stride-dimension byte offset `sbo` (the next 8 rows), the fixed version
// bits.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 16;
    d |= (uint64_t)(sbo >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, fp16 A and B (the
// same type), both K-major, M = 128, the given N.
__host__ __device__ constexpr uint32_t idesc_of(int n)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kGM >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the
// tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 TMEM lanes x 32 consecutive 32-bit columns into 32 registers per lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

constexpr int kTK = 64;                  // inputs per operand slice: two blocks
// Decoder groups of four warps, taking slices round-robin.  A group's waits
// stay within one phase of each ring barrier only while the groups are no
// more than the ring's slots (checked per instantiation).
constexpr int kDecGroups = 3;
constexpr int kTThreads = 128 + 128 * kDecGroups;   // 4 role warps + the decoders
constexpr int kATileT = kGM * kTK * 2;   // fp16 weight tile of one slice (16 KB)
constexpr int kDecWarp0 = 4;             // warps 4.. decode, then read out

// Raw chunk of each format: BPC blocks (of BE weights, BS bytes) of each of
// the 128 rows per tensor copy (BPC * BS is a multiple of 16, so every chunk
// starts on a 16-byte boundary of a 16-byte aligned row), R chunks in
// flight; a chunk holds QPC 64-input slices.
template <int FMT> struct RawCfg;
template <> struct RawCfg<RF_Q4_0> { static constexpr int BS = 18, BE = 32, BPC = 8, R = 3; };
template <> struct RawCfg<RF_Q8_0> { static constexpr int BS = 34, BE = 32, BPC = 8, R = 2; };
template <> struct RawCfg<RF_MXFP4> { static constexpr int BS = 17, BE = 32, BPC = 16, R = 2; };
template <> struct RawCfg<RF_Q4_K> { static constexpr int BS = 144, BE = 256, BPC = 1, R = 3; };

// Slots of the operand ring (a decoded-weight tile and an activation tile
// each) for a token tile of N.  The decoder groups take the slices
// round-robin, so a ring of at least as many slots as groups keeps every
// parity wait within one phase of its barrier.
// DIRECT: the decoders read the raw rows themselves (no raw ring), so the
// operand ring can be deeper.
template <int N, bool DIRECT> __host__ __device__ constexpr int tc_stages()
{
    return DIRECT ? (N == 256 ? 4 : (N == 128 ? 6 : 8)) : (N == 256 ? 3 : (N == 128 ? 4 : 6));
}

// MMA issue threads.  One thread's chain per slice (barrier wait, fence,
// four MMAs, commit: about 750 cycles) exceeds the tensor work of a slice
// below N = 256, so where the ring allows, two threads take alternate slices
// into two accumulators that the epilogue adds.  Issuer i then owns the slots
// of parity i (an even ring), and each waits only on its own slots'
// barriers, in order.  The decoder groups, which no longer see one global
// consumption order, stay within one phase of a slot only with at least
// six slots: a group's fill of slice b - 6 needed slice b - 6 - S consumed,
// which by its issuer's order covers slice b - 2S when S >= 6.
template <int N, bool DIRECT> __host__ __device__ constexpr int tc_issuers()
{
    return tc_stages<N, DIRECT>() % 2 == 0 && tc_stages<N, DIRECT>() >= 6 ? 2 : 1;
}

template <int FMT, int N, bool DIRECT>
constexpr size_t tc_smem()
{
    using RC = RawCfg<FMT>;
    return (size_t)tc_stages<N, DIRECT>() * (kATileT + N * kTK * 2) +
           (DIRECT ? 0 : (size_t)RC::R * kGM * RC::BPC * RC::BS) + 16 +
           (size_t)(3 * tc_stages<N, DIRECT>() + 2 * RC::R + 3) * 8 + 16;
}

struct TcParams {
    CUtensorMap wmap;   // the window's rows as uint16 columns; boxes of one chunk x 128 rows
    const uint8_t *Wd;  // direct mode: row 0 of the window
    int64_t rb;         // direct mode: bytes per row
    const uint8_t *Xp;  // fp16 activation tiles: [token tile][slice][N x 64]
    float *Y;
    int64_t ldy;
    int32_t rows, n_tok, nst, nch;   // nst: 64-input slices; nch: raw chunks (slices if direct)
    int32_t ntt;                     // token tiles; tile index = token tile + ntt * row tile
    int32_t full_tiles;              // tiles [0, full_tiles) take one CTA each; the rest two,
    int32_t split_c;                 // chunks [0, split_c) and [split_c, nch), summed into Y
    int32_t withhold;                // test hook: CTA 0 never copies this slice's activations
    unsigned long long limit;
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    return (uint32_t)__half_as_ushort(__low2half(h)) | ((uint32_t)__half_as_ushort(__high2half(h)) << 16);
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Bytes [OFF, OFF + NB) of a 16-byte aligned row slot: the 16-byte units
// holding them, as words; word<P>, half<P> and byte<P> read at OFF + P.
template <int OFF, int NB>
struct RawWin {
    static constexpr int A = OFF & ~15;
    static constexpr int NU = (OFF + NB - 1 - A) / 16 + 1;
    uint32_t w[4 * NU];
    __device__ __forceinline__ void load(const uint8_t *slot)
    {
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const uint4 v = *reinterpret_cast<const uint4 *>(slot + A + 16 * u);
            w[4 * u] = v.x;
            w[4 * u + 1] = v.y;
            w[4 * u + 2] = v.z;
            w[4 * u + 3] = v.w;
        }
    }
    template <int P> __device__ __forceinline__ uint32_t word() const
    {
        constexpr int B = OFF - A + P;
        if constexpr (B % 4 == 0) return w[B / 4];
        else return __funnelshift_r(w[B / 4], w[B / 4 + 1], 8 * (B % 4));
    }
    template <int P> __device__ __forceinline__ uint32_t half() const
    {
        constexpr int B = OFF - A + P;
        static_assert(B % 2 == 0, "fp16 scale at an odd byte");
        return (w[B / 4] >> (8 * (B % 4))) & 0xFFFFu;
    }
    template <int P> __device__ __forceinline__ uint32_t byte() const
    {
        constexpr int B = OFF - A + P;
        return (w[B / 4] >> (8 * (B % 4))) & 0xFFu;
    }
};

// One block of 32 weights as 16 fp16 pairs (out[m] holds elements 2m and
// 2m+1).  Q4_0: element j < 16 is the low nibble of byte j, j + 16 its high
// nibble; 0x6400 | n is the fp16 value 1024 + n, so subtracting 1032 gives
// n - 8 exactly and one multiply by d rounds the weight once.
__device__ __forceinline__ void q4_0_pairs(uint32_t d, const uint32_t (&qs)[4], uint32_t *out)
{
    const uint32_t dd = d | (d << 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t t01 = prmt(qs[j], 0u, 0x4140u), t23 = prmt(qs[j], 0u, 0x4342u);
        out[2 * j] = hmul2(hsub2((t01 & 0x000F000Fu) | 0x64006400u, 0x64086408u), dd);
        out[2 * j + 1] = hmul2(hsub2((t23 & 0x000F000Fu) | 0x64006400u, 0x64086408u), dd);
        out[8 + 2 * j] = hmul2(hsub2(((t01 >> 4) & 0x000F000Fu) | 0x64006400u, 0x64086408u), dd);
        out[9 + 2 * j] = hmul2(hsub2(((t23 >> 4) & 0x000F000Fu) | 0x64006400u, 0x64086408u), dd);
    }
}
// Q8_0: byte j is element j (int8); with the sign bit flipped, 0x6400 | u is
// 1024 + q + 128, so subtracting 1152 gives q exactly.
__device__ __forceinline__ void q8_0_pairs(uint32_t d, const uint32_t (&qs)[8], uint32_t *out)
{
    const uint32_t dd = d | (d << 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t v = qs[j] ^ 0x80808080u;
        out[2 * j] = hmul2(hsub2(prmt(v, 0x64646464u, 0x5140u), 0x64806480u), dd);
        out[2 * j + 1] = hmul2(hsub2(prmt(v, 0x64646464u, 0x7362u), 0x64806480u), dd);
    }
}
// fp16 bits of 2^k: normal for k >= -14, subnormal down to 2^-24, 0 below,
// infinity above 2^15.
__device__ __forceinline__ uint32_t pow2_h(int k)
{
    if (k > 15) return 0x7C00u;
    if (k >= -14) return (uint32_t)(k + 15) << 10;
    if (k >= -24) return 1u << (k + 24);
    return 0u;
}
// Two E2M1 codes (the low 8 bits of `lo8`: low nibble, high nibble) as an
// fp16 pair (low half, high half), exactly.
__device__ __forceinline__ uint32_t e2m1x2_h2(uint32_t lo8)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(r)
        : "r"(lo8));
    return r;
}
// MXFP4: byte j holds element j (low nibble) and j + 16 (high nibble), as
// Q4_0.  Adjacent elements are paired into one byte (x | x >> 4 puts the
// nibbles of bytes 2i and 2i+1 together in byte 2i), converted exactly, and
// scaled by 2^(E-127): one exact multiply whenever the product is
// representable; outside fp16's exponent range the scale goes in two steps
// (2^15 then the rest, or 2^-12 then the rest), so the weight is rounded
// once.
__device__ __forceinline__ void mxfp4_pairs(uint32_t E, const uint32_t (&qs)[4], uint32_t *out)
{
    uint32_t s1, s2 = 0u;
    const int k = (int)E - 127;
    if (E == 255u) s1 = 0x7E00u;                       // NaN scale
    else if (k >= -24 && k <= 15) s1 = pow2_h(k);
    else if (k > 15) { s1 = 0x7800u; s2 = pow2_h(min(k - 15, 15)); }
    else { s1 = 0x0C00u; s2 = k + 12 >= -24 ? pow2_h(k + 12) : 0u; }
    const uint32_t ss = s1 | (s1 << 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = qs[j] & 0x0F0F0F0Fu, hi = (qs[j] >> 4) & 0x0F0F0F0Fu;
        const uint32_t pl = lo | (lo >> 4), ph = hi | (hi >> 4);
        out[2 * j] = hmul2(e2m1x2_h2(pl), ss);
        out[2 * j + 1] = hmul2(e2m1x2_h2(pl >> 16), ss);
        out[8 + 2 * j] = hmul2(e2m1x2_h2(ph), ss);
        out[9 + 2 * j] = hmul2(e2m1x2_h2(ph >> 16), ss);
    }
    if (E != 255u && (k < -24 || k > 15)) {
        const uint32_t s22 = s2 | (s2 << 16);
#pragma unroll
        for (int m = 0; m < 16; ++m) out[m] = hmul2(out[m], s22);
    }
}

// Q4_K slice Q of a 256-weight super-block (16-byte aligned in its slot):
// sub-blocks 2Q (low nibbles of quant bytes 32Q..32Q+31) and 2Q+1 (their high
// nibbles).  Scale and min of sub-block j are 6-bit fields of the 12 scale
// bytes: j < 4 the low 6 bits of bytes j and j+4; j >= 4 a nibble of byte j+4
// with the top two bits of bytes j-4 and j.  Each weight is d*sc*q - dmin*m
// by one fused multiply-add in fp32 (d*sc, dmin*m and d*sc*q are exact),
// then rounded to fp16.
template <int Q>
__device__ __forceinline__ void q4k_slice(const uint8_t *slot, uint32_t (&out)[32])
{
    const uint4 h = *reinterpret_cast<const uint4 *>(slot);
    const uint4 qa = *reinterpret_cast<const uint4 *>(slot + 16 + 32 * Q);
    const uint4 qb = *reinterpret_cast<const uint4 *>(slot + 32 + 32 * Q);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const uint32_t sw[3] = {h.y, h.z, h.w};   // the 12 scale bytes
    auto sb = [&](int i) -> uint32_t { return (sw[i >> 2] >> (8 * (i & 3))) & 0xFFu; };
    float ds[2], dm[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        constexpr int j0 = 2 * Q;
        const int j = j0 + t;
        uint32_t sc, m;
        if (j < 4) {
            sc = sb(j) & 63u;
            m = sb(j + 4) & 63u;
        } else {
            sc = (sb(j + 4) & 15u) | ((sb(j - 4) >> 6) << 4);
            m = (sb(j + 4) >> 4) | ((sb(j) >> 6) << 4);
        }
        ds[t] = d * (float)sc;
        dm[t] = dmin * (float)m;
    }
    const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    // 0x4B000000 | n is the fp32 value 2^23 + n, so subtracting 2^23 gives n.
    auto w = [](uint32_t nib, float s, float mm) {
        return fmaf(s, __uint_as_float(0x4B000000u | nib) - 8388608.f, -mm);
    };
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t v = qw[k];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t b0 = (v >> (16 * e)) & 0xFFu, b1 = (v >> (16 * e + 8)) & 0xFFu;
            out[2 * k + e] = h2_bits(__floats2half2_rn(w(b0 & 15u, ds[0], dm[0]), w(b1 & 15u, ds[0], dm[0])));
            out[16 + 2 * k + e] =
                h2_bits(__floats2half2_rn(w(b0 >> 4, ds[1], dm[1]), w(b1 >> 4, ds[1], dm[1])));
        }
    }
}

// One slice (two 32-weight blocks) as 32 fp16 pairs, from a window whose
// word<P>, half<P> and byte<P> read the slice's byte P.
template <int FMT, class Win>
__device__ __forceinline__ void decode_win(const Win &win, uint32_t (&out)[32])
{
    if constexpr (FMT == RF_Q4_0) {
        const uint32_t q0[4] = {win.template word<2>(), win.template word<6>(),
                                win.template word<10>(), win.template word<14>()};
        const uint32_t q1[4] = {win.template word<20>(), win.template word<24>(),
                                win.template word<28>(), win.template word<32>()};
        q4_0_pairs(win.template half<0>(), q0, out);
        q4_0_pairs(win.template half<18>(), q1, out + 16);
    } else if constexpr (FMT == RF_Q8_0) {
        const uint32_t q0[8] = {win.template word<2>(),  win.template word<6>(),
                                win.template word<10>(), win.template word<14>(),
                                win.template word<18>(), win.template word<22>(),
                                win.template word<26>(), win.template word<30>()};
        const uint32_t q1[8] = {win.template word<36>(), win.template word<40>(),
                                win.template word<44>(), win.template word<48>(),
                                win.template word<52>(), win.template word<56>(),
                                win.template word<60>(), win.template word<64>()};
        q8_0_pairs(win.template half<0>(), q0, out);
        q8_0_pairs(win.template half<34>(), q1, out + 16);
    } else {
        const uint32_t q0[4] = {win.template word<1>(), win.template word<5>(),
                                win.template word<9>(), win.template word<13>()};
        const uint32_t q1[4] = {win.template word<18>(), win.template word<22>(),
                                win.template word<26>(), win.template word<30>()};
        mxfp4_pairs(win.template byte<0>(), q0, out);
        mxfp4_pairs(win.template byte<17>(), q1, out + 16);
    }
}

// Slice Q of a raw chunk (blocks 2Q and 2Q+1 of one row, or a quarter of a
// Q4_K super-block) as 32 fp16 pairs.
template <int FMT, int Q>
__device__ __forceinline__ void decode_slice(const uint8_t *slot, uint32_t (&out)[32])
{
    if constexpr (FMT == RF_Q4_K) {
        q4k_slice<Q>(slot, out);
    } else {
        using RC = RawCfg<FMT>;
        RawWin<Q * 2 * RC::BS, 2 * RC::BS> win;
        win.load(slot);
        decode_win<FMT>(win, out);
    }
}

// A slice's NB bytes as words starting at its first byte (one word of
// slack for the funnel of the last unaligned read).
template <int NB>
struct SliceWin {
    uint32_t w[(NB + 3) / 4 + 1];
    template <int P> __device__ __forceinline__ uint32_t word() const
    {
        if constexpr (P % 4 == 0) return w[P / 4];
        else return __funnelshift_r(w[P / 4], w[P / 4 + 1], 8 * (P % 4));
    }
    template <int P> __device__ __forceinline__ uint32_t half() const
    {
        static_assert(P % 2 == 0, "fp16 scale at an odd byte");
        return (w[P / 4] >> (8 * (P % 4))) & 0xFFFFu;
    }
    template <int P> __device__ __forceinline__ uint32_t byte() const
    {
        return (w[P / 4] >> (8 * (P % 4))) & 0xFFu;
    }
};

// Rows whose byte length is not a multiple of 16 cannot be described by a
// tensor map, so their decoders read the raw bytes themselves: the aligned
// 4-byte words that hold a slice's nb bytes (never a word past the one
// holding its last byte; bytes past nb are cleared, so a final slice of one
// block decodes zeros for its second), read through the non-coherent path,
// then shifted by the slice's byte phase into a window that starts at it.
template <int FMT>
struct DirectSlice {
    static constexpr int NB = 2 * RawCfg<FMT>::BS;
    static constexpr int NW = (3 + NB + 3) / 4;   // words covering NB bytes at any phase
    uint32_t w[NW];
    uint32_t sh;
    __device__ __forceinline__ void load(const uint8_t *a, int nb)
    {
        const uintptr_t ua = reinterpret_cast<uintptr_t>(a);
        const uint32_t *a4 = reinterpret_cast<const uint32_t *>(ua & ~(uintptr_t)3);
        sh = 8u * (uint32_t)(ua & 3);
        const int end = (int)(ua & 3) + nb;   // bytes from the first word's start to the slice's end
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const int rem = end - 4 * j;      // bytes of word j that belong to the slice
            const uint32_t v = rem > 0 ? __ldg(a4 + j) : 0u;
            w[j] = rem >= 4 ? v : v & ((1u << (8 * (rem > 0 ? rem : 0))) - 1u);
        }
    }
    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int j = 0; j < NW; ++j) w[j] = 0u;
        sh = 0u;
    }
    // Slice b of a row of rb bytes at `row`: NB bytes, or one block at the
    // end of a row whose inputs are an odd number of blocks; zeros for a
    // row past the window.
    __device__ __forceinline__ void fetch(const uint8_t *row, int b, int64_t rb, bool row_ok)
    {
        const int64_t off = (int64_t)b * NB;
        if (row_ok) load(row + off, rb - off < NB ? (int)(rb - off) : NB);
        else zero();
    }
    __device__ __forceinline__ void to(SliceWin<NB> &win) const
    {
        constexpr int NO = (NB + 3) / 4 + 1;
        static_assert(NO <= NW, "window wider than the words read");
#pragma unroll
        for (int j = 0; j < NO; ++j)
            win.w[j] = __funnelshift_r(w[j], j + 1 < NW ? w[j + 1] : 0u, sh);
    }
};

// Compile-time loop over the slices of a chunk: f(integral_constant<Q>) for
// Q = Q0 .. QN-1 while it returns true.
template <int Q0, int QN>
struct SliceLoop {
    template <class F> __device__ __forceinline__ static bool run(F &f)
    {
        if (!f(std::integral_constant<int, Q0>())) return false;
        return SliceLoop<Q0 + 1, QN>::run(f);
    }
};
template <int QN>
struct SliceLoop<QN, QN> {
    template <class F> __device__ __forceinline__ static bool run(F &) { return true; }
};

template <int FMT, int N, bool DIRECT>
__global__ void __launch_bounds__(kTThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p)
{
    using RC = RawCfg<FMT>;
    constexpr int S = tc_stages<N, DIRECT>(), R = RC::R, CB = RC::BPC * RC::BS;
    // Slices per raw chunk; in direct mode every slice is its own "chunk"
    // (the unit of the last-wave K split).
    constexpr int QPC = DIRECT ? 1 : RC::BPC * RC::BE / kTK;
    constexpr int NI = tc_issuers<N, DIRECT>();
    constexpr uint32_t kCols = (uint32_t)(NI * N);   // accumulator i at columns [i*N, (i+1)*N)
    constexpr int BT = N * kTK * 2;   // fp16 activation tile of one slice
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *a_t = smem;                 // [S][16 KB]
    uint8_t *b_t = a_t + S * kATileT;    // [S][BT]
    uint8_t *raw = b_t + S * BT;         // [R][128 rows][CB] (none in direct mode)
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw + (DIRECT ? 0 : (size_t)R * kGM * CB) + 16);
    // full: the slot's weights decoded and its activations landed (one
    // arrival per decoder warp); bfull: the activation copy's bytes; empty:
    // the slot's MMAs done.
    uint64_t *full = bars, *bfull = bars + S, *empty = bars + 2 * S;
    uint64_t *rfull = bars + 3 * S, *rempty = rfull + R;
    uint64_t *accf = rempty + R, *mdone = accf + 1;   // mdone: one per issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 2);
    volatile int *stop = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // This CTA's tile and K range: a whole tile, or one half of a tile of
    // the last partial wave (split at a raw-chunk boundary; the two halves
    // add their sums into a zeroed Y, which is exact in order: a + b = b + a).
    int tile = (int)blockIdx.x, half = -1;
    if (tile >= p.full_tiles) {
        const int j = tile - p.full_tiles;
        tile = p.full_tiles + (j >> 1);
        half = j & 1;
    }
    const int tt = tile % p.ntt, rt = tile / p.ntt;
    const int c_lo = half == 1 ? p.split_c : 0;
    const int c_hi = half == 0 ? p.split_c : p.nch;
    const int b_lo = c_lo * QPC;
    const int b_hi = min(c_hi * QPC, p.nst);
    const int ni = b_hi - b_lo >= 2 ? NI : 1;   // issuers with slices (b_hi > b_lo always)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 4);
            mbar_init(&bfull[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&rfull[r], 1);
            mbar_init(&rempty[r], 4 * kDecGroups);
        }
        mbar_init(accf, (uint32_t)ni);
        mbar_init(&mdone[0], 1);
        mbar_init(&mdone[1], 1);
        *stop = 0;
        fence_barrier_init();
    }
    if (warp == 3) {
        tmem_alloc(tmem_slot, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*stop) return false;
        if (mbar_wait_bounded(bar, parity, &g_gemm_status, p.limit)) return true;
        *stop = 1;
        return false;
    };

    if (warp == 0) {
        // Raw rows: one 2-D tensor copy per chunk of 128 rows.
        if (!DIRECT && lane == 0) {
            int issued = 0;   // chunks c_lo .. c_lo + issued - 1; ring position = c - c_lo
            for (int c = c_lo; c < c_hi; ++c) {
                const int cl = c - c_lo, rs = cl % R;
                if (!wait(&rempty[rs], ((cl / R) & 1) ^ 1)) break;
                mbar_arrive_expect_tx(&rfull[rs], (uint32_t)(kGM * CB));
                tma_2d_g2s(raw + (size_t)rs * kGM * CB, &p.wmap, c * (CB / 2), rt * kGM, &rfull[rs]);
                ++issued;
            }
            for (int cl = max(0, issued - R); cl < issued; ++cl)
                mbar_drain(&rfull[cl % R], (cl / R) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // Activation tiles: one 1-D bulk copy per slice.
        if (lane == 0) {
            const uint8_t *xs = p.Xp + (size_t)tt * p.nst * BT;
            const int skip = blockIdx.x == 0 ? p.withhold : -1;
            int next = 0;   // local slices [0, next) have been issued (but `skip`)
            for (int b = b_lo; b < b_hi; ++b) {
                const int bl = b - b_lo, s = bl % S;
                if (!wait(&empty[s], ((bl / S) & 1) ^ 1)) break;
                next = bl + 1;
                if (b == skip) continue;
                mbar_arrive_expect_tx(&bfull[s], (uint32_t)BT);
                bulk_g2s(b_t + (size_t)s * BT, xs + (size_t)b * BT, (uint32_t)BT, &bfull[s]);
            }
            // Every copy issued lands before the CTA can exit.
            for (int bl = max(0, next - S); bl < next; ++bl)
                if (b_lo + bl != skip) mbar_drain(&bfull[bl % S], (bl / S) & 1);
        }
        __syncwarp();
    } else if (warp == 2 || (NI == 2 && warp == 3)) {
        // MMA issue: four K=16 steps per slice into issuer iss's
        // accumulator, slices iss, iss + NI, ...  The descriptors of slot 0
        // are built once; a slot and a K step move the start-address field
        // (address / 16, well inside its 14 bits).
        const int iss = warp - 2;
        if (lane == 0 && iss < ni) {
            int issued = 0;
            bool failed = false;
            const uint64_t ad0 = smem_desc(smem_addr(a_t), 1024);
            const uint64_t bd0 = smem_desc(smem_addr(b_t), 1024);
            const uint32_t acc = tmem + (uint32_t)(iss * N);
            int s = iss;   // NI divides S
            uint32_t ph = 0;
            for (int b = b_lo + iss; b < b_hi; b += NI) {
                if (!wait(&full[s], ph)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = ad0 + (uint64_t)((s * kATileT) >> 4);
                const uint64_t bd = bd0 + (uint64_t)((s * BT) >> 4);
                tc_mma(acc, ad, bd, idesc_of(N), b != b_lo + iss);
#pragma unroll
                for (int kk = 1; kk < kTK / 16; ++kk)
                    tc_mma(acc, ad + 16 * kk, bd + 16 * kk, idesc_of(N), 1u);
                tc_commit(&empty[s]);
                ++issued;
                if ((s += NI) >= S) {
                    s -= S;
                    ph ^= 1u;
                }
            }
            if (!failed) {
                tc_commit(accf);
            } else if (issued) {
                // Every issued MMA completes before tensor memory is freed.
                tc_commit(&mdone[iss]);
                mbar_drain(&mdone[iss], 0);
            }
        }
        __syncwarp();
    } else if (warp >= kDecWarp0) {
        // Decoders: warp group `grp` takes every kDecGroups-th slice; thread
        // i of a group owns row i of the tile (tensor-memory lane i).
        const int dw = warp - kDecWarp0;
        const int grp = dw >> 2;
        const int i = (dw & 3) * 32 + lane;
        // The decoded weight tile of slot s and this row, written in the
        // core-matrix layout, fenced to the async proxy; once the slot's
        // activation tile has landed too, one arrival per warp.
        auto publish = [&](int s, uint32_t ph, const uint32_t (&out)[32]) -> bool {
            uint8_t *at = a_t + (size_t)s * kATileT + (i >> 3) * 1024 + (i & 7) * 16;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4 *>(at + c8 * 128) =
                    make_uint4(out[4 * c8], out[4 * c8 + 1], out[4 * c8 + 2], out[4 * c8 + 3]);
            fence_async_smem();
            if (!__all_sync(0xffffffffu, wait(&bfull[s], ph))) return false;
            if (lane == 0) mbar_arrive(&full[s]);
            return true;
        };
        if constexpr (DIRECT) {
            // This group's slices b_lo + grp, + kDecGroups, ...; the raw
            // words of the next one are read before this one is decoded.
            constexpr int SB = 2 * RC::BS;   // bytes per slice
            const int64_t row = (int64_t)rt * kGM + i;
            const bool row_ok = row < p.rows;   // rows past the window decode zeros
            const uint8_t *rowp = p.Wd + (row_ok ? row : 0) * p.rb;
            DirectSlice<FMT> nxt;
            int bl = grp;
            if (b_lo + bl < b_hi) nxt.fetch(rowp, b_lo + bl, p.rb, row_ok);
            for (; b_lo + bl < b_hi; bl += kDecGroups) {
                const DirectSlice<FMT> cur = nxt;
                const int bn = b_lo + bl + kDecGroups;
                if (bn < b_hi) nxt.fetch(rowp, bn, p.rb, row_ok);
                const int s = bl % S;
                const uint32_t ph = (bl / S) & 1;
                if (!__all_sync(0xffffffffu, wait(&empty[s], ph ^ 1))) break;
                SliceWin<SB> win;
                cur.to(win);
                uint32_t out[32];
                decode_win<FMT>(win, out);
                if (!publish(s, ph, out)) break;
            }
        }
        bool ok = !DIRECT;
        for (int c = c_lo; c < c_hi && ok; ++c) {
            const int cl = c - c_lo, rs = cl % R;
            if (!__all_sync(0xffffffffu, wait(&rfull[rs], (cl / R) & 1))) break;
            const uint8_t *slot = raw + (size_t)rs * kGM * CB + (size_t)i * CB;
            auto one = [&](auto qc) -> bool {
                constexpr int Q = decltype(qc)::value;
                const int b = c * QPC + Q;
                if (b >= b_hi) return true;
                const int bl = b - b_lo;   // ring position of the slice
                if (bl % kDecGroups != grp) return true;
                const int s = bl % S;
                const uint32_t ph = (bl / S) & 1;
                if (!__all_sync(0xffffffffu, wait(&empty[s], ph ^ 1))) return false;
                uint32_t out[32];
                decode_slice<FMT, Q>(slot, out);
                return publish(s, ph, out);
            };
            ok = SliceLoop<0, QPC>::run(one);
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[rs]);
        }
        // Epilogue: the group's share of the accumulator columns (with two
        // issuers, the sum of both accumulators: one fp32 addition).
        if (__all_sync(0xffffffffu, wait(accf, 0))) {
            tc_fence_after();
            const int64_t row = (int64_t)rt * kGM + i;
            const bool row_ok = row < p.rows;
            const uint32_t tb = tmem + ((uint32_t)((dw & 3) * 32) << 16);
            const int tok0 = tt * N;
#pragma unroll 1
            for (int cc = grp * 32; cc < N; cc += 32 * kDecGroups) {
                uint32_t v[32];
                if constexpr (NI == 1) {
                    tmem_ld32(tb + (uint32_t)cc, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int h = 0; h < 32; h += 16) {
                        uint32_t a[16], c[16];
                        tmem_ld16(tb + (uint32_t)(cc + h), a);
                        if (ni == 2) tmem_ld16(tb + (uint32_t)(N + cc + h), c);
                        tmem_ld_wait();
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            v[h + n] = ni == 2 ? __float_as_uint(__uint_as_float(a[n]) + __uint_as_float(c[n]))
                                               : a[n];
                    }
                }
                if (row_ok) {
#pragma unroll
                    for (int n = 0; n < 32; ++n)
                        if (tok0 + cc + n < p.n_tok) {
                            float *y = p.Y + (int64_t)(tok0 + cc + n) * p.ldy + row;
                            if (half < 0) *y = __uint_as_float(v[n]);
                            else atomicAdd(y, __uint_as_float(v[n]));
                        }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 3) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

struct PrepParams {
    const float *X;
    int64_t ldx, in_dim, units;
    int n_tok, nst;
    uint8_t *Xp;
    int xb;              // blocks [0, xb) convert X, the rest zero Y
    float *Y;
    int64_t ldy;
    int rows, ntt, t0, ntiles;
};

// The pre-pass of a call, one launch:
//  * blocks [0, xb): X (fp32 rows ldx apart) -> fp16 tiles [token tile]
//    [slice][N x 64] in the K-major core-matrix layout: element (t, k) of a
//    tile at (t/8)*1024 + (k/8)*128 + (t%8)*16 + (k%8)*2; 16-byte unit u of
//    the whole buffer holds tokens and inputs such that the unit index within
//    a tile is (t/8)*64 + (k/8)*8 + t%8.  Tokens past n_tok and inputs past
//    in_dim are 0.
//  * the other blocks: Y = 0 over tiles [t0, t0 + ntiles) (tile = token tile
//    + ntt * row tile), whose two K halves are then added into it.
template <int N>
__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ PrepParams q)
{
    if ((int)blockIdx.x < q.xb) {
        for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < q.units;
             u += (int64_t)q.xb * blockDim.x) {
            const int64_t tile = u / (N * 8);
            const int w = (int)(u % (N * 8));
            const int t = (w >> 6) * 8 + (w & 7), c = (w >> 3) & 7;
            const int64_t tok = (tile / q.nst) * N + t;
            const int64_t k0 = (tile % q.nst) * kTK + c * 8;
            uint32_t h[4] = {0u, 0u, 0u, 0u};
            if (tok < q.n_tok && k0 < q.in_dim) {   // k0 + 8 <= in_dim (a multiple of 32)
                const float *x = q.X + tok * q.ldx + k0;
                float f[8];
                if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
                    const float4 a = reinterpret_cast<const float4 *>(x)[0];
                    const float4 b = reinterpret_cast<const float4 *>(x)[1];
                    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
                } else {
#pragma unroll
                    for (int m = 0; m < 8; ++m) f[m] = x[m];
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    h[m] = (uint32_t)__half_as_ushort(__float2half_rn(f[2 * m])) |
                           ((uint32_t)__half_as_ushort(__float2half_rn(f[2 * m + 1])) << 16);
            }
            *reinterpret_cast<uint4 *>(q.Xp + u * 16) = make_uint4(h[0], h[1], h[2], h[3]);
        }
    } else {
        const int64_t per = (int64_t)N * kGM;
        const int zb = (int)gridDim.x - q.xb;
        for (int64_t u = (int64_t)(blockIdx.x - q.xb) * blockDim.x + threadIdx.x;
             u < (int64_t)q.ntiles * per; u += (int64_t)zb * blockDim.x) {
            const int tile = q.t0 + (int)(u / per);
            const int w = (int)(u % per);
            const int tok = (tile % q.ntt) * N + w / kGM;
            const int row = (tile / q.ntt) * kGM + w % kGM;
            if (tok < q.n_tok && row < q.rows) q.Y[(int64_t)tok * q.ldy + row] = 0.f;
        }
    }
}

// Token tile of the main path for a chunk of n_tok tokens.
int tc_n(int n_tok) { return n_tok <= 64 ? 64 : (n_tok <= 128 ? 128 : 256); }

// Rows whose byte length is a multiple of 16 (always true for Q4_K's
// 144-byte super-blocks) are copied by tensor maps; others are read directly.
bool tc_rows_ok(int fmt, int64_t in_dim)
{
    return ((in_dim / block_elems_of(fmt)) * (int64_t)block_bytes_of(fmt)) % 16 == 0;
}

bool gemm_fmt_ok(int fmt)
{
    return fmt == RF_Q4_0 || fmt == RF_Q8_0 || fmt == RF_MXFP4 || fmt == RF_Q4_K;
}

size_t tc_workspace(int64_t in_dim, int n_tok)
{
    const int64_t N = tc_n(n_tok);
    const int64_t ntt = (n_tok + N - 1) / N, nst = (in_dim + kTK - 1) / kTK;
    return (size_t)(ntt * N) * (size_t)nst * kTK * 2;
}

template <int FMT, int N, bool DIRECT>
rf_status launch_tc_n(const TcParams &p, const float *X, int64_t ldx, int64_t in_dim,
                      uint8_t *Xp, dim3 grid, cudaStream_t s)
{
    static_assert(tc_smem<FMT, N, DIRECT>() <= 232448, "rings exceed the 227 KB of shared memory");
    static_assert(kDecGroups <= tc_stages<N, DIRECT>(), "more decoder groups than ring slots");
    static std::once_flag once[64];
    static bool ok[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    std::call_once(once[dev & 63], [dev] {
        ok[dev & 63] = cudaFuncSetAttribute(gemm_tc_kernel<FMT, N, DIRECT>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)tc_smem<FMT, N, DIRECT>()) == cudaSuccess;
        cudaGetLastError();
    });
    if (!ok[dev & 63]) return RF_ERR_CUDA;
    PrepParams q;
    q.X = X;
    q.ldx = ldx;
    q.in_dim = in_dim;
    q.units = (int64_t)p.ntt * N * p.nst * 8;
    q.n_tok = p.n_tok;
    q.nst = p.nst;
    q.Xp = Xp;
    q.Y = p.Y;
    q.ldy = p.ldy;
    q.rows = p.rows;
    q.ntt = p.ntt;
    q.t0 = p.full_tiles;
    q.ntiles = ((int)grid.x - p.full_tiles) / 2;   // CTAs past the whole tiles, two per split tile
    const int64_t cap = (int64_t)num_sms() * 8;
    q.xb = (int)std::min<int64_t>((q.units + 255) / 256, cap);
    const int zb = q.ntiles > 0 ? (int)std::min<int64_t>(((int64_t)q.ntiles * N * kGM + 255) / 256, cap) : 0;
    prep_kernel<N><<<q.xb + zb, 256, 0, s>>>(q);
    if (last_cuda_error() != RF_OK) return RF_ERR_CUDA;
    gemm_tc_kernel<FMT, N, DIRECT><<<grid, kTThreads, tc_smem<FMT, N, DIRECT>(), s>>>(p);
    return last_cuda_error();
}

template <int FMT, bool DIRECT>
rf_status launch_tc(const TcParams &p, const float *X, int64_t ldx, int64_t in_dim, uint8_t *Xp,
                    dim3 grid, cudaStream_t s)
{
    switch (tc_n(p.n_tok)) {
    case 64: return launch_tc_n<FMT, 64, DIRECT>(p, X, ldx, in_dim, Xp, grid, s);
    case 128: return launch_tc_n<FMT, 128, DIRECT>(p, X, ldx, in_dim, Xp, grid, s);
    default: return launch_tc_n<FMT, 256, DIRECT>(p, X, ldx, in_dim, Xp, grid, s);
    }
}

}  // namespace

rf_status read_and_clear_gemm_status()
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int)) != cudaSuccess)
            return RF_ERR_CUDA;
    }
    return static_cast<rf_status>(v);
}

}  // namespace rf

using namespace rf;

extern "C" {

size_t rf_gemm_workspace_bytes(int fmt, int64_t in_dim, int n_tok)
{
    if (!gemm_fmt_ok(fmt) || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || n_tok <= 0)
        return 0;
    return tc_workspace(in_dim, n_tok);
}

rf_status rf_gemm(int fmt, const void *W, int64_t row_start, int64_t row_end, int64_t in_dim,
                  int n_tok, const float *X, int64_t ldx, float *Y, int64_t ldy, void *workspace,
                  size_t workspace_bytes, void *stream)
{
    if (!gemm_fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!W || !X || !Y || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || row_start < 0 ||
        row_end < row_start || n_tok < 0 || ldx < in_dim || ldy < row_end - row_start)
        return RF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return RF_ERR_MISALIGNED;
    const int N = tc_n(n_tok);
    const int64_t ntt = (n_tok + N - 1) / N, nrt = (row_end - row_start + kGM - 1) / kGM;
    if (in_dim / 32 > 0x7fffffffLL || row_end - row_start > 0x7fffffffLL || ntt * nrt > 0x3fffffffLL)
        return RF_ERR_TOO_LARGE;
    const size_t need = n_tok > 0 ? tc_workspace(in_dim, n_tok) : 0;
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return RF_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return RF_ERR_MISALIGNED;
    }
    if (row_end == row_start || n_tok == 0) return RF_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t rb = (in_dim / block_elems_of(fmt)) * (int64_t)block_bytes_of(fmt);
    const bool direct = !tc_rows_ok(fmt, in_dim);
    TcParams p;
    std::memset(&p, 0, sizeof(p));
    const int cb = fmt == RF_Q4_0 || fmt == RF_Q4_K ? 144 : 272;   // chunk bytes (tensor maps)
    const uint8_t *W0 = static_cast<const uint8_t *>(W) + row_start * rb;
    if (!direct && !encode_u16_map(&p.wmap, W0, (uint64_t)(rb / 2), (uint64_t)(row_end - row_start),
                                   (uint64_t)rb, (uint32_t)(cb / 2), (uint32_t)kGM))
        return RF_ERR_CUDA;
    p.Wd = W0;
    p.rb = rb;
    p.Xp = static_cast<const uint8_t *>(workspace);
    p.Y = Y;
    p.ldy = ldy;
    p.rows = (int32_t)(row_end - row_start);
    p.n_tok = n_tok;
    p.nst = (int32_t)((in_dim + kTK - 1) / kTK);
    // The unit of the K split: a raw chunk, or a slice when rows are read directly.
    p.nch = direct ? p.nst : (int32_t)((rb + cb - 1) / cb);
    p.limit = 2000000000ull;
    p.withhold = -1;
    if (const unsigned long long lim = take_wait_fault()) {
        p.limit = lim;
        p.withhold = p.nst > 1 ? 1 : 0;
    }
    p.ntt = (int32_t)ntt;
    const int64_t tiles = ntt * nrt;
    // A last partial wave of at most half the SMs is split in K, so that it
    // takes half a tile's time instead of a whole one (with fewer tiles than
    // SMs, every tile).
    const int sms = num_sms();
    const int64_t last = tiles % sms;
    p.full_tiles = (int32_t)tiles;
    p.split_c = p.nch / 2;
    if (last > 0 && 2 * last <= sms && p.nch >= 2) p.full_tiles = (int32_t)(tiles - last);
    const dim3 grid((unsigned)(p.full_tiles + 2 * (tiles - p.full_tiles)));
    uint8_t *Xp = static_cast<uint8_t *>(workspace);
    if (direct) {
        switch (fmt) {   // Q4_K rows are always aligned
        case RF_Q4_0: return launch_tc<RF_Q4_0, true>(p, X, ldx, in_dim, Xp, grid, s);
        case RF_Q8_0: return launch_tc<RF_Q8_0, true>(p, X, ldx, in_dim, Xp, grid, s);
        case RF_MXFP4: return launch_tc<RF_MXFP4, true>(p, X, ldx, in_dim, Xp, grid, s);
        default: return RF_ERR_UNSUPPORTED_FMT;
        }
    }
    switch (fmt) {
    case RF_Q4_0: return launch_tc<RF_Q4_0, false>(p, X, ldx, in_dim, Xp, grid, s);
    case RF_Q8_0: return launch_tc<RF_Q8_0, false>(p, X, ldx, in_dim, Xp, grid, s);
    case RF_Q4_K: return launch_tc<RF_Q4_K, false>(p, X, ldx, in_dim, Xp, grid, s);
    default: return launch_tc<RF_MXFP4, false>(p, X, ldx, in_dim, Xp, grid, s);
    }
}

}  // extern "C"
