/*
 * rf_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously-correct CPU implementation of what the row-window
 * dequant-GEMV path computes.  Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference leg may load it.  It shares no code,
 * header, table or constant with the CUDA library: everything here is written
 * out from the format and algorithm definitions on the source pages.
 *
 * Sources (page title, section):
 *   [RF-M5]  RAMforge, "Milestone 5 - Native Quantized Tensor Support":
 *            Q4_0 = 32 elements in 18 B (2 B half scale d, 16 B of 4-bit quants,
 *            value d*(q-8)); Q8_0 = 32 elements in 34 B (2 B half scale d,
 *            32 int8 quants, value d*q).
 *   [RF-M6]  RAMforge, "Milestone 6 - True Out-of-Core Integrity", matrix
 *            layout: shape [in,out], buffer row-major [out][in],
 *            y[o] = sum_i W[o*in+i] * x[i].
 *   [NS-IDEA] neurostream, "The idea": rows are output neurons, a row is a
 *            whole number of quantization blocks; blocks shrink so that
 *            lookahead+1 raw buffers fit the arena; an expert e owns rows
 *            [e*out,(e+1)*out) of the stacked tensor; a 2,880-row MXFP4
 *            expert is 4.41 MB and streams 128 rows at a time at 0.39 MB.
 *   [NS-HOW] neurostream, "How it works" (2. routing, 4. stream_linear,
 *            6. arena) and the two-phase FFN paragraph.
 *   [NS-BUGS] neurostream, "Bugs worth knowing about": the pipeline holds
 *            depth+1 blocks, not depth.
 *   [RF-M5K] RAMforge, "Milestone 5 - Native Quantized Tensor Support": Q4_K =
 *            256 elements in 144 B: 2 B half d, 2 B half dmin, 12 B of scales
 *            (8 scales and 8 mins packed as 6-bit values), 128 B of 4-bit
 *            quants; an element is d*sc*q - dmin*m with (sc, m) its
 *            sub-block's scale and min.
 *   [NS-OSS] neurostream, "GPT-OSS-120B": GPT-OSS adds biased projections and
 *            experts and a clamped SwiGLU (no constants printed).
 *   [RF-M5Q6] RAMforge, "Milestone 5 - Native Quantized Tensor Support" (and
 *            its legacy tensor list): Q6_K is one of the K-quant block
 *            layouts; neurostream, "Supported" models list: Q6_K decoded
 *            bit-exact against the reference GGUF implementation.  Neither
 *            page prints the layout.
 *
 * Readings where the pages are silent:
 *   - fp16 scale: IEEE-754 binary16, little endian, first two bytes.
 *   - Q4_0 nibble order: element j (j<16) is the low nibble of quant byte j,
 *     element j+16 is its high nibble (the GGUF convention).
 *   - MXFP4 block (17 B, no page prints its layout): byte 0 is an E8M0 scale
 *     exponent E (scale 2^(E-127)), bytes 1..16 hold 32 FP4 E2M1 codes in the
 *     same nibble order as Q4_0.  E2M1 code bits are s e1 e0 m with exponent
 *     bias 1.  PARITY UNPINNED by the pages (only the 17-byte size is pinned,
 *     through the 4.41 MB figure); pinned here by the OCP MX definition.
 *   - Q4_K (the pages name the unpacking get_scale_min_k4 but print neither
 *     it nor the quant order; reading: the GGML layout).  Sub-block j (32
 *     elements, j = 0..7) has a 6-bit scale and a 6-bit min.  For j < 4 they
 *     are the low 6 bits of scale bytes j and j+4; for j >= 4 the scale is
 *     the low nibble of byte j+4 plus the top two bits of byte j-4 (as bits
 *     4-5), and the min is the high nibble of byte j+4 plus the top two bits
 *     of byte j (as bits 4-5).  Quant byte 32*i + l holds element 64*i + l in
 *     its low nibble (sub-block 2i) and element 64*i + 32 + l in its high
 *     nibble (sub-block 2i+1).  The value d*sc*q - dmin*m is computed
 *     exactly (fp64) and rounded once to float.  PARITY UNPINNED by the pages
 *     for the scale packing and the quant order (the 144-byte size and the
 *     formula are theirs); pinned here by a reduction to Q4_0.
 *   - GEMV accumulation: fp64, index order.
 *   - Router: the k largest fp32 logits, ties to the lower expert index,
 *     weights = softmax over the k selected logits.
 *   - SwiGLU: silu(g)*u with silu(z) = z/(1+exp(-z)); GELU (erf form) for the
 *     host-streamed dense FFN, whose activation no page states: PARITY
 *     UNPINNED by the pages (pinned by the GELU identities).
 *   - Q6_K (the GGML layout; PARITY UNPINNED by the pages, which name the
 *     format only): 256 elements in 210 B -- 128 B of low 4-bit quant parts
 *     (ql), 64 B of high 2-bit parts (qh), 16 signed 8-bit scales, then an
 *     fp16 d.  Element e = 128*n + 32*k + l (half n, quarter k, lane l < 32)
 *     has q = low | high << 4 with low the low nibble (k = 0, 1) or high
 *     nibble (k = 2, 3) of ql[64*n + l + 32*(k & 1)] and high = bits
 *     2k..2k+1 of qh[32*n + l]; its value is d * scale[e / 16] * (q - 32).
 *     Every such value needs at most 24 significant bits (11 + 8 + 6 bits),
 *     so it is exact in float.  Pinned in tests by hand-worked bytes and by
 *     a reduction to Q8_0.
 *
 *   - Biased experts with the clamped SwiGLU ([NS-OSS]; PARITY UNPINNED by
 *     the pages, which print no formula or constant).  Reading, from the
 *     public GPT-OSS reference release (its model code's swiglu and MoE
 *     block): per expert, g = G x + b_g, u = U x + b_u, then
 *     g' = min(g, limit), u' = max(-limit, min(u, limit)),
 *     h = g' * sigmoid(alpha * g') * (u' + 1), and the expert's output is
 *     D h + b_d; the combine is sum_k w_k (D_k h_k + b_d,k).  The release's
 *     constants are alpha = 1.702 and limit = 7.0; both are arguments here.
 *     Pinned in tests by a reduction to the plain SwiGLU MoE (alpha = 1,
 *     limit = +inf, b_u = -1, other biases 0), by bias-only closed forms and
 *     by the clamp making the output independent of weights it cuts off.
 *
 * Floating point: all arithmetic in double; dequantized weights are returned
 * as float (every value d*q, d*(q-8) and e2m1*2^k is exactly representable).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q4_0 2
#define ORC_Q8_0 8
#define ORC_MXFP4 39
#define ORC_Q4_K 12
#define ORC_Q6_K 14

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2
#define ORC_EARENA 3

/* ---------------------------------------------------------------- scalars */

/* IEEE-754 binary16 -> double, decoded field by field. */
double orc_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);          /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* E8M0 scale exponent -> 2^(E-127); 0xFF is NaN in the format. */
double orc_e8m0_to_double(uint8_t E)
{
    if (E == 255)
        return NAN;
    return ldexp(1.0, (int)E - 127);
}

/* FP4 E2M1 code (low 4 bits) -> value.  Bits: s e1 e0 m, exponent bias 1,
 * e == 0 is subnormal (0 or 0.5). */
double orc_e2m1_to_double(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* ------------------------------------------------------------ block sizes */

int64_t orc_block_bytes(int fmt)
{
    switch (fmt) {
    case ORC_Q8_0: return 34;   /* [RF-M5] */
    case ORC_Q4_0: return 18;   /* [RF-M5] */
    case ORC_MXFP4: return 17;  /* 1 scale byte + 16 code bytes */
    case ORC_Q4_K: return 144;  /* [RF-M5K] */
    case ORC_Q6_K: return 210;  /* 128 + 64 + 16 + 2, the Q6_K reading */
    default: return 0;
    }
}

/* Elements per block: 32, or 256 for the K-quant super-blocks. */
int64_t orc_block_elems(int fmt)
{
    if (fmt == ORC_Q4_K || fmt == ORC_Q6_K)
        return 256;
    return orc_block_bytes(fmt) ? 32 : 0;
}

/* Q6_K element e's 6-bit quant (0..63) from the ql and qh parts. */
int orc_q6k_quant(const uint8_t *blk, int e)
{
    int n = e / 128, k = (e % 128) / 32, l = e % 32;
    int lowbyte = blk[64 * n + l + 32 * (k & 1)];
    int low = k < 2 ? (lowbyte & 15) : (lowbyte >> 4);
    int high = (blk[128 + 32 * n + l] >> (2 * k)) & 3;
    return low | (high << 4);
}

int64_t orc_row_bytes(int fmt, int64_t in_dim)
{
    int64_t bb = orc_block_bytes(fmt), be = orc_block_elems(fmt);
    if (bb == 0 || in_dim <= 0 || in_dim % be != 0)
        return 0;
    return (in_dim / be) * bb;
}

/* Q4_K sub-block j's 6-bit scale and min from the 12 scale bytes. */
void orc_q4k_scale_min(const uint8_t *sc12, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = sc12[j] & 63;
        *m = sc12[j + 4] & 63;
    } else {
        *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        *m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

/* ------------------------------------------------------- block dequantize */

/* Decode one block into out[0..elems-1] (float; Q8_0, Q4_0 and MXFP4 values
 * are exact, Q4_K values are the exact value rounded once). */
int orc_dequant_block(int fmt, const uint8_t *blk, float *out)
{
    int j;
    if (fmt == ORC_Q4_K) {
        double d = orc_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        double dmin = orc_fp16_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
        const uint8_t *sc12 = blk + 4, *qs = blk + 16;
        int i, l;
        for (i = 0; i < 4; i++) {
            int sc0, m0, sc1, m1;
            orc_q4k_scale_min(sc12, 2 * i, &sc0, &m0);
            orc_q4k_scale_min(sc12, 2 * i + 1, &sc1, &m1);
            for (l = 0; l < 32; l++) {
                int lo = qs[32 * i + l] & 15, hi = qs[32 * i + l] >> 4;
                out[64 * i + l] = (float)(d * sc0 * lo - dmin * m0);
                out[64 * i + 32 + l] = (float)(d * sc1 * hi - dmin * m1);
            }
        }
        return ORC_OK;
    }
    if (fmt == ORC_Q6_K) {
        double d = orc_fp16_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
        const int8_t *scale = (const int8_t *)(blk + 192);
        for (j = 0; j < 256; j++)
            out[j] = (float)(d * (double)scale[j / 16] * (double)(orc_q6k_quant(blk, j) - 32));
        return ORC_OK;
    }
    if (fmt == ORC_Q8_0) {
        double d = orc_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        for (j = 0; j < 32; j++) {
            int q = (int)(int8_t)blk[2 + j];
            out[j] = (float)(d * (double)q);
        }
        return ORC_OK;
    }
    if (fmt == ORC_Q4_0) {
        double d = orc_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        for (j = 0; j < 16; j++) {
            int lo = blk[2 + j] & 15;
            int hi = blk[2 + j] >> 4;
            out[j] = (float)(d * (double)(lo - 8));
            out[j + 16] = (float)(d * (double)(hi - 8));
        }
        return ORC_OK;
    }
    if (fmt == ORC_MXFP4) {
        double scale = orc_e8m0_to_double(blk[0]);
        for (j = 0; j < 16; j++) {
            uint8_t lo = blk[1 + j] & 15;
            uint8_t hi = blk[1 + j] >> 4;
            out[j] = (float)(orc_e2m1_to_double(lo) * scale);
            out[j + 16] = (float)(orc_e2m1_to_double(hi) * scale);
        }
        return ORC_OK;
    }
    return ORC_EINVAL;
}

/* Dequantize n_blocks consecutive blocks into out[32*n_blocks]. */
int orc_dequantize(int fmt, const uint8_t *W, int64_t n_blocks, float *out)
{
    int64_t bb = orc_block_bytes(fmt), be = orc_block_elems(fmt), b;
    if (bb == 0 || n_blocks < 0)
        return ORC_EINVAL;
    for (b = 0; b < n_blocks; b++) {
        int rc = orc_dequant_block(fmt, W + b * bb, out + be * b);
        if (rc)
            return rc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------- GEMV */

/* y[r - row_start] = sum_i w[r,i] * x[i] for r in [row_start, row_end),
 * with W the [out][in] row-major raw matrix starting at row 0 ([RF-M6]).
 * Accumulated in double in index order; x given in double. */
int orc_gemv_d(int fmt, const uint8_t *W, int64_t row_start, int64_t row_end,
               int64_t in_dim, const double *x, double *y)
{
    int64_t rb = orc_row_bytes(fmt, in_dim), bb = orc_block_bytes(fmt);
    int64_t be = orc_block_elems(fmt);
    int64_t r, b, nb = be ? in_dim / be : 0;
    float w[256];
    int j;
    if (rb == 0 || row_start < 0 || row_end < row_start)
        return ORC_EINVAL;
    for (r = row_start; r < row_end; r++) {
        const uint8_t *row = W + r * rb;
        double acc = 0.0;
        for (b = 0; b < nb; b++) {
            orc_dequant_block(fmt, row + b * bb, w);
            for (j = 0; j < be; j++)
                acc += (double)w[j] * x[b * be + j];
        }
        y[r - row_start] = acc;
    }
    return ORC_OK;
}

/* Same, with the fp32 activation vector every caller of the GPU path has. */
int orc_gemv(int fmt, const uint8_t *W, int64_t row_start, int64_t row_end,
             int64_t in_dim, const float *x, double *y)
{
    int64_t i;
    int rc;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(in_dim > 0 ? in_dim : 1));
    if (!xd)
        return ORC_ENOMEM;
    for (i = 0; i < in_dim; i++)
        xd[i] = (double)x[i];
    rc = orc_gemv_d(fmt, W, row_start, row_end, in_dim, xd, y);
    free(xd);
    return rc;
}

/* Euclidean norm of each dequantized row (used by the parity tolerance). */
int orc_row_norms(int fmt, const uint8_t *W, int64_t row_start, int64_t row_end,
                  int64_t in_dim, double *norms)
{
    int64_t rb = orc_row_bytes(fmt, in_dim), bb = orc_block_bytes(fmt);
    int64_t be = orc_block_elems(fmt);
    int64_t r, b, nb = be ? in_dim / be : 0;
    float w[256];
    int j;
    if (rb == 0 || row_start < 0 || row_end < row_start)
        return ORC_EINVAL;
    for (r = row_start; r < row_end; r++) {
        double s = 0.0;
        for (b = 0; b < nb; b++) {
            orc_dequant_block(fmt, W + r * rb + b * bb, w);
            for (j = 0; j < be; j++)
                s += (double)w[j] * (double)w[j];
        }
        norms[r - row_start] = sqrt(s);
    }
    return ORC_OK;
}

/* --------------------------------------------------- streaming emulation */

/* Block planning ([NS-IDEA], [NS-BUGS]): a window of n_rows rows is walked in
 * blocks of block_rows rows (0 = the whole window); a block shrinks until
 * depth+1 raw buffers fit the arena.  Returns the effective rows per block or
 * a negative value when even a one-row block does not fit. */
int64_t orc_plan_block_rows(int64_t row_bytes, int64_t n_rows, int64_t block_rows,
                            int depth, int64_t arena_bytes)
{
    int64_t want, fit;
    if (row_bytes <= 0 || n_rows < 0 || block_rows < 0 || depth < 0 || arena_bytes < 0)
        return -1;
    want = (block_rows == 0 || block_rows > n_rows) ? n_rows : block_rows;
    if (want < 1)
        want = 1;
    fit = arena_bytes / ((int64_t)(depth + 1) * row_bytes);
    if (fit < 1)
        return -1;
    return want < fit ? want : fit;
}

/* stream_linear ([NS-HOW] 4 and 6): walk [row_start,row_end) of a matrix held
 * in slow memory.  Keep up to depth blocks reserved ahead of the one being
 * multiplied; each reservation holds its bytes in an arena ring of depth+1
 * slots until its output exists.  Every block's bytes are copied into its
 * slot and multiplied from there.  *peak_bytes receives the largest number of
 * arena bytes reserved at once. */
int orc_stream_linear(int fmt, const uint8_t *W, int64_t row_start, int64_t row_end,
                      int64_t in_dim, int64_t block_rows, int depth, int64_t arena_bytes,
                      const float *x, double *y, int64_t *eff_rows, int64_t *n_blocks,
                      int64_t *peak_bytes)
{
    int64_t rb = orc_row_bytes(fmt, in_dim);
    int64_t n_rows = row_end - row_start, br, nblk, slot_bytes;
    int64_t next_fetch = 0, i, reserved = 0, peak = 0;
    int64_t *slot_of = NULL, *bytes_of = NULL;
    uint8_t *arena = NULL;
    int rc = ORC_OK;

    if (rb == 0 || row_start < 0 || n_rows < 0 || depth < 0)
        return ORC_EINVAL;
    br = orc_plan_block_rows(rb, n_rows, block_rows, depth, arena_bytes);
    if (br < 0)
        return ORC_EARENA;
    nblk = n_rows == 0 ? 0 : (n_rows + br - 1) / br;
    slot_bytes = br * rb;
    arena = (uint8_t *)malloc((size_t)(slot_bytes * (depth + 1) + 1));
    slot_of = (int64_t *)calloc((size_t)(nblk + 1), sizeof(int64_t));
    bytes_of = (int64_t *)calloc((size_t)(nblk + 1), sizeof(int64_t));
    if (!arena || !slot_of || !bytes_of) {
        rc = ORC_ENOMEM;
        goto out;
    }
    for (i = 0; i < nblk; i++) {
        int64_t r0, r1;
        /* Fetch ahead: blocks i .. i+depth are reserved while block i is
         * multiplied (the multiplied block still owns its lease). */
        while (next_fetch < nblk && next_fetch <= i + depth) {
            int64_t f0 = row_start + next_fetch * br;
            int64_t f1 = f0 + br < row_end ? f0 + br : row_end;
            slot_of[next_fetch] = next_fetch % (depth + 1);
            bytes_of[next_fetch] = (f1 - f0) * rb;
            memcpy(arena + slot_of[next_fetch] * slot_bytes, W + f0 * rb,
                   (size_t)bytes_of[next_fetch]);
            reserved += bytes_of[next_fetch];
            if (reserved > peak)
                peak = reserved;
            next_fetch++;
        }
        r0 = row_start + i * br;
        r1 = r0 + br < row_end ? r0 + br : row_end;
        /* Multiply the block from its arena slot: rows r0..r1 sit at the
         * start of the slot, so the slot is a matrix of (r1-r0) rows. */
        rc = orc_gemv(fmt, arena + slot_of[i] * slot_bytes, 0, r1 - r0, in_dim, x,
                      y + (r0 - row_start));
        if (rc)
            goto out;
        reserved -= bytes_of[i];   /* retire: release the lease */
    }
    if (eff_rows)
        *eff_rows = br;
    if (n_blocks)
        *n_blocks = nblk;
    if (peak_bytes)
        *peak_bytes = peak;
out:
    free(arena);
    free(slot_of);
    free(bytes_of);
    return rc;
}

/* ------------------------------------------------------------ activations */

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

double orc_gelu(double z) { return 0.5 * z * (1.0 + erf(z / sqrt(2.0))); }

/* Clamped SwiGLU of the biased experts ([NS-OSS] reading above). */
double orc_swiglu_clamped(double g, double u, double alpha, double limit)
{
    double gc = g < limit ? g : limit;
    double uc = u < -limit ? -limit : (u > limit ? limit : u);
    return gc / (1.0 + exp(-alpha * gc)) * (uc + 1.0);
}

/* ----------------------------------------------------------------- router */

/* [NS-HOW] 2: the router names the k active experts.  Pick the k largest
 * logits (ties to the lower index) in descending order, then weight them by a
 * softmax over the selected logits.  The pages say nothing of NaN logits: a
 * NaN counts as -infinity, for the ranking and for the weights. */
static double router_value(float v) { return isnan(v) ? -INFINITY : (double)v; }

int orc_router_topk(const float *logits, int n_expert, int top_k, int *idx, double *w)
{
    int k, e;
    char *taken;
    double m, s = 0.0;
    if (n_expert <= 0 || top_k <= 0 || top_k > n_expert)
        return ORC_EINVAL;
    taken = (char *)calloc((size_t)n_expert, 1);
    if (!taken)
        return ORC_ENOMEM;
    for (k = 0; k < top_k; k++) {
        int best = -1;
        for (e = 0; e < n_expert; e++) {
            if (taken[e])
                continue;
            if (best < 0 || router_value(logits[e]) > router_value(logits[best]))
                best = e;   /* strict '>' keeps the lower index on ties */
        }
        taken[best] = 1;
        idx[k] = best;
    }
    free(taken);
    m = router_value(logits[idx[0]]);
    for (k = 0; k < top_k; k++) {
        w[k] = exp(router_value(logits[idx[k]]) - m);
        s += w[k];
    }
    for (k = 0; k < top_k; k++)
        w[k] /= s;
    return ORC_OK;
}

/* -------------------------------------------------------------- FFN / MoE */

/* Two-phase SwiGLU FFN ([NS-HOW], FFN paragraph): walk gate and up by neuron
 * to get h = silu(gate.x) * (up.x), then walk down by output dimension.
 * gate/up are [n_ff][n_embd] starting at row g0/u0, down is [n_embd][n_ff]
 * starting at row d0.  h_out (n_ff doubles, may be NULL) receives h. */
int orc_ffn_swiglu(int fmt, const uint8_t *gate, int64_t g0, const uint8_t *up, int64_t u0,
                   const uint8_t *down, int64_t d0, int64_t n_ff, int64_t n_embd,
                   const float *x, double *y, double *h_out)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)n_ff);
    double *u = (double *)malloc(sizeof(double) * (size_t)n_ff);
    int64_t i;
    int rc = ORC_ENOMEM;
    if (!g || !u)
        goto out;
    rc = orc_gemv(fmt, gate, g0, g0 + n_ff, n_embd, x, g);
    if (!rc)
        rc = orc_gemv(fmt, up, u0, u0 + n_ff, n_embd, x, u);
    if (rc)
        goto out;
    for (i = 0; i < n_ff; i++)
        g[i] = orc_silu(g[i]) * u[i];
    if (h_out)
        memcpy(h_out, g, sizeof(double) * (size_t)n_ff);
    rc = orc_gemv_d(fmt, down, d0, d0 + n_embd, n_ff, g, y);
out:
    free(g);
    free(u);
    return rc;
}

/* MoE FFN over stacked (n_expert, out, in) tensors ([NS-IDEA], [NS-HOW] 2-4):
 * route, then for each selected expert (in selection order) run the
 * two-phase SwiGLU FFN on its row windows, and sum the outputs weighted by
 * the router weights.  gate/up are (n_expert, n_ff, n_embd), down is
 * (n_expert, n_embd, n_ff).  idx/w receive the routing (top_k entries). */
int orc_moe_ffn(int fmt, const float *logits, int n_expert, int top_k,
                const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                int64_t n_ff, int64_t n_embd, const float *x, double *y,
                int *idx, double *w)
{
    double *yk = (double *)malloc(sizeof(double) * (size_t)n_embd);
    int k, rc;
    int64_t r;
    if (!yk)
        return ORC_ENOMEM;
    rc = orc_router_topk(logits, n_expert, top_k, idx, w);
    if (rc)
        goto out;
    for (r = 0; r < n_embd; r++)
        y[r] = 0.0;
    for (k = 0; k < top_k; k++) {
        int64_t e = idx[k];
        rc = orc_ffn_swiglu(fmt, gate, e * n_ff, up, e * n_ff, down, e * n_embd, n_ff,
                            n_embd, x, yk, NULL);
        if (rc)
            goto out;
        for (r = 0; r < n_embd; r++)
            y[r] += w[k] * yk[r];
    }
out:
    free(yk);
    return rc;
}

/* Routed MoE over biased experts with the clamped SwiGLU ([NS-OSS] reading
 * above; [NS-IDEA], [NS-HOW] 2-4 for the routing and row windows).  gate/up
 * are (n_expert, n_ff, n_embd), down is (n_expert, n_embd, n_ff); gate_bias
 * and up_bias are (n_expert, n_ff) and down_bias (n_expert, n_embd) doubles,
 * any of them NULL for zero.  y = sum_k w_k (D_k h_k + b_d,k) in selection
 * order; idx/w receive the routing; h_out (top_k * n_ff, may be NULL)
 * receives each selected expert's h. */
int orc_moe_ffn_biased(int fmt, const float *logits, int n_expert, int top_k,
                       const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                       const double *gate_bias, const double *up_bias,
                       const double *down_bias, double alpha, double limit,
                       int64_t n_ff, int64_t n_embd, const float *x, double *y,
                       int *idx, double *w, double *h_out)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)n_ff);
    double *u = (double *)malloc(sizeof(double) * (size_t)n_ff);
    double *yk = (double *)malloc(sizeof(double) * (size_t)n_embd);
    int k, rc = ORC_ENOMEM;
    int64_t i, r;
    if (!g || !u || !yk)
        goto out;
    rc = orc_router_topk(logits, n_expert, top_k, idx, w);
    if (rc)
        goto out;
    for (r = 0; r < n_embd; r++)
        y[r] = 0.0;
    for (k = 0; k < top_k; k++) {
        int64_t e = idx[k];
        rc = orc_gemv(fmt, gate, e * n_ff, (e + 1) * n_ff, n_embd, x, g);
        if (!rc)
            rc = orc_gemv(fmt, up, e * n_ff, (e + 1) * n_ff, n_embd, x, u);
        if (rc)
            goto out;
        for (i = 0; i < n_ff; i++) {
            double gb = g[i] + (gate_bias ? gate_bias[e * n_ff + i] : 0.0);
            double ub = u[i] + (up_bias ? up_bias[e * n_ff + i] : 0.0);
            g[i] = orc_swiglu_clamped(gb, ub, alpha, limit);
        }
        if (h_out)
            memcpy(h_out + (int64_t)k * n_ff, g, sizeof(double) * (size_t)n_ff);
        rc = orc_gemv_d(fmt, down, e * n_embd, (e + 1) * n_embd, n_ff, g, yk);
        if (rc)
            goto out;
        for (r = 0; r < n_embd; r++)
            y[r] += w[k] * (yk[r] + (down_bias ? down_bias[e * n_embd + r] : 0.0));
    }
out:
    free(g);
    free(u);
    free(yk);
    return rc;
}
