/*
 * rf.h -- C ABI of the row-window dequant-GEMV library for GB300 (sm_103a).
 *
 * Batch-1 decode multiplies quantized weights straight from their raw
 * GGUF-style block bytes, one row window of output neurons at a time.  A
 * weight matrix is row-major [out][in] (RAMforge, "Milestone 6 - True
 * Out-of-Core Integrity", matrix layout: y[o] = sum_i W[o*in+i] * x[i]); a row
 * is a whole number of 32-element blocks (neurostream, "The idea").
 *
 * Conventions for every call:
 *   - W, x, y, logits, workspace and out are CUDA device pointers unless the
 *     name says host.  All buffers belong to the caller; the library keeps no
 *     pointer past the call except inside an rf_arena it created.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     stream ordered and return after enqueueing.  These calls block the host
 *     on GPU work, and no others do:
 *       rf_device_status        (synchronizes the device),
 *       rf_arena_destroy        (waits for the arena's copies and readers),
 *       rf_arena_wait           (waits, up to its deadline, for the same),
 *       rf_expert_cache_destroy (waits for the cache's copies and readers),
 *       rf_moe_ffn_streamed     (waits for its routing result: the host plan
 *                                needs the expert ids).
 *   - Argument errors are detected on the host before anything is enqueued;
 *     the call then returns an error and enqueues nothing.  Launch errors
 *     return RF_ERR_CUDA.  Kernels never trap: a kernel whose internal wait
 *     exceeds its time limit records RF_ERR_TIMEOUT in a device status word
 *     that rf_device_status reports, issues no further copies, waits for the
 *     ones it issued and ends.  The word is sticky: while it is set, every
 *     bounded wait of later kernels ends at once (their outputs are
 *     undefined), until rf_device_status reads and clears it.
 *   - Weight pointers must be 16-byte aligned.  A kernel may read whole
 *     16-byte aligned chunks that contain bytes of the rows it was given (so
 *     up to 15 bytes before the first and after the last row byte, never in
 *     another 16-byte chunk); it never writes weight memory.
 *   - There is no CPU fallback: without a CUDA device every compute call
 *     returns RF_ERR_CUDA.
 */
#ifndef RF_H
#define RF_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RF_API __attribute__((visibility("default")))
#else
#define RF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- formats */
/* Block formats, numbered like the GGML type ids.
 *   RF_Q4_0 : 18 B per 32 weights: fp16 scale d, then 16 bytes of 4-bit q;
 *             w = d*(q-8) (RAMforge, "Milestone 5 - Native Quantized Tensor
 *             Support").  Element j<16 is the low nibble of quant byte j and
 *             element j+16 its high nibble.
 *   RF_Q8_0 : 34 B per 32 weights: fp16 scale d, then 32 int8 q; w = d*q
 *             (same section).
 *   RF_MXFP4: 17 B per 32 weights: E8M0 scale byte E, then 16 bytes of FP4
 *             E2M1 codes in the Q4_0 nibble order; w = e2m1(c) * 2^(E-127)
 *             (named by neurostream, "The idea"; layout per the OCP MX
 *             definition, which the pages do not print).
 *   RF_Q4_K : 144 B per 256 weights (a super-block of eight 32-weight
 *             sub-blocks): fp16 d, fp16 dmin, 12 bytes of 6-bit scales and
 *             mins, 128 bytes of 4-bit q; w = d*sc*q - dmin*m with (sc, m)
 *             the sub-block's scale and min (RAMforge, "Milestone 5 - Native
 *             Quantized Tensor Support").  The unpacking and quant order
 *             follow the GGML layout (the page names but does not print
 *             them): sub-block j < 4 takes the low 6 bits of scale bytes j
 *             and j+4; j >= 4 the low/high nibble of byte j+4 plus the top
 *             two bits of bytes j-4 / j; quant byte 32i+l holds weight 64i+l
 *             (low nibble) and 64i+32+l (high nibble).  in_dim must be a
 *             multiple of 256 for this format.
 *   RF_Q6_K : 210 B per 256 weights: 128 bytes of low 4-bit quant parts (ql),
 *             64 bytes of high 2-bit parts (qh), 16 signed 8-bit scales (one
 *             per 16 weights), fp16 d last; w = d*scale*(q-32).  RAMforge
 *             ("Milestone 5 - Native Quantized Tensor Support") lists the
 *             format and neurostream's model list decodes it, but neither
 *             prints the layout; it follows the GGML layout: weight
 *             128n+32k+l takes the low (k < 2) or high (k >= 2) nibble of ql
 *             byte 64n+32(k&1)+l and bit pair 2k of qh byte 32n+l as its top
 *             two bits.  Every value is exact in fp32.  in_dim must be a
 *             multiple of 256; rows never take tensor copies (210-byte
 *             super-blocks), so they are staged whole or copied per lane. */
#define RF_Q4_0 2
#define RF_Q8_0 8
#define RF_MXFP4 39
#define RF_Q4_K 12
#define RF_Q6_K 14

typedef enum rf_status {
    RF_OK = 0,
    RF_ERR_INVALID_ARG = 1,     /* null pointer, bad size, in_dim not a whole number of blocks, ... */
    RF_ERR_UNSUPPORTED_FMT = 2, /* fmt is not one of RF_Q4_0, RF_Q8_0, RF_MXFP4, RF_Q4_K, RF_Q6_K */
    RF_ERR_NOT_PINNED = 3,      /* a host weight pointer is not page-locked */
    RF_ERR_ARENA_TOO_SMALL = 4, /* depth+1 one-row blocks do not fit the arena */
    RF_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed */
    RF_ERR_TIMEOUT = 6,         /* a device wait exceeded its limit */
    RF_ERR_OOM = 7,             /* device or host allocation failed */
    RF_ERR_MISALIGNED = 8,      /* a weight pointer is not 16-byte aligned */
    RF_ERR_TOO_LARGE = 9        /* a size exceeds a documented kernel limit */
} rf_status;

/* Human-readable name of a status code (static string, never NULL). */
RF_API const char *rf_status_str(int status);

/* Library ABI version (major*10000 + minor*100 + patch). */
RF_API int rf_version(void);

/* Bytes per block: 18 (Q4_0), 34 (Q8_0), 17 (MXFP4) per 32 weights, 144 (Q4_K)
 * and 210 (Q6_K) per 256 weights; 0 if unknown. */
RF_API size_t rf_block_bytes(int fmt);

/* Bytes per row of in_dim weights (in_dim/32 blocks, in_dim/256 for Q4_K and
 * Q6_K); 0
 * if fmt is unknown or in_dim is not a positive whole number of blocks. */
RF_API size_t rf_row_bytes(int fmt, int64_t in_dim);

/* Largest in_dim the GEMV kernels accept for `fmt` with `n_x` distinct
 * activation vectors in one launch (their fixed-point digits are kept in
 * shared memory); 0 without a CUDA device. */
RF_API int64_t rf_max_in_dim(int fmt, int n_x);

/* ------------------------------------------------------------- dequantize */
/* Decode n_blocks consecutive blocks at W (device) into out (device,
 * 32*n_blocks floats, 256*n_blocks for Q4_K and Q6_K).  Q8_0, Q4_0, MXFP4
 * and Q6_K values are exactly representable in fp32; a Q4_K value is the
 * exact d*sc*q - dmin*m rounded once; so the result is bit-exact against
 * that definition.  Errors: RF_ERR_UNSUPPORTED_FMT,
 * RF_ERR_INVALID_ARG (null pointer, n_blocks < 0). */
RF_API rf_status rf_dequantize(int fmt, const void *W, int64_t n_blocks, float *out,
                               void *stream);

/* ------------------------------------------------------------------- GEMV */
/* Fused dequant-GEMV over one row window (neurostream, "How it works" 4-5:
 * stream_linear walks [row_start,row_end) and the fused kernel multiplies
 * straight from the quantized bytes):
 *     y[r - row_start] = sum_i w[r,i] * x[i]   for r in [row_start, row_end)
 * W   : device, 16-byte aligned, row 0 of a row-major matrix of
 *       rf_row_bytes(fmt,in_dim)-byte rows; only the window's rows are read.
 * x   : device, in_dim floats.   y : device, row_end-row_start floats.
 * The result of a row depends only on that row and x, never on the window,
 * so any split of a matrix into windows gives bit-identical outputs.
 * Errors: RF_ERR_UNSUPPORTED_FMT; RF_ERR_INVALID_ARG (null pointer,
 * in_dim % 32 != 0, row_start < 0, row_end < row_start); RF_ERR_MISALIGNED;
 * RF_ERR_TOO_LARGE (in_dim > rf_max_in_dim(fmt,1)).  An empty window is a
 * no-op. */
RF_API rf_status rf_gemv(int fmt, const void *W, int64_t row_start, int64_t row_end,
                         int64_t in_dim, const float *x, float *y, void *stream);

/* One row window for rf_gemv_batch (all device pointers). */
typedef struct rf_window {
    const void *W;      /* row 0 of the matrix (16-byte aligned) */
    int64_t row_start;  /* first row of the window */
    int64_t row_end;    /* one past the last row */
    const float *x;     /* in_dim floats */
    float *y;           /* row_end-row_start floats */
} rf_window;

/* Several row windows of matrices with the same fmt and in_dim in ONE kernel
 * launch (e.g. the Q, K and V projections of a decode step).  `windows` is a
 * host array; at most 8 distinct x pointers per call.  Each window's output is
 * bit-identical to rf_gemv on it.  Errors as rf_gemv, plus RF_ERR_TOO_LARGE
 * for more than 64 windows or 8 distinct x. */
RF_API rf_status rf_gemv_batch(int fmt, int64_t in_dim, int n_windows,
                               const rf_window *windows, void *stream);

/* Launch flags for the *_ex variants.
 * RF_CHAIN: no kernel still pending on `stream` writes the weights of this call
 *   (weights are static during inference).  The launch may then start before
 *   the previous kernel on the stream finishes and copy its weights while that
 *   kernel drains (programmatic dependent launch); it still waits for that
 *   kernel before reading x.  Copies and memsets are never overtaken.  Without
 *   the flag a launch starts only after the previous work completes. */
#define RF_CHAIN 1u

/* rf_gemv / rf_gemv_batch with launch flags (RF_CHAIN); otherwise identical,
 * including bit-identical results. */
RF_API rf_status rf_gemv_ex(int fmt, const void *W, int64_t row_start, int64_t row_end,
                            int64_t in_dim, const float *x, float *y, unsigned flags,
                            void *stream);
RF_API rf_status rf_gemv_batch_ex(int fmt, int64_t in_dim, int n_windows,
                                  const rf_window *windows, unsigned flags, void *stream);

/* ------------------------------------------------------------ activations */
/* h[i] = silu(g[i]) * u[i], silu(z) = z/(1+exp(-z)) (RAMforge, "Milestone 3";
 * the SwiGLU between gate/up and down).  Device pointers, n >= 0. */
RF_API rf_status rf_swiglu(const float *g, const float *u, float *h, int64_t n, void *stream);

/* h[i] = 0.5*z[i]*(1+erf(z[i]/sqrt(2))) (erf form of GELU).  Device. */
RF_API rf_status rf_gelu(const float *z, float *h, int64_t n, void *stream);

/* --------------------------------------------------------- dense SwiGLU FFN */
/* Two-phase FFN (neurostream, "How it works", FFN paragraph): walk gate and up
 * by neuron to get h = silu(gate.x) * (up.x) (one launch, SwiGLU fused into
 * its epilogue), then walk down by output dimension (one launch).
 * gate, up: [n_ff][n_embd]; down: [n_embd][n_ff]; x: n_embd; y: n_embd;
 * h: n_ff floats of caller memory that receives the activations.
 * All device.  Errors as rf_gemv. */
RF_API rf_status rf_ffn_swiglu(int fmt, const void *gate, const void *up, const void *down,
                               int64_t n_ff, int64_t n_embd, const float *x, float *y,
                               float *h, void *stream);

/* rf_ffn_swiglu with launch flags: RF_CHAIN applies to its first launch (the
 * second one is always chained to the first). */
RF_API rf_status rf_ffn_swiglu_ex(int fmt, const void *gate, const void *up, const void *down,
                                  int64_t n_ff, int64_t n_embd, const float *x, float *y,
                                  float *h, unsigned flags, void *stream);

/* Bytes of workspace rf_ffn_swiglu_ws takes for n_ff activations (80 bytes
 * per 32); 0 if n_ff is not a positive multiple of 32. */
RF_API size_t rf_ffn_workspace_bytes(int64_t n_ff);

/* rf_ffn_swiglu_ex with a device workspace of rf_ffn_workspace_bytes(n_ff)
 * bytes (16-byte aligned; NULL = none): the first launch also writes the
 * fixed-point digits of h that the second launch multiplies by, so the down
 * projection copies them instead of rebuilding them from h.  Results are
 * bit-identical to rf_ffn_swiglu_ex.  The workspace is overwritten. */
RF_API rf_status rf_ffn_swiglu_ws(int fmt, const void *gate, const void *up, const void *down,
                                  int64_t n_ff, int64_t n_embd, const float *x, float *y,
                                  float *h, void *workspace, unsigned flags, void *stream);

/* Several tokens through one row window (a decode batch, or a small prefill
 * chunk): Y[t][r - row_start] = sum_i W[r,i] * X[t][i] for t < n_tok, all in
 * ONE launch that walks the window's rows once (neurostream, "What the
 * numbers taught us": tokens that share one pass over the weights cost
 * little more than one).  The rows are copied to shared memory once per
 * token from L2, so HBM sees each weight byte about once per call.  Every
 * token's row is bit-identical to rf_gemv on that token alone.
 * X: n_tok rows of in_dim floats, ldx floats apart; Y: n_tok rows of
 * row_end-row_start floats, ldy floats apart.  All device.  flags as
 * rf_gemv_ex.  Errors: as rf_gemv; RF_ERR_TOO_LARGE for n_tok > 8;
 * RF_ERR_INVALID_ARG for n_tok < 1, ldx < in_dim or ldy < rows. */
RF_API rf_status rf_gemv_multi(int fmt, const void *W, int64_t row_start, int64_t row_end,
                               int64_t in_dim, int n_tok, const float *X, int64_t ldx, float *Y,
                               int64_t ldy, unsigned flags, void *stream);

/* Prefill dequant-GEMM on the tensor cores (neurostream, "What the numbers
 * taught us": a prompt or an image prefills through one pass over the
 * weights for the whole chunk of tokens):
 *     Y[t][r - row_start] = sum_i W[r,i] * X[t][i],  r in [row_start, row_end),
 *                                                    t < n_tok.
 * Formats: RF_Q4_0, RF_Q8_0, RF_MXFP4, RF_Q4_K (others:
 * RF_ERR_UNSUPPORTED_FMT; for one to eight tokens rf_gemv_multi serves every
 * format).  X is first rounded to fp16 into `workspace`, each weight is
 * decoded to fp16 as d * q with one rounding (MXFP4 values are exact;
 * Q4_K's d*sc*q - dmin*m is rounded to fp32, then to fp16), and
 * tcgen05.mma accumulates the whole row in fp32.  Rows whose byte length is
 * a multiple of 16 (in_dim a multiple of 256 for Q4_0/Q8_0, of 512 for
 * MXFP4, any Q4_K width) are staged by tensor copies; other rows are read
 * by the decoding threads directly, with the same arithmetic.  |X| and |w|
 * must stay below 65504.
 * W: device, row 0 of the [out][in] matrix, 16-byte aligned; X: n_tok rows
 * of in_dim floats, ldx floats apart; Y: n_tok rows, ldy floats apart;
 * workspace: device, 16-byte aligned, at least
 * rf_gemm_workspace_bytes(fmt, in_dim, n_tok) bytes (may be NULL when
 * n_tok is 0),
 * owned by the caller and overwritten; it must not be used by another call
 * that is in flight.  All device.  Errors: RF_ERR_INVALID_ARG (null
 * pointer, in_dim not a positive multiple of the format's block (32, or
 * 256 for Q4_K), bad window, n_tok < 0, ldx < in_dim, ldy < rows,
 * workspace missing or too small);
 * RF_ERR_MISALIGNED (W or workspace not 16-byte aligned); RF_ERR_TOO_LARGE
 * (more than 2^31 - 1 rows, or ceil(rows / 128) * ceil(n_tok / T) above
 * 2^30 - 1, T the token tile: 64 up to 64 tokens, 128 up to 128, else 256).
 * Empty work is a no-op.
 * A bounded internal wait that gives up is reported by rf_device_status as
 * RF_ERR_TIMEOUT. */
RF_API rf_status rf_gemm(int fmt, const void *W, int64_t row_start, int64_t row_end,
                         int64_t in_dim, int n_tok, const float *X, int64_t ldx, float *Y,
                         int64_t ldy, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace rf_gemm needs for (fmt, in_dim, n_tok): the fp16
 * activation tiles, T * ceil(n_tok / T) tokens x ceil(in_dim / 64) * 64
 * inputs x 2 bytes (T as above); 0 when the arguments are invalid. */
RF_API size_t rf_gemm_workspace_bytes(int fmt, int64_t in_dim, int n_tok);

/* Zero-copy variant of rf_gemv (hipfire PR #793, "Summary": the "pcie"
 * execution of a spilled layer, where the GPU kernels read host-mapped
 * weights over the link; "Design notes": the host memory is allocated mapped
 * and the device pointer is its host-mapped alias): the kernel reads the rows
 * straight from page-locked host memory over the link, with no arena and no
 * copy engine.  host_W: page-locked, device-mapped host
 * pointer to row 0 of the [out][in] matrix (16-byte aligned); x, y: device.
 * Output is bit-identical to rf_gemv on the same bytes.
 * Errors: as rf_gemv; RF_ERR_NOT_PINNED if host_W is not page-locked and
 * mapped. */
RF_API rf_status rf_gemv_host(int fmt, const void *host_W, int64_t row_start, int64_t row_end,
                              int64_t in_dim, const float *x, float *y, void *stream);

/* ------------------------------------------- host-streamed row windows */
/* An arena is a bounded ring of device memory plus a copy stream and events
 * (neurostream, "How it works" 6: each block in flight takes arena space,
 * and a fetch that finds none free waits for a block to be given back).
 * rf_arena_create allocates `bytes` (plus a little alignment slack) of
 * device memory on the chosen device.  An arena is used by one host thread
 * at a time. */
typedef struct rf_arena rf_arena;
/* device: the CUDA device the arena lives on, or -1 for the current one.  The
 * arena's memory, copy stream and events belong to that device; every call
 * that uses the arena must be made with it current (else
 * RF_ERR_INVALID_ARG).  Errors: RF_ERR_INVALID_ARG (bytes == 0, out NULL,
 * no such device), RF_ERR_OOM, RF_ERR_CUDA. */
RF_API rf_status rf_arena_create(size_t bytes, int device, rf_arena **out);
/* Waits for the arena's outstanding eager copies and readers, then frees it
 * (launches of graphs captured with it must have finished).  NULL is a
 * no-op. */
RF_API void rf_arena_destroy(rf_arena *arena);

/* Arena options (rf_arena_configure), each on by default:
 *   RF_ARENA_MERGE_RUNS -- a walk whose blocks all fit the ring at once goes
 *                          over the link as one copy and through one launch
 *                          (each block still its own window; results are
 *                          bit-identical either way).  Off: one copy and one
 *                          launch per block, the per-block pipeline.
 *   RF_ARENA_LANES      -- walks of 8 or more blocks of at most 1 MiB run
 *                          their GEMVs round-robin on the arena's four lane
 *                          streams.  Off: every GEMV on the caller's stream.
 * value 0 turns an option off, 1 on.  Errors: RF_ERR_INVALID_ARG (NULL
 * arena, unknown option, value not 0 or 1). */
#define RF_ARENA_MERGE_RUNS 1
#define RF_ARENA_LANES 2
RF_API rf_status rf_arena_configure(rf_arena *arena, int option, int value);

/* Host wait with a deadline: blocks until every copy the arena has enqueued
 * and every launch that read one of its slots (eager use) has finished, or
 * until timeout_ms milliseconds have passed (neurostream, "Bugs worth
 * knowing about": a prefetcher that can stall must not stall its caller for
 * ever).  Returns RF_OK, RF_ERR_TIMEOUT (work still outstanding; call again
 * to keep waiting), RF_ERR_CUDA (the device reported an error) or
 * RF_ERR_INVALID_ARG (NULL arena, timeout_ms < 0, the arena's device is not
 * current, or a capture is using the arena's streams). */
RF_API rf_status rf_arena_wait(rf_arena *arena, int timeout_ms);

/* Host-side failure injection for tests (the pages have no counterpart; it
 * lets the failure path be exercised without faulting a GPU).  Arms a
 * one-shot fault for the next rf_stream_linear walk on the arena, at the
 * walk's block `block` (0-based):
 *   RF_FAULT_COPY_FAIL  -- that block's copy reports a failure, as a failed
 *                          cudaMemcpyAsync would: the walk stops enqueueing,
 *                          the blocks already enqueued keep their order on
 *                          the caller's stream (lane streams are joined
 *                          back), every slot stays reusable, and the call
 *                          returns RF_ERR_CUDA;
 *   RF_FAULT_COPY_STALL -- the copy stream stalls for `ms` milliseconds on
 *                          the host before that block's copy (a slow link);
 *                          the walk itself succeeds.
 * An armed fault also turns off the one-copy path for walks that fit the
 * ring, so the fault lands on a real per-block copy.  RF_FAULT_NONE
 * disarms.  Errors: RF_ERR_INVALID_ARG (NULL arena, unknown kind, block < 0,
 * ms outside 0..10000). */
#define RF_FAULT_NONE 0
#define RF_FAULT_COPY_FAIL 1
#define RF_FAULT_COPY_STALL 2
RF_API rf_status rf_arena_inject_fault(rf_arena *arena, int kind, int64_t block, int ms);

/* Host-side block plan for walking n_rows rows of rf_row_bytes(fmt,in_dim)
 * bytes in blocks of block_rows rows (0 = the whole window) with `depth`
 * blocks in flight: blocks shrink until depth+1 of them fit arena_bytes
 * (neurostream, "The idea"; "Bugs worth knowing about": the pipeline holds
 * depth+1 blocks).  Outputs (each may be NULL) the effective rows per block,
 * the block count and the peak arena bytes.  RF_ERR_ARENA_TOO_SMALL if one
 * row per block does not fit; never touches a GPU. */
RF_API rf_status rf_stream_plan(int fmt, int64_t in_dim, int64_t n_rows, int64_t block_rows,
                                int depth, size_t arena_bytes, int64_t *eff_rows,
                                int64_t *n_blocks, size_t *peak_bytes);

/* stream_linear over weights held in page-locked host memory (neurostream,
 * "How it works" 3-4 and 6): for each planned block of rows in
 * [row_start,row_end), copy its raw bytes host->arena slot on the arena's copy
 * stream, then run the fused GEMV on that slot in `stream`; a slot is reused
 * only after the GEMV that read it has finished, so at most `depth` copies
 * run ahead of the multiply and depth+1 slots are held.  The host never
 * blocks.  host_W: page-locked host pointer to row 0 of the [out][in] matrix
 * (16-byte aligned); x, y: device.  Output is bit-identical to rf_gemv on the
 * same rows for every block_rows and depth.
 * The call may be made while `stream` is being captured into a CUDA graph:
 * the copies and GEMVs become graph nodes with the same dependencies, and
 * later captured calls on the same arena keep prefetching across call
 * boundaries.  The first call after a switch between eager use and a capture
 * (or between two captures) is ordered after all work already on `stream`;
 * a graph must be launched on the stream it was captured from (or after the
 * arena's earlier work has finished), and one capture at a time may use an
 * arena.
 * Errors: as rf_gemv; RF_ERR_NOT_PINNED if host_W is not page-locked;
 * RF_ERR_ARENA_TOO_SMALL; RF_ERR_INVALID_ARG for depth < 0 or depth > 64. */
RF_API rf_status rf_stream_linear(int fmt, const void *host_W, int64_t in_dim,
                                  int64_t row_start, int64_t row_end, int64_t block_rows,
                                  int depth, rf_arena *arena, const float *x, float *y,
                                  void *stream);

/* Counters of an arena (each one is exercised by a test). */
typedef struct rf_stream_stats_t {
    uint64_t calls;          /* rf_stream_linear calls enqueued */
    uint64_t blocks;         /* blocks copied and multiplied */
    uint64_t bytes_copied;   /* host->device bytes enqueued */
    uint64_t peak_bytes;     /* largest arena bytes reserved at once (planned) */
    uint64_t slot_bytes;     /* bytes per slot in the last call */
    uint64_t arena_bytes;    /* arena capacity */
    int32_t slots;           /* slots (depth+1) in the last call */
    int32_t last_block_rows; /* effective rows per block in the last call */
} rf_stream_stats_t;
/* Copies the arena's counters to *out.  Errors: RF_ERR_INVALID_ARG (NULL). */
RF_API rf_status rf_stream_stats(const rf_arena *arena, rf_stream_stats_t *out);

/* ------------------------------------------------------------------- MoE */
/* Device top-k router (neurostream, "How it works" 2: the router names the
 * active experts and only those are read): idx[k] = the k-th largest logit's
 * expert (ties to the lower index), w[k] = softmax over the selected logits.
 * A NaN logit counts as -inf (the pages leave NaN undefined), so the k
 * indices are always distinct experts in [0, n_expert).  The routed FFNs
 * below rank their logits the same way.
 * logits: device n_expert floats; idx: device top_k int32; w: device top_k
 * floats.  1 <= top_k <= min(n_expert, 8), n_expert <= 1024. */
RF_API rf_status rf_moe_route(const float *logits, int n_expert, int top_k, int32_t *idx,
                              float *w, void *stream);

/* Bytes of caller scratch rf_moe_ffn needs (routing result, activations and
 * their fixed-point digits); 0 if top_k is out of range or n_ff is not a
 * positive multiple of 32. */
RF_API size_t rf_moe_workspace_bytes(int top_k, int64_t n_ff, int64_t n_embd,
                                     int64_t block_rows);

/* Routed MoE SwiGLU FFN over stacked expert tensors (neurostream, "The idea"
 * and "How it works" 2-5): route on device, then walk each selected expert's
 * row windows [e*out + j*block_rows, ...) of gate and up in ONE launch (SwiGLU
 * in the epilogue), then the down windows of all selected experts in ONE
 * launch that also forms y = sum_k w_k * down_k(h_k) in selection order.
 * No host synchronisation.  gate, up: (n_expert, n_ff, n_embd);
 * down: (n_expert, n_embd, n_ff); router_logits: n_expert floats; x, y:
 * n_embd floats; workspace: rf_moe_workspace_bytes(...) bytes, 256-byte
 * aligned.  All device.  block_rows 0 = whole expert.  Errors as rf_gemv and
 * rf_moe_route. */
RF_API rf_status rf_moe_ffn(int fmt, const float *router_logits, int n_expert, int top_k,
                            const void *gate, const void *up, const void *down, int64_t n_ff,
                            int64_t n_embd, int64_t block_rows, const float *x, float *y,
                            void *workspace, void *stream);

/* rf_moe_ffn over stacked expert tensors held in page-locked, device-mapped
 * host memory (neurostream, "How it works" 2: only the routed experts' rows
 * are read; hipfire PR #793, "Summary": GPU kernels reading host-mapped
 * weights over the link).  The kernels read the selected experts' rows in
 * place over the host link; routing never leaves the device, so no host
 * round trip decides what to read.  Results are bit-identical to rf_moe_ffn
 * on the same bytes.  Errors: as rf_moe_ffn; RF_ERR_NOT_PINNED if a tensor is
 * not page-locked and mapped. */
RF_API rf_status rf_moe_ffn_host(int fmt, const float *router_logits, int n_expert, int top_k,
                                 const void *host_gate, const void *host_up,
                                 const void *host_down, int64_t n_ff, int64_t n_embd,
                                 int64_t block_rows, const float *x, float *y, void *workspace,
                                 void *stream);

/* Routed FFN over biased experts with the clamped SwiGLU (neurostream,
 * "GPT-OSS-120B": GPT-OSS adds biased projections and experts and a clamped
 * SwiGLU; the page prints no formula, so the form follows the public GPT-OSS
 * reference release): for each selected expert e (weight w_k),
 *     g = G_e x + gate_bias[e],  u = U_e x + up_bias[e],
 *     g' = min(g, limit),  u' = min(max(u, -limit), limit),
 *     h = g' * sigmoid(alpha * g') * (u' + 1),
 *     y = sum_k w_k * (D_e h + down_bias[e])      (selection order).
 * The release uses alpha = 1.702 and limit = 7.  Routing, layouts, launches
 * (two: gate/up with this epilogue, then down) and the workspace are those
 * of rf_moe_ffn; with alpha = 1, limit = +inf, up_bias = -1 and no other
 * bias the result is rf_moe_ffn's.  gate_bias, up_bias: (n_expert, n_ff)
 * fp32; down_bias: (n_expert, n_embd) fp32; device, 4-byte aligned; any may
 * be NULL (no bias).  NaN activations are outside the contract.
 * Errors: as rf_moe_ffn; RF_ERR_INVALID_ARG for a NaN or infinite alpha or a
 * limit that is not positive (+inf is allowed: no clamp); RF_ERR_MISALIGNED
 * for a misaligned bias. */
RF_API rf_status rf_moe_ffn_biased(int fmt, const float *router_logits, int n_expert,
                                   int top_k, const void *gate, const void *up, const void *down,
                                   const float *gate_bias, const float *up_bias,
                                   const float *down_bias, float alpha, float limit,
                                   int64_t n_ff, int64_t n_embd, int64_t block_rows,
                                   const float *x, float *y, void *workspace, void *stream);

/* --------------------------------------------- host-streamed MoE experts */
/* Expert cache: device memory for `slots` whole experts (each expert's n_ff
 * gate rows, n_ff up rows and n_embd down rows, raw block bytes) of one fmt
 * and shape, with a host-side directory keyed by (host gate tensor, expert
 * index) and least-recently-used replacement (neurostream, "How it works" 1
 * and 3: the slab cache of expert windows; windows it holds are not read
 * again).  Owns its device memory and events; used by one host thread at a
 * time.  Errors: RF_ERR_INVALID_ARG for a bad shape or slots < 1,
 * RF_ERR_UNSUPPORTED_FMT, RF_ERR_OOM. */
typedef struct rf_expert_cache rf_expert_cache;
RF_API rf_status rf_expert_cache_create(int fmt, int64_t n_ff, int64_t n_embd, int slots,
                                        rf_expert_cache **out);
/* Waits for the cache's outstanding copies and readers, then frees it.  NULL
 * is a no-op. */
RF_API void rf_expert_cache_destroy(rf_expert_cache *cache);

typedef struct rf_expert_cache_stats_t {
    uint64_t lookups;          /* selected experts looked up */
    uint64_t hits;             /* ... found in the cache (nothing read from the host) */
    uint64_t fills;            /* ... streamed into a cache slot */
    uint64_t bypasses;         /* ... streamed through the arena (no free slot) */
    uint64_t evictions;        /* fills that replaced another expert */
    uint64_t bytes_streamed;   /* host->device expert bytes enqueued */
    uint64_t bytes_cached;     /* expert bytes read from the cache instead */
    int32_t slots, used;       /* capacity and occupied slots */
} rf_expert_cache_stats_t;
/* Copies the cache's counters to *out.  Errors: RF_ERR_INVALID_ARG (NULL). */
RF_API rf_status rf_expert_cache_stats(const rf_expert_cache *cache,
                                       rf_expert_cache_stats_t *out);

/* Routed SwiGLU FFN with the stacked expert tensors in page-locked host
 * memory, read through one layer-wide prefetch plan (neurostream, "How it
 * works" 3: once routing has named the layer's experts, a single block list
 * covers their gate, up and down rows in the order the launches read them,
 * with at most `depth` blocks fetched ahead, so copies run on into down's
 * rows while gate/up computes; rows the cache holds are not copied; "What
 * the numbers taught us": separate per-projection pipelines drain between
 * projections, the single list does not).
 *
 * Steps: the router kernel writes the top_k experts and weights to the
 * workspace; their ids are copied to the host (the call blocks until the
 * routing result and everything before it on `stream` is done; it is not
 * capturable in a CUDA graph); the host then enqueues, without blocking:
 *   gate/up -- one launch for the cached experts; for every other expert,
 *              per block of block_rows rows its gate and up rows (copied
 *              into a cache slot, or through the arena when no slot is
 *              free) and a launch with the SwiGLU epilogue;
 *   down    -- per block of block_rows output rows, the rows of every
 *              selected expert (from the cache or copied) in one launch that
 *              forms sum_k w_k * down_k . h_k in selection order.
 * All copies go through the arena's copy stream in that order; a slot is
 * reused only after the launch reading it.  Outputs are bit-identical to
 * rf_moe_ffn on the same bytes.
 *
 * host_gate, host_up: (n_expert, n_ff, n_embd); host_down: (n_expert,
 * n_embd, n_ff); page-locked, 16-byte aligned.  block_rows: a multiple of 32
 * (0 = whole windows), shrunk to a multiple of 32 until depth+1 blocks of
 * the longer rows fit the arena.  depth: 1..64 with depth+1 >= max(2,
 * top_k) (a down launch holds top_k blocks at once).  cache: NULL (every
 * expert streams through the arena) or a cache of the same fmt and shape.
 * workspace: rf_moe_workspace_bytes(top_k, n_ff, n_embd, block_rows) bytes
 * of device memory, 256-byte aligned; it receives the routing result and h as
 * rf_moe_ffn's does.
 * Errors: as rf_moe_ffn; RF_ERR_NOT_PINNED for pageable tensors;
 * RF_ERR_ARENA_TOO_SMALL if 32-row blocks do not fit; RF_ERR_INVALID_ARG if
 * `stream` is capturing or the cache's shape differs. */
RF_API rf_status rf_moe_ffn_streamed(int fmt, const float *router_logits, int n_expert,
                                     int top_k, const void *host_gate, const void *host_up,
                                     const void *host_down, int64_t n_ff, int64_t n_embd,
                                     int64_t block_rows, int depth, rf_arena *arena,
                                     rf_expert_cache *cache, const float *x, float *y,
                                     void *workspace, void *stream);

/* rf_moe_ffn without a workspace argument, for callers that cannot allocate
 * device memory: for example an engine that plans all of its device memory
 * once at start-up and forbids allocations afterwards, or a decode loop that
 * must not call cudaMalloc/cudaFree because those synchronize the device.
 * (The source pages have no counterpart to this entry point.)
 * The scratch it needs lives in a fixed device array inside the library,
 * RF_MOE_STATIC_MAX_H floats of activations, their digits (80 bytes per 32)
 * and the routing result, which
 * every GPU that loads the library keeps until the process exits.  Limit:
 * top_k * n_ff <= RF_MOE_STATIC_MAX_H, else RF_ERR_TOO_LARGE before any work
 * (n_ff <= rf_max_in_dim(fmt, top_k) applies as for rf_moe_ffn, which with
 * 4 experts caps the activations at 53,120 on a GB300).
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; make that first call before any stream capture.  A caller that
 * resets the device (cudaDeviceReset) invalidates that address: do not call
 * this entry point on the device afterwards.  All calls share the one array and it keeps the last call's
 * contents; nothing in it needs to start at zero.  Calls whose kernels
 * overlap on the GPU (different streams, or different host threads) race on
 * it: serialise them.  Arguments and results otherwise as rf_moe_ffn. */
#define RF_MOE_STATIC_MAX_H 65536
RF_API rf_status rf_moe_ffn_noalloc(int fmt, const float *router_logits, int n_expert, int top_k,
                                    const void *gate, const void *up, const void *down,
                                    int64_t n_ff, int64_t n_embd, int64_t block_rows,
                                    const float *x, float *y, void *stream);

/* --------------------------------------------------------------- status */
/* Synchronizes the current device, then reports and clears the device status
 * word that kernels set when a bounded wait times out (RF_OK if none).
 * Returns RF_ERR_CUDA if the device reports an error. */
RF_API rf_status rf_device_status(void);

/* Test hook for the kernels' bounded waits (the pages have no counterpart; it
 * lets the failure path be exercised without faulting a GPU).  Arms a
 * one-shot fault for the next launch on this process that copies with
 * tensor or bulk copies: a GEMV over device memory whose rows are 16-byte
 * aligned or take per-row bulk copies, or an rf_gemm.  In
 * that launch one copy of its first CTA is never issued (a stage of the
 * GEMV's weights; the GEMM's second activation tile), so the warps waiting
 * for it give up after limit_us microseconds,
 * record RF_ERR_TIMEOUT, and the launch ends with nothing in flight (its
 * outputs are undefined).
 * limit_us = 0 disarms.  Errors: RF_ERR_INVALID_ARG for limit_us above
 * 2,000,000. */
RF_API rf_status rf_debug_arm_wait_fault(uint32_t limit_us);

#ifdef __cplusplus
}
#endif
#endif /* RF_H */
