// rf_internal.h -- host-side interface between the C ABI entry points and the
// row-window GEMV launcher.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "rf.h"

namespace rf {

constexpr int kMaxTerms = 8;   // matrices combined per output row (top-k of a MoE down)
constexpr int kMaxJobs = 64;   // row windows per launch
constexpr int kMaxX = 8;       // distinct activation vectors per launch

// How the per-term row dots of a job become the output row.
enum Combine : int32_t {
    kCombineSum = 0,     // y = sum_t weight_t * dot_t (weight 1 when weights == nullptr)
    kCombineSwiGLU = 1,  // y = silu(dot_0) * dot_1  (gate, up)
    kCombineRouted = 2,  // y = sum_t w[expert_slot_t] * dot_t, w from the launch's own routing
    kCombineEach = 3,    // y[t * y_stride + r] = dot_t: one output row per term (batched tokens)
};
// Activation of the output row.  kActClampSwiGLU changes kCombineSwiGLU to
// the biased experts' clamped form: g' = min(g, limit), u' = clamp(u, -limit,
// limit), y = g' * sigmoid(alpha * g') * (u' + 1).
enum Act : int32_t { kActNone = 0, kActGelu = 1, kActClampSwiGLU = 2 };

struct Term {
    const uint8_t *W;     // row 0 of the matrix (or of the stacked tensor)
    int32_t xslot;        // which activation vector multiplies this matrix
    int32_t expert_slot;  // >= 0: add expert_idx[expert_slot]*expert_rows rows to W
    int32_t tmap;         // filled by the launcher: tensor map of W (aligned rows)
    int32_t pad;
    const float *bias;    // or nullptr: added to the row's dot (indexed like W's rows)
};

// One window of rows [row0, row0+n_rows) taken from every term's matrix.
struct Job {
    Term term[kMaxTerms];
    float *y;               // n_rows outputs
    const float *weights;   // per-term weights (device) for kCombineSum, or nullptr
    int64_t row0;
    int64_t expert_rows;
    int64_t expert_count;   // experts in the stacked tensor (expert terms)
    int64_t y_stride;       // kCombineEach: floats between the terms' output rows
    int32_t n_rows;
    int32_t n_terms;
    int32_t combine;
    int32_t act;
    int32_t group_begin;    // filled by the launcher
    int32_t aligned;        // filled by the launcher
    float alpha, limit;     // kActClampSwiGLU constants
};

struct LaunchDesc {
    int fmt = 0;
    int64_t in_dim = 0;
    const Job *jobs = nullptr;
    int n_jobs = 0;
    const float *x[kMaxX] = {};
    int n_x = 0;
    const int32_t *expert_idx = nullptr;   // device, for expert_slot terms
    bool pdl = false;                      // programmatic dependent launch
    bool any_expert = false;               // some term resolves an expert on device
    bool host_weights = false;             // weights are mapped page-locked host memory
    // Routing computed inside the launch (instead of expert_idx): top route_k
    // of route_n logits (ties to the lower index) and a softmax over the k
    // selected; CTA 0 also stores them to route_idx_out / route_w_out.  The
    // logits must not be written by the kernel this launch is chained to.
    const float *route_logits = nullptr;
    int route_n = 0, route_k = 0;
    int32_t *route_idx_out = nullptr;
    float *route_w_out = nullptr;
    // Activation digits (80 bytes per 32 activations) written by this launch
    // for every full 32-output block of its jobs, indexed by the outputs'
    // position from xr_y_base (jobs must start and end on 32-output
    // boundaries from it), and digits read instead of built: slot s of the
    // launch's activations is records [s*in_dim/32, (s+1)*in_dim/32) of xr_in.
    void *xr_out = nullptr;
    const float *xr_y_base = nullptr;
    const void *xr_in = nullptr;
};

// Bytes of activation digits for n activations (n a multiple of 32).
constexpr size_t xrec_bytes(int64_t n) { return (size_t)(n / 32) * 80; }

// Validates and launches the row-window GEMV kernel (in batches of kMaxJobs
// windows).  Host-side argument checks return an error before anything is
// enqueued.
rf_status launch_rowwin(const LaunchDesc &d, cudaStream_t stream);

bool fmt_ok(int fmt);
size_t block_bytes_of(int fmt);
// Weights per block: 32, or 256 for the K-quant super-blocks.
inline int64_t block_elems_of(int fmt) { return fmt == RF_Q4_K || fmt == RF_Q6_K ? 256 : 32; }
rf_status last_cuda_error();
rf_status read_and_clear_device_status();
// 2-D tiled tensor map of uint16 elements: `rows` rows of `cols` elements,
// `row_bytes` apart (a multiple of 16), boxes of box_cols x box_rows, no
// swizzle, zero fill outside.  False if the driver refuses it.
bool encode_u16_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows);
// The prefill GEMM's own status word (bounded waits), read and cleared.
rf_status read_and_clear_gemm_status();
// Arms the one-shot wait fault of the next producer-mode launch
// (rf_debug_arm_wait_fault).
rf_status arm_wait_fault(uint32_t limit_us);
// The armed wait limit in ns (0 if none), disarming it: the next launch
// that takes it withholds one copy.
unsigned long long take_wait_fault();
int num_sms();
int64_t max_in_dim(int fmt, int n_x);
// RF_OK, RF_ERR_TOO_LARGE (in_dim above max_in_dim) or RF_ERR_CUDA (no device).
rf_status check_in_dim(int fmt, int64_t in_dim, int n_x);

rf_status launch_router(const float *logits, int n_expert, int top_k, int32_t *idx, float *w,
                        cudaStream_t stream);

}  // namespace rf
