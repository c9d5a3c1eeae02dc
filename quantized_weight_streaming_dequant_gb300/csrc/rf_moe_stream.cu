// rf_moe_stream.cu -- the routed MoE FFN with host-resident experts, read
// through one layer-wide prefetch plan, and the device expert cache.
//
// What it follows (neurostream, "How it works" 1-3 and 6; "What the numbers
// taught us"): quantized expert rows may stay cached on the device; routing
// comes first and fixes which experts a token touches; a single block list
// for the whole layer orders every active expert's gate, up and down rows as
// the launches will read them, and the copy engine runs through that list a
// bounded number of blocks ahead, so it moves on to down's rows while
// gate/up still computes instead of draining between projections; rows the
// cache already holds are not copied; each block in flight occupies arena
// space until its reader is done.
//
// GB300 form: the router kernel's result is read back to the host (the one
// synchronisation), the host plans, and everything else is stream-ordered:
// copies on the arena's copy stream in plan order (into a cache slot, or an
// arena slot when no cache slot is free), each launch waits for its blocks'
// copies, and each slot is reused only after the launches that read it.  The
// launches are the resident MoE's: a 2-term SwiGLU job per gate/up block, and
// per down block one job whose top_k terms are combined with the router's
// weights in selection order -- so outputs are bit-identical to rf_moe_ffn.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "rf_arena.h"

using namespace rf;

struct rf_expert_cache {
    int fmt = 0;
    int64_t n_ff = 0, n_embd = 0;
    int slots = 0;
    int64_t rb_g = 0, rb_d = 0;   // gate/up row bytes, down row bytes
    uint8_t *gate = nullptr, *up = nullptr, *down = nullptr;   // [slots][rows][row bytes]
    int device = 0;
    // Directory: which (host gate tensor, expert) each slot holds.
    std::vector<const void *> key_tensor;
    std::vector<int> key_expert;
    std::vector<uint64_t> last_use;
    std::vector<cudaEvent_t> freed;   // recorded after the last launch reading the slot
    std::vector<bool> freed_recorded;
    std::vector<cudaEvent_t> ready;   // recorded after the last copy filling the slot
    std::vector<bool> ready_recorded;
    cudaEvent_t copied = nullptr;     // block copy into a slot done (re-recorded per block)
    uint64_t clock = 0;
    rf_expert_cache_stats_t stats = {};
};

namespace {

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

bool pinned(const void *p)
{
    cudaPointerAttributes attr;
    if (!p || cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

rf_status rf_expert_cache_create(int fmt, int64_t n_ff, int64_t n_embd, int slots,
                                 rf_expert_cache **out)
{
    if (!out) return RF_ERR_INVALID_ARG;
    *out = nullptr;
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (n_ff <= 0 || n_embd <= 0 || n_ff % block_elems_of(fmt) != 0 ||
        n_embd % block_elems_of(fmt) != 0 || n_ff % 32 != 0 || n_embd % 32 != 0 || slots < 1 ||
        slots > 1024)
        return RF_ERR_INVALID_ARG;
    rf_expert_cache *c = new (std::nothrow) rf_expert_cache();
    if (!c) return RF_ERR_OOM;
    c->fmt = fmt;
    c->n_ff = n_ff;
    c->n_embd = n_embd;
    c->slots = slots;
    c->rb_g = n_embd / block_elems_of(fmt) * (int64_t)block_bytes_of(fmt);
    c->rb_d = n_ff / block_elems_of(fmt) * (int64_t)block_bytes_of(fmt);
    if (cudaGetDevice(&c->device) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return RF_ERR_CUDA;
    }
    const size_t gsz = (size_t)slots * (size_t)n_ff * (size_t)c->rb_g;
    const size_t dsz = (size_t)slots * (size_t)n_embd * (size_t)c->rb_d;
    bool ok = cudaMalloc(&c->gate, gsz) == cudaSuccess && cudaMalloc(&c->up, gsz) == cudaSuccess &&
              cudaMalloc(&c->down, dsz) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&c->copied, cudaEventDisableTiming) == cudaSuccess;
    c->freed.assign(slots, nullptr);
    c->ready.assign(slots, nullptr);
    for (int i = 0; ok && i < slots; ++i)
        ok = cudaEventCreateWithFlags(&c->freed[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&c->ready[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        rf_expert_cache_destroy(c);
        return RF_ERR_OOM;
    }
    c->key_tensor.assign(slots, nullptr);
    c->key_expert.assign(slots, -1);
    c->last_use.assign(slots, 0);
    c->freed_recorded.assign(slots, false);
    c->ready_recorded.assign(slots, false);
    c->stats.slots = slots;
    *out = c;
    return RF_OK;
}

void rf_expert_cache_destroy(rf_expert_cache *c)
{
    if (!c) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(c->device);
    if (c->copied) {
        cudaEventSynchronize(c->copied);
        cudaEventDestroy(c->copied);
    }
    for (size_t i = 0; i < c->freed.size(); ++i) {
        if (!c->freed[i]) continue;
        if (i < c->freed_recorded.size() && c->freed_recorded[i]) cudaEventSynchronize(c->freed[i]);
        cudaEventDestroy(c->freed[i]);
    }
    for (size_t i = 0; i < c->ready.size(); ++i)
        if (c->ready[i]) cudaEventDestroy(c->ready[i]);
    if (c->gate) cudaFree(c->gate);
    if (c->up) cudaFree(c->up);
    if (c->down) cudaFree(c->down);
    cudaGetLastError();
    cudaSetDevice(prev);
    delete c;
}

rf_status rf_expert_cache_stats(const rf_expert_cache *c, rf_expert_cache_stats_t *out)
{
    if (!c || !out) return RF_ERR_INVALID_ARG;
    *out = c->stats;
    out->used = (int32_t)std::count_if(c->key_expert.begin(), c->key_expert.end(),
                                       [](int e) { return e >= 0; });
    return RF_OK;
}

rf_status rf_moe_ffn_streamed(int fmt, const float *router_logits, int n_expert, int top_k,
                              const void *host_gate, const void *host_up, const void *host_down,
                              int64_t n_ff, int64_t n_embd, int64_t block_rows, int depth,
                              rf_arena *a, rf_expert_cache *cache, const float *x, float *y,
                              void *workspace, void *stream)
{
    // ---- checks (nothing is enqueued before they pass)
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!router_logits || !host_gate || !host_up || !host_down || !a || !x || !y || !workspace)
        return RF_ERR_INVALID_ARG;
    if (n_expert < 1 || n_expert > 1024 || top_k < 1 || top_k > kMaxTerms || top_k > n_expert)
        return RF_ERR_INVALID_ARG;
    if (n_ff <= 0 || n_embd <= 0 || n_ff % block_elems_of(fmt) != 0 ||
        n_embd % block_elems_of(fmt) != 0 || n_ff % 32 != 0 || n_embd % 32 != 0)
        return RF_ERR_INVALID_ARG;
    if (block_rows < 0 || block_rows % 32 != 0 || depth < 1 || depth > rf_arena::kMaxSlots - 1 ||
        depth + 1 < std::max(2, top_k))
        return RF_ERR_INVALID_ARG;
    if (n_ff > 0x7fffffffLL || n_embd > 0x7fffffffLL) return RF_ERR_TOO_LARGE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RF_ERR_MISALIGNED;
    for (const void *p : {host_gate, host_up, host_down})
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (!pinned(host_gate) || !pinned(host_up) || !pinned(host_down)) return RF_ERR_NOT_PINNED;
    if (cache && (cache->fmt != fmt || cache->n_ff != n_ff || cache->n_embd != n_embd))
        return RF_ERR_INVALID_ARG;
    if (const rf_status c = check_in_dim(fmt, n_embd, 1)) return c;
    if (const rf_status c = check_in_dim(fmt, n_ff, top_k)) return c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return RF_ERR_INVALID_ARG;

    const int64_t rb_g = n_embd / block_elems_of(fmt) * (int64_t)block_bytes_of(fmt);
    const int64_t rb_d = n_ff / block_elems_of(fmt) * (int64_t)block_bytes_of(fmt);
    const int64_t rb_max = std::max(rb_g, rb_d);
    const int64_t rows_max = std::max(n_ff, n_embd);
    int64_t eff = arena_plan_rows(rb_max, rows_max, block_rows, depth, a->bytes);
    if (eff < 32) return RF_ERR_ARENA_TOO_SMALL;
    eff = eff / 32 * 32;   // blocks start on 32-row (16-byte aligned) boundaries
    const int slots = depth + 1;
    const size_t stride = align256((size_t)(eff * rb_max));
    if ((size_t)slots * stride > a->alloc_bytes) return RF_ERR_ARENA_TOO_SMALL;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *idx = reinterpret_cast<int32_t *>(ws);
    float *wts = reinterpret_cast<float *>(ws + align256(sizeof(int32_t) * kMaxTerms));
    float *h = reinterpret_cast<float *>(ws + align256(sizeof(int32_t) * kMaxTerms) +
                                         align256(sizeof(float) * kMaxTerms));
    void *hdig = ws + align256(sizeof(int32_t) * kMaxTerms) + align256(sizeof(float) * kMaxTerms) +
                 align256(sizeof(float) * (size_t)top_k * (size_t)n_ff);

    std::lock_guard<std::mutex> lock(a->mu);

    // ---- routing, read back for the plan
    if (const rf_status st = launch_router(router_logits, n_expert, top_k, idx, wts, s)) return st;
    if (cudaMemcpyAsync(a->route_host, idx, sizeof(int32_t) * top_k, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return RF_ERR_CUDA;
    int experts[kMaxTerms];
    for (int k = 0; k < top_k; ++k) {
        experts[k] = a->route_host[k];
        if (experts[k] < 0 || experts[k] >= n_expert) return RF_ERR_CUDA;
    }

    // ---- cache directory: hits, and a slot for every miss that can have one
    int slot_of[kMaxTerms];    // cache slot of expert k, or -1 (arena)
    bool fill[kMaxTerms];      // the slot is filled by this call
    bool taken_slot[1024] = {};
    if (cache) {
        cache->clock += 1;
        for (int k = 0; k < top_k; ++k) {
            slot_of[k] = -1;
            fill[k] = false;
            for (int c = 0; c < cache->slots; ++c)
                if (cache->key_expert[c] == experts[k] && cache->key_tensor[c] == host_gate) {
                    slot_of[k] = c;
                    break;
                }
            if (slot_of[k] >= 0 && slot_of[k] < 1024) taken_slot[slot_of[k]] = true;
        }
        for (int k = 0; k < top_k; ++k) {
            cache->stats.lookups += 1;
            if (slot_of[k] >= 0) {
                cache->stats.hits += 1;
                cache->last_use[slot_of[k]] = cache->clock;
                continue;
            }
            // Victim: an empty slot, else the least recently used one that
            // this call does not use.
            int v = -1;
            for (int c = 0; c < cache->slots && c < 1024; ++c) {
                if (taken_slot[c]) continue;
                if (v < 0 || (cache->key_expert[c] < 0 && cache->key_expert[v] >= 0) ||
                    ((cache->key_expert[c] >= 0) == (cache->key_expert[v] >= 0) &&
                     cache->last_use[c] < cache->last_use[v]))
                    v = c;
            }
            if (v < 0) {
                cache->stats.bypasses += 1;
                continue;
            }
            if (cache->key_expert[v] >= 0) cache->stats.evictions += 1;
            cache->stats.fills += 1;
            taken_slot[v] = true;
            slot_of[k] = v;
            fill[k] = true;
            cache->key_tensor[v] = host_gate;
            cache->key_expert[v] = experts[k];
            cache->last_use[v] = cache->clock;
        }
    } else {
        for (int k = 0; k < top_k; ++k) {
            slot_of[k] = -1;
            fill[k] = false;
        }
    }

    if (const rf_status st = arena_prepare(a, s, slots, stride)) return st;
    const uint8_t *hg = static_cast<const uint8_t *>(host_gate);
    const uint8_t *hu = static_cast<const uint8_t *>(host_up);
    const uint8_t *hd = static_cast<const uint8_t *>(host_down);
    int64_t blocks = 0;

    // A block of `bytes` from host `src` into cache slot memory `dst` (after
    // the slot's last reader, for the first block of a fill).
    auto fetch_cache = [&](int c, bool first, uint8_t *dst, const uint8_t *src,
                           size_t bytes) -> rf_status {
        if (first && cache->freed_recorded[c] &&
            cudaStreamWaitEvent(a->copy_stream, cache->freed[c], 0) != cudaSuccess)
            return RF_ERR_CUDA;
        if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, a->copy_stream) !=
                cudaSuccess ||
            cudaEventRecord(cache->copied, a->copy_stream) != cudaSuccess ||
            cudaStreamWaitEvent(s, cache->copied, 0) != cudaSuccess)
            return RF_ERR_CUDA;
        cache->stats.bytes_streamed += bytes;
        return RF_OK;
    };
    auto launch = [&](Job *jobs, int n_jobs, int64_t in_dim, const float *const *xs, int n_x,
                      bool gate_up) -> rf_status {
        LaunchDesc d;
        d.fmt = fmt;
        d.in_dim = in_dim;
        d.jobs = jobs;
        d.n_jobs = n_jobs;
        for (int i = 0; i < n_x; ++i) d.x[i] = xs[i];
        d.n_x = n_x;
        if (gate_up) {
            d.xr_out = hdig;   // h's digits for the down launches
            d.xr_y_base = h;
        } else {
            d.xr_in = hdig;
        }
        return launch_rowwin(d, s);
    };

    // Cached experts may have been filled from another stream.
    for (int k = 0; k < top_k; ++k)
        if (slot_of[k] >= 0 && !fill[k] && cache->ready_recorded[slot_of[k]] &&
            cudaStreamWaitEvent(s, cache->ready[slot_of[k]], 0) != cudaSuccess)
            return RF_ERR_CUDA;

    // ---- gate/up: the cached experts in one launch, then block by block
    Job jobs[kMaxTerms];
    int nj = 0;
    for (int k = 0; k < top_k; ++k) {
        if (slot_of[k] < 0 || fill[k]) continue;
        const int c = slot_of[k];
        Job &J = jobs[nj++];
        std::memset(&J, 0, sizeof(J));
        J.term[0] = Term{cache->gate + (size_t)c * n_ff * rb_g, 0, -1, 0, 0};
        J.term[1] = Term{cache->up + (size_t)c * n_ff * rb_g, 0, -1, 0, 0};
        J.y = h + (int64_t)k * n_ff;
        J.n_rows = (int32_t)n_ff;
        J.n_terms = 2;
        J.combine = kCombineSwiGLU;
        cache->stats.bytes_cached += (uint64_t)(2 * n_ff * rb_g + n_embd * rb_d);
    }
    if (nj > 0)
        if (const rf_status st = launch(jobs, nj, n_embd, &x, 1, true)) return st;
    for (int k = 0; k < top_k; ++k) {
        if (slot_of[k] >= 0 && !fill[k]) continue;
        const int64_t e = experts[k];
        for (int64_t r0 = 0; r0 < n_ff; r0 += eff) {
            const int64_t nr = std::min(eff, n_ff - r0);
            const size_t bytes = (size_t)(nr * rb_g);
            const uint8_t *sg = hg + ((size_t)e * n_ff + r0) * rb_g;
            const uint8_t *su = hu + ((size_t)e * n_ff + r0) * rb_g;
            uint8_t *dg = nullptr, *du = nullptr;
            int slot_g = -1, slot_u = -1;
            if (fill[k]) {
                const int c = slot_of[k];
                dg = cache->gate + ((size_t)c * n_ff + r0) * rb_g;
                du = cache->up + ((size_t)c * n_ff + r0) * rb_g;
                if (const rf_status st = fetch_cache(c, r0 == 0, dg, sg, bytes)) return st;
                if (const rf_status st = fetch_cache(c, false, du, su, bytes)) return st;
            } else {
                if (const rf_status st = arena_fetch(a, s, sg, bytes, &slot_g, &dg)) return st;
                if (const rf_status st = arena_fetch(a, s, su, bytes, &slot_u, &du)) return st;
                if (cache) cache->stats.bytes_streamed += 2 * bytes;
            }
            Job &J = jobs[0];
            std::memset(&J, 0, sizeof(J));
            J.term[0] = Term{dg, 0, -1, 0, 0};
            J.term[1] = Term{du, 0, -1, 0, 0};
            J.y = h + (int64_t)k * n_ff + r0;
            J.n_rows = (int32_t)nr;
            J.n_terms = 2;
            J.combine = kCombineSwiGLU;
            if (const rf_status st = launch(jobs, 1, n_embd, &x, 1, true)) return st;
            if (slot_g >= 0)
                if (arena_release(a, s, slot_g) != RF_OK || arena_release(a, s, slot_u) != RF_OK)
                    return RF_ERR_CUDA;
            blocks += 2;
        }
    }

    // ---- down: per output row block, every selected expert's rows in one
    // launch, combined with the router's weights in selection order
    const float *hk[kMaxTerms];
    for (int k = 0; k < top_k; ++k) hk[k] = h + (int64_t)k * n_ff;
    for (int64_t r0 = 0; r0 < n_embd; r0 += eff) {
        const int64_t nr = std::min(eff, n_embd - r0);
        const size_t bytes = (size_t)(nr * rb_d);
        int slot_a[kMaxTerms];
        Job &J = jobs[0];
        std::memset(&J, 0, sizeof(J));
        for (int k = 0; k < top_k; ++k) {
            slot_a[k] = -1;
            const uint8_t *src = hd + ((size_t)experts[k] * n_embd + r0) * rb_d;
            uint8_t *dst = nullptr;
            if (slot_of[k] >= 0) {
                const int c = slot_of[k];
                dst = cache->down + ((size_t)c * n_embd + r0) * rb_d;
                if (fill[k])
                    if (const rf_status st = fetch_cache(c, false, dst, src, bytes)) return st;
            } else {
                if (const rf_status st = arena_fetch(a, s, src, bytes, &slot_a[k], &dst)) return st;
                if (cache) cache->stats.bytes_streamed += bytes;
            }
            J.term[k] = Term{dst, k, -1, 0, 0};
        }
        J.y = y + r0;
        J.n_rows = (int32_t)nr;
        J.n_terms = top_k;
        J.combine = kCombineSum;
        J.weights = wts;
        if (const rf_status st = launch(jobs, 1, n_ff, hk, top_k, false)) return st;
        for (int k = 0; k < top_k; ++k) {
            if (slot_a[k] >= 0 && arena_release(a, s, slot_a[k]) != RF_OK) return RF_ERR_CUDA;
            if (slot_a[k] >= 0) ++blocks;
            if (fill[k]) ++blocks;
        }
    }
    // The cache slots this call read are free again after its last launch;
    // the slots it filled are complete after its last copy.
    if (cache)
        for (int k = 0; k < top_k; ++k) {
            const int c = slot_of[k];
            if (c < 0) continue;
            if (cudaEventRecord(cache->freed[c], s) != cudaSuccess) return RF_ERR_CUDA;
            cache->freed_recorded[c] = true;
            if (fill[k]) {
                if (cudaEventRecord(cache->ready[c], a->copy_stream) != cudaSuccess)
                    return RF_ERR_CUDA;
                cache->ready_recorded[c] = true;
            }
        }
    a->stats.calls += 1;
    a->stats.blocks += (uint64_t)blocks;
    a->stats.slot_bytes = stride;
    a->stats.slots = slots;
    a->stats.last_block_rows = (int32_t)eff;
    a->stats.peak_bytes = std::max<uint64_t>(a->stats.peak_bytes, (uint64_t)slots * stride);
    return RF_OK;
}

}  // extern "C"
