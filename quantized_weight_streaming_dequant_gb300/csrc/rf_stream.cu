// rf_stream.cu -- bounded device arena and host-streamed row windows.
//
// What it follows (neurostream, "How it works" 3, 4 and 6; "Bugs worth
// knowing about"): a row window is walked block by block -- fetch, multiply,
// add to the outputs, give the block back -- with a bounded number of blocks
// fetched ahead of the one being multiplied; each fetched block takes arena
// space, and a fetch that finds no free space waits for a block to be given
// back, so the prefetcher cannot run away.  A block keeps its space until
// its outputs exist, so a walk with `depth` blocks ahead holds depth+1.
//
// GB300 form: the arena is one device allocation cut into depth+1 slots.  The
// prefetcher is a dedicated copy stream; each block is a cudaMemcpyAsync from
// page-locked host memory into its slot, followed by an event that the
// block's GEMV waits on before it reads the slot.  The GEMVs of a walk of 8
// or more small blocks go round-robin to the arena's lane streams (rows are
// disjoint), so a block whose copy has landed does not queue behind the
// previous block's GEMV; the lanes start after the caller's stream and the
// caller's stream waits for all of them at the end of the walk.  After a
// GEMV a "slot free" event is recorded on its lane; the copy that next
// reuses the slot waits on it.  Reservations and back-pressure are therefore
// stream-ordered dependencies: the host enqueues a whole walk without
// blocking, and consecutive calls keep the copy engine busy across call
// boundaries (no drain between projections).
//
// A walk can also be captured into a CUDA graph (the copy stream joins the
// capture through a fork event), so a whole token's walks replay with one
// host call.  Slot-free events only order walks of the same epoch: the eager
// epoch, or one capture.  The first walk of a new epoch starts after
// everything already enqueued on its stream instead.
#include <algorithm>
#include <chrono>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>

#include "rf_arena.h"

using namespace rf;

namespace rf {

namespace {
// Host function of an injected stall: holds the copy stream for `ms` ms.
void CUDART_CB stall_host(void *ms)
{
    std::this_thread::sleep_for(std::chrono::milliseconds((int)(intptr_t)ms));
}
}  // namespace

int64_t arena_plan_rows(int64_t row_bytes, int64_t n_rows, int64_t block_rows, int depth,
                        size_t arena_bytes)
{
    int64_t want = (block_rows == 0 || block_rows > n_rows) ? n_rows : block_rows;
    if (want < 1) want = 1;
    const int64_t fit = (int64_t)(arena_bytes / ((size_t)(depth + 1) * (size_t)row_bytes));
    if (fit < 1) return -1;
    return std::min(want, fit);
}

rf_status arena_prepare(rf_arena *a, cudaStream_t s, int slots, size_t stride)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    unsigned long long cap_id = 0;
    if (cudaStreamGetCaptureInfo(s, &cap, &cap_id) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    if (cap == cudaStreamCaptureStatusInvalidated) return RF_ERR_CUDA;
    const unsigned long long epoch = cap == cudaStreamCaptureStatusActive ? cap_id : 0;
    if (epoch != a->epoch) {
        // The slot-free events belong to another epoch: order this walk
        // after all work already enqueued on `s` (which includes every
        // earlier reader of the slots when the graph is launched there).
        if (cudaEventRecord(a->fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(a->copy_stream, a->fork, 0) != cudaSuccess)
            return RF_ERR_CUDA;
        for (int i = 0; i < rf_arena::kMaxSlots; ++i) a->freed_recorded[i] = false;
        a->next_slot = 0;
        a->last_slots = slots;
        a->last_stride = stride;
        a->epoch = epoch;
    }
    // A new slot layout overlaps the old one: the copy stream first waits for
    // every old slot's last reader.
    if (a->last_slots != slots || a->last_stride != stride) {
        for (int i = 0; i < rf_arena::kMaxSlots; ++i)
            if (a->freed_recorded[i] &&
                cudaStreamWaitEvent(a->copy_stream, a->freed[i], 0) != cudaSuccess)
                return RF_ERR_CUDA;
        a->next_slot = 0;
        a->last_slots = slots;
        a->last_stride = stride;
    }
    return RF_OK;
}

rf_status arena_fetch(rf_arena *a, cudaStream_t s, const void *src, size_t bytes, int *slot_out,
                      uint8_t **dst_out)
{
    const int slot = a->next_slot;
    a->next_slot = (a->next_slot + 1) % a->last_slots;
    uint8_t *dst = a->base + (size_t)slot * a->last_stride;
    // Reservation: the slot's previous readers must have finished with it.
    if (a->freed_recorded[slot] &&
        cudaStreamWaitEvent(a->copy_stream, a->freed[slot], 0) != cudaSuccess)
        return RF_ERR_CUDA;
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, a->copy_stream) != cudaSuccess ||
        cudaEventRecord(a->copied[slot], a->copy_stream) != cudaSuccess ||
        cudaStreamWaitEvent(s, a->copied[slot], 0) != cudaSuccess)
        return RF_ERR_CUDA;
    a->stats.bytes_copied += bytes;
    *slot_out = slot;
    *dst_out = dst;
    return RF_OK;
}

rf_status arena_release(rf_arena *a, cudaStream_t s, int slot)
{
    if (cudaEventRecord(a->freed[slot], s) != cudaSuccess) return RF_ERR_CUDA;
    a->freed_recorded[slot] = true;
    return RF_OK;
}

rf_status arena_fetch_run(rf_arena *a, cudaStream_t s, const void *src, size_t block_bytes,
                          int n, size_t last_bytes, int *first_slot, uint8_t **base)
{
    const int first = a->next_slot + n <= a->last_slots ? a->next_slot : 0;
    a->next_slot = (first + n) % a->last_slots;
    for (int k = first; k < first + n; ++k)
        if (a->freed_recorded[k] && cudaStreamWaitEvent(a->copy_stream, a->freed[k], 0) != cudaSuccess)
            return RF_ERR_CUDA;
    uint8_t *dst = a->base + (size_t)first * a->last_stride;
    const uint8_t *hsrc = static_cast<const uint8_t *>(src);
    const size_t full = (size_t)(n - 1) * block_bytes;
    if (a->last_stride == block_bytes) {
        // Slots packed back to back: the whole run is one contiguous copy.
        if (cudaMemcpyAsync(dst, hsrc, full + last_bytes, cudaMemcpyHostToDevice,
                            a->copy_stream) != cudaSuccess)
            return RF_ERR_CUDA;
    } else {
        if ((n > 1 && cudaMemcpy2DAsync(dst, a->last_stride, hsrc, block_bytes, block_bytes,
                                        (size_t)(n - 1), cudaMemcpyHostToDevice,
                                        a->copy_stream) != cudaSuccess) ||
            cudaMemcpyAsync(dst + (size_t)(n - 1) * a->last_stride, hsrc + full, last_bytes,
                            cudaMemcpyHostToDevice, a->copy_stream) != cudaSuccess)
            return RF_ERR_CUDA;
    }
    if (cudaEventRecord(a->copied[first], a->copy_stream) != cudaSuccess ||
        cudaStreamWaitEvent(s, a->copied[first], 0) != cudaSuccess)
        return RF_ERR_CUDA;
    a->stats.bytes_copied += full + last_bytes;
    *first_slot = first;
    *base = dst;
    return RF_OK;
}

rf_status arena_release_run(rf_arena *a, cudaStream_t s, int first_slot, int n)
{
    for (int k = first_slot; k < first_slot + n; ++k)
        if (const rf_status st = arena_release(a, s, k)) return st;
    return RF_OK;
}

rf_status LaneFan::begin()
{
    if (on && cudaEventRecord(a->lane_start, s) != cudaSuccess) return RF_ERR_CUDA;
    return RF_OK;
}

rf_status LaneFan::stream(int64_t i, cudaStream_t *out)
{
    if (!on) {
        *out = s;
        return RF_OK;
    }
    const int l = (int)(i % rf_arena::kLanes);
    if (!(used & (1u << l))) {
        if (cudaStreamWaitEvent(a->lane[l], a->lane_start, 0) != cudaSuccess) return RF_ERR_CUDA;
        used |= 1u << l;
    }
    *out = a->lane[l];
    return RF_OK;
}

rf_status LaneFan::end()
{
    for (int l = 0; l < rf_arena::kLanes; ++l)
        if (used & (1u << l))
            if (cudaEventRecord(a->lane_done[l], a->lane[l]) != cudaSuccess ||
                cudaStreamWaitEvent(s, a->lane_done[l], 0) != cudaSuccess)
                return RF_ERR_CUDA;
    used = 0;
    return RF_OK;
}

}  // namespace rf

extern "C" {

rf_status rf_stream_plan(int fmt, int64_t in_dim, int64_t n_rows, int64_t block_rows, int depth,
                         size_t arena_bytes, int64_t *eff_rows, int64_t *n_blocks,
                         size_t *peak_bytes)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || n_rows < 0 || block_rows < 0 || depth < 0 ||
        depth > rf_arena::kMaxSlots - 1)
        return RF_ERR_INVALID_ARG;
    const int64_t rb = (in_dim / block_elems_of(fmt)) * (int64_t)block_bytes_of(fmt);
    const int64_t eff = arena_plan_rows(rb, n_rows, block_rows, depth, arena_bytes);
    if (eff < 0) return RF_ERR_ARENA_TOO_SMALL;
    const int64_t nblk = n_rows == 0 ? 0 : (n_rows + eff - 1) / eff;
    // Peak: the bytes of a block being multiplied plus the depth blocks
    // fetched ahead of it, maximised over the walk.
    size_t peak = 0;
    for (int64_t i = 0; i < nblk; ++i) {
        size_t held = 0;
        for (int64_t k = i; k < std::min(nblk, i + depth + 1); ++k)
            held += (size_t)(std::min(eff, n_rows - k * eff) * rb);
        peak = std::max(peak, held);
        if (i + depth + 1 >= nblk) break;   // later windows are subsets
    }
    if (eff_rows) *eff_rows = eff;
    if (n_blocks) *n_blocks = nblk;
    if (peak_bytes) *peak_bytes = peak;
    return RF_OK;
}

namespace {

// Makes `dev` current for the life of the guard and restores the previous
// device afterwards.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        ok = dev == prev || cudaSetDevice(dev) == cudaSuccess;
        if (!ok) cudaGetLastError();
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

rf_status create_arena(size_t bytes, rf_arena **out);

}  // namespace

rf_status rf_arena_create(size_t bytes, int device, rf_arena **out)
{
    if (!out || bytes == 0 || device < -1) return RF_ERR_INVALID_ARG;
    *out = nullptr;
    if (device >= 0) {
        int n = 0;
        if (cudaGetDeviceCount(&n) != cudaSuccess) {
            cudaGetLastError();
            return RF_ERR_CUDA;
        }
        if (device >= n) return RF_ERR_INVALID_ARG;
        DeviceGuard g(device);
        if (!g.ok) return RF_ERR_CUDA;
        return create_arena(bytes, out);
    }
    return create_arena(bytes, out);
}

namespace {

rf_status create_arena(size_t bytes, rf_arena **out)
{
    rf_arena *a = new (std::nothrow) rf_arena();
    if (!a) return RF_ERR_OOM;
    if (cudaGetDevice(&a->device) != cudaSuccess) {
        cudaGetLastError();
        delete a;
        return RF_ERR_CUDA;
    }
    // Slack for rounding every slot up to 256 bytes.
    a->bytes = bytes;
    a->alloc_bytes = bytes + 256 * rf_arena::kMaxSlots;
    if (cudaMalloc(&a->base, a->alloc_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete a;
        return RF_ERR_OOM;
    }
    if (cudaStreamCreateWithFlags(&a->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(a->base);
        delete a;
        return RF_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&a->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&a->lane_start, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        rf_arena_destroy(a);
        return RF_ERR_CUDA;
    }
    for (int l = 0; l < rf_arena::kLanes; ++l)
        if (cudaStreamCreateWithFlags(&a->lane[l], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&a->lane_done[l], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            rf_arena_destroy(a);
            return RF_ERR_CUDA;
        }
    if (cudaMallocHost(&a->route_host, sizeof(int32_t) * kMaxTerms) != cudaSuccess) {
        cudaGetLastError();
        a->route_host = nullptr;
        rf_arena_destroy(a);
        return RF_ERR_OOM;
    }
    for (int i = 0; i < rf_arena::kMaxSlots; ++i) {
        if (cudaEventCreateWithFlags(&a->copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&a->freed[i], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            rf_arena_destroy(a);
            return RF_ERR_CUDA;
        }
    }
    a->stats.arena_bytes = bytes;
    *out = a;
    return RF_OK;
}

}  // namespace

void rf_arena_destroy(rf_arena *a)
{
    if (!a) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(a->device);
    // Copies may still be writing the arena and GEMVs may still read it:
    // wait for both before freeing.  (Launches of captured graphs are the
    // caller's to finish.)
    if (a->copy_stream) cudaStreamSynchronize(a->copy_stream);
    for (int l = 0; l < rf_arena::kLanes; ++l)
        if (a->lane[l]) cudaStreamSynchronize(a->lane[l]);
    if (a->fork) cudaEventDestroy(a->fork);
    if (a->lane_start) cudaEventDestroy(a->lane_start);
    for (int l = 0; l < rf_arena::kLanes; ++l) {
        if (a->lane_done[l]) cudaEventDestroy(a->lane_done[l]);
        if (a->lane[l]) cudaStreamDestroy(a->lane[l]);
    }
    for (int i = 0; i < rf_arena::kMaxSlots; ++i) {
        if (a->freed[i]) {
            if (a->freed_recorded[i] && a->epoch == 0) cudaEventSynchronize(a->freed[i]);
            cudaEventDestroy(a->freed[i]);
        }
        if (a->copied[i]) cudaEventDestroy(a->copied[i]);
    }
    if (a->copy_stream) cudaStreamDestroy(a->copy_stream);
    if (a->base) cudaFree(a->base);
    if (a->route_host) cudaFreeHost(a->route_host);
    cudaSetDevice(prev);
    delete a;
}

rf_status rf_stream_stats(const rf_arena *a, rf_stream_stats_t *out)
{
    if (!a || !out) return RF_ERR_INVALID_ARG;
    *out = a->stats;
    return RF_OK;
}

rf_status rf_arena_wait(rf_arena *a, int timeout_ms)
{
    if (!a || timeout_ms < 0) return RF_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_CUDA;
    }
    if (cur != a->device) return RF_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(a->mu);
    // Marks at the end of the copy stream and of every lane stream, plus the
    // slot-free events of eager walks (readers on the callers' streams).
    cudaEvent_t marks[1 + rf_arena::kLanes];
    cudaStream_t streams[1 + rf_arena::kLanes] = {a->copy_stream};
    for (int l = 0; l < rf_arena::kLanes; ++l) streams[1 + l] = a->lane[l];
    int n_marks = 0;
    rf_status st = RF_OK;
    for (cudaStream_t cs : streams) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) {
            cudaGetLastError();
            st = RF_ERR_CUDA;
            break;
        }
        if (cap != cudaStreamCaptureStatusNone) {
            st = RF_ERR_INVALID_ARG;
            break;
        }
        if (cudaEventCreateWithFlags(&marks[n_marks], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            st = RF_ERR_CUDA;
            break;
        }
        ++n_marks;
        if (cudaEventRecord(marks[n_marks - 1], cs) != cudaSuccess) {
            cudaGetLastError();
            st = RF_ERR_CUDA;
            break;
        }
    }
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
    auto done = [&](cudaEvent_t e) -> rf_status {
        const cudaError_t q = cudaEventQuery(e);
        if (q == cudaSuccess) return RF_OK;
        if (q == cudaErrorNotReady) return RF_ERR_TIMEOUT;
        cudaGetLastError();
        return RF_ERR_CUDA;
    };
    while (st == RF_OK) {
        rf_status all = RF_OK;
        for (int i = 0; i < n_marks && all != RF_ERR_CUDA; ++i)
            if (const rf_status q = done(marks[i])) all = q;
        if (a->epoch == 0)
            for (int i = 0; i < rf_arena::kMaxSlots && all != RF_ERR_CUDA; ++i)
                if (a->freed_recorded[i])
                    if (const rf_status q = done(a->freed[i])) all = q;
        if (all != RF_ERR_TIMEOUT) {
            st = all;
            break;
        }
        if (std::chrono::steady_clock::now() >= deadline) {
            st = RF_ERR_TIMEOUT;
            break;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    for (int i = 0; i < n_marks; ++i) cudaEventDestroy(marks[i]);
    return st;
}

rf_status rf_arena_configure(rf_arena *a, int option, int value)
{
    if (!a || (value != 0 && value != 1)) return RF_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(a->mu);
    if (option == RF_ARENA_MERGE_RUNS)
        a->merge_runs = value != 0;
    else if (option == RF_ARENA_LANES)
        a->use_lanes = value != 0;
    else
        return RF_ERR_INVALID_ARG;
    return RF_OK;
}

rf_status rf_arena_inject_fault(rf_arena *a, int kind, int64_t block, int ms)
{
    if (!a || block < 0 || ms < 0 || ms > 10000) return RF_ERR_INVALID_ARG;
    if (kind != RF_FAULT_NONE && kind != RF_FAULT_COPY_FAIL && kind != RF_FAULT_COPY_STALL)
        return RF_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(a->mu);
    a->fault_kind = kind;
    a->fault_block = block;
    a->fault_ms = ms;
    return RF_OK;
}

rf_status rf_stream_linear(int fmt, const void *host_W, int64_t in_dim, int64_t row_start,
                           int64_t row_end, int64_t block_rows, int depth, rf_arena *a,
                           const float *x, float *y, void *stream)
{
    if (!fmt_ok(fmt)) return RF_ERR_UNSUPPORTED_FMT;
    if (!host_W || !a || !x || !y || in_dim <= 0 || in_dim % block_elems_of(fmt) != 0 || row_start < 0 ||
        row_end < row_start || block_rows < 0 || depth < 0 || depth > rf_arena::kMaxSlots - 1)
        return RF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(host_W) & 15u) != 0) return RF_ERR_MISALIGNED;
    if (const rf_status c = check_in_dim(fmt, in_dim, 1)) return c;
    {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess) {
            cudaGetLastError();
            return RF_ERR_CUDA;
        }
        if (cur != a->device) return RF_ERR_INVALID_ARG;
    }
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_W) != cudaSuccess) {
        cudaGetLastError();
        return RF_ERR_NOT_PINNED;
    }
    if (attr.type != cudaMemoryTypeHost) return RF_ERR_NOT_PINNED;
    const int64_t n_rows = row_end - row_start;
    const int64_t rb = (in_dim / block_elems_of(fmt)) * (int64_t)block_bytes_of(fmt);
    const int64_t eff = arena_plan_rows(rb, std::max<int64_t>(n_rows, 1), block_rows, depth, a->bytes);
    if (eff < 0) return RF_ERR_ARENA_TOO_SMALL;
    if (n_rows == 0) return RF_OK;
    if (eff > 0x7fffffffLL) return RF_ERR_TOO_LARGE;

    std::lock_guard<std::mutex> lock(a->mu);
    const int slots = depth + 1;
    const size_t stride = ((size_t)(eff * rb) + 255) & ~(size_t)255;
    if ((size_t)slots * stride > a->alloc_bytes) return RF_ERR_ARENA_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (const rf_status st = arena_prepare(a, s, slots, stride)) return st;
    const uint8_t *hw = static_cast<const uint8_t *>(host_W);
    size_t peak = 0;
    rf_stream_plan(fmt, in_dim, n_rows, block_rows, depth, a->bytes, nullptr, nullptr, &peak);

    // A walk whose blocks all fit in the ring at once (at most depth+1 of
    // them) needs no slot reuse: its blocks go over the link as one copy and
    // through one launch (each block its own window: with packed slots they
    // are consecutive rows of one matrix and merge into one window; else at
    // most 16 distinct slot bases, the tensor maps a launch holds).  Per-block
    // copies and launches would only add their fixed costs.
    const int64_t nblk = (n_rows + eff - 1) / eff;
    const bool packed = stride == (size_t)(eff * rb);
    // A one-shot injected fault, taken by this walk.
    const int fault = a->fault_kind;
    const int64_t fault_at = a->fault_block;
    const int fault_ms = a->fault_ms;
    a->fault_kind = RF_FAULT_NONE;
    if (nblk > 1 && nblk <= slots && (packed || nblk <= 16) && fault == RF_FAULT_NONE &&
        a->merge_runs) {
        int first = 0;
        uint8_t *base = nullptr;
        const int64_t last_rows = n_rows - (nblk - 1) * eff;
        if (const rf_status st = arena_fetch_run(a, s, hw + row_start * rb, (size_t)(eff * rb),
                                                 (int)nblk, (size_t)(last_rows * rb), &first, &base))
            return st;
        static thread_local Job run_jobs[rf_arena::kMaxSlots];
        for (int64_t i = 0; i < nblk; ++i) {
            Job &J = run_jobs[i];
            std::memset(&J, 0, sizeof(J));
            J.term[0] = Term{packed ? base : base + (size_t)i * stride, 0, -1, 0, 0};
            J.row0 = packed ? i * eff : 0;
            J.y = y + i * eff;
            J.n_rows = (int32_t)(i + 1 < nblk ? eff : last_rows);
            J.n_terms = 1;
            J.combine = kCombineSum;
        }
        LaunchDesc d;
        d.fmt = fmt;
        d.in_dim = in_dim;
        d.jobs = run_jobs;
        d.n_jobs = (int)nblk;
        d.x[0] = x;
        d.n_x = 1;
        if (const rf_status st = launch_rowwin(d, s)) return st;
        if (const rf_status st = arena_release_run(a, s, first, (int)nblk)) return st;
        a->stats.calls += 1;
        a->stats.blocks += (uint64_t)nblk;
        a->stats.peak_bytes = std::max<uint64_t>(a->stats.peak_bytes, peak);
        a->stats.slot_bytes = stride;
        a->stats.slots = slots;
        a->stats.last_block_rows = (int32_t)eff;
        return RF_OK;
    }

    // Blocks run side by side on the lane streams (their rows are disjoint)
    // when they are small (at most 1 MiB: a block's GEMV, a few CTAs, then
    // takes longer than its copy) and the walk has at least two blocks per
    // lane (a fan-out costs a fork and a join per walk, which a short walk
    // does not earn back; in a CUDA graph each is a cross-branch dependency).
    LaneFan fan{a, s,
                a->use_lanes && eff * rb <= (int64_t)(1 << 20) &&
                    (n_rows + eff - 1) / eff >= 2 * rf_arena::kLanes};
    if (const rf_status st = fan.begin()) return st;
    int64_t blocks = 0;
    rf_status err = RF_OK;
    for (int64_t r0 = row_start; r0 < row_end; r0 += eff) {
        const int64_t nr = std::min(eff, row_end - r0);
        int slot = 0;
        uint8_t *dst = nullptr;
        cudaStream_t cs = s;
        if ((err = fan.stream(blocks, &cs)) != RF_OK) break;
        if (fault != RF_FAULT_NONE && blocks == fault_at) {
            if (fault == RF_FAULT_COPY_FAIL) {   // as if this block's copy had failed
                err = RF_ERR_CUDA;
                break;
            }
            if (cudaLaunchHostFunc(a->copy_stream, stall_host, reinterpret_cast<void *>(
                                                                    (intptr_t)fault_ms)) !=
                cudaSuccess) {
                cudaGetLastError();
                err = RF_ERR_CUDA;
                break;
            }
        }
        if ((err = arena_fetch(a, cs, hw + r0 * rb, (size_t)(nr * rb), &slot, &dst)) != RF_OK)
            break;
        Job J;
        std::memset(&J, 0, sizeof(J));
        J.term[0] = Term{dst, 0, -1, 0, 0};
        J.y = y + (r0 - row_start);
        J.n_rows = (int32_t)nr;
        J.n_terms = 1;
        J.combine = kCombineSum;
        LaunchDesc d;
        d.fmt = fmt;
        d.in_dim = in_dim;
        d.jobs = &J;
        d.n_jobs = 1;
        d.x[0] = x;
        d.n_x = 1;
        err = launch_rowwin(d, cs);
        // Retire: the slot is free once this GEMV has run (or, when the launch
        // failed, once the work before it on the stream has).
        const rf_status rel = arena_release(a, cs, slot);
        if (err != RF_OK) break;
        if ((err = rel) != RF_OK) break;
        ++blocks;
    }
    // On an error the walk stops enqueueing; the blocks already enqueued keep
    // their slots' release events, and the lanes rejoin the caller's stream,
    // so later work on `stream` and on the arena stays ordered after them.
    const rf_status joined = fan.end();
    if (err == RF_OK) err = joined;
    a->stats.blocks += (uint64_t)blocks;
    if (err != RF_OK) return err;
    a->stats.calls += 1;
    a->stats.peak_bytes = std::max<uint64_t>(a->stats.peak_bytes, peak);
    a->stats.slot_bytes = stride;
    a->stats.slots = slots;
    a->stats.last_block_rows = (int32_t)eff;
    return RF_OK;
}

}  // extern "C"
