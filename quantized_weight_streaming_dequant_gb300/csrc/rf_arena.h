// rf_arena.h -- the bounded device arena shared by the host-streamed walks
// (rf_stream_linear, rf_moe_ffn_streamed).
//
// neurostream, "How it works" 3 and 6: a prefetcher keeps `depth` blocks in
// flight, every in-flight block holds a reservation in a bounded arena, and
// allocation waits until a block retires.  Here the arena is one device
// allocation cut into slots; the prefetcher is a copy stream; a block's copy
// waits (stream-ordered, never on the host) for the event recorded after the
// last launch that read its slot.
#pragma once

#include <cstdint>
#include <mutex>

#include "rf_internal.h"

struct rf_arena {
    static constexpr int kMaxSlots = 65;   // depth <= 64
    uint8_t *base = nullptr;
    size_t bytes = 0;          // capacity promised to the caller
    size_t alloc_bytes = 0;    // allocation (capacity + alignment slack)
    int device = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied[kMaxSlots] = {};
    cudaEvent_t freed[kMaxSlots] = {};
    bool freed_recorded[kMaxSlots] = {};
    cudaEvent_t fork = nullptr;       // joins the copy stream to the caller's stream
    unsigned long long epoch = 0;     // 0: eager; else the id of the capture
    int next_slot = 0;
    int last_slots = 0;
    size_t last_stride = 0;
    rf_stream_stats_t stats = {};
    bool merge_runs = true;           // RF_ARENA_MERGE_RUNS
    bool use_lanes = true;            // RF_ARENA_LANES
    // One-shot host-side failure injection (rf_arena_inject_fault).
    int fault_kind = 0;
    int64_t fault_block = 0;
    int fault_ms = 0;
    int32_t *route_host = nullptr;    // page-locked: routing ids read back for planning
    // Lane streams: the launches of one walk's blocks go round-robin to them,
    // so that blocks whose copies have landed run side by side.
    static constexpr int kLanes = 4;
    cudaStream_t lane[kLanes] = {};
    cudaEvent_t lane_start = nullptr;         // the caller's stream at the walk's start
    cudaEvent_t lane_done[kLanes] = {};       // a lane's last launch of the walk
    std::mutex mu;
};

namespace rf {

// Block rows for walking n_rows rows of row_bytes bytes in blocks of
// block_rows (0 = all) with depth+1 slots of the arena: the request, shrunk
// until depth+1 blocks fit; -1 if one row does not.
int64_t arena_plan_rows(int64_t row_bytes, int64_t n_rows, int64_t block_rows, int depth,
                        size_t arena_bytes);

// Starts a walk on `s` with `slots` slots of `stride` bytes (caller holds
// a->mu): joins the copy stream to `s` when the capture epoch changed, and
// orders the first copies after every reader of the old slots when the slot
// layout changed.
rf_status arena_prepare(rf_arena *a, cudaStream_t s, int slots, size_t stride);

// Takes the next slot, enqueues the copy of `bytes` bytes from page-locked
// host memory `src` into it on the copy stream (after the slot's previous
// reader), and makes `s` wait for the copy.  *slot_out / *dst_out receive the
// slot and its device address.
rf_status arena_fetch(rf_arena *a, cudaStream_t s, const void *src, size_t bytes, int *slot_out,
                      uint8_t **dst_out);

// Every launch that reads `slot` is enqueued on `s`: the slot is free once
// they have run.
rf_status arena_release(rf_arena *a, cudaStream_t s, int slot);

// A walk whose n blocks (n <= slots) all fit in the ring at once: takes n
// consecutive slots (from the next slot when they do not wrap, else from
// slot 0), copies the blocks -- contiguous host rows: n-1 blocks of
// block_bytes, then last_bytes -- with one copy (two when the slot pitch
// exceeds the block) after the slots' previous readers, and makes `s` wait
// for it.  Block i lands at *base + i * slot pitch; *first_slot is the first
// slot taken.
rf_status arena_fetch_run(rf_arena *a, cudaStream_t s, const void *src, size_t block_bytes,
                          int n, size_t last_bytes, int *first_slot, uint8_t **base);

// Releases the n slots from first_slot once the launches on `s` have run.
rf_status arena_release_run(rf_arena *a, cudaStream_t s, int first_slot, int n);

// Fan-out of a walk's launches over the lane streams.  begin() records the
// caller's stream; stream(i) is the stream for the walk's i-th block (a lane,
// which first waits for the caller's stream); end() makes the caller's stream
// wait for every lane used.  With `on` false everything stays on the
// caller's stream.
struct LaneFan {
    rf_arena *a;
    cudaStream_t s;
    bool on;
    unsigned used = 0;
    rf_status begin();
    rf_status stream(int64_t i, cudaStream_t *out);
    rf_status end();
};

}  // namespace rf
