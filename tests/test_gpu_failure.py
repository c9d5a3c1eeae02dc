"""Failure paths on the GPU, made without faulting it (neurostream, "Bugs
worth knowing about": a stalled prefetcher must neither deadlock nor
poison the arena).

* A kernel's bounded wait: a test hook makes one launch withhold one
  stage's copy (the GEMV's producer warp, a warp of a GEMV whose rows take
  per-row bulk copies, or the prefill GEMM's activation copier), with the
  wait limit cut to 1 ms.  The launch
  must end quickly with RF_ERR_TIMEOUT in the device status word and nothing
  in flight, and the next call on the device must be correct.
* The host streamer: an injected copy failure at block k stops the walk,
  returns RF_ERR_CUDA, keeps the k blocks already enqueued correct and
  leaves every slot reusable; an injected copy stall makes the host wait
  with a deadline (rf_arena_wait) time out, then succeed.
"""
import time

import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import assert_gemv_close, dev_tensor, gemv_tol

pytestmark = pytest.mark.gpu

TIMEOUT = 6


@pytest.fixture(scope="module")
def rf():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import quantized_weight_streaming_dequant_gb300 as m
    from quantized_weight_streaming_dequant_gb300 import build
    build.build()
    m.lib()
    yield m
    m.debug_arm_wait_fault(0)
    assert m.device_status() == m.OK


def bits(t):
    return t.detach().cpu().numpy().astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("rows", [4096, 64 * 152 * 2])   # static, and ticket-scheduled groups
def test_kernel_wait_timeout_ends_launch_and_device_recovers(rf, rows):
    import torch
    fmt, in_dim = syn.Q4_0, 4096   # 2,304-byte rows: tensor copies, producer warp
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=300)
    x_np = syn.normal_f32(in_dim, 301)
    W, x = dev_tensor(W_np), dev_tensor(x_np)
    y_ok = rf.gemv(fmt, W, 0, rows, in_dim, x)
    assert rf.device_status() == rf.OK
    ref = oracle.gemv(fmt, W_np, 0, rows, in_dim, x_np)
    assert_gemv_close(y_ok.cpu().numpy(), ref, gemv_tol(fmt, W_np, 0, rows, in_dim, x_np))

    rf.debug_arm_wait_fault(1000)    # one-shot: 1 ms limit, one stage never filled
    t0 = time.perf_counter()
    rf.gemv(fmt, W, 0, rows, in_dim, x)
    status = rf.device_status()      # synchronizes the device
    dt = time.perf_counter() - t0
    assert status == TIMEOUT
    assert dt < 1.0, f"the failed launch took {dt:.3f} s: waits did not end early"
    assert rf.device_status() == rf.OK   # read and cleared

    # the device and the ticket slots are clean: later launches are correct
    for _ in range(3):
        y = rf.gemv(fmt, W, 0, rows, in_dim, x)
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), bits(y_ok))
    assert rf.device_status() == rf.OK


def test_per_lane_bulk_wait_timeout_ends_launch_and_device_recovers(rf):
    """The same hook on a launch whose rows take per-row bulk copies (Q6_K
    rows of 9,030 bytes): warp 0 of the first CTA never arms its first
    stage, gives up after 1 ms, and every warp drains the stages it armed;
    the next calls give the bits of the call before the fault."""
    import torch
    fmt, rows, in_dim = syn.Q6_K, 512, 11008
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=330)
    x_np = syn.normal_f32(in_dim, 331)
    W, x = dev_tensor(W_np), dev_tensor(x_np)
    y_ok = rf.gemv(fmt, W, 0, rows, in_dim, x)
    assert rf.device_status() == rf.OK
    ref = oracle.gemv(fmt, W_np, 0, rows, in_dim, x_np)
    assert_gemv_close(y_ok.cpu().numpy(), ref, gemv_tol(fmt, W_np, 0, rows, in_dim, x_np))

    rf.debug_arm_wait_fault(1000)
    t0 = time.perf_counter()
    rf.gemv(fmt, W, 0, rows, in_dim, x)
    status = rf.device_status()
    dt = time.perf_counter() - t0
    assert status == TIMEOUT
    assert dt < 1.0, f"the failed launch took {dt:.3f} s: waits did not end early"
    assert rf.device_status() == rf.OK

    for _ in range(3):
        y = rf.gemv(fmt, W, 0, rows, in_dim, x)
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), bits(y_ok))
    assert rf.device_status() == rf.OK


def test_gemm_wait_timeout_ends_launch_and_device_recovers(rf):
    """The prefill GEMM under the same hook: CTA (0, 0) never copies slice 1's
    activation tile, its decoders give up after 1 ms, every role stops,
    drains what it issued and frees its tensor memory; the next calls are
    bit-identical to the call before the fault."""
    import torch
    fmt, rows, in_dim, n_tok = syn.Q4_0, 384, 1024, 70
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=310)
    X_np = np.stack([syn.normal_f32(in_dim, 320 + t) for t in range(n_tok)])
    W, X = dev_tensor(W_np), dev_tensor(X_np)
    Y_ok = rf.gemm(fmt, W, 0, rows, in_dim, X)
    assert rf.device_status() == rf.OK
    for t in (0, n_tok - 1):
        ref = oracle.gemv(fmt, W_np, 0, rows, in_dim, X_np[t])
        assert_gemv_close(Y_ok[t].cpu().numpy(), ref,
                          gemv_tol(fmt, W_np, 0, rows, in_dim, X_np[t]), f"token {t}")

    rf.debug_arm_wait_fault(1000)
    t0 = time.perf_counter()
    rf.gemm(fmt, W, 0, rows, in_dim, X)
    status = rf.device_status()
    dt = time.perf_counter() - t0
    assert status == TIMEOUT
    assert dt < 1.0, f"the failed launch took {dt:.3f} s: waits did not end early"
    assert rf.device_status() == rf.OK

    for _ in range(3):
        Y = rf.gemm(fmt, W, 0, rows, in_dim, X)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), bits(Y_ok))
    assert rf.device_status() == rf.OK


def test_stream_copy_failure_stops_walk_and_keeps_arena_usable(rf):
    import torch
    fmt, rows, in_dim, br, depth = syn.Q8_0, 512, 2048, 32, 2
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=310)
    x_np = syn.normal_f32(in_dim, 311)
    host = torch.from_numpy(W_np).pin_memory()
    x = dev_tensor(x_np)
    y_res = rf.gemv(fmt, dev_tensor(W_np), 0, rows, in_dim, x)
    arena = rf.Arena(8 << 20)
    try:
        k = 5
        y = torch.full((rows,), float("nan"), device="cuda")
        arena.inject_fault(rf.FAULT_COPY_FAIL, k)
        with pytest.raises(rf.RFError) as e:
            arena.stream_linear(fmt, host, in_dim, 0, rows, br, depth, x, y)
        assert e.value.code == 5
        assert arena.wait(5000) == rf.OK        # what was enqueued drains
        torch.cuda.synchronize()
        assert arena.stats()["blocks"] == k and arena.stats()["calls"] == 0
        # the k blocks enqueued before the failure ran, on the caller's stream
        assert np.array_equal(bits(y[:k * br]), bits(y_res[:k * br]))
        assert bool(torch.isnan(y[k * br:]).all())
        # every slot is reusable: the next walks are correct, blocks and whole
        for block_rows in (br, 128, 0):
            y2 = arena.stream_linear(fmt, host, in_dim, 0, rows, block_rows, depth, x)
            torch.cuda.synchronize()
            assert np.array_equal(bits(y2), bits(y_res)), block_rows
        ref = oracle.gemv(fmt, W_np, 0, rows, in_dim, x_np)
        assert_gemv_close(y2.cpu().numpy(), ref, gemv_tol(fmt, W_np, 0, rows, in_dim, x_np))
    finally:
        torch.cuda.synchronize()
        arena.close()


def test_stream_copy_stall_host_wait_deadline(rf):
    import torch
    fmt, rows, in_dim, br, depth = syn.Q4_0, 1024, 4096, 128, 2
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=320)
    host = torch.from_numpy(W_np).pin_memory()
    x = dev_tensor(syn.normal_f32(in_dim, 321))
    y_res = rf.gemv(fmt, dev_tensor(W_np), 0, rows, in_dim, x)
    torch.cuda.synchronize()
    arena = rf.Arena(8 << 20)
    try:
        arena.inject_fault(rf.FAULT_COPY_STALL, 1, 400)
        t0 = time.perf_counter()
        y = arena.stream_linear(fmt, host, in_dim, 0, rows, br, depth, x)
        assert time.perf_counter() - t0 < 0.3     # enqueueing never blocks the host
        assert arena.wait(20) == TIMEOUT          # the stalled copy is still pending
        assert arena.wait(10000) == rf.OK
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), bits(y_res))
        # injection is one-shot: the next walk takes the fast path again
        t0 = time.perf_counter()
        arena.stream_linear(fmt, host, in_dim, 0, rows, br, depth, x, y)
        assert arena.wait(10000) == rf.OK
        assert time.perf_counter() - t0 < 0.3
    finally:
        torch.cuda.synchronize()
        arena.close()


def test_arena_options_keep_bits(rf):
    """Turning off the one-copy merge of walks that fit the ring, or the lane
    streams, changes how blocks are copied and launched, not the result."""
    import torch
    fmt, rows, in_dim = syn.Q8_0, 512, 2048
    W_np = syn.quant_matrix(fmt, rows, in_dim, seed=330)
    host = torch.from_numpy(W_np).pin_memory()
    x = dev_tensor(syn.normal_f32(in_dim, 331))
    y_res = rf.gemv(fmt, dev_tensor(W_np), 0, rows, in_dim, x)
    arena = rf.Arena(8 << 20)
    try:
        for merge in (True, False):
            for lanes in (True, False):
                arena.configure(rf.ARENA_MERGE_RUNS, merge)
                arena.configure(rf.ARENA_LANES, lanes)
                for br, depth in ((128, 4), (32, 8), (16, 2)):
                    b0 = arena.stats()["blocks"]
                    y = arena.stream_linear(fmt, host, in_dim, 0, rows, br, depth, x)
                    torch.cuda.synchronize()
                    assert np.array_equal(bits(y), bits(y_res)), (merge, lanes, br, depth)
                    assert arena.stats()["blocks"] - b0 == rows // br
    finally:
        torch.cuda.synchronize()
        arena.close()
