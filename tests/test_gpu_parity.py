"""GPU parity: every CUDA entry point against the CPU oracle on the same
seeded inputs.  Dequantized values must be bit-exact; GEMV rows must satisfy
|y_gpu - y_ref| <= 1e-3 * ||W_r||_2 * ||x||_2; row results must not depend
on the window, the batch or the streaming block size (bit-identical)."""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import (assert_gemv_close, check_moe, dev_tensor, ffn_reference, gemv_tol,
                         moe_reference)

pytestmark = pytest.mark.gpu

FMTS = [syn.Q8_0, syn.Q4_0, syn.MXFP4]


@pytest.fixture(scope="module")
def rf():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import quantized_weight_streaming_dequant_gb300 as m
    from quantized_weight_streaming_dequant_gb300 import build
    build.build()
    m.lib()
    yield m
    assert m.device_status() == m.OK


def bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------- dequantize

def test_dequantize_hand_blocks_bit_exact(rf, golden_dir):
    from test_oracle_pins import parse_blocks
    for name, fmt, raw, values in parse_blocks(golden_dir):
        W = dev_tensor(np.frombuffer(raw, np.uint8))
        got = rf.dequantize(fmt, W, 1).cpu().numpy()
        assert np.array_equal(bits(got), bits(np.array(values, np.float32))), name


@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_random_bit_exact(rf, fmt):
    n = 20_011
    W = syn.quant_matrix(fmt, 1, 32 * n, seed=77)
    # add edge scales: fp16 subnormal/zero/negative, E8M0 extremes
    blk = W.reshape(n, syn.block_bytes(fmt))
    if fmt == syn.MXFP4:
        blk[:8, 0] = [0, 1, 2, 126, 127, 128, 200, 254]
    else:
        blk[:6, 0:2] = np.array([[0, 0], [1, 0], [0xff, 0x03], [0, 0x80], [0, 0xbc], [0xff, 0x7b]],
                                np.uint8)
    got = rf.dequantize(fmt, dev_tensor(W), n).cpu().numpy()
    ref = oracle.dequantize(fmt, W, n)
    assert np.array_equal(bits(got), bits(ref))


# ------------------------------------------------------------------ GEMV

SHAPES = [  # (rows, in_dim, window) -- several 32-row groups, ragged tails,
    (1000, 4096, (0, 1000)),     # 16-byte aligned rows (static decode)
    (1000, 2880, (3, 997)),      # unaligned rows (generic decode)
    (257, 11008, (0, 257)),
    (70, 32, (1, 70)),           # one block per row
    (300, 96, (5, 299)),         # nb = 3 < warps
    (64, 24576, (0, 64)),        # the host-streamed FFN's down width
    (100, 3104, (2, 99)),        # whole-group staging with one CTA per SM
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,in_dim,win", SHAPES)
def test_gemv_parity(rf, fmt, rows, in_dim, win):
    W = syn.quant_matrix(fmt, rows, in_dim, seed=rows + in_dim + fmt)
    x = syn.normal_f32(in_dim, seed=in_dim)
    r0, r1 = win
    y = rf.gemv(fmt, dev_tensor(W), r0, r1, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(fmt, W, r0, r1, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(fmt, W, r0, r1, in_dim, x), f"fmt {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_x_with_wide_dynamic_range(rf, fmt):
    rows, in_dim = 96, 1024
    W = syn.quant_matrix(fmt, rows, in_dim, seed=3)
    x = syn.normal_f32(in_dim, seed=4)
    x[::7] *= 1e6
    x[3::11] *= 1e-9
    x[64:96] = 0.0          # an all-zero activation block
    y = rf.gemv(fmt, dev_tensor(W), 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(fmt, W, 0, rows, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(fmt, W, 0, rows, in_dim, x), "dynamic range")


@pytest.mark.parametrize("fmt", FMTS + [syn.Q4_K])
def test_gemv_activation_rounding_aligned_with_weights(rf, fmt):
    """The kernel turns each 32-element activation block into fixed-point
    digits X = rint(x * 2^s), |X| < 2^15, s set by the block maximum.  Here
    every block's maximum is exactly 1.0 (so s = 14) and every other x_j sits
    (0.5 -+ 2^-8) units of 2^-14 off the grid, on the side that makes its
    rounding error carry the sign of w_j: the errors add up instead of
    cancelling.  The measured error must stay within the stated bound
    sqrt(32) * 2^-15 * ||W_r|| * ||x|| (and so within 1e-3 * ||W_r|| * ||x||),
    and must be the aligned error the rounding predicts (at least half of
    2^-14 * (0.5 - 2^-8) * sum_j |w_j|), which shows that the rounding, and
    not something coarser or finer, is what the kernel does."""
    rows, in_dim = 96, 1024
    W = syn.quant_matrix(fmt, rows, in_dim, seed=130 + fmt)
    dense = oracle.dequantize(fmt, W).reshape(rows, in_dim).astype(np.float64)
    rng = np.random.default_rng(131)
    for r in (0, 37, 95):
        w = dense[r]
        sig = rng.choice([-1.0, 1.0], size=in_dim)
        n = rng.integers(1 << 13, (1 << 14) - 1, size=in_dim).astype(np.float64)
        up = np.where(sig * np.sign(w) > 0, 1.0, -1.0)   # round away or toward zero
        x = sig * (n + 0.5 + up * 2.0 ** -8) * 2.0 ** -14
        x[::32] = 1.0                                      # each block's maximum
        x = x.astype(np.float32)
        assert np.all(x.astype(np.float64) * 2 ** 14 % 1 != 0.5)   # no ties
        y = rf.gemv(fmt, dev_tensor(W), r, r + 1, in_dim, dev_tensor(x)).cpu().numpy()
        ref = oracle.gemv(fmt, W, r, r + 1, in_dim, x)
        err = abs(float(y[0]) - float(ref[0]))
        nw, nx = float(np.linalg.norm(w)), float(np.linalg.norm(x.astype(np.float64)))
        bound = math.sqrt(32) * 2.0 ** -15 * nw * nx
        assert err <= bound and err <= 1e-3 * nw * nx, (r, err, bound)
        aligned = 2.0 ** -14 * (0.5 - 2.0 ** -8) * float(np.abs(w).sum())
        assert err >= 0.5 * aligned, (r, err, aligned)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_one_hot_exact(rf, fmt):
    rows, in_dim = 65, 512
    W = syn.quant_matrix(fmt, rows, in_dim, seed=9)
    D = oracle.dequantize(fmt, W).reshape(rows, in_dim)
    Wd = dev_tensor(W)
    for i in (0, 31, 32, 200, 511):
        x = np.zeros(in_dim, np.float32)
        x[i] = 1.0
        y = rf.gemv(fmt, Wd, 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
        assert np.array_equal(y, D[:, i])      # == (signed zeros compare equal)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("in_dim", [2880, 4096])
def test_window_and_batch_invariance_bit_exact(rf, fmt, in_dim):
    import torch
    rows = 700
    W = syn.quant_matrix(fmt, rows, in_dim, seed=5)
    x = dev_tensor(syn.normal_f32(in_dim, 6))
    Wd = dev_tensor(W)
    full = rf.gemv(fmt, Wd, 0, rows, in_dim, x).cpu().numpy()
    cuts = [0, 1, 33, 100, 101, 450, 699, 700]
    parts = [rf.gemv(fmt, Wd, a, b, in_dim, x).cpu().numpy() for a, b in zip(cuts, cuts[1:])]
    assert np.array_equal(bits(np.concatenate(parts)), bits(full))
    outs = [torch.empty(b - a, device="cuda") for a, b in zip(cuts, cuts[1:])]
    rf.gemv_batch(fmt, in_dim, [(Wd, a, b, x, o) for (a, b), o in zip(zip(cuts, cuts[1:]), outs)])
    assert np.array_equal(bits(torch.cat(outs).cpu().numpy()), bits(full))


def test_gemv_batch_distinct_x(rf):
    import torch
    fmt, in_dim = syn.Q4_0, 1024
    mats = [syn.quant_matrix(fmt, 100 + 13 * i, in_dim, seed=i) for i in range(5)]
    xs = [syn.normal_f32(in_dim, 10 + i) for i in range(5)]
    outs = [torch.empty(m.shape[0], device="cuda") for m in mats]
    rf.gemv_batch(fmt, in_dim, [(dev_tensor(m), 0, m.shape[0], dev_tensor(x), o)
                                for m, x, o in zip(mats, xs, outs)])
    for m, x, o in zip(mats, xs, outs):
        ref = oracle.gemv(fmt, m, 0, m.shape[0], in_dim, x)
        assert_gemv_close(o.cpu().numpy(), ref, gemv_tol(fmt, m, 0, m.shape[0], in_dim, x))


def test_gemv_errors(rf):
    import torch
    W = dev_tensor(syn.quant_matrix(syn.Q8_0, 4, 64, 1))
    x = torch.zeros(64, device="cuda")
    with pytest.raises(rf.RFError) as e:
        rf.gemv(syn.Q8_0, W, 0, 4, 48, x)
    assert e.value.code == 1
    with pytest.raises(rf.RFError) as e:
        rf.gemv(syn.Q8_0, W, 0, 4, rf.max_in_dim(syn.Q8_0) + 32, x)
    assert e.value.code == 9
    assert rf.gemv(syn.Q8_0, W, 2, 2, 64, x).numel() == 0


# --------------------------------------------------------- activations

def test_swiglu_and_gelu_kernels(rf):
    z = syn.normal_f32(10_000, 1) * 4
    u = syn.normal_f32(10_000, 2)
    h = rf.swiglu(dev_tensor(z), dev_tensor(u)).cpu().numpy().astype(np.float64)
    ref = oracle.silu_vec(z) * u
    assert np.allclose(h, ref, rtol=1e-5, atol=1e-6)
    g = rf.gelu(dev_tensor(z)).cpu().numpy().astype(np.float64)
    assert np.allclose(g, oracle.gelu_vec(z), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------------ FFN

@pytest.mark.parametrize("fmt,n_ff,n_embd", [(syn.Q4_0, 1376, 512), (syn.MXFP4, 2880, 2880),
                                             (syn.Q8_0, 672, 1056)])
def test_ffn_swiglu_parity(rf, fmt, n_ff, n_embd):
    G = syn.quant_matrix(fmt, n_ff, n_embd, 21)
    U = syn.quant_matrix(fmt, n_ff, n_embd, 22)
    D = syn.quant_matrix(fmt, n_embd, n_ff, 23)
    x = syn.normal_f32(n_embd, 24)
    y, h = rf.ffn_swiglu(fmt, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                         dev_tensor(x))
    y, h = y.cpu().numpy(), h.cpu().numpy()
    # the oracle's own chain, with bounds derived from the per-GEMV tolerance
    ref = ffn_reference(fmt, G, U, D, n_ff, n_embd, x)
    assert_gemv_close(h, ref["h"], ref["tol_h"], "h")
    assert_gemv_close(y, ref["y"], ref["tol_y"], "y")
    # with the digit hand-off workspace: the same bits (the digits gate/up
    # writes are the ones down would build from h)
    ws = rf.ffn_workspace(n_ff, "cuda")
    for _ in range(2):
        y2, h2 = rf.ffn_swiglu(fmt, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                               dev_tensor(x), workspace=ws)
        assert np.array_equal(h2.cpu().numpy().view(np.uint32), h.view(np.uint32))
        assert np.array_equal(y2.cpu().numpy().view(np.uint32), y.view(np.uint32))


# ------------------------------------------------------------ streaming

@pytest.mark.parametrize("fmt", FMTS)
def test_stream_linear_bit_identical_to_resident(rf, fmt):
    import torch
    rows, in_dim = 900, 2880 if fmt == syn.MXFP4 else 2048
    W = syn.quant_matrix(fmt, rows, in_dim, seed=31)
    x = dev_tensor(syn.normal_f32(in_dim, 32))
    resident = rf.gemv(fmt, dev_tensor(W), 7, rows, in_dim, x).cpu().numpy()
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(64 * rf.row_bytes(fmt, in_dim))
    try:
        calls = 0
        for block_rows, depth in [(1, 0), (7, 1), (32, 4), (128, 1), (0, 0), (0, 3)]:
            y = arena.stream_linear(fmt, host, in_dim, 7, rows, block_rows, depth, x)
            calls += 1
            assert np.array_equal(bits(y.cpu().numpy()), bits(resident)), (block_rows, depth)
            st = arena.stats()
            eff, nblk, peak = rf.stream_plan(fmt, in_dim, rows - 7, block_rows, depth,
                                             arena.nbytes)
            assert st["last_block_rows"] == eff and st["slots"] == depth + 1
            assert st["calls"] == calls
        st = arena.stats()
        assert st["bytes_copied"] >= 6 * (rows - 7) * rf.row_bytes(fmt, in_dim)
        assert st["blocks"] > 893 and st["peak_bytes"] <= arena.nbytes
    finally:
        arena.close()


def test_stream_linear_captured_in_cuda_graph(rf):
    """Walks captured into a CUDA graph (two calls with different slot layouts
    in one capture) replay to the same bits as the eager walk, several times
    in a row, and eager use of the arena works again afterwards."""
    import torch
    fmt, rows, in_dim = syn.Q8_0, 1000, 1024
    W = syn.quant_matrix(fmt, rows, in_dim, seed=91)
    xd = dev_tensor(syn.normal_f32(in_dim, 92))
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(400 * rf.row_bytes(fmt, in_dim))
    try:
        eager = arena.stream_linear(fmt, host, in_dim, 0, rows, 96, 3, xd).cpu().numpy()
        ref = oracle.gemv(fmt, W, 0, rows, in_dim, syn.normal_f32(in_dim, 92))
        assert_gemv_close(eager, ref, gemv_tol(fmt, W, 0, rows, in_dim, syn.normal_f32(in_dim, 92)))
        s = torch.cuda.Stream()
        yg = torch.full((rows,), float("nan"), device="cuda")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            # 10 blocks (fanned out over the lane streams), then 4 (one stream)
            arena.stream_linear(fmt, host, in_dim, 0, 600, 64, 3, xd, yg[:600], stream=s)
            arena.stream_linear(fmt, host, in_dim, 600, rows, 128, 2, xd, yg[600:], stream=s)
        for rep in range(3):
            yg.fill_(float("nan"))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(bits(yg.cpu().numpy()), bits(eager)), rep
        again = arena.stream_linear(fmt, host, in_dim, 0, rows, 64, 4, xd).cpu().numpy()
        assert np.array_equal(bits(again), bits(eager))
        del g
    finally:
        torch.cuda.synchronize()
        arena.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_stream_linear_whole_walk_in_ring(rf, fmt):
    """Walks whose blocks all fit in the ring at once take one copy and one
    launch: packed slots (128-row blocks, 7 blocks in 8 slots) and slots with
    a pitch above the block (7-row blocks, 15 blocks in 16 slots); bit-exact
    against the resident GEMV, eager twice in a row and replayed from a graph."""
    import torch
    in_dim = 2880 if fmt == syn.MXFP4 else 2048
    W = syn.quant_matrix(fmt, 900, in_dim, seed=41)
    x = dev_tensor(syn.normal_f32(in_dim, 42))
    Wd = dev_tensor(W)
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(256 << 20)
    s = torch.cuda.Stream()
    try:
        for r0, r1, block_rows, depth in ((7, 900, 128, 7), (3, 103, 7, 15)):
            want = rf.gemv(fmt, Wd, r0, r1, in_dim, x).cpu().numpy()
            copied0 = arena.stats()["bytes_copied"]
            for _ in range(2):
                y = arena.stream_linear(fmt, host, in_dim, r0, r1, block_rows, depth, x)
                assert np.array_equal(bits(y.cpu().numpy()), bits(want)), (block_rows, depth)
            st = arena.stats()
            assert st["last_block_rows"] == block_rows and st["slots"] == depth + 1
            assert st["bytes_copied"] - copied0 == 2 * (r1 - r0) * rf.row_bytes(fmt, in_dim)
            yg = torch.full((r1 - r0,), float("nan"), device="cuda")
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                arena.stream_linear(fmt, host, in_dim, r0, r1, block_rows, depth, x, yg, stream=s)
            for _ in range(2):
                yg.fill_(float("nan"))
                torch.cuda.synchronize()
                with torch.cuda.stream(s):
                    g.replay()
                torch.cuda.synchronize()
                assert np.array_equal(bits(yg.cpu().numpy()), bits(want)), (block_rows, "graph")
            del g
    finally:
        torch.cuda.synchronize()
        arena.close()


@pytest.mark.parametrize("captured", [False, True])
def test_stream_linear_lanes_ordered_with_caller_stream(rf, captured):
    """A walk of many blocks (fanned out over the arena's lane streams) sees
    activations written on the caller's stream just before it, and work on the
    caller's stream just after it sees every block's rows."""
    import torch
    fmt, rows, in_dim = syn.Q4_0, 4096, 4096
    W = syn.quant_matrix(fmt, rows, in_dim, seed=93)
    xs = [dev_tensor(syn.normal_f32(in_dim, 94 + i)) for i in range(3)]
    Wd = dev_tensor(W)
    want = [rf.gemv(fmt, Wd, 0, rows, in_dim, x).cpu().numpy() for x in xs]
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(256 << 20)
    s = torch.cuda.Stream()
    x = torch.empty(in_dim, device="cuda")
    y = torch.empty(rows, device="cuda")
    big = torch.empty(64 << 20, device="cuda")
    outs = [torch.empty(rows, device="cuda") for _ in xs]

    def walk():
        for i, xi in enumerate(xs):
            big.fill_(float(i))                    # a slow kernel ahead of x
            x.copy_(xi)
            arena.stream_linear(fmt, host, in_dim, 0, rows, 64, 4, x, y, stream=s)
            outs[i].copy_(y)
            y.fill_(float("nan"))
    try:
        torch.cuda.synchronize()
        if captured:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                walk()
            for _ in range(2):
                with torch.cuda.stream(s):
                    g.replay()
                torch.cuda.synchronize()
            del g
        else:
            with torch.cuda.stream(s):
                walk()
            torch.cuda.synchronize()
        for i in range(len(xs)):
            assert np.array_equal(bits(outs[i].cpu().numpy()), bits(want[i])), i
    finally:
        torch.cuda.synchronize()
        arena.close()


def test_stream_linear_refusals(rf):
    import torch
    fmt, in_dim = syn.Q8_0, 256
    W = syn.quant_matrix(fmt, 64, in_dim, 1)
    x = torch.zeros(in_dim, device="cuda")
    arena = rf.Arena(3 * rf.row_bytes(fmt, in_dim))
    try:
        with pytest.raises(rf.RFError) as e:      # pageable host memory
            arena.stream_linear(fmt, torch.from_numpy(W), in_dim, 0, 64, 8, 1, x)
        assert e.value.code == 3
        host = torch.from_numpy(W).pin_memory()
        with pytest.raises(rf.RFError) as e:      # depth+1 one-row blocks do not fit
            arena.stream_linear(fmt, host, in_dim, 0, 64, 8, 3, x)
        assert e.value.code == 4
        y = arena.stream_linear(fmt, host, in_dim, 0, 64, 8, 2, x)   # shrinks to 1 row
        assert arena.stats()["last_block_rows"] == 1 and arena.stats()["blocks"] == 64
        assert np.all(y.cpu().numpy() == 0)
    finally:
        arena.close()


# ------------------------------------------------------------------ MoE

@pytest.mark.parametrize("n_expert,top_k", [(128, 4), (8, 8), (33, 3), (1, 1)])
def test_moe_route_matches_oracle(rf, n_expert, top_k):
    for seed in range(5):
        logits = syn.router_logits(n_expert, seed)
        if seed == 1 and n_expert > 3:
            logits[2] = logits[0] = logits.max()     # exact ties
        idx, w = rf.moe_route(dev_tensor(logits), top_k)
        idx_ref, w_ref = oracle.router_topk(logits, top_k)
        assert idx.cpu().numpy().tolist() == idx_ref.tolist()
        assert np.allclose(w.cpu().numpy(), w_ref, rtol=1e-6, atol=1e-7)


def special_logits(n_expert, trial, rng):
    """Logits mixing NaN, -inf, signed zeros and numbers (down to a single
    finite one), for the routing edge cases."""
    lg = rng.standard_normal(n_expert).astype(np.float32)
    kind = rng.integers(0, 4, n_expert)
    lg[kind == 0] = np.nan
    lg[kind == 1] = -np.inf
    if trial % 4 == 0:
        lg[:] = np.nan
        lg[rng.integers(n_expert)] = 2.0
    if trial % 4 == 1:
        lg[:] = np.nan
        lg[0], lg[-1] = -0.0, 0.0
    return lg


@pytest.mark.parametrize("n_expert,top_k", [(128, 4), (8, 8), (300, 8), (33, 3)])
def test_route_nan_and_infinite_logits(rf, n_expert, top_k):
    """A NaN logit counts as -inf: the standalone router and the routing inside
    the MoE launch both name the oracle's experts (always distinct and in
    range, even with fewer finite logits than top_k) and the same weights."""
    rng = np.random.default_rng(n_expert * 31 + top_k)
    fmt, n_ff, n_embd = syn.Q4_0, 64, 64
    G = dev_tensor(syn.stacked_experts(fmt, n_expert, n_ff, n_embd, 1))
    U = dev_tensor(syn.stacked_experts(fmt, n_expert, n_ff, n_embd, 2))
    D = dev_tensor(syn.stacked_experts(fmt, n_expert, n_embd, n_ff, 3))
    x = dev_tensor(syn.normal_f32(n_embd, 4))
    for trial in range(8):
        lg = special_logits(n_expert, trial, rng)
        idx_ref, w_ref = oracle.router_topk(lg, top_k)
        idx, w = rf.moe_route(dev_tensor(lg), top_k)
        _, ws = rf.moe_ffn(fmt, dev_tensor(lg), top_k, G, U, D, n_ff, n_embd, 0, x)
        idx2, w2, _ = rf.moe_workspace_views(ws, top_k, n_ff)
        assert idx.cpu().numpy().tolist() == idx_ref.tolist(), trial
        assert idx2.cpu().numpy().tolist() == idx_ref.tolist(), trial
        wa, wb = w.cpu().numpy(), w2.cpu().numpy()
        assert np.array_equal(np.isnan(wa), np.isnan(w_ref)), trial
        ok = ~np.isnan(w_ref)
        assert np.allclose(wa[ok], w_ref[ok], rtol=1e-6, atol=1e-7), trial
        assert np.array_equal(wa.view(np.uint32), wb.view(np.uint32)), trial
    assert rf.device_status() == rf.OK


def moe_check(rf, fmt, E, n_ff, n_embd, top_k, block_rows, seed):
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, seed)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, seed + 1)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, seed + 2)
    x = syn.normal_f32(n_embd, seed + 3)
    logits = syn.router_logits(E, seed + 4)
    y, ws = rf.moe_ffn(fmt, dev_tensor(logits), top_k, dev_tensor(G), dev_tensor(U),
                       dev_tensor(D), n_ff, n_embd, block_rows, dev_tensor(x))
    idx, w, h = (t.cpu().numpy() for t in rf.moe_workspace_views(ws, top_k, n_ff))
    y = y.cpu().numpy()
    # the oracle alone, with bounds derived from the per-GEMV tolerance
    check_moe(moe_reference(fmt, G, U, D, n_ff, n_embd, x, logits, top_k), y, idx, w, h,
              what="moe")
    # end to end against the oracle's own fp64 chain (router weights in fp64)
    y_e2e, _, _ = oracle.moe_ffn(fmt, logits, top_k, G, U, D, n_ff, n_embd, x)
    scale = float(np.abs(y_e2e).max())
    assert np.max(np.abs(y - y_e2e)) <= 2e-3 * scale


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_ffn_small(rf, fmt):
    moe_check(rf, fmt, 16, 320, 256, 4, 64, seed=40 + fmt)


def test_moe_ffn_whole_expert_windows(rf):
    moe_check(rf, syn.MXFP4, 12, 2880, 2880, 2, 0, seed=50)


# ------------------------------------------------------------- zero copy

@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_host_zero_copy_bit_identical_to_resident(rf, fmt):
    """The zero-copy arm reads page-locked host memory in place and gives the
    resident GEMV's bits, for aligned and misaligned rows and a ragged window."""
    import torch
    for rows, in_dim, (r0, r1) in ((700, 4096, (3, 700)), (300, 2880, (0, 299))):
        W = syn.quant_matrix(fmt, rows, in_dim, seed=61)
        x = dev_tensor(syn.normal_f32(in_dim, 62))
        resident = rf.gemv(fmt, dev_tensor(W), r0, r1, in_dim, x).cpu().numpy()
        host = torch.from_numpy(W).pin_memory()
        y = rf.gemv_host(fmt, host, r0, r1, in_dim, x).cpu().numpy()
        assert np.array_equal(bits(y), bits(resident)), (rows, in_dim)
        ref = oracle.gemv(fmt, W, r0, r1, in_dim, syn.normal_f32(in_dim, 62))
        assert_gemv_close(y, ref, gemv_tol(fmt, W, r0, r1, in_dim, syn.normal_f32(in_dim, 62)))
    with pytest.raises(rf.RFError) as e:   # pageable memory is refused
        rf.gemv_host(fmt, torch.from_numpy(W), 0, 8, in_dim, x)
    assert e.value.code == 3


def test_moe_ffn_host_zero_copy_bit_identical(rf):
    """The routed FFN over expert tensors in page-locked host memory, read in
    place, gives rf_moe_ffn's bits (two tokens with different routing)."""
    import torch
    fmt, E, n_ff, n_embd, top_k, br = syn.MXFP4, 16, 320, 2880, 4, 64
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, 80)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, 81)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, 82)
    x_np = syn.normal_f32(n_embd, 83)
    x = dev_tensor(x_np)
    hg, hu, hd = (torch.from_numpy(a).pin_memory() for a in (G, U, D))
    Gd, Ud, Dd = dev_tensor(G), dev_tensor(U), dev_tensor(D)
    for seed in (84, 85):
        lg = syn.router_logits(E, seed)
        logits = dev_tensor(lg)
        y_dev, _ = rf.moe_ffn(fmt, logits, top_k, Gd, Ud, Dd, n_ff, n_embd, br, x)
        y_host, ws = rf.moe_ffn_host(fmt, logits, top_k, hg, hu, hd, n_ff, n_embd, br, x)
        # against the oracle on the same bytes, then bit-identical to resident
        idx, w, h = (t.cpu().numpy() for t in rf.moe_workspace_views(ws, top_k, n_ff))
        check_moe(moe_reference(fmt, G, U, D, n_ff, n_embd, x_np, lg, top_k),
                  y_host.cpu().numpy(), idx, w, h, what=f"zero copy {seed}")
        assert np.array_equal(bits(y_host.cpu().numpy()), bits(y_dev.cpu().numpy())), seed
    with pytest.raises(rf.RFError) as e:   # pageable memory is refused
        rf.moe_ffn_host(fmt, logits, top_k, torch.from_numpy(G), hu, hd, n_ff, n_embd, br, x)
    assert e.value.code == 3
