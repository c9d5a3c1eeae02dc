"""GPU parity of the Q6_K super-block path (256 weights in 210 B, value
d*scale*(q-32), one signed scale per 16 weights; the GGML layout, which the
pages name but do not print) against the CPU oracle: dequantized values
bit-exact, GEMV rows within |y_gpu - y_ref| <= 1e-3 * ||W_r||_2 * ||x||_2,
results independent of the window, the batch, streaming and zero-copy reads
(bit-identical), and the FFN and routed MoE on Q6_K weights against the
oracle's own chain."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import (assert_gemv_close, check_moe, dev_tensor, ffn_reference, gemv_tol,
                         moe_reference)

pytestmark = pytest.mark.gpu

Q6_K = syn.Q6_K


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


def test_q6k_constants(rf):
    assert rf.Q6_K == Q6_K == oracle.Q6_K
    assert rf.block_bytes(Q6_K) == 210
    assert rf.row_bytes(Q6_K, 4096) == 16 * 210
    assert rf.row_bytes(Q6_K, 4096 + 32) == 0
    assert rf.max_in_dim(Q6_K) % 256 == 0 and rf.max_in_dim(Q6_K) >= 24576


def test_dequantize_hand_blocks(rf, golden_dir):
    from test_oracle_q6k import hand_blocks
    for blk, want in hand_blocks(golden_dir):
        got = rf.dequantize(Q6_K, dev_tensor(blk), 1).cpu().numpy()
        assert np.array_equal(bits(got), bits(np.array(want, np.float32)))


def test_dequantize_random_bit_exact(rf):
    n = 5_003
    W = syn.quant_matrix(Q6_K, 1, 256 * n, seed=171).reshape(n, 210)
    # edge scales: fp16 d zero, subnormal, largest subnormal, -0, -1, largest
    # finite; scales -128 and 127; all quants 0 and 63
    W[:6, 208:210] = np.array([[0, 0], [1, 0], [0xff, 0x03], [0, 0x80], [0, 0xbc], [0xff, 0x7b]],
                              np.uint8)
    W[6, 192:208] = 0x80
    W[7, 192:208] = 0x7f
    W[8, :192] = 0x00
    W[9, :192] = 0xff
    got = rf.dequantize(Q6_K, dev_tensor(W), n).cpu().numpy()
    ref = oracle.dequantize(Q6_K, W, n)
    assert np.array_equal(bits(got), bits(ref))


SHAPES = [  # (rows, in_dim, window): several 32-row groups, ragged tails
    (1000, 4096, (0, 1000)),     # 3,360-byte rows (16-byte multiple): staged whole
    (257, 11008, (0, 257)),      # 9,030-byte rows: not a 16-byte multiple
    (70, 256, (1, 70)),          # one super-block per row
    (300, 768, (5, 299)),        # 3 super-blocks < 8 warps
    (64, 24576, (0, 64)),        # a 24576-wide down projection: per-lane copies
    (100, 2816, (2, 99)),
]


@pytest.mark.parametrize("rows,in_dim,win", SHAPES)
def test_gemv_parity(rf, rows, in_dim, win):
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=rows + in_dim + 1)
    x = syn.normal_f32(in_dim, seed=in_dim + 3)
    r0, r1 = win
    y = rf.gemv(Q6_K, dev_tensor(W), r0, r1, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(Q6_K, W, r0, r1, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(Q6_K, W, r0, r1, in_dim, x), "Q6_K")


def test_gemv_edge_scales_and_dynamic_range(rf):
    rows, in_dim = 96, 2048
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=173)
    blk = W.reshape(rows * 8, 210)
    blk[::5, 192:208] = 0x80               # every scale -128
    blk[1::7, 192:208] = 0x7f              # every scale 127
    blk[2::11, 208:210] = [0x00, 0x80]     # d = -0
    blk[3::13, :192] = 0xff                # every quant 63
    x = syn.normal_f32(in_dim, seed=174)
    x[::7] *= 1e5
    x[3::11] *= 1e-9
    x[256:288] = 0.0                       # an all-zero activation block
    y = rf.gemv(Q6_K, dev_tensor(W), 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(Q6_K, W, 0, rows, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(Q6_K, W, 0, rows, in_dim, x), "edge scales")


def test_gemv_one_hot_exact(rf):
    """A one-hot x picks one column exactly as the dequantizer gives it (the
    digit of 1.0 is a power of two and every Q6_K weight is exact in fp32)."""
    rows, in_dim = 65, 512
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=175)
    D = oracle.dequantize(Q6_K, W).reshape(rows, in_dim)
    Wd = dev_tensor(W)
    for i in (0, 15, 16, 31, 32, 63, 64, 127, 128, 200, 255, 256, 511):
        x = np.zeros(in_dim, np.float32)
        x[i] = 1.0
        y = rf.gemv(Q6_K, Wd, 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
        assert np.array_equal(y, D[:, i]), i


def test_window_and_batch_invariance_bit_exact(rf):
    import torch
    rows, in_dim = 700, 4096
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=176)
    x = dev_tensor(syn.normal_f32(in_dim, 177))
    Wd = dev_tensor(W)
    full = rf.gemv(Q6_K, Wd, 0, rows, in_dim, x).cpu().numpy()
    cuts = [0, 1, 33, 100, 101, 450, 699, 700]
    for a, b in zip(cuts, cuts[1:]):
        part = rf.gemv(Q6_K, Wd, a, b, in_dim, x).cpu().numpy()
        assert np.array_equal(bits(part), bits(full[a:b])), (a, b)
    ys = [torch.empty(b - a, device="cuda") for a, b in zip(cuts, cuts[1:])]
    rf.gemv_batch(Q6_K, in_dim, [(Wd, a, b, x, y) for (a, b), y in zip(zip(cuts, cuts[1:]), ys)])
    assert np.array_equal(bits(torch.cat(ys).cpu().numpy()), bits(full))


def test_ffn_swiglu_parity(rf):
    n_ff, n_embd = 1536, 512
    G = syn.quant_matrix(Q6_K, n_ff, n_embd, 181)
    U = syn.quant_matrix(Q6_K, n_ff, n_embd, 182)
    D = syn.quant_matrix(Q6_K, n_embd, n_ff, 183)
    x = syn.normal_f32(n_embd, 184)
    y, h = rf.ffn_swiglu(Q6_K, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                         dev_tensor(x))
    y, h = y.cpu().numpy(), h.cpu().numpy()
    ref = ffn_reference(Q6_K, G, U, D, n_ff, n_embd, x)
    assert_gemv_close(h, ref["h"], ref["tol_h"], "h")
    assert_gemv_close(y, ref["y"], ref["tol_y"], "y")
    # the digit hand-off (gate/up writes h's digits, with both 16-element sums)
    ws = rf.ffn_workspace(n_ff, "cuda")
    y2, h2 = rf.ffn_swiglu(Q6_K, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                           dev_tensor(x), workspace=ws)
    assert np.array_equal(bits(h2.cpu().numpy()), bits(h))
    assert np.array_equal(bits(y2.cpu().numpy()), bits(y))


def test_stream_linear_and_zero_copy_bit_identical_to_resident(rf):
    import torch
    rows, in_dim, r0 = 900, 2048, 7
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=185)
    x = dev_tensor(syn.normal_f32(in_dim, 186))
    resident = rf.gemv(Q6_K, dev_tensor(W), r0, rows, in_dim, x).cpu().numpy()
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(64 * rf.row_bytes(Q6_K, in_dim))
    try:
        for block_rows, depth in [(1, 0), (7, 1), (32, 4), (0, 3)]:
            y = arena.stream_linear(Q6_K, host, in_dim, r0, rows, block_rows, depth, x)
            assert np.array_equal(bits(y.cpu().numpy()), bits(resident)), (block_rows, depth)
    finally:
        arena.close()
    y = rf.gemv_host(Q6_K, host, r0, rows, in_dim, x).cpu().numpy()
    assert np.array_equal(bits(y), bits(resident))


def test_gemv_multi_tokens_bit_identical(rf):
    rows, in_dim = 300, 1024
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=187)
    X = np.stack([syn.normal_f32(in_dim, 190 + t) for t in range(5)])
    Wd = dev_tensor(W)
    Y = rf.gemv_multi(Q6_K, Wd, 0, rows, in_dim, dev_tensor(X)).cpu().numpy()
    for t in range(5):
        one = rf.gemv(Q6_K, Wd, 0, rows, in_dim, dev_tensor(X[t])).cpu().numpy()
        assert np.array_equal(bits(Y[t]), bits(one)), t


def test_moe_ffn(rf):
    E, n_ff, n_embd, top_k, br = 16, 512, 256, 4, 64
    G = syn.stacked_experts(Q6_K, E, n_ff, n_embd, 190)
    U = syn.stacked_experts(Q6_K, E, n_ff, n_embd, 191)
    D = syn.stacked_experts(Q6_K, E, n_embd, n_ff, 192)
    x = syn.normal_f32(n_embd, 193)
    logits = syn.router_logits(E, 194)
    y, ws = rf.moe_ffn(Q6_K, dev_tensor(logits), top_k, dev_tensor(G), dev_tensor(U),
                       dev_tensor(D), n_ff, n_embd, br, dev_tensor(x))
    idx, w, h = (t.cpu().numpy() for t in rf.moe_workspace_views(ws, top_k, n_ff))
    check_moe(moe_reference(Q6_K, G, U, D, n_ff, n_embd, x, logits, top_k), y.cpu().numpy(),
              idx, w, h, what="Q6_K moe")
