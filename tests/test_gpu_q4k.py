"""GPU parity of the Q4_K super-block path (RAMforge, "Milestone 5 - Native
Quantized Tensor Support": 256 elements in 144 B, value d*sc*q - dmin*m)
against the CPU oracle: dequantized values bit-exact, GEMV rows within
|y_gpu - y_ref| <= 1e-3 * ||W_r||_2 * ||x||_2, and results independent of
the window, the batch, streaming and zero-copy reads (bit-identical)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import (assert_gemv_close, check_moe, dev_tensor, ffn_reference, gemv_tol,
                         moe_reference)

pytestmark = pytest.mark.gpu

Q4_K = syn.Q4_K


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


def test_q4k_constants(rf):
    assert rf.Q4_K == Q4_K == oracle.Q4_K
    assert rf.block_bytes(Q4_K) == 144
    assert rf.row_bytes(Q4_K, 4096) == 16 * 144
    assert rf.row_bytes(Q4_K, 4096 + 32) == 0
    assert rf.max_in_dim(Q4_K) % 256 == 0 and rf.max_in_dim(Q4_K) >= 24576


def test_dequantize_hand_block(rf, golden_dir):
    from test_oracle_q4k import hand_block
    blk, want = hand_block(golden_dir)
    got = rf.dequantize(Q4_K, dev_tensor(blk), 1).cpu().numpy()
    assert np.array_equal(bits(got), bits(np.array(want, np.float32)))


def test_dequantize_random_bit_exact(rf):
    n = 5_003
    W = syn.quant_matrix(Q4_K, 1, 256 * n, seed=71).reshape(n, 144)
    # edge scales: fp16 zero, subnormal, negative, largest finite; all-ones
    # packed scale bytes (every sc and m 63)
    W[:6, 0:2] = np.array([[0, 0], [1, 0], [0xff, 0x03], [0, 0x80], [0, 0xbc], [0xff, 0x7b]],
                          np.uint8)
    W[6:12, 2:4] = np.array([[0, 0], [1, 0], [0xff, 0x03], [0, 0x80], [0, 0xbc], [0xff, 0x7b]],
                            np.uint8)
    W[12, 4:16] = 0xff
    got = rf.dequantize(Q4_K, dev_tensor(W), n).cpu().numpy()
    ref = oracle.dequantize(Q4_K, W, n)
    assert np.array_equal(bits(got), bits(ref))


SHAPES = [  # (rows, in_dim, window): several 32-row groups, ragged tails
    (1000, 4096, (0, 1000)),
    (257, 11008, (0, 257)),
    (70, 256, (1, 70)),          # one super-block per row
    (300, 768, (5, 299)),        # 3 super-blocks < 8 warps
    (64, 24576, (0, 64)),        # a 24576-wide down projection
    (100, 2816, (2, 99)),
]


@pytest.mark.parametrize("rows,in_dim,win", SHAPES)
def test_gemv_parity(rf, rows, in_dim, win):
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=rows + in_dim)
    x = syn.normal_f32(in_dim, seed=in_dim + 1)
    r0, r1 = win
    y = rf.gemv(Q4_K, dev_tensor(W), r0, r1, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(Q4_K, W, r0, r1, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(Q4_K, W, r0, r1, in_dim, x), "Q4_K")


def test_gemv_edge_scales_and_dynamic_range(rf):
    rows, in_dim = 96, 2048
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=73)
    blk = W.reshape(rows * 8, 144)
    blk[::5, 4:16] = 0xff                 # largest sub-block scales and mins
    blk[1::7, 2:4] = 0                    # dmin = 0
    blk[2::11, 0:2] = [0x00, 0x80]        # d = -0
    x = syn.normal_f32(in_dim, seed=74)
    x[::7] *= 1e5
    x[3::11] *= 1e-9
    x[256:288] = 0.0                      # an all-zero activation block
    y = rf.gemv(Q4_K, dev_tensor(W), 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
    ref = oracle.gemv(Q4_K, W, 0, rows, in_dim, x)
    assert_gemv_close(y, ref, gemv_tol(Q4_K, W, 0, rows, in_dim, x), "edge scales")


def test_gemv_one_hot_exact(rf):
    """A one-hot x picks one column: d*sc*q - dmin*m rounded once, as the
    dequantizer gives it (the activation digit of 1.0 is a power of two)."""
    rows, in_dim = 65, 512
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=75)
    D = oracle.dequantize(Q4_K, W).reshape(rows, in_dim)
    Wd = dev_tensor(W)
    for i in (0, 31, 32, 63, 64, 200, 255, 256, 511):
        x = np.zeros(in_dim, np.float32)
        x[i] = 1.0
        y = rf.gemv(Q4_K, Wd, 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
        assert np.array_equal(y, D[:, i]), i


def test_window_and_batch_invariance_bit_exact(rf):
    rows, in_dim = 700, 4096
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=76)
    x = dev_tensor(syn.normal_f32(in_dim, 77))
    Wd = dev_tensor(W)
    full = rf.gemv(Q4_K, Wd, 0, rows, in_dim, x).cpu().numpy()
    cuts = [0, 1, 33, 100, 101, 450, 699, 700]
    for a, b in zip(cuts, cuts[1:]):
        part = rf.gemv(Q4_K, Wd, a, b, in_dim, x).cpu().numpy()
        assert np.array_equal(bits(part), bits(full[a:b])), (a, b)
    import torch
    ys = [torch.empty(b - a, device="cuda") for a, b in zip(cuts, cuts[1:])]
    rf.gemv_batch(Q4_K, in_dim, [(Wd, a, b, x, y) for (a, b), y in zip(zip(cuts, cuts[1:]), ys)])
    got = torch.cat(ys).cpu().numpy()
    assert np.array_equal(bits(got), bits(full))


def test_ffn_swiglu_parity(rf):
    n_ff, n_embd = 1536, 512
    G = syn.quant_matrix(Q4_K, n_ff, n_embd, 81)
    U = syn.quant_matrix(Q4_K, n_ff, n_embd, 82)
    D = syn.quant_matrix(Q4_K, n_embd, n_ff, 83)
    x = syn.normal_f32(n_embd, 84)
    y, h = rf.ffn_swiglu(Q4_K, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                         dev_tensor(x))
    y, h = y.cpu().numpy(), h.cpu().numpy()
    ref = ffn_reference(Q4_K, G, U, D, n_ff, n_embd, x)
    assert_gemv_close(h, ref["h"], ref["tol_h"], "h")
    assert_gemv_close(y, ref["y"], ref["tol_y"], "y")
    ws = rf.ffn_workspace(n_ff, "cuda")
    y2, h2 = rf.ffn_swiglu(Q4_K, dev_tensor(G), dev_tensor(U), dev_tensor(D), n_ff, n_embd,
                           dev_tensor(x), workspace=ws)
    assert np.array_equal(bits(h2.cpu().numpy()), bits(h))
    assert np.array_equal(bits(y2.cpu().numpy()), bits(y))


def test_stream_linear_and_zero_copy_bit_identical_to_resident(rf):
    import torch
    rows, in_dim, r0 = 900, 2048, 7
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=85)
    x = dev_tensor(syn.normal_f32(in_dim, 86))
    resident = rf.gemv(Q4_K, dev_tensor(W), r0, rows, in_dim, x).cpu().numpy()
    host = torch.from_numpy(W).pin_memory()
    arena = rf.Arena(64 * rf.row_bytes(Q4_K, in_dim))
    try:
        for block_rows, depth in [(1, 0), (7, 1), (32, 4), (0, 3)]:
            y = arena.stream_linear(Q4_K, host, in_dim, r0, rows, block_rows, depth, x)
            assert np.array_equal(bits(y.cpu().numpy()), bits(resident)), (block_rows, depth)
    finally:
        arena.close()
    y = rf.gemv_host(Q4_K, host, r0, rows, in_dim, x).cpu().numpy()
    assert np.array_equal(bits(y), bits(resident))


def test_moe_ffn(rf):
    E, n_ff, n_embd, top_k, br = 16, 512, 256, 4, 64
    G = syn.stacked_experts(Q4_K, E, n_ff, n_embd, 90)
    U = syn.stacked_experts(Q4_K, E, n_ff, n_embd, 91)
    D = syn.stacked_experts(Q4_K, E, n_embd, n_ff, 92)
    x = syn.normal_f32(n_embd, 93)
    logits = syn.router_logits(E, 94)
    y, ws = rf.moe_ffn(Q4_K, dev_tensor(logits), top_k, dev_tensor(G), dev_tensor(U),
                       dev_tensor(D), n_ff, n_embd, br, dev_tensor(x))
    idx, w, h = (t.cpu().numpy() for t in rf.moe_workspace_views(ws, top_k, n_ff))
    check_moe(moe_reference(Q4_K, G, U, D, n_ff, n_embd, x, logits, top_k), y.cpu().numpy(),
              idx, w, h, what="Q4_K moe")
