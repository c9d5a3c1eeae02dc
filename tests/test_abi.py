"""The C ABI library: loads, exports every declared symbol, and its host-side
logic (sizes, block planning, argument validation) -- no GPU needed."""
import ctypes
import subprocess

import numpy as np
import pytest

import oracle
import quantized_weight_streaming_dequant_gb300 as rf

FMTS = [rf.Q8_0, rf.Q4_0, rf.MXFP4]


@pytest.fixture(scope="module")
def L():
    from quantized_weight_streaming_dequant_gb300 import build
    build.build()
    return rf.lib()


def has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_exports_every_declared_symbol(L):
    declared = rf.header_symbols()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", str(rf.SO)], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert set(declared) <= exported
    # the binding declares a signature for each of them
    assert set(declared) == set(rf._SIGS)


def test_status_strings(L):
    for code, name in rf.STATUS.items():
        assert rf.status_str(code) == name
    assert rf.status_str(12345) == "RF_ERR_UNKNOWN"
    assert L.rf_version() >= 100


@pytest.mark.parametrize("fmt", FMTS + [rf.Q4_K])
def test_sizes_match_oracle(L, fmt):
    assert rf.block_bytes(fmt) == oracle.block_bytes(fmt)
    for in_dim in (32, 64, 256, 2048, 2880, 4096, 11008, 24576):
        assert rf.row_bytes(fmt, in_dim) == oracle.row_bytes(fmt, in_dim)
    assert rf.row_bytes(fmt, 33) == 0 and rf.row_bytes(fmt, 0) == 0
    assert rf.block_bytes(7) == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n_rows,block_rows,depth,arena_rows", [
    (2880, 128, 1, 1000), (2880, 1024, 4, 10000), (37, 3, 0, 64), (37, 0, 4, 64),
    (512, 128, 4, 100000), (24576, 512, 4, 2600), (5, 8, 1, 2), (1, 1, 0, 1), (0, 4, 2, 50)])
def test_stream_plan_matches_oracle(L, fmt, n_rows, block_rows, depth, arena_rows):
    in_dim = 2880
    rb = oracle.row_bytes(fmt, in_dim)
    arena = arena_rows * rb + 7
    want = oracle.plan_block_rows(rb, n_rows, block_rows, depth, arena)
    if want < 0:
        with pytest.raises(rf.RFError) as e:
            rf.stream_plan(fmt, in_dim, n_rows, block_rows, depth, arena)
        assert e.value.code == 4
        return
    eff, nblk, peak = rf.stream_plan(fmt, in_dim, n_rows, block_rows, depth, arena)
    assert eff == want
    assert nblk == (0 if n_rows == 0 else -(-n_rows // eff))
    if n_rows:
        W = np.zeros((n_rows, rb), np.uint8)
        _, e2, n2, p2 = oracle.stream_linear(fmt, W, 0, n_rows, in_dim, block_rows, depth,
                                             arena, np.zeros(in_dim, np.float32))
        assert (e2, n2, p2) == (eff, nblk, peak)
        assert peak <= arena


def test_stream_plan_page_example(L):
    """2,880-row MXFP4 expert, 128-row blocks, one block of lookahead: 0.39 MB."""
    eff, nblk, peak = rf.stream_plan(rf.MXFP4, 2880, 2880, 128, 1, 1 << 20)
    assert (eff, nblk, peak) == (128, 23, 391_680)


def test_argument_errors_before_any_gpu_work(L):
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.addressof(buf)
    p16 = (p + 15) & ~15
    # unknown format
    assert L.rf_gemv(7, p16, 0, 1, 32, p16, p16, None) == 2
    assert L.rf_dequantize(7, p16, 1, p16, None) == 2
    # null pointers / bad sizes
    assert L.rf_gemv(rf.Q8_0, None, 0, 1, 32, p16, p16, None) == 1
    assert L.rf_gemv(rf.Q8_0, p16, 0, 1, 33, p16, p16, None) == 1
    assert L.rf_gemv(rf.Q8_0, p16, 5, 4, 32, p16, p16, None) == 1
    assert L.rf_gemv(rf.Q8_0, p16, -1, 4, 32, p16, p16, None) == 1
    assert L.rf_dequantize(rf.Q8_0, p16, -1, p16, None) == 1
    # misaligned weights
    assert L.rf_gemv(rf.Q8_0, p16 + 2, 0, 1, 32, p16, p16, None) == 8
    # empty window: no-op
    assert L.rf_gemv(rf.Q8_0, p16, 3, 3, 32, p16, p16, None) == 0
    assert L.rf_dequantize(rf.Q4_0, p16, 0, p16, None) == 0
    # router / MoE argument checks
    assert L.rf_moe_route(p16, 4, 5, p16, p16, None) == 1
    assert L.rf_moe_route(p16, 4, 0, p16, p16, None) == 1
    assert L.rf_moe_route(p16, 2000, 2, p16, p16, None) == 1
    # routing (2 x 256 B), h (top_k x n_ff floats), h's digits (80 B per 32)
    assert L.rf_moe_workspace_bytes(4, 2880, 2880, 512) == 256 + 256 + 4 * 2880 * 4 + 4 * 2880 // 32 * 80
    assert L.rf_moe_workspace_bytes(4, 2890, 2880, 512) == 0
    assert L.rf_ffn_workspace_bytes(11008) == 11008 // 32 * 80
    assert L.rf_ffn_workspace_bytes(100) == 0 and L.rf_ffn_workspace_bytes(0) == 0
    assert L.rf_moe_workspace_bytes(0, 2880, 2880, 512) == 0
    # activations
    assert L.rf_swiglu(None, p16, p16, 4, None) == 1
    assert L.rf_gelu(p16, p16, 0, None) == 0
    # stream: bad depth
    assert L.rf_stream_linear(rf.Q8_0, p16, 32, 0, 1, 1, -1, p16, p16, p16, None) == 1
    assert L.rf_stream_linear(rf.Q8_0, p16, 32, 0, 1, 1, 65, p16, p16, p16, None) == 1


def test_newer_entry_points_check_arguments_first(L):
    """rf_gemv_multi, the expert cache and rf_moe_ffn_streamed refuse bad
    arguments before touching the GPU."""
    buf = (ctypes.c_uint8 * 8192)()
    p = (ctypes.addressof(buf) + 255) & ~255
    # rf_gemv_multi(fmt, W, r0, r1, in_dim, n_tok, X, ldx, Y, ldy, flags, stream)
    assert L.rf_gemv_multi(7, p, 0, 4, 32, 2, p, 32, p, 4, 0, None) == 2
    assert L.rf_gemv_multi(rf.Q4_0, p, 0, 4, 32, 0, p, 32, p, 4, 0, None) == 1
    assert L.rf_gemv_multi(rf.Q4_0, p, 0, 4, 32, 2, p, 31, p, 4, 0, None) == 1
    assert L.rf_gemv_multi(rf.Q4_0, p, 0, 4, 32, 2, p, 32, p, 3, 0, None) == 1
    assert L.rf_gemv_multi(rf.Q4_0, p, 0, 4, 32, 9, p, 32, p, 4, 0, None) == 9
    assert L.rf_gemv_multi(rf.Q4_0, p + 4, 0, 4, 32, 2, p, 32, p, 4, 0, None) == 8
    assert L.rf_gemv_multi(rf.Q4_0, p, 4, 4, 32, 2, p, 32, p, 4, 0, None) == 0   # no rows
    assert L.rf_gemv_multi(rf.Q4_K, p, 0, 4, 288, 2, p, 288, p, 4, 0, None) == 1  # not 256-multiple
    # rf_expert_cache_create(fmt, n_ff, n_embd, slots, out)
    h = ctypes.c_void_p()
    assert L.rf_expert_cache_create(7, 64, 64, 2, ctypes.byref(h)) == 2
    assert L.rf_expert_cache_create(rf.Q4_0, 48, 64, 2, ctypes.byref(h)) == 1
    assert L.rf_expert_cache_create(rf.Q4_0, 64, 64, 0, ctypes.byref(h)) == 1
    assert L.rf_expert_cache_create(rf.Q4_0, 64, 64, 1025, ctypes.byref(h)) == 1
    assert L.rf_expert_cache_create(rf.Q4_0, 64, 64, 2, None) == 1
    assert L.rf_expert_cache_stats(None, ctypes.byref(rf.ExpertCacheStats())) == 1
    L.rf_expert_cache_destroy(None)   # no-op
    # rf_moe_ffn_streamed(fmt, logits, E, k, hG, hU, hD, n_ff, n_embd, br, depth, arena, cache,
    #                     x, y, workspace, stream)
    ms = L.rf_moe_ffn_streamed
    assert ms(7, p, 8, 2, p, p, p, 64, 64, 32, 3, p, None, p, p, p, None) == 2
    assert ms(rf.Q4_0, p, 8, 2, p, p, p, 64, 64, 32, 3, None, None, p, p, p, None) == 1  # arena
    assert ms(rf.Q4_0, p, 8, 9, p, p, p, 64, 64, 32, 8, p, None, p, p, p, None) == 1     # k > E
    assert ms(rf.Q4_0, p, 8, 2, p, p, p, 64, 64, 48, 3, p, None, p, p, p, None) == 1     # rows
    assert ms(rf.Q4_0, p, 8, 4, p, p, p, 64, 64, 32, 2, p, None, p, p, p, None) == 1     # depth
    assert ms(rf.Q4_0, p, 8, 2, p, p, p, 64, 64, 32, 3, p, None, p, p, p + 16, None) == 8
    assert ms(rf.Q4_0, p, 8, 2, p + 8, p, p, 64, 64, 32, 3, p, None, p, p, p, None) == 8


def test_gemm_checks_arguments_first(L):
    """rf_gemm refuses bad arguments, and returns for empty work, before any
    device call; rf_gemm_workspace_bytes covers at least the fp16 activation
    tiles (tokens rounded up to the token tile, inputs to 64)."""
    buf = (ctypes.c_uint8 * 16384)()
    p = (ctypes.addressof(buf) + 255) & ~255
    g = L.rf_gemm
    ws = 8192   # 64 tokens x 64 inputs x 2 bytes: enough for in_dim 32, up to 64 tokens
    # rf_gemm(fmt, W, r0, r1, in_dim, n_tok, X, ldx, Y, ldy, workspace, workspace_bytes, stream)
    assert g(rf.Q6_K, p, 0, 4, 256, 4, p, 256, p, 4, p, ws, None) == 2     # not served
    assert g(7, p, 0, 4, 32, 4, p, 32, p, 4, p, ws, None) == 2
    assert g(rf.Q4_0, p, 0, 4, 48, 4, p, 48, p, 4, p, ws, None) == 1       # not whole blocks
    assert g(rf.Q4_K, p, 0, 4, 288, 4, p, 288, p, 4, p, ws, None) == 1     # not whole super-blocks
    assert g(rf.Q4_0, None, 0, 4, 32, 4, p, 32, p, 4, p, ws, None) == 1
    assert g(rf.Q4_0, p, 4, 3, 32, 4, p, 32, p, 4, p, ws, None) == 1       # row_end < row_start
    assert g(rf.Q4_0, p, 0, 4, 32, -1, p, 32, p, 4, p, ws, None) == 1
    assert g(rf.Q4_0, p, 0, 4, 32, 4, p, 31, p, 4, p, ws, None) == 1       # ldx < in_dim
    assert g(rf.Q4_0, p, 0, 4, 32, 4, p, 32, p, 3, p, ws, None) == 1       # ldy < rows
    assert g(rf.Q4_0, p + 4, 0, 4, 32, 4, p, 32, p, 4, p, ws, None) == 8   # W not 16-byte aligned
    assert g(rf.Q4_0, p, 0, 4, 32, 4, p, 32, p, 4, None, 0, None) == 1     # no workspace
    assert g(rf.Q4_0, p, 0, 4, 32, 4, p, 32, p, 4, p, ws - 1, None) == 1   # too small
    assert g(rf.Q4_0, p, 0, 4, 32, 4, p, 32, p, 4, p + 8, ws, None) == 8   # misaligned
    big = 1 << 40
    assert g(rf.Q4_0, p, 0, big, 32, 4, p, 32, p, big, p, ws, None) == 9   # too many tiles
    assert g(rf.Q4_0, p, 0, 1 << 31, 32, 1, p, 32, p, 1 << 31, p, ws, None) == 9   # rows > 2^31 - 1
    assert g(rf.Q4_0, p, 5, 5, 32, 4, p, 32, p, 4, p, ws, None) == 0       # no rows
    assert g(rf.Q4_0, p, 0, 4, 32, 0, p, 32, p, 4, None, 0, None) == 0     # no tokens
    wb = L.rf_gemm_workspace_bytes
    assert wb(rf.Q6_K, 256, 4) == 0 and wb(rf.Q4_0, 48, 4) == 0 and wb(rf.Q4_0, 64, 0) == 0
    for fmt, in_dim, n_tok, tile in ((rf.Q4_0, 4096, 8, 64), (rf.MXFP4, 2880, 100, 128),
                                     (rf.Q4_K, 4096, 300, 256)):
        xp = -(-n_tok // tile) * tile * -(-in_dim // 64) * 64 * 2
        assert wb(fmt, in_dim, n_tok) >= xp


@pytest.mark.skipif(has_gpu(), reason="checks the behaviour on a machine without a GPU")
def test_no_gpu_means_cuda_error_not_fallback(L):
    buf = (ctypes.c_uint8 * 4096)()
    p16 = (ctypes.addressof(buf) + 15) & ~15
    assert L.rf_gemv(rf.Q8_0, p16, 0, 1, 32, p16, p16, None) == 5
    assert L.rf_max_in_dim(rf.Q8_0, 1) == 0
    h = ctypes.c_void_p()
    assert L.rf_arena_create(1 << 20, -1, ctypes.byref(h)) in (5, 7)


def test_boundary_names_and_conventions():
    """The boundary keeps the survey's names and signatures: rf_arena_create
    takes the device, the arena counters are read by rf_stream_stats, and the
    header's convention block lists every call that blocks the host."""
    text = rf.HEADER.read_text()
    decl = " ".join(text.split())
    assert "rf_status rf_arena_create(size_t bytes, int device, rf_arena **out);" in decl
    assert "rf_status rf_stream_stats(const rf_arena *arena, rf_stream_stats_t *out);" in decl
    assert "rf_status rf_arena_wait(rf_arena *arena, int timeout_ms);" in decl
    conv = text[:text.index("#ifndef RF_H")]
    for name in ("rf_device_status", "rf_arena_destroy", "rf_arena_wait",
                 "rf_expert_cache_destroy", "rf_moe_ffn_streamed"):
        assert name in conv, name
    for name in ("rf_stream_stats", "rf_arena_wait", "rf_arena_inject_fault",
                 "rf_debug_arm_wait_fault", "rf_expert_cache_stats"):
        assert name in rf.header_symbols(), name


def test_failure_hooks_check_arguments(L):
    """The test hooks and the deadline wait refuse bad arguments on the host."""
    assert L.rf_arena_wait(None, 10) == 1
    assert L.rf_arena_inject_fault(None, 1, 0, 0) == 1
    assert L.rf_arena_configure(None, 1, 0) == 1
    assert L.rf_debug_arm_wait_fault(2000001) == 1
    assert L.rf_debug_arm_wait_fault(0) == 0   # disarm
    h = ctypes.c_void_p()
    assert L.rf_arena_create(0, -1, ctypes.byref(h)) == 1
    assert L.rf_arena_create(1 << 20, -2, ctypes.byref(h)) == 1
    assert L.rf_arena_create(1 << 20, -1, None) == 1
