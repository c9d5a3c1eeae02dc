"""rf_moe_ffn_noalloc: the MoE FFN entry point for callers that cannot
allocate device memory (an engine that fixes its memory plan at start-up, or
a decode loop that must not call cudaMalloc/cudaFree because they synchronize
the device).  It keeps its scratch in a fixed array inside the library, so
the caller passes only inputs and outputs.

Checked through the C ABI against rf_moe_ffn (which takes a caller-allocated
workspace) and against the CPU oracle on the same bytes, on two calls in a
row with different routing, so the second call runs on scratch the first one
left behind; once at the largest size the kernels take (81 % of the array);
and one 32-row step over the array's limit must be refused.  This file is collected last; it
passes on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

import synthetic as syn
from gpu_helpers import check_moe, moe_reference

pytestmark = pytest.mark.gpu

MAX_H = 65536   # RF_MOE_STATIC_MAX_H in include/rf.h


@pytest.fixture(scope="module")
def rf():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import quantized_weight_streaming_dequant_gb300 as m
    from quantized_weight_streaming_dequant_gb300 import build
    build.build()
    m.lib()
    return m


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _run_twice(rf, fmt, E, n_ff, n_embd, top_k, block_rows, seed):
    import torch
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, seed)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, seed + 1)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, seed + 2)
    x_np = syn.normal_f32(n_embd, seed + 3)
    Gd, Ud, Dd, x = _dev(G), _dev(U), _dev(D), _dev(x_np)
    L = rf.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call, lseed in enumerate((seed + 4, seed + 5)):
        lg = syn.router_logits(E, lseed)
        logits = _dev(lg)
        y_ref, _ = rf.moe_ffn(fmt, logits, top_k, Gd, Ud, Dd, n_ff, n_embd, block_rows, x)
        y = torch.full((n_embd,), float("nan"), device="cuda")
        rc = L.rf_moe_ffn_noalloc(fmt, logits.data_ptr(), E, top_k, Gd.data_ptr(), Ud.data_ptr(),
                                  Dd.data_ptr(), n_ff, n_embd, block_rows, x.data_ptr(),
                                  y.data_ptr(), ctypes.c_void_p(stream))
        assert rc == 0, rf.status_str(rc)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy().astype(np.float64), y_ref.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a)), f"call {call}"
        # against the oracle on the same bytes, within the derived bound
        check_moe(moe_reference(fmt, G, U, D, n_ff, n_embd, x_np, lg, top_k), a,
                  what=f"noalloc call {call}")
        # against the workspace entry point, within the tests' tolerance ...
        scale = float(np.abs(b).max())
        assert np.max(np.abs(a - b)) <= 2e-3 * scale, f"call {call}"
        # ... and, being the same kernels on the same inputs, bit for bit
        assert np.array_equal(a, b), f"call {call}"
    assert rf.device_status() == rf.OK


@pytest.mark.parametrize("fmt", [syn.MXFP4, syn.Q4_0])
def test_noalloc_matches_workspace_entry_point_twice(rf, fmt):
    _run_twice(rf, fmt, 16, 320, 256, 4, 64, seed=70)


def test_noalloc_at_the_largest_size_the_kernels_take(rf):
    # The down launch keeps all top_k activation vectors' digits in shared
    # memory, so n_ff is also capped by rf_max_in_dim(fmt, top_k): with 4
    # experts that is 13,280 on a GB300, so 4 * 13,280 = 53,120 of the
    # array's 65,536 activations (81 %) are used.
    top_k = 4
    n_ff = min(MAX_H // top_k, rf.max_in_dim(syn.Q4_0, top_k)) // 32 * 32
    assert top_k * n_ff > 0.75 * MAX_H
    _run_twice(rf, syn.Q4_0, 8, n_ff, 256, top_k, 0, seed=90)


def test_noalloc_rejects_sizes_beyond_its_scratch(rf):
    L = rf.lib()
    p = ctypes.c_void_p(16)
    # one 32-row step over the limit: 4 * 16,416 = 65,664 activations
    rc = L.rf_moe_ffn_noalloc(syn.Q4_0, p, 8, 4, p, p, p, MAX_H // 4 + 32, 256, 0, p, p, None)
    assert rc == 9   # RF_ERR_TOO_LARGE, before any work is enqueued
    rc = L.rf_moe_ffn_noalloc(syn.MXFP4, p, 8, 5, p, p, p, 16384, 256, 0, p, p, None)
    assert rc == 9
    # inside the array but above the kernels' in_dim limit: refused as well
    n_ff = MAX_H // 4
    assert n_ff > rf.max_in_dim(syn.Q4_0, 4)
    rc = L.rf_moe_ffn_noalloc(syn.Q4_0, p, 8, 4, p, p, p, n_ff, 256, 0, p, p, None)
    assert rc == 9
