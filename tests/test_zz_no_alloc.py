"""rf_moe_ffn_noalloc: the MoE FFN entry point for callers that cannot
allocate device memory (an engine that fixes its memory plan at start-up, or
a decode loop that must not call cudaMalloc/cudaFree because they synchronize
the device).  It keeps its scratch in a fixed array inside the library, so
the caller passes only inputs and outputs.

Checked through the C ABI against rf_moe_ffn (which takes a caller-allocated
workspace) on two calls in a row with different routing, so the second call
runs on scratch the first one left behind.  This file is collected last; it
passes on its own in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

import synthetic as syn

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("fmt", [syn.MXFP4, syn.Q4_0])
def test_noalloc_matches_workspace_entry_point_twice(rf, fmt):
    import torch
    E, n_ff, n_embd, top_k, block_rows = 16, 320, 256, 4, 64
    G = _dev(syn.stacked_experts(fmt, E, n_ff, n_embd, 70))
    U = _dev(syn.stacked_experts(fmt, E, n_ff, n_embd, 71))
    D = _dev(syn.stacked_experts(fmt, E, n_embd, n_ff, 72))
    x = _dev(syn.normal_f32(n_embd, 73))
    L = rf.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((74, 75)):
        logits = _dev(syn.router_logits(E, seed))
        y_ref, _ = rf.moe_ffn(fmt, logits, top_k, G, U, D, n_ff, n_embd, block_rows, x)
        y = torch.full((n_embd,), float("nan"), device="cuda")
        rc = L.rf_moe_ffn_noalloc(fmt, logits.data_ptr(), E, top_k, G.data_ptr(), U.data_ptr(),
                                  D.data_ptr(), n_ff, n_embd, block_rows, x.data_ptr(),
                                  y.data_ptr(), ctypes.c_void_p(stream))
        assert rc == 0, rf.status_str(rc)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy().astype(np.float64), y_ref.cpu().numpy().astype(np.float64)
        scale = float(np.abs(b).max())
        assert np.all(np.isfinite(a)), f"call {call}"
        assert np.max(np.abs(a - b)) <= 2e-3 * scale, f"call {call}"
        # same kernels on the same inputs: the results agree bit for bit
        assert np.array_equal(a, b), f"call {call}"
    assert rf.device_status() == rf.OK


def test_noalloc_rejects_sizes_beyond_its_scratch(rf):
    L = rf.lib()
    p = ctypes.c_void_p(16)
    n_ff = 16384   # top_k * n_ff = 65,536 + 16,384 floats: above the fixed scratch
    rc = L.rf_moe_ffn_noalloc(syn.MXFP4, p, 8, 5, p, p, p, n_ff, 256, 0, p, p, None)
    assert rc == 9   # RF_ERR_TOO_LARGE, before any work is enqueued
