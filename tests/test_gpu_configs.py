"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times, against the oracle on every row (the oracle is fast enough
for these) or on sampled rows (host-streamed FFN)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import assert_gemv_close, dev_tensor, ffn_reference, gemv_tol

pytestmark = pytest.mark.gpu


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


def test_streamed_q8_0_gemv_512x2048(rf):
    """512x2048 Q8_0 streamed from pinned host memory in 128-row blocks."""
    import torch
    c = syn.C1
    fmt, rows, in_dim = c["fmt"], c["out_dim"], c["in_dim"]
    W = syn.quant_matrix(fmt, rows, in_dim, c["seed"])
    x = syn.normal_f32(in_dim, c["seed"] + 1)
    arena = rf.Arena(c["arena_bytes"])
    try:
        host = torch.from_numpy(W).pin_memory()
        for depth in (c["depth"], 1):
            y = arena.stream_linear(fmt, host, in_dim, 0, rows, c["block_rows"], depth,
                                    dev_tensor(x)).cpu().numpy()
            ref = oracle.gemv(fmt, W, 0, rows, in_dim, x)
            assert_gemv_close(y, ref, gemv_tol(fmt, W, 0, rows, in_dim, x), f"depth {depth}")
            assert arena.stats()["last_block_rows"] == 128
        resident = rf.gemv(fmt, dev_tensor(W), 0, rows, in_dim, dev_tensor(x)).cpu().numpy()
        assert np.array_equal(bits(y), bits(resident))
    finally:
        arena.close()


@pytest.mark.parametrize("fmt", [syn.Q4_0, syn.Q4_K])
def test_dense_layer_4096_11008(rf, fmt):
    """One dense decode layer (Q4_0, and the same layer in Q4_K): QKV batched,
    O, gate/up + SwiGLU, down; every row of every projection against the
    oracle; chained and unchained launches, and the FFN with and without the
    digit hand-off workspace, give identical bits."""
    import torch
    from quantized_weight_streaming_dequant_gb300.layer import DenseLayer
    d, f = syn.C2["d_model"], syn.C2["d_ff"]
    s = syn.C2["seed"] * 1000
    mats = [syn.quant_matrix(fmt, d, d, s + i, threads=8) for i in range(4)]
    mats += [syn.quant_matrix(fmt, f, d, s + 4, threads=8), syn.quant_matrix(fmt, f, d, s + 5, threads=8),
             syn.quant_matrix(fmt, d, f, s + 6, threads=8)]
    L = DenseLayer(fmt, d, f, *[dev_tensor(m) for m in mats])
    x, attn, x_ffn = (syn.normal_f32(d, 101), syn.normal_f32(d, 102), syn.normal_f32(d, 103))
    outs = []
    for chain, digits in ((False, False), (True, False), (True, True)):
        out = {k: torch.empty(n, device="cuda") for k, n in
               (("q", d), ("k", d), ("v", d), ("o", d), ("h", f), ("y", d))}
        if digits:   # gate/up hands h's digits to down through a workspace
            out["hd"] = rf.ffn_workspace(f, "cuda")
        L.step(dev_tensor(x), dev_tensor(attn), dev_tensor(x_ffn), out, chain=chain)
        torch.cuda.synchronize()
        outs.append({k: v.cpu().numpy() for k, v in out.items() if k != "hd"})
    for other in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(bits(outs[0][k]), bits(other[k])), k
    o = outs[2]
    for name, M, inp in (("q", mats[0], x), ("k", mats[1], x), ("v", mats[2], x),
                         ("o", mats[3], attn)):
        assert_gemv_close(o[name], oracle.gemv(fmt, M, 0, d, d, inp), gemv_tol(fmt, M, 0, d, d, inp),
                          name)
    ref = ffn_reference(fmt, mats[4], mats[5], mats[6], f, d, x_ffn)
    assert_gemv_close(o["h"], ref["h"], ref["tol_h"], "h")
    assert_gemv_close(o["y"], ref["y"], ref["tol_y"], "y")


def test_moe_mxfp4_128x2880x2880_top4(rf):
    from test_gpu_parity import moe_check
    c = syn.C3
    moe_check(rf, c["fmt"], c["n_expert"], c["n_ff"], c["n_embd"], c["top_k"], c["block_rows"],
              seed=c["seed"])


def test_moe_mxfp4_128x2880x2880_streamed_as_benched(rf):
    """The routed MoE with its experts in page-locked host memory, through the
    layer-wide prefetch plan in the benchmark's configuration (whole windows,
    depth 4, 256 MiB arena, a 32-expert cache, popular experts): every token
    bit-identical to the resident rf_moe_ffn, which the test above checks
    against the oracle."""
    import torch
    c = syn.C3
    fmt, E, n_ff, n_embd, k = c["fmt"], c["n_expert"], c["n_ff"], c["n_embd"], c["top_k"]
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, c["seed"], threads=8)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, c["seed"] + 1, threads=8)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, c["seed"] + 2, threads=8)
    Gd, Ud, Dd = (dev_tensor(a) for a in (G, U, D))
    hG, hU, hD = (torch.from_numpy(a).pin_memory() for a in (G, U, D))
    x = dev_tensor(syn.normal_f32(n_embd, c["seed"] + 3))
    logits = torch.from_numpy(syn.skewed_router_logits(E, 12, 11)).cuda()
    arena = rf.Arena(256 << 20)
    cache = rf.ExpertCache(fmt, n_ff, n_embd, 32)
    try:
        for t in range(12):
            y_ref, _ = rf.moe_ffn(fmt, logits[t], k, Gd, Ud, Dd, n_ff, n_embd, c["block_rows"], x)
            y, _ = rf.moe_ffn_streamed(fmt, logits[t], k, hG, hU, hD, n_ff, n_embd, 0, 4, arena,
                                       x, cache=cache)
            assert np.array_equal(bits(y.cpu().numpy()), bits(y_ref.cpu().numpy())), t
        st = cache.stats()
        assert st["lookups"] == 12 * k and st["hits"] + st["fills"] + st["bypasses"] == 12 * k
    finally:
        torch.cuda.synchronize()
        cache.close()
        arena.close()


def test_streamed_ffn_q8_0_24576x6144_sampled(rf):
    """Two layers of the host-streamed FFN at full size (256 MiB arena,
    512-row blocks, depth 4) against the oracle's own chain (up, GELU, down):
    256 sampled rows of up, every activation, 256 sampled rows of down, with
    bounds derived from the per-GEMV tolerance."""
    import torch
    from quantized_weight_streaming_dequant_gb300.layer import StreamedFFN
    c = syn.C4
    fmt, d, f = c["fmt"], c["d_model"], c["d_ff"]
    rng = np.random.default_rng(0)
    arena = rf.Arena(c["arena_bytes"])
    try:
        for l in range(2):
            up = torch.empty((f, rf.row_bytes(fmt, d)), dtype=torch.uint8).pin_memory()
            dn = torch.empty((d, rf.row_bytes(fmt, f)), dtype=torch.uint8).pin_memory()
            syn.quant_matrix(fmt, f, d, c["seed"] * 1000 + 2 * l, out=up.numpy(), threads=8)
            syn.quant_matrix(fmt, d, f, c["seed"] * 1000 + 2 * l + 1, out=dn.numpy(), threads=8)
            layer = StreamedFFN(fmt, d, f, up, dn)
            x = syn.normal_f32(d, 5000 + l)
            u = torch.empty(f, device="cuda")
            h = torch.empty(f, device="cuda")
            y = torch.empty(d, device="cuda")
            layer.step(arena, dev_tensor(x), u, h, y, c["block_rows"], c["depth"])
            torch.cuda.synchronize()
            u_, h_, y_ = u.cpu().numpy(), h.cpu().numpy(), y.cpu().numpy()
            W_up, W_dn = up.numpy(), dn.numpy()
            rows_dn = np.sort(rng.choice(d, 256, replace=False))
            ref = ffn_reference(fmt, None, W_up, W_dn, f, d, x, act="gelu", rows=rows_dn)
            rows_up = rng.choice(f, 256, replace=False)
            assert_gemv_close(u_[rows_up], ref["u"][rows_up], ref["tol_u"][rows_up], "up")
            assert_gemv_close(h_, ref["h"], ref["tol_h"], "gelu")
            assert_gemv_close(y_[rows_dn], ref["y"], ref["tol_y"], "down")
        st = arena.stats()
        assert st["last_block_rows"] == 512 and st["slots"] == 5
        assert st["peak_bytes"] == 5 * 512 * rf.row_bytes(fmt, f)
    finally:
        arena.close()


@pytest.mark.parametrize("fmt,in_dim,out_dim", sorted({(c["fmt"], c["in_dim"], c["out_dim"])
                                                       for c in syn.sweep_cells()}))
def test_sweep_shapes_resident_windows_and_streamed(rf, fmt, in_dim, out_dim):
    """Every format x shape of the sweep at 512-row windows: the resident
    batch of windows and the host-streamed walk both match the oracle on every
    row and agree with each other bit for bit."""
    import torch
    cell = next(c for c in syn.sweep_cells() if (c["fmt"], c["in_dim"], c["out_dim"],
                                                  c["block_rows"]) == (fmt, in_dim, out_dim, 512))
    W = syn.quant_matrix(fmt, out_dim, in_dim, cell["seed"], threads=8)
    x = syn.normal_f32(in_dim, cell["seed"] + 1)
    Wd, xd = dev_tensor(W), dev_tensor(x)
    y = torch.empty(out_dim, device="cuda")
    rf.gemv_batch(fmt, in_dim, [(Wd, r0, min(out_dim, r0 + 512), xd, y[r0:min(out_dim, r0 + 512)])
                                for r0 in range(0, out_dim, 512)])
    resident = y.cpu().numpy()
    ref = oracle.gemv(fmt, W, 0, out_dim, in_dim, x)
    assert_gemv_close(resident, ref, gemv_tol(fmt, W, 0, out_dim, in_dim, x), "resident")
    arena = rf.Arena(256 << 20)
    try:
        host = torch.from_numpy(W).pin_memory()
        streamed = arena.stream_linear(fmt, host, in_dim, 0, out_dim, 512, 4, xd).cpu().numpy()
    finally:
        arena.close()
    assert np.array_equal(bits(streamed), bits(resident))
