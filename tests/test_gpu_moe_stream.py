"""GPU tests of the routed MoE FFN read from page-locked host memory through
one layer-wide prefetch plan (rf_moe_ffn_streamed) and of the expert cache:
outputs bit-identical to the resident rf_moe_ffn for every block size, depth
and cache size; cache hits, fills and evictions as the directory says; the
streamed bytes are exactly the missed experts' bytes; refusals."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import check_moe, dev_tensor, moe_reference

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


def bits(t):
    return t.detach().cpu().numpy().astype(np.float32).view(np.uint32)


def experts(fmt, E, n_ff, n_embd, seed):
    import torch
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, seed)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, seed + 1)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, seed + 2)
    dev = [dev_tensor(a) for a in (G, U, D)]
    host = [torch.from_numpy(a).pin_memory() for a in (G, U, D)]
    return (G, U, D), dev, host


CASES = [  # fmt, E, n_ff, n_embd, top_k
    (syn.MXFP4, 16, 320, 2880, 4),   # 1,530-byte rows: whole-group staging
    (syn.Q4_0, 8, 512, 256, 2),      # 16-byte aligned rows: producer mode
    (syn.Q4_K, 6, 512, 512, 3),
]


@pytest.mark.parametrize("fmt,E,n_ff,n_embd,top_k", CASES)
def test_streamed_moe_bit_identical_to_resident(rf, fmt, E, n_ff, n_embd, top_k):
    import torch
    (G, U, D), (Gd, Ud, Dd), (Gh, Uh, Dh) = experts(fmt, E, n_ff, n_embd, 100 + fmt)
    x_np = syn.normal_f32(n_embd, 5)
    x = dev_tensor(x_np)
    arena = rf.Arena(8 << 20)
    caches = [None, rf.ExpertCache(fmt, n_ff, n_embd, 2), rf.ExpertCache(fmt, n_ff, n_embd, E)]
    refs = {}
    try:
        for seed in range(4):
            lg = syn.router_logits(E, 40 + seed % 2)   # tokens repeat routing
            logits = dev_tensor(lg)
            if seed % 2 not in refs:   # the oracle on the same bytes, nothing from the GPU
                refs[seed % 2] = moe_reference(fmt, G, U, D, n_ff, n_embd, x_np, lg, top_k)
            ref = refs[seed % 2]
            y_ref, ws_ref = rf.moe_ffn(fmt, logits, top_k, Gd, Ud, Dd, n_ff, n_embd, 0, x)
            h_ref = rf.moe_workspace_views(ws_ref, top_k, n_ff)[2]
            for cache in caches:
                for block_rows, depth in ((0, max(top_k, 2) - 1), (64, 4), (32, 7)):
                    y, ws = rf.moe_ffn_streamed(fmt, logits, top_k, Gh, Uh, Dh, n_ff, n_embd,
                                                block_rows, depth, arena, x, cache=cache)
                    idx, w, h = rf.moe_workspace_views(ws, top_k, n_ff)
                    what = (seed, None if cache is None else cache.stats()["slots"], block_rows)
                    # against the oracle on its own bytes (hits, fills and
                    # bypasses all included) ...
                    check_moe(ref, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(),
                              h.cpu().numpy(), what=str(what))
                    # ... and bit-identical to the resident path
                    assert np.array_equal(bits(y), bits(y_ref)), what
                    assert np.array_equal(bits(h), bits(h_ref)), what
    finally:
        torch.cuda.synchronize()
        for c in caches:
            if c is not None:
                c.close()
        arena.close()


def test_expert_cache_directory_and_bytes(rf):
    """Streamed bytes are exactly the bytes of the experts not served from the
    cache; hits, fills and evictions follow the least-recently-used directory
    (top-1 tokens, so every token touches one slot and the order is unique)."""
    import torch
    fmt, E, n_ff, n_embd = syn.Q4_0, 8, 512, 256
    (G, U, D), (Gd, Ud, Dd), (Gh, Uh, Dh) = experts(fmt, E, n_ff, n_embd, 7)
    per_expert = 2 * n_ff * rf.row_bytes(fmt, n_embd) + n_embd * rf.row_bytes(fmt, n_ff)
    x = dev_tensor(syn.normal_f32(n_embd, 8))
    arena = rf.Arena(4 << 20)
    cache = rf.ExpertCache(fmt, n_ff, n_embd, 3)
    try:
        # expert per token, and what the directory does with it
        plan = [(0, "fill"), (1, "fill"), (0, "hit"), (2, "fill"), (3, "evict 1"),
                (1, "evict 0"), (2, "hit"), (0, "evict 3")]
        for t, (e, _) in enumerate(plan):
            lg = np.zeros(E, np.float32)
            lg[e] = 5.0
            logits = dev_tensor(lg)
            y, _ = rf.moe_ffn_streamed(fmt, logits, 1, Gh, Uh, Dh, n_ff, n_embd, 128, 3, arena, x,
                                       cache=cache)
            y_ref, _ = rf.moe_ffn(fmt, logits, 1, Gd, Ud, Dd, n_ff, n_embd, 0, x)
            assert np.array_equal(bits(y), bits(y_ref)), t
        torch.cuda.synchronize()
        st = cache.stats()
        assert (st["lookups"], st["hits"], st["fills"], st["evictions"], st["bypasses"]) == \
            (8, 2, 6, 3, 0)
        assert st["bytes_streamed"] == 6 * per_expert
        assert st["bytes_cached"] == 2 * per_expert
        assert st["used"] == 3 and st["slots"] == 3
    finally:
        torch.cuda.synchronize()
        cache.close()
        arena.close()


def test_cache_smaller_than_top_k_bypasses(rf):
    import torch
    fmt, E, n_ff, n_embd, k = syn.MXFP4, 16, 320, 2880, 4
    (G, U, D), (Gd, Ud, Dd), (Gh, Uh, Dh) = experts(fmt, E, n_ff, n_embd, 20)
    x_np, lg = syn.normal_f32(n_embd, 21), syn.router_logits(E, 22)
    x, logits = dev_tensor(x_np), dev_tensor(lg)
    ref = moe_reference(fmt, G, U, D, n_ff, n_embd, x_np, lg, k)
    arena = rf.Arena(8 << 20)
    cache = rf.ExpertCache(fmt, n_ff, n_embd, 1)
    try:
        y_ref, _ = rf.moe_ffn(fmt, logits, k, Gd, Ud, Dd, n_ff, n_embd, 0, x)
        for _ in range(2):
            y, ws = rf.moe_ffn_streamed(fmt, logits, k, Gh, Uh, Dh, n_ff, n_embd, 64, 3, arena,
                                        x, cache=cache)
            idx, w, h = rf.moe_workspace_views(ws, k, n_ff)
            check_moe(ref, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), h.cpu().numpy(),
                      what="hit and bypasses")
            assert np.array_equal(bits(y), bits(y_ref))
        st = cache.stats()
        assert (st["lookups"], st["hits"], st["fills"], st["bypasses"]) == (8, 1, 1, 6)
    finally:
        torch.cuda.synchronize()
        cache.close()
        arena.close()


def test_streamed_moe_refusals(rf):
    import torch
    fmt, E, n_ff, n_embd, k = syn.Q4_0, 8, 512, 256, 2
    (G, U, D), _, (Gh, Uh, Dh) = experts(fmt, E, n_ff, n_embd, 30)
    x = dev_tensor(syn.normal_f32(n_embd, 31))
    logits = dev_tensor(syn.router_logits(E, 32))
    y = torch.full((n_embd,), 7.0, device="cuda")
    arena = rf.Arena(4 << 20)
    try:
        def call(**kw):
            a = dict(host_gate=Gh, host_up=Uh, host_down=Dh, block_rows=128, depth=3, arena=arena,
                     top_k=k, cache=None)
            a.update(kw)
            rf.moe_ffn_streamed(fmt, logits, a["top_k"], a["host_gate"], a["host_up"],
                                a["host_down"], n_ff, n_embd, a["block_rows"], a["depth"],
                                a["arena"], x, cache=a["cache"], y=y)

        with pytest.raises(rf.RFError) as e:      # pageable host memory
            call(host_down=torch.from_numpy(D))
        assert e.value.code == 3
        with pytest.raises(rf.RFError) as e:      # block rows not a multiple of 32
            call(block_rows=48)
        assert e.value.code == 1
        with pytest.raises(rf.RFError) as e:      # a down launch holds top_k blocks
            call(top_k=4, depth=2)
        assert e.value.code == 1
        cache = rf.ExpertCache(fmt, n_ff, n_embd * 2, 2)
        with pytest.raises(rf.RFError) as e:      # cache of another shape
            call(cache=cache)
        assert e.value.code == 1
        cache.close()
        small = rf.Arena(4 * 32 * rf.row_bytes(fmt, n_ff) - 1)
        with pytest.raises(rf.RFError) as e:      # 4 blocks of 32 rows do not fit
            call(arena=small)
        assert e.value.code == 4
        small.close()
        torch.cuda.synchronize()
        assert bool((y == 7.0).all())             # nothing was enqueued
    finally:
        torch.cuda.synchronize()
        arena.close()
