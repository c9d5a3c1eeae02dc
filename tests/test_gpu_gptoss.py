"""GPU parity of the routed FFN over biased experts with the clamped SwiGLU
(rf_moe_ffn_biased; neurostream, "GPT-OSS-120B"; form and constants from the
public GPT-OSS reference release: alpha 1.702, limit 7) against the CPU
oracle's own chain, at small sizes and at the full 128-expert 2880x2880
MXFP4 MoE in its benchmark configuration (top-4, 512-row windows)."""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import check_moe, dev_tensor, moe_reference_biased

pytestmark = pytest.mark.gpu

ALPHA, LIMIT = 1.702, 7.0


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


def biases(E, n_ff, n_embd, seed, scale=1.0):
    rng = np.random.default_rng([seed, 0xB1A5])
    return tuple((scale * rng.standard_normal(s)).astype(np.float32)
                 for s in ((E, n_ff), (E, n_ff), (E, n_embd)))


def run_case(rf, fmt, E, n_ff, n_embd, top_k, br, seed, with_bias=(True, True, True),
             alpha=ALPHA, limit=LIMIT, threads=1, bias_scale=3.0):
    G = syn.stacked_experts(fmt, E, n_ff, n_embd, seed, threads=threads)
    U = syn.stacked_experts(fmt, E, n_ff, n_embd, seed + 1, threads=threads)
    D = syn.stacked_experts(fmt, E, n_embd, n_ff, seed + 2, threads=threads)
    x, lg = syn.normal_f32(n_embd, seed + 3), syn.router_logits(E, seed + 4)
    bs = [b if on else None for b, on in zip(biases(E, n_ff, n_embd, seed, bias_scale),
                                             with_bias)]
    dev = [None if b is None else dev_tensor(b) for b in bs]
    y, ws = rf.moe_ffn_biased(fmt, dev_tensor(lg), top_k, dev_tensor(G), dev_tensor(U),
                              dev_tensor(D), *dev, alpha, limit, n_ff, n_embd, br,
                              dev_tensor(x))
    idx, w, h = (t.cpu().numpy() for t in rf.moe_workspace_views(ws, top_k, n_ff))
    ref = moe_reference_biased(fmt, G, U, D, n_ff, n_embd, x, lg, top_k, *bs, alpha, limit)
    check_moe(ref, y.cpu().numpy(), idx, w, h, what=f"biased fmt {fmt}")
    return ref, h


@pytest.mark.parametrize("fmt", [syn.MXFP4, syn.Q4_0, syn.Q8_0, syn.Q6_K])
def test_biased_clamped_moe_small(rf, fmt):
    n_embd = 256 if fmt == syn.Q6_K else 2880 if fmt == syn.MXFP4 else 512
    ref, _ = run_case(rf, fmt, 16, 512, n_embd, 4, 64, seed=400 + fmt)
    assert ref["clamped"] > 0   # the clamp is in play on these inputs


@pytest.mark.parametrize("with_bias", [(True, False, False), (False, True, False),
                                       (False, False, True), (False, False, False)])
def test_each_bias_alone(rf, with_bias):
    run_case(rf, syn.Q4_0, 8, 256, 256, 2, 0, seed=420, with_bias=with_bias)


def test_no_clamp_plain_sigmoid_form(rf):
    # limit = +inf, alpha = 1: h = silu(g) (u + 1), no clamp anywhere
    run_case(rf, syn.MXFP4, 8, 320, 2880, 3, 64, seed=430, alpha=1.0, limit=math.inf)


def test_bias_only_closed_form(rf):
    """Every weight 0 (fp16 d = 0): y = sum_k w_k down_bias[e_k]."""
    fmt, E, n_ff, n_embd, k = syn.Q4_0, 8, 256, 256, 3
    mats = []
    for rows, cols in ((E * n_ff, n_embd), (E * n_ff, n_embd), (E * n_embd, n_ff)):
        W = syn.quant_matrix(fmt, rows, cols, seed=5)
        W.reshape(-1, 18)[:, 0:2] = 0
        mats.append(dev_tensor(W))
    bg, bu, bd = biases(E, n_ff, n_embd, 440, scale=6.0)
    lg = syn.router_logits(E, 441)
    x = dev_tensor(syn.normal_f32(n_embd, 442))
    y, _ = rf.moe_ffn_biased(fmt, dev_tensor(lg), k, *mats, dev_tensor(bg), dev_tensor(bu),
                             dev_tensor(bd), ALPHA, LIMIT, n_ff, n_embd, 0, x)
    idx, w = oracle.router_topk(lg, k)
    want = sum(w[j] * bd[idx[j]].astype(np.float64) for j in range(k))
    np.testing.assert_allclose(y.cpu().numpy(), want, rtol=1e-6, atol=1e-7)


def test_refusals(rf):
    import torch
    fmt, E, n_ff, n_embd = syn.Q4_0, 4, 64, 64
    W = dev_tensor(syn.stacked_experts(fmt, E, n_ff, n_embd, 1))
    lg, x = dev_tensor(syn.router_logits(E, 2)), dev_tensor(syn.normal_f32(n_embd, 3))
    y = torch.full((n_embd,), 7.0, device="cuda")
    b = torch.zeros(E * n_ff, device="cuda")
    odd = torch.zeros(4 * E * n_ff + 1, dtype=torch.uint8, device="cuda")[1:]   # misaligned
    for alpha, limit, bias, code in ((math.nan, LIMIT, b, 1), (math.inf, LIMIT, b, 1),
                                     (ALPHA, 0.0, b, 1), (ALPHA, math.nan, b, 1),
                                     (ALPHA, LIMIT, odd, 8)):
        with pytest.raises(rf.RFError) as e:
            rf.moe_ffn_biased(fmt, lg, 2, W, W, W, bias, None, None, alpha, limit, n_ff, n_embd,
                              0, x, y=y)
        assert e.value.code == code
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())   # nothing was enqueued


def test_biased_clamped_moe_128x2880x2880_top4(rf):
    c = syn.C3
    ref, _ = run_case(rf, c["fmt"], c["n_expert"], c["n_ff"], c["n_embd"], c["top_k"],
                      c["block_rows"], seed=c["seed"] + 50, threads=8, bias_scale=1.0)
    assert ref["clamped"] > 0
