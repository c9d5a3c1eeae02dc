"""Pins of the oracle's biased experts with the clamped SwiGLU (neurostream,
"GPT-OSS-120B": GPT-OSS adds biased projections and experts and a clamped
SwiGLU; the page prints neither formula nor constants).

Reading (from the public GPT-OSS reference release): g = G x + b_g,
u = U x + b_u, h = min(g, L) * sigmoid(a * min(g, L)) * (clamp(u, -L, L) + 1),
expert output D h + b_d, combined as sum_k w_k (D_k h_k + b_d,k); the
release's constants are a = 1.702 and L = 7.  Parity is unpinned by the
pages; these tests pin the oracle to things other than itself: a reduction
to the already pinned plain SwiGLU MoE, closed forms with zero weights, the
clamp cutting whole weight matrices off, and the sigmoid form of GELU."""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn

ALPHA, LIMIT = 1.702, 7.0


def experts(fmt, E, n_ff, n_embd, seed):
    return (syn.stacked_experts(fmt, E, n_ff, n_embd, seed),
            syn.stacked_experts(fmt, E, n_ff, n_embd, seed + 1),
            syn.stacked_experts(fmt, E, n_embd, n_ff, seed + 2))


@pytest.mark.parametrize("fmt", [oracle.MXFP4, oracle.Q4_0])
def test_reduces_to_the_plain_swiglu_moe(fmt):
    """a = 1, L = +inf, b_u = -1 and the other biases 0 make h = silu(g) * u:
    the plain routed SwiGLU FFN (pinned elsewhere)."""
    E, n_ff, n_embd, k = 8, 96, 64, 3
    G, U, D = experts(fmt, E, n_ff, n_embd, 11)
    x, lg = syn.normal_f32(n_embd, 12), syn.router_logits(E, 13)
    y0, idx0, w0 = oracle.moe_ffn(fmt, lg, k, G, U, D, n_ff, n_embd, x)
    y1, idx1, w1, _ = oracle.moe_ffn_biased(fmt, lg, k, G, U, D, None, -np.ones((E, n_ff)),
                                            None, 1.0, math.inf, n_ff, n_embd, x)
    assert idx0.tolist() == idx1.tolist() and np.array_equal(w0, w1)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-12 * np.abs(y0).max())


def zero_weights(fmt, rows, in_dim):
    W = syn.quant_matrix(fmt, rows, in_dim, seed=5)
    blk = W.reshape(-1, syn.block_bytes(fmt))
    blk[:, 0:2] = 0       # fp16 d = 0: every Q4_0 weight is 0
    return W


def test_bias_only_closed_forms():
    """With every weight 0: g = b_g, u = b_u, and y = sum_k w_k b_d[e_k]; h of
    each selected expert is the clamped SwiGLU of its own biases."""
    fmt, E, n_ff, n_embd, k = oracle.Q4_0, 6, 64, 32, 3
    G, U, D = (zero_weights(fmt, E * n_ff, n_embd), zero_weights(fmt, E * n_ff, n_embd),
               zero_weights(fmt, E * n_embd, n_ff))
    rng = np.random.default_rng(3)
    bg, bu = rng.normal(0, 6, (E, n_ff)), rng.normal(0, 6, (E, n_ff))
    bd = rng.normal(0, 1, (E, n_embd))
    x, lg = syn.normal_f32(n_embd, 4), syn.router_logits(E, 5)
    y, idx, w, h = oracle.moe_ffn_biased(fmt, lg, k, G, U, D, bg, bu, bd, ALPHA, LIMIT, n_ff,
                                         n_embd, x)
    idx_r, w_r = oracle.router_topk(lg, k)
    assert idx.tolist() == idx_r.tolist()
    want = sum(w_r[j] * bd[idx_r[j]] for j in range(k))
    np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-15)
    for j, e in enumerate(idx_r):
        for i in range(0, n_ff, 7):
            assert h[j, i] == oracle.swiglu_clamped(bg[e, i], bu[e, i], ALPHA, LIMIT)


def test_clamp_cuts_weights_off():
    """A gate bias far above L clamps every g to L, so the gate weights stop
    mattering; an up bias far outside [-L, L] does the same for up."""
    fmt, E, n_ff, n_embd, k = oracle.MXFP4, 4, 64, 64, 2
    G, U, D = experts(fmt, E, n_ff, n_embd, 21)
    G2, U2, _ = experts(fmt, E, n_ff, n_embd, 31)
    x, lg = syn.normal_f32(n_embd, 22), syn.router_logits(E, 23)
    big = np.full((E, n_ff), 1e3)
    for bu in (big, -big):
        ya = oracle.moe_ffn_biased(fmt, lg, k, G, U, D, big, bu, None, ALPHA, LIMIT, n_ff,
                                   n_embd, x)[0]
        yb = oracle.moe_ffn_biased(fmt, lg, k, G2, U2, D, big, bu, None, ALPHA, LIMIT, n_ff,
                                   n_embd, x)[0]
        assert np.array_equal(ya, yb)
        # and h is the constant L * sigmoid(a L) * (+-L + 1)
        h = oracle.moe_ffn_biased(fmt, lg, k, G, U, D, big, bu, None, ALPHA, LIMIT, n_ff,
                                  n_embd, x)[3]
        c = LIMIT / (1 + math.exp(-ALPHA * LIMIT)) * (math.copysign(LIMIT, bu[0, 0]) + 1)
        np.testing.assert_allclose(h, c, rtol=1e-15)


def test_clamped_swiglu_scalar_properties():
    scipy_special = pytest.importorskip("scipy.special")
    # against a library sigmoid, inside and outside the clamp
    for g in (-30.0, -7.5, -1.0, -1e-3, 0.0, 0.5, 3.0, 6.999, 7.0, 7.001, 50.0):
        for u in (-9.0, -7.0, -1.0, 0.0, 0.3, 6.5, 7.0, 12.0):
            gc, uc = min(g, LIMIT), max(-LIMIT, min(u, LIMIT))
            want = gc * scipy_special.expit(ALPHA * gc) * (uc + 1.0)
            assert oracle.swiglu_clamped(g, u, ALPHA, LIMIT) == pytest.approx(want, rel=1e-14,
                                                                               abs=1e-300)
    # zeros: g = 0, or u = -1
    assert oracle.swiglu_clamped(0.0, 3.0, ALPHA, LIMIT) == 0.0
    assert oracle.swiglu_clamped(2.0, -1.0, ALPHA, LIMIT) == 0.0
    # the gate's lower side is not clamped: a very negative g gives ~0, not a
    # clamped -L value
    assert abs(oracle.swiglu_clamped(-60.0, 0.0, ALPHA, LIMIT)) < 1e-40
    # with u = 0, g * sigmoid(1.702 g) is the sigmoid form of GELU: within
    # 0.021 of the erf GELU for every g (its known accuracy), which places
    # the factor 1.702 inside the sigmoid
    for g in np.linspace(-6, 6, 241):
        assert abs(oracle.swiglu_clamped(float(g), 0.0, ALPHA, LIMIT) - oracle.gelu(float(g))) < 0.021
