"""CPU check of the error bound the prefill GEMM's GPU tests use.

rf_gemm's arithmetic, emulated with numpy: every weight rounded once to
fp16 (Q4_K's to fp32 first, as its fused multiply-add does), every
activation rounded to fp16, fp16 x fp16 products (exact in fp32), fp32
accumulation in an arbitrary order.  The emulated result must stay inside
the derived bound for every (token, row), the bound must be tighter than the
path's parity bar 1e-3 * ||W_r|| * ||x||, and a case built to round every
activation the same way must need the bound's fp16 term (so a bound that
dropped it would fail here)."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import derived_gemm_bound, gemv_tol


def emulate(fmt, W, rows, in_dim, X, order):
    Wd = oracle.dequantize(fmt, W).astype(np.float64).reshape(rows, in_dim)
    w32 = Wd.astype(np.float32) if fmt == syn.Q4_K else Wd
    w16 = w32.astype(np.float16).astype(np.float32)
    x16 = np.asarray(X, dtype=np.float32).astype(np.float16).astype(np.float32)
    acc = np.zeros((x16.shape[0], rows), dtype=np.float32)
    for k in order:                      # fp32 adds, one input at a time
        acc += x16[:, k][:, None] * w16[:, k][None, :]
    return acc


@pytest.mark.parametrize("fmt,rows,in_dim", [(syn.Q4_0, 40, 2048), (syn.Q8_0, 32, 1024),
                                              (syn.MXFP4, 24, 2880), (syn.Q4_K, 24, 2048)])
def test_emulated_arithmetic_stays_inside_the_bound(fmt, rows, in_dim):
    W = syn.quant_matrix(fmt, rows, in_dim, seed=rows + in_dim)
    X = np.stack([syn.normal_f32(in_dim, 500 + t) for t in range(4)])
    bound = derived_gemm_bound(fmt, W, 0, rows, in_dim, X)
    rng = np.random.default_rng(fmt)
    for order in (np.arange(in_dim), np.arange(in_dim)[::-1], rng.permutation(in_dim)):
        Y = emulate(fmt, W, rows, in_dim, X, order)
        for t in range(X.shape[0]):
            ref = oracle.gemv(fmt, W, 0, rows, in_dim, X[t])
            err = np.abs(Y[t].astype(np.float64) - ref)
            assert np.all(err <= bound[t])
            assert np.all(bound[t] < gemv_tol(fmt, W, 0, rows, in_dim, X[t]))


def test_the_fp16_term_is_needed():
    """Q8_0 weights of exactly 1 (d = 1, q = 1) and activations 1 + 2^-11 +
    2^-13, which all round up to 1 + 2^-10 in fp16: the error is 0.75 * 2^-11
    per input, inside the bound, and above what the bound's accumulation and
    absolute terms alone allow."""
    in_dim = 1024
    block = np.array([0x00, 0x3C] + [1] * 32, dtype=np.uint8)
    W = np.tile(block, in_dim // 32)[None, :]   # one row of 32 blocks
    x = np.full(in_dim, 1.0 + 2.0 ** -11 + 2.0 ** -13, dtype=np.float32)
    X = x[None, :]
    Y = emulate(syn.Q8_0, W, 1, in_dim, X, np.arange(in_dim))
    ref = oracle.gemv(syn.Q8_0, W, 0, 1, in_dim, x)
    err = abs(float(Y[0, 0]) - float(ref[0]))
    S = float(np.abs(x.astype(np.float64)).sum())
    assert err == 0.75 * 2.0 ** -11 * in_dim   # each activation off by 2^-11 - 2^-13
    assert err <= derived_gemm_bound(syn.Q8_0, W, 0, 1, in_dim, X)[0, 0]
    without_fp16 = (2.0 ** -22 + in_dim * 2.0 ** -23) * S + 2.0 ** -25 * 1.001 * 2 * S
    assert err > without_fp16
