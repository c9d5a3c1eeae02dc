"""GPU tests of rf_gemm, the prefill dequant-GEMM on the tensor cores
(neurostream, "What the numbers taught us": a chunk of tokens shares one pass
over the weights).  Every (token, row) output is compared with the oracle's
fp64 row-window matvec of that token.

Rows whose byte length is not a multiple of 16 are read by the decoders
directly instead of by tensor copies; the arithmetic is the same.

Tolerance, derived from that arithmetic:
  * w and x each take one fp16 rounding: |dw| <= 2^-11 |w| + 2^-25,
    |dx| <= 2^-11 |x| + 2^-25 (half an fp16 subnormal step);
  * fp16 x fp16 products are exact in fp32;
  * fp32 accumulation over in_dim terms, bounded loosely by in_dim * 2^-23
    times the sum of |products| (allowing truncating adds).
  So |y - y_ref| <= (2^-10 + 2^-22 + in_dim * 2^-23) * S
                    + 2^-25 * 1.001 * (sum|w| + sum|x|),
  with S = sum_i |w_i| |x_i|.  Q4_K weights take one fp32 rounding (the
  fused d*sc*q - dmin*m) before the fp16 one, which adds 2^-23 * S.  The
  path's parity bar, 1e-3 * ||W_r|| * ||x||, is checked as well.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import derived_gemm_bound as derived_bound, dev_tensor, gemv_tol

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


def check_gemm(fmt, W, r0, r1, in_dim, X, Y):
    """Every (token, row) within the derived bound and within the path's
    parity bar; returns the largest error as a fraction of the parity bar."""
    bound = derived_bound(fmt, W, r0, r1, in_dim, X)
    worst = 0.0
    for t in range(X.shape[0]):
        ref = oracle.gemv(fmt, W, r0, r1, in_dim, X[t])
        err = np.abs(np.asarray(Y[t], dtype=np.float64) - ref)
        bad = np.nonzero(~(err <= bound[t]))[0]
        assert bad.size == 0, (f"token {t}: {bad.size} rows above the derived bound, row "
                               f"{bad[0]}: gpu {Y[t][bad[0]]} ref {ref[bad[0]]}")
        bar = gemv_tol(fmt, W, r0, r1, in_dim, X[t])
        bad = np.nonzero(~(err <= bar))[0]
        assert bad.size == 0, (f"token {t}: {bad.size} rows above 1e-3*|W_r|*|x|, row "
                               f"{bad[0]}: gpu {Y[t][bad[0]]} ref {ref[bad[0]]}")
        worst = max(worst, float((err / np.maximum(bar, 1e-300)).max()))
    return worst


CASES = [  # fmt, rows, in_dim, window, n_tok
    (syn.Q4_0, 128, 256, (0, 128), 64),      # one CTA, one raw chunk
    (syn.Q4_0, 300, 4096, (5, 300), 70),     # ragged row tile, 128-token tile
    (syn.Q8_0, 257, 2048, (1, 257), 130),    # 256-token tile, ragged
    (syn.MXFP4, 200, 4096, (3, 200), 65),
    (syn.Q4_0, 64, 2304, (0, 64), 300),      # two 256-token tiles, nine chunks
    (syn.Q8_0, 512, 1024, (0, 512), 1),      # one token
    (syn.MXFP4, 200, 2880, (0, 200), 40),    # 1,530-byte rows: direct loads
    (syn.Q4_0, 96, 4064, (0, 96), 9),        # 2,286-byte rows, odd block count: direct
    (syn.Q8_0, 130, 2080, (2, 130), 66),     # 2,210-byte rows, odd block count: direct
    (syn.Q4_0, 300, 2336, (7, 300), 200),    # 1,314-byte rows (phase 2 mod 4): direct
    (syn.Q4_0, 100, 64, (0, 100), 5),        # one slice: the second MMA issuer has none
    (syn.Q8_0, 70, 32, (3, 70), 3),          # one block per row: a half slice
    (syn.MXFP4, 140, 128, (0, 140), 100),    # two slices split in K: one per CTA, N = 128
    (syn.Q4_K, 128, 256, (0, 128), 64),      # one super-block per row
    (syn.Q4_K, 300, 4096, (5, 300), 70),
    (syn.Q4_K, 257, 2048, (1, 257), 300),    # two 256-token tiles, ragged
]


@pytest.mark.parametrize("fmt,rows,in_dim,win,n_tok", CASES)
def test_gemm_matches_oracle(rf, fmt, rows, in_dim, win, n_tok):
    W = syn.quant_matrix(fmt, rows, in_dim, seed=rows * 7 + in_dim)
    X = np.stack([syn.normal_f32(in_dim, 900 + t) for t in range(n_tok)])
    r0, r1 = win
    assert rf.gemm_workspace_bytes(fmt, in_dim, n_tok) > 0
    Y = rf.gemm(fmt, dev_tensor(W), r0, r1, in_dim, dev_tensor(X)).cpu().numpy()
    assert Y.shape == (n_tok, r1 - r0)
    check_gemm(fmt, W, r0, r1, in_dim, X, Y)


def test_gemm_strided_views_and_untouched_margins(rf):
    import torch
    fmt, rows, in_dim, n_tok = syn.Q4_0, 160, 1024, 20
    W = syn.quant_matrix(fmt, rows, in_dim, 3)
    Xbig = torch.randn(n_tok, in_dim + 64, device="cuda")
    X = Xbig[:, 32:32 + in_dim]                    # rows 1,088 floats apart
    Ybig = torch.full((n_tok, rows + 40), float("nan"), device="cuda")
    Y = Ybig[:, 8:8 + rows]
    rf.gemm(fmt, dev_tensor(W), 0, rows, in_dim, X, Y)
    torch.cuda.synchronize()
    check_gemm(fmt, W, 0, rows, in_dim, X.cpu().numpy(), Y.cpu().numpy())
    assert torch.isnan(Ybig[:, :8]).all() and torch.isnan(Ybig[:, 8 + rows:]).all()


def test_gemm_mxfp4_extreme_scales(rf):
    """Scale exponents at the edges of the fp16 decode: 2^(E-127) below the
    fp16 range (weights round to zero), on its subnormals, and above 2^1
    (the two-step multiply)."""
    fmt, rows, in_dim, n_tok = syn.MXFP4, 128, 512, 8
    W = syn.quant_matrix(fmt, rows, in_dim, 5)
    blocks = W.reshape(rows, in_dim // 32, 17)
    E = np.array([70, 95, 104, 113, 120, 127, 129, 135, 140], dtype=np.uint8)
    blocks[:, :, 0] = E[(np.arange(rows)[:, None] + np.arange(in_dim // 32)[None, :]) % E.size]
    X = np.stack([syn.normal_f32(in_dim, 40 + t) for t in range(n_tok)])
    Y = rf.gemm(fmt, dev_tensor(W), 0, rows, in_dim, dev_tensor(X)).cpu().numpy()
    check_gemm(fmt, W, 0, rows, in_dim, X, Y)


def test_gemm_full_size_sampled(rf):
    """The 11008 x 4096 Q4_0 projection at 512 tokens, in the launch
    configuration the prefill bench line times; 64 sampled rows of 8 tokens
    against the oracle, every output finite."""
    import torch
    fmt, rows, in_dim, n_tok = syn.Q4_0, 11008, 4096, 512
    W = syn.quant_matrix(fmt, rows, in_dim, 11, threads=8)
    X = np.stack([syn.normal_f32(in_dim, 70 + t) for t in range(n_tok)])
    Y = rf.gemm(fmt, dev_tensor(W), 0, rows, in_dim, dev_tensor(X))
    torch.cuda.synchronize()
    Y = Y.cpu().numpy()
    assert np.isfinite(Y).all()
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(n_tok, 8, replace=False))
    for r in np.sort(rng.choice(rows, 64, replace=False)):
        r = int(r)
        check_gemm(fmt, W, r, r + 1, in_dim, X[toks], Y[toks][:, r:r + 1])


def test_gemm_direct_full_size_sampled(rf):
    """The 5760 x 2880 MXFP4 expert projection (1,530-byte rows, read
    directly) at 512 tokens: 90 whole tiles, no K split; 64 sampled rows of
    8 tokens against the oracle, every output finite."""
    import torch
    fmt, rows, in_dim, n_tok = syn.MXFP4, 5760, 2880, 512
    W = syn.quant_matrix(fmt, rows, in_dim, 13, threads=8)
    X = np.stack([syn.normal_f32(in_dim, 170 + t) for t in range(n_tok)])
    Y = rf.gemm(fmt, dev_tensor(W), 0, rows, in_dim, dev_tensor(X))
    torch.cuda.synchronize()
    Y = Y.cpu().numpy()
    assert np.isfinite(Y).all()
    rng = np.random.default_rng(4)
    toks = np.sort(rng.choice(n_tok, 8, replace=False))
    for r in np.sort(rng.choice(rows, 64, replace=False)):
        r = int(r)
        check_gemm(fmt, W, r, r + 1, in_dim, X[toks], Y[toks][:, r:r + 1])


def test_gemm_refusals_and_empty_work(rf):
    import torch
    fmt, rows, in_dim = syn.Q4_0, 64, 256
    W = dev_tensor(syn.quant_matrix(fmt, rows, in_dim, 2))
    X = torch.zeros(4, in_dim, device="cuda")
    with pytest.raises(rf.RFError) as e:                       # Q6_K: not served
        rf.gemm(syn.Q6_K, W, 0, rows, in_dim, X)
    assert e.value.code == 2   # RF_ERR_UNSUPPORTED_FMT
    with pytest.raises(rf.RFError) as e:                       # workspace too small
        rf.gemm(fmt, W, 0, rows, in_dim, X, workspace=torch.empty(16, dtype=torch.uint8,
                                                                    device="cuda"))
    assert e.value.code == 1   # RF_ERR_INVALID_ARG
    raw = torch.empty(W.numel() + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rf.RFError) as e:                       # W not 16-byte aligned
        rf.gemm(fmt, raw[1:1 + W.numel()], 0, rows, in_dim, X)
    assert e.value.code == 8   # RF_ERR_MISALIGNED
    # Empty work (an empty window, no tokens) is a no-op that writes nothing.
    Ybuf = torch.full((4, rows), 1.0, device="cuda")
    ws = torch.empty(rf.gemm_workspace_bytes(fmt, in_dim, 4), dtype=torch.uint8, device="cuda")
    L = rf.lib()
    for r0, r1, n in ((5, 5, 4), (0, rows, 0)):
        assert L.rf_gemm(fmt, W.data_ptr(), r0, r1, in_dim, n, X.data_ptr(), in_dim,
                         Ybuf.data_ptr(), rows, ws.data_ptr(), ws.numel(), None) == rf.OK
    torch.cuda.synchronize()
    assert bool((Ybuf == 1.0).all())
