"""GPU tests of rf_gemv_multi (several tokens through one row window in one
launch): every token's row bit-identical to rf_gemv on that token alone and
within the oracle's tolerance; strided inputs and outputs; refusals."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import assert_gemv_close, dev_tensor, gemv_tol

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


CASES = [  # fmt, rows, in_dim, window
    (syn.Q4_0, 1000, 4096, (0, 1000)),     # 16-byte aligned rows
    (syn.Q4_0, 300, 2880, (3, 299)),       # misaligned rows
    (syn.Q8_0, 257, 2048, (1, 257)),
    (syn.MXFP4, 200, 2880, (0, 200)),
    (syn.Q4_K, 130, 1024, (2, 130)),
]


@pytest.mark.parametrize("fmt,rows,in_dim,win", CASES)
@pytest.mark.parametrize("n_tok", [1, 2, 5, 8])
def test_multi_token_rows_bit_identical_to_single(rf, fmt, rows, in_dim, win, n_tok):
    import torch
    W = syn.quant_matrix(fmt, rows, in_dim, seed=rows + in_dim)
    Wd = dev_tensor(W)
    X = np.stack([syn.normal_f32(in_dim, 500 + t) for t in range(n_tok)])
    Xd = dev_tensor(X)
    r0, r1 = win
    Y = rf.gemv_multi(fmt, Wd, r0, r1, in_dim, Xd).cpu().numpy()
    assert Y.shape == (n_tok, r1 - r0)
    for t in range(n_tok):
        single = rf.gemv(fmt, Wd, r0, r1, in_dim, Xd[t].contiguous()).cpu().numpy()
        assert np.array_equal(bits(Y[t]), bits(single)), t
    t = n_tok - 1
    ref = oracle.gemv(fmt, W, r0, r1, in_dim, X[t])
    assert_gemv_close(Y[t], ref, gemv_tol(fmt, W, r0, r1, in_dim, X[t]), f"token {t}")
    torch.cuda.synchronize()


def test_multi_token_strided(rf):
    import torch
    fmt, rows, in_dim, n_tok = syn.Q4_0, 96, 512, 3
    W = dev_tensor(syn.quant_matrix(fmt, rows, in_dim, 1))
    Xbig = torch.randn(n_tok, in_dim + 64, device="cuda")
    X = Xbig[:, 32:32 + in_dim]                    # rows 576 floats apart
    Ybig = torch.full((n_tok, rows + 40), float("nan"), device="cuda")
    Y = Ybig[:, 8:8 + rows]
    rf.gemv_multi(fmt, W, 0, rows, in_dim, X, Y)
    for t in range(n_tok):
        single = rf.gemv(fmt, W, 0, rows, in_dim, X[t].contiguous())
        assert np.array_equal(bits(Y[t].cpu().numpy()), bits(single.cpu().numpy()))
    assert torch.isnan(Ybig[:, :8]).all() and torch.isnan(Ybig[:, 8 + rows:]).all()


def test_multi_token_refusals(rf):
    import torch
    fmt, rows, in_dim = syn.Q4_0, 64, 256
    W = dev_tensor(syn.quant_matrix(fmt, rows, in_dim, 2))
    with pytest.raises(rf.RFError) as e:          # more than 8 tokens
        rf.gemv_multi(fmt, W, 0, rows, in_dim, torch.zeros(9, in_dim, device="cuda"))
    assert e.value.code == 9
    Y = torch.zeros(2, rows, device="cuda")
    X = torch.zeros(2, in_dim, device="cuda")
    w = W.data_ptr()
    for args in ((fmt, w, 0, rows, in_dim, 0, X.data_ptr(), in_dim, Y.data_ptr(), rows),  # no tokens
                 (fmt, w, 0, rows, in_dim, 2, X.data_ptr(), in_dim - 1, Y.data_ptr(), rows),
                 (fmt, w, 0, rows, in_dim, 2, X.data_ptr(), in_dim, Y.data_ptr(), rows - 1)):
        assert rf.lib().rf_gemv_multi(*args, 0, None) == 1
