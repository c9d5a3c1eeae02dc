"""Pins for the CPU oracle against things other than itself.

Each test fixes the oracle to a value printed on the pages, a hand-worked
block derived from the format definitions, a library routine, a closed form,
an invariant or brute force on tiny inputs.  No GPU needed.
"""
import itertools
import math
import struct

import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle import MXFP4, Q4_0, Q8_0

FMTS = [Q8_0, Q4_0, MXFP4]


def f32_bits(v) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def load_page_figures(golden_dir):
    vals = {}
    for line in (golden_dir / "page_figures.txt").read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()
            vals[k] = float(v)
    return vals


# ------------------------------------------------------------------ scalars

def test_fp16_exhaustive_matches_numpy():
    """Every binary16 bit pattern decodes like numpy's float16 (a library
    implementation of IEEE-754 binary16)."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero is part of bit-exactness
    assert math.copysign(1.0, oracle.fp16_to_double(0x8000)) == -1.0


def test_e2m1_matches_ocp_table(golden_dir):
    for line in (golden_dir / "e2m1_ocp.txt").read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        code, val = line.split()
        got = oracle.e2m1_to_double(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e8m0_closed_forms():
    assert oracle.e8m0_to_double(127) == 1.0
    assert oracle.e8m0_to_double(0) == 2.0 ** -127
    assert oracle.e8m0_to_double(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_to_double(255))
    for E in range(0, 254):
        assert oracle.e8m0_to_double(E + 1) == 2.0 * oracle.e8m0_to_double(E)


# ---------------------------------------------------------- hand blocks

def parse_blocks(golden_dir):
    names = {"Q8_0": Q8_0, "Q4_0": Q4_0, "MXFP4": MXFP4}
    cases = []
    for line in (golden_dir / "blocks.txt").read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        fmt_s, hexbytes, expect = (p.strip() for p in line.split("|"))
        fmt = names[fmt_s]
        raw = bytes(int(h, 16) for h in hexbytes.split())
        raw = raw + bytes(syn.block_bytes(fmt) - len(raw))
        exp = {}
        rest = None
        for item in expect.split():
            k, v = item.split("=")
            fv = {"zero": 0.0, "negzero": -0.0}.get(v)
            fv = float.fromhex(v) if fv is None else fv
            if k == "rest":
                rest = fv
            else:
                exp[int(k)] = fv
        values = [exp.get(j, rest) for j in range(32)]
        cases.append((fmt_s, fmt, raw, values))
    return cases


def test_hand_blocks_bit_exact(golden_dir):
    cases = parse_blocks(golden_dir)
    assert len(cases) >= 10
    for name, fmt, raw, values in cases:
        out = oracle.dequantize(fmt, np.frombuffer(raw, dtype=np.uint8), 1)
        got = [f32_bits(float(v)) for v in out]
        want = [f32_bits(v) for v in values]
        assert got == want, f"{name} block {raw.hex()}"


# ------------------------------------------------- figures on the pages

def test_block_bytes_match_pages(golden_dir):
    pf = load_page_figures(golden_dir)
    assert oracle.block_bytes(Q4_0) == pf["q4_0_block_bytes"]
    assert oracle.block_bytes(Q8_0) == pf["q8_0_block_bytes"]
    assert oracle.block_bytes(MXFP4) == 17


def test_expert_matrix_is_4_41_mb(golden_dir):
    pf = load_page_figures(golden_dir)
    rows, in_dim = int(pf["expert_rows"]), int(pf["expert_in_dim"])
    total = rows * oracle.row_bytes(MXFP4, in_dim)
    assert total == 4_406_400
    assert round(total / 1e6, 2) == pf["expert_matrix_mb"]


def test_arena_peak_0_39_mb_and_bit_identical(golden_dir):
    """Streaming one expert 128 rows at a time (one block of lookahead) peaks
    at 0.39 MB of arena and gives the same output bit for bit."""
    pf = load_page_figures(golden_dir)
    rows, in_dim = int(pf["expert_rows"]), int(pf["expert_in_dim"])
    W = syn.quant_matrix(MXFP4, rows, in_dim, seed=11)
    x = syn.normal_f32(in_dim, seed=12)
    y_whole = oracle.gemv(MXFP4, W, 0, rows, in_dim, x)
    y, eff, nblk, peak = oracle.stream_linear(MXFP4, W, 0, rows, in_dim,
                                              int(pf["stream_block_rows"]), 1, 1 << 20, x)
    assert eff == 128 and nblk == math.ceil(rows / 128)
    assert peak == 2 * 128 * oracle.row_bytes(MXFP4, in_dim) == 391_680
    assert round(peak / 1e6, 2) == pf["arena_peak_mb"]
    assert round(rows * oracle.row_bytes(MXFP4, in_dim) / peak) == pf["memory_ratio"]
    assert np.array_equal(y.view(np.uint64), y_whole.view(np.uint64))


def test_expert_bytes_per_token_1_9_gb(golden_dir):
    pf = load_page_figures(golden_dir)
    per_matrix = int(pf["expert_rows"]) * oracle.row_bytes(MXFP4, int(pf["expert_in_dim"]))
    total = pf["gptoss_layers"] * pf["gptoss_active"] * 3 * per_matrix
    assert round(total / 1e9, 1) == pf["expert_gb_per_token"]


def test_window_of_2880_rows_at_1024_is_three_blocks(golden_dir):
    pf = load_page_figures(golden_dir)
    rb = oracle.row_bytes(MXFP4, 2880)
    eff = oracle.plan_block_rows(rb, int(pf["window_rows"]), int(pf["window_block_rows"]), 4,
                                 1 << 30)
    assert eff == 1024
    assert math.ceil(pf["window_rows"] / eff) == pf["window_blocks"]


# --------------------------------------------------------- GEMV pins

def dense(fmt, W, rows, in_dim):
    return oracle.dequantize(fmt, W, rows * in_dim // 32).astype(np.float64).reshape(rows,
                                                                                      in_dim)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,in_dim", [(1, 32), (5, 64), (7, 96), (3, 256)])
def test_gemv_matches_bruteforce_fsum(fmt, rows, in_dim):
    W = syn.quant_matrix(fmt, rows, in_dim, seed=rows * 1000 + in_dim)
    x = syn.normal_f32(in_dim, seed=in_dim)
    y = oracle.gemv(fmt, W, 0, rows, in_dim, x)
    D = dense(fmt, W, rows, in_dim)
    for r in range(rows):
        terms = [D[r, i] * float(x[i]) for i in range(in_dim)]   # exact products
        ref = math.fsum(terms)
        scale = math.fsum(abs(t) for t in terms)
        assert abs(y[r] - ref) <= 1e-12 * scale


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_one_hot_column_exact(fmt):
    rows, in_dim = 9, 128
    W = syn.quant_matrix(fmt, rows, in_dim, seed=5)
    D = dense(fmt, W, rows, in_dim)
    for i in (0, 17, 31, 32, 100, 127):
        x = np.zeros(in_dim, dtype=np.float32)
        x[i] = 1.0
        y = oracle.gemv(fmt, W, 0, rows, in_dim, x)
        assert np.array_equal(y, D[:, i])


def test_gemv_constant_quants_closed_form():
    """Q8_0 rows whose quants all equal c and whose blocks share d:
    y = d * c * sum(x)."""
    rows, in_dim = 4, 256
    W = np.zeros((rows, oracle.row_bytes(Q8_0, in_dim)), dtype=np.uint8)
    blk = W.reshape(rows, in_dim // 32, 34)
    ds = [0.5, 0.25, 2.0, 0.125]
    cs = [3, -7, 1, 127]
    for r in range(rows):
        blk[r, :, 0:2] = np.frombuffer(np.float16(ds[r]).tobytes(), dtype=np.uint8)
        blk[r, :, 2:] = np.uint8(cs[r] & 0xFF)
    x = syn.normal_f32(in_dim, seed=3)
    y = oracle.gemv(Q8_0, W, 0, rows, in_dim, x)
    sx = math.fsum(float(v) for v in x)
    for r in range(rows):
        assert abs(y[r] - ds[r] * cs[r] * sx) <= 1e-12 * abs(ds[r] * cs[r]) * float(
            np.abs(x).sum())


def test_gemv_zero_scale_gives_zero():
    rows, in_dim = 3, 64
    W = syn.quant_matrix(Q4_0, rows, in_dim, seed=1, scale_range=(0.0, 0.0))
    y = oracle.gemv(Q4_0, W, 0, rows, in_dim, syn.normal_f32(in_dim, 1))
    assert np.all(y == 0.0)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_linear_in_x(fmt):
    rows, in_dim = 6, 160
    W = syn.quant_matrix(fmt, rows, in_dim, seed=8)
    x1 = syn.normal_f32(in_dim, 1).astype(np.float64)
    x2 = syn.normal_f32(in_dim, 2).astype(np.float64)
    y1 = oracle.gemv(fmt, W, 0, rows, in_dim, x1)
    y2 = oracle.gemv(fmt, W, 0, rows, in_dim, x2)
    y12 = oracle.gemv(fmt, W, 0, rows, in_dim, 2.0 * x1 - 3.0 * x2)
    assert np.allclose(y12, 2.0 * y1 - 3.0 * y2, rtol=0, atol=1e-10)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_window_is_slice_of_whole(fmt):
    rows, in_dim = 20, 96
    W = syn.quant_matrix(fmt, rows, in_dim, seed=4)
    x = syn.normal_f32(in_dim, 4)
    full = oracle.gemv(fmt, W, 0, rows, in_dim, x)
    for r0, r1 in [(0, 1), (3, 11), (19, 20), (5, 5)]:
        assert np.array_equal(oracle.gemv(fmt, W, r0, r1, in_dim, x), full[r0:r1])


# ------------------------------------------------------ streaming pins

def expected_peak(n_rows, eff, row_bytes, depth):
    sizes = [min(eff, n_rows - s) * row_bytes for s in range(0, n_rows, eff)]
    return max((sum(sizes[i:i + depth + 1]) for i in range(len(sizes))), default=0)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("block_rows", [1, 3, 16, 128, 0])
@pytest.mark.parametrize("depth", [0, 1, 4])
def test_stream_linear_invariance(fmt, block_rows, depth):
    """Any block size and lookahead gives the whole-matrix output bit for bit
    (neurostream, "The idea"; "Results", P1 row)."""
    rows, in_dim = 37, 128
    W = syn.quant_matrix(fmt, rows, in_dim, seed=21)
    x = syn.normal_f32(in_dim, 21)
    ref = oracle.gemv(fmt, W, 2, rows, in_dim, x)
    rb = oracle.row_bytes(fmt, in_dim)
    y, eff, nblk, peak = oracle.stream_linear(fmt, W, 2, rows, in_dim, block_rows, depth,
                                              64 * rb, x)
    assert np.array_equal(y.view(np.uint64), ref.view(np.uint64))
    want = rows - 2 if block_rows == 0 else min(block_rows, rows - 2)
    want = min(want, 64 // (depth + 1))
    assert eff == want
    assert nblk == math.ceil((rows - 2) / eff)
    assert peak == expected_peak(rows - 2, eff, rb, depth)
    assert peak <= 64 * rb


def test_plan_shrink_and_refusal():
    # Host-streamed FFN shapes: 512-row blocks, depth 4, 256 MiB arena fit as is.
    for in_dim in (6144, 24576):
        rb = oracle.row_bytes(Q8_0, in_dim)
        assert oracle.plan_block_rows(rb, 24576, 512, 4, 256 << 20) == 512
    # Shrink until depth+1 buffers fit.
    assert oracle.plan_block_rows(100, 1000, 8, 1, 1000) == 5
    # Sized for depth blocks instead of depth+1 (the deadlock on the pages):
    # the plan shrinks rather than overcommitting.
    assert oracle.plan_block_rows(100, 1000, 10, 3, 3 * 10 * 100) == 7
    # Not even one row per buffer: refuse.
    assert oracle.plan_block_rows(100, 1000, 8, 1, 199) == -1
    with pytest.raises(MemoryError):
        oracle.stream_linear(Q8_0, syn.quant_matrix(Q8_0, 4, 32, 1), 0, 4, 32, 2, 1, 67,
                             np.zeros(32, np.float32))


# ---------------------------------------------------------- router pins

@pytest.mark.parametrize("n_expert,top_k", [(1, 1), (5, 2), (8, 4), (16, 4), (128, 4)])
def test_router_topk_bruteforce(n_expert, top_k):
    from scipy.special import softmax
    rng = np.random.default_rng(n_expert * 7 + top_k)
    for trial in range(20):
        logits = rng.standard_normal(n_expert).astype(np.float32)
        if trial % 3 == 0 and n_expert > 2:          # plant exact ties
            logits[rng.integers(n_expert)] = logits[0]
            logits[n_expert - 1] = logits[1]
        idx, w = oracle.router_topk(logits, top_k)
        want = sorted(range(n_expert), key=lambda e: (-float(logits[e]), e))[:top_k]
        assert list(idx) == want
        p = softmax(logits.astype(np.float64))
        assert np.allclose(w, p[want] / p[want].sum(), rtol=1e-12, atol=0)
        assert abs(w.sum() - 1.0) < 1e-12
        assert all(w[i] >= w[i + 1] for i in range(top_k - 1))


@pytest.mark.parametrize("n_expert,top_k", [(4, 4), (8, 3), (40, 8), (128, 4)])
def test_router_nan_counts_as_minus_infinity(n_expert, top_k):
    """Reading: a NaN logit ranks as -inf (ties to the lower index) and weighs
    as -inf.  Brute force over inputs mixing NaN, -inf, +-0 and numbers, down to
    fewer finite logits than top_k."""
    rng = np.random.default_rng(n_expert + 100 * top_k)
    for trial in range(30):
        logits = rng.standard_normal(n_expert).astype(np.float32)
        kind = rng.integers(0, 4, n_expert)
        logits[kind == 0] = np.nan
        logits[kind == 1] = -np.inf
        if trial % 5 == 0:
            logits[:] = np.nan
            logits[rng.integers(n_expert)] = 1.0
        if trial % 7 == 1:
            logits[0], logits[-1] = -0.0, 0.0            # signed zeros tie
            logits[1:-1] = np.nan
        idx, w = oracle.router_topk(logits, top_k)
        rank = np.where(np.isnan(logits), -np.inf, logits.astype(np.float64))
        want = sorted(range(n_expert), key=lambda e: (-rank[e], e))[:top_k]
        assert list(idx) == want, trial
        sel = rank[want]
        if np.isfinite(sel[0]):
            ex = np.exp(sel - sel[0])
            assert np.allclose(w, ex / ex.sum(), rtol=1e-12, atol=0)
            assert all(w[i] == 0.0 for i in range(top_k) if sel[i] == -np.inf)
        else:                                             # every selected logit is -inf
            assert np.isnan(w).all()


def test_router_equal_logits_uniform():
    idx, w = oracle.router_topk(np.full(128, 0.25, np.float32), 4)
    assert list(idx) == [0, 1, 2, 3]
    assert np.allclose(w, 0.25, rtol=0, atol=1e-15)
    idx, w = oracle.router_topk(np.zeros(6, np.float32), 6)
    assert list(idx) == list(range(6)) and np.allclose(w, 1 / 6)


# ------------------------------------------------------ activation pins

def test_activation_identities_and_constants():
    for z in (-30.0, -3.5, -1.0, -1e-3, 0.0, 0.3, 1.0, 2.5, 40.0):
        assert abs((oracle.silu(z) - oracle.silu(-z)) - z) <= 1e-14 * max(1.0, abs(z))
        assert abs((oracle.gelu(z) - oracle.gelu(-z)) - z) <= 1e-14 * max(1.0, abs(z))
    assert oracle.silu(0.0) == 0.0 and oracle.gelu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 0.7310585786300049) < 1e-15      # 1/(1+1/e)
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15      # Phi(1)
    assert abs(oracle.gelu(-1.0) + 0.15865525393145707) < 1e-15    # -(1-Phi(1))
    assert abs(oracle.silu(50.0) - 50.0) < 1e-12 and abs(oracle.silu(-50.0)) < 1e-18
    assert abs(oracle.gelu(10.0) - 10.0) < 1e-12 and abs(oracle.gelu(-10.0)) < 1e-18


# ----------------------------------------------------------- FFN / MoE

def test_ffn_swiglu_matches_dense_matmul():
    fmt, n_ff, n_embd = Q4_0, 96, 64
    G = syn.quant_matrix(fmt, n_ff, n_embd, 31)
    U = syn.quant_matrix(fmt, n_ff, n_embd, 32)
    D = syn.quant_matrix(fmt, n_embd, n_ff, 33)
    x = syn.normal_f32(n_embd, 34)
    y, h = oracle.ffn_swiglu(fmt, G, U, D, n_ff, n_embd, x)
    Gd, Ud, Dd = dense(fmt, G, n_ff, n_embd), dense(fmt, U, n_ff, n_embd), dense(fmt, D, n_embd,
                                                                                     n_ff)
    g = Gd @ x.astype(np.float64)
    u = Ud @ x.astype(np.float64)
    h_ref = np.array([oracle.silu(v) for v in g]) * u
    assert np.allclose(h, h_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(y, Dd @ h_ref, rtol=1e-10, atol=1e-10)


def _moe_tensors(fmt, n_expert, n_ff, n_embd, seed):
    G = syn.stacked_experts(fmt, n_expert, n_ff, n_embd, seed)
    U = syn.stacked_experts(fmt, n_expert, n_ff, n_embd, seed + 1)
    D = syn.stacked_experts(fmt, n_expert, n_embd, n_ff, seed + 2)
    return G, U, D


def test_moe_expert_rows_and_top1():
    """Expert e owns rows [e*out,(e+1)*out) of each stacked tensor; top-1
    routing returns that expert's FFN with weight 1."""
    fmt, E, n_ff, n_embd = MXFP4, 6, 64, 32
    G, U, D = _moe_tensors(fmt, E, n_ff, n_embd, 40)
    x = syn.normal_f32(n_embd, 41)
    for e in range(E):
        logits = np.zeros(E, np.float32)
        logits[e] = 5.0
        y, idx, w = oracle.moe_ffn(fmt, logits, 1, G, U, D, n_ff, n_embd, x)
        assert list(idx) == [e] and w[0] == 1.0
        y_ref, _ = oracle.ffn_swiglu(fmt, G[e * n_ff:(e + 1) * n_ff], U[e * n_ff:(e + 1) * n_ff],
                                     D[e * n_embd:(e + 1) * n_embd], n_ff, n_embd, x)
        assert np.array_equal(y, y_ref)


def test_moe_identical_experts_weights_sum_to_one():
    fmt, E, n_ff, n_embd = Q8_0, 8, 64, 64
    G1, U1, D1 = _moe_tensors(fmt, 1, n_ff, n_embd, 50)
    G, U, D = (np.tile(a, (E, 1)) for a in (G1, U1, D1))
    x = syn.normal_f32(n_embd, 51)
    y_one, _ = oracle.ffn_swiglu(fmt, G1, U1, D1, n_ff, n_embd, x)
    y, idx, w = oracle.moe_ffn(fmt, syn.router_logits(E, 52), 4, G, U, D, n_ff, n_embd, x)
    assert len(set(idx.tolist())) == 4
    assert np.allclose(y, y_one, rtol=1e-12, atol=1e-12)


def test_moe_is_weighted_sum_of_selected_experts():
    fmt, E, n_ff, n_embd = Q4_0, 10, 32, 64
    G, U, D = _moe_tensors(fmt, E, n_ff, n_embd, 60)
    x = syn.normal_f32(n_embd, 61)
    logits = syn.router_logits(E, 62)
    y, idx, w = oracle.moe_ffn(fmt, logits, 3, G, U, D, n_ff, n_embd, x)
    parts = []
    for e in range(E):
        ye, _ = oracle.ffn_swiglu(fmt, G[e * n_ff:(e + 1) * n_ff], U[e * n_ff:(e + 1) * n_ff],
                                  D[e * n_embd:(e + 1) * n_embd], n_ff, n_embd, x)
        parts.append(ye)
    best = max(itertools.combinations(range(E), 3), key=lambda s: sum(logits[list(s)]))
    assert sorted(idx.tolist()) == sorted(best)
    ref = sum(wk * parts[e] for wk, e in zip(w, idx))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- row norms
# Every GPU parity tolerance is 1e-3 * ||W_r||_2 * ||x||_2 with W_r the
# dequantized row, so the oracle's row norms are pinned on their own: by
# hand-worked blocks, by a library norm of the (separately pinned) dequantized
# rows, and by closed forms.

def _row(*blocks):
    return np.frombuffer(b"".join(blocks), dtype=np.uint8)


def test_row_norms_hand_blocks():
    # Q8_0, d = 0.5, q = 1, -1, 127, -128: values 0.5, -0.5, 63.5, -64, rest 0
    q8 = bytes([0x00, 0x38, 0x01, 0xFF, 0x7F, 0x80]) + bytes(28)
    assert oracle.row_norms(Q8_0, _row(q8), 0, 1, 32)[0] == math.sqrt(
        0.25 + 0.25 + 63.5 ** 2 + 64.0 ** 2)
    # two Q4_0 blocks in one row: (d = 1: e0 = 7, e1 = -8, e17 = -7, rest 0)
    # and (d = 2, every quant 0: 32 values of -16)
    a = bytes([0x00, 0x3C, 0x8F, 0x10]) + bytes([0x88] * 14)
    b = bytes([0x00, 0x40]) + bytes(16)
    assert oracle.row_norms(Q4_0, _row(a, b), 0, 1, 64)[0] == math.sqrt(
        49 + 64 + 49 + 32 * 256)
    # MXFP4, scale 1: 0.5, 6, -0, -6, rest 0
    mx = bytes([0x7F, 0x71, 0xF8]) + bytes(14)
    assert oracle.row_norms(MXFP4, _row(mx), 0, 1, 32)[0] == math.sqrt(0.25 + 36 + 36)


def test_row_norms_closed_forms():
    # constant quants: |d * c| * sqrt(in_dim); d = 0.25, c = -3, in_dim = 256
    blk = bytes([0x00, 0x34]) + bytes([0xFD] * 32)
    assert oracle.row_norms(Q8_0, _row(*[blk] * 8), 0, 1, 256)[0] == 0.75 * 16
    # zero scale: every value is 0 whatever the quants
    zero = bytes([0x00, 0x00]) + bytes([0x7F] * 32)
    assert oracle.row_norms(Q8_0, _row(*[zero] * 4), 0, 1, 128)[0] == 0.0
    # Q4_0 quants all 8 (value 0) except one nibble 15 (value 7*d), d = 2
    one = bytes([0x00, 0x40, 0x8F]) + bytes([0x88] * 15)
    assert oracle.row_norms(Q4_0, _row(one, one, one, one), 0, 1, 128)[0] == math.sqrt(4 * 196)


@pytest.mark.parametrize("fmt", FMTS + [oracle.Q4_K, oracle.Q6_K])
def test_row_norms_match_library_norm_of_dequantized_rows(fmt):
    rows, in_dim = 37, 512
    W = syn.quant_matrix(fmt, rows, in_dim, seed=90 + fmt)
    dense = oracle.dequantize(fmt, W).reshape(rows, in_dim).astype(np.float64)
    ref = np.linalg.norm(dense, axis=1)
    got = oracle.row_norms(fmt, W, 0, rows, in_dim)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=0)
    # a window reports the same rows, in window order
    assert np.array_equal(oracle.row_norms(fmt, W, 5, 20, in_dim), got[5:20])
