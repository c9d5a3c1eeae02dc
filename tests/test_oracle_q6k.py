"""Pins of the oracle's Q6_K decoder.

RAMforge ("Milestone 5 - Native Quantized Tensor Support") lists Q6_K among
its K-quant block layouts and neurostream's model list says its Q6_K decode
is bit-exact against the reference GGUF implementation; neither page prints
the layout, so the GGML layout is the reading (parity unpinned by the
pages).  Pinned here by hand-worked bytes (tests/golden/q6k.txt), by a
reduction to the already pinned Q8_0 decoder through an encoder written
from the layout in this file, and by the exactness of every value in fp32."""
import math
import struct

import numpy as np
import pytest

import oracle
import synthetic as syn

Q6_K, Q8_0 = oracle.Q6_K, oracle.Q8_0


def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def parse_value(v):
    if v == "zero":
        return 0.0
    if v == "negzero":
        return -0.0
    return float.fromhex(v)


def hand_blocks(golden_dir):
    out = []
    for line in (golden_dir / "q6k.txt").read_text().splitlines():
        if not line.startswith("block |"):
            continue
        _, raw, expect = (p.strip() for p in line.split("|"))
        blk = np.zeros(210, dtype=np.uint8)
        for item in raw.split():
            i, v = item.split(":")
            blk[int(i)] = int(v, 16)
        vals = [None] * 256
        for item in expect.split():
            rng, v = item.split("=")
            a, _, b = rng.partition("-")
            for e in range(int(a), int(b or a) + 1):
                vals[e] = parse_value(v)
        assert None not in vals
        out.append((blk, vals))
    return out


def test_block_size_and_row_bytes():
    assert oracle.block_bytes(Q6_K) == 210
    assert oracle.block_elems(Q6_K) == 256
    assert oracle.row_bytes(Q6_K, 4096) == 16 * 210
    assert oracle.row_bytes(Q6_K, 4096 + 32) == 0          # not a whole super-block
    assert syn.row_bytes(Q6_K, 2048) == oracle.row_bytes(Q6_K, 2048)


def test_hand_blocks_bit_exact(golden_dir):
    blocks = hand_blocks(golden_dir)
    assert len(blocks) == 2
    for blk, vals in blocks:
        got = oracle.dequantize(Q6_K, blk)
        for e, v in enumerate(vals):
            assert f32_bits(got[e]) == f32_bits(v), (e, got[e], v)


def encode(q, scales, d_bits):
    """A Q6_K block from 256 quants (0..63), 16 scales and fp16 d bits, laid
    out per the layout reading: the inverse of the decoder, written here from
    the layout rather than from the oracle."""
    blk = np.zeros(210, dtype=np.uint8)
    for n in range(2):
        for k in range(4):
            for l in range(32):
                v = int(q[128 * n + 32 * k + l])
                i = 64 * n + l + 32 * (k & 1)
                blk[i] |= (v & 15) << (4 if k >= 2 else 0)
                blk[128 + 32 * n + l] |= (v >> 4) << (2 * k)
    blk[192:208] = np.asarray(scales, dtype=np.int8).view(np.uint8)
    blk[208], blk[209] = d_bits & 0xFF, d_bits >> 8
    return blk


def test_quant_positions_round_trip():
    rng = np.random.default_rng(5)
    q = rng.integers(0, 64, size=256)
    blk = encode(q, np.zeros(16), 0x3C00)
    assert [oracle.q6k_quant(blk, e) for e in range(256)] == q.tolist()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_reduction_to_q8_0(seed):
    """With d = 2^-4 and the two scales of every 32-element run equal, a Q6_K
    super-block holds the same values as eight Q8_0 blocks with d_j =
    scale_2j / 16 (exact in fp16) and quants q - 32 (int8)."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 64, size=256)
    pair = rng.integers(-128, 128, size=8)
    scales = np.repeat(pair, 2)
    blk = encode(q, scales, 0x2C00)    # fp16 0x2c00 = 2^-4
    q8 = np.zeros((8, 34), dtype=np.uint8)
    for j in range(8):
        q8[j, 0:2] = np.frombuffer(np.float16(pair[j] / 16).tobytes(), dtype=np.uint8)
        q8[j, 2:] = (q[32 * j:32 * j + 32] - 32).astype(np.int8).view(np.uint8)
    a = oracle.dequantize(Q6_K, blk)
    b = oracle.dequantize(Q8_0, q8.reshape(-1))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_every_value_exact_in_fp32():
    """|d * scale * (q - 32)| needs at most 11 + 8 + 6 significant bits, so
    the float result equals the exact product (checked in fp64 over random
    blocks, subnormal d included)."""
    W = syn.quant_matrix(Q6_K, 64, 1024, seed=7)
    W[:4, 208::210] = 0x01      # subnormal d in the first rows' blocks
    W[:4, 209::210] = 0x00
    got = oracle.dequantize(Q6_K, W).astype(np.float64).reshape(-1, 256)
    blocks = W.reshape(-1, 210)
    for b in range(0, blocks.shape[0], 7):
        blk = blocks[b]
        d = float(np.frombuffer(blk[208:210].tobytes(), dtype="<f2")[0])
        sc = blk[192:208].view(np.int8).astype(np.float64)
        for e in range(0, 256, 5):
            exact = d * sc[e // 16] * (oracle.q6k_quant(blk, e) - 32)
            assert got[b, e] == exact


@pytest.mark.parametrize("rows,in_dim", [(1, 256), (4, 512), (3, 1024)])
def test_gemv_matches_bruteforce_fsum(rows, in_dim):
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=rows * 100 + in_dim)
    x = syn.normal_f32(in_dim, seed=in_dim + 2)
    y = oracle.gemv(Q6_K, W, 0, rows, in_dim, x)
    D = oracle.dequantize(Q6_K, W).astype(np.float64).reshape(rows, in_dim)
    for r in range(rows):
        terms = [D[r, i] * float(x[i]) for i in range(in_dim)]   # exact products
        assert abs(y[r] - math.fsum(terms)) <= 1e-12 * math.fsum(abs(t) for t in terms)


def test_gemv_one_hot_column_exact():
    rows, in_dim = 5, 512
    W = syn.quant_matrix(Q6_K, rows, in_dim, seed=4)
    D = oracle.dequantize(Q6_K, W).reshape(rows, in_dim)
    for i in (0, 15, 16, 31, 32, 127, 128, 255, 256, 511):
        x = np.zeros(in_dim, dtype=np.float32)
        x[i] = 1.0
        assert np.array_equal(oracle.gemv(Q6_K, W, 0, rows, in_dim, x), D[:, i])
