"""Pins of the oracle's Q4_K decoder (the K-quant of RAMforge, "Milestone 5
- Native Quantized Tensor Support").

The page gives the block size (256 elements in 144 B), the fields (half d,
half dmin, 12 B of packed 6-bit scales and mins, 128 B of 4-bit quants) and
the value d*sc*q - dmin*m.  It names but does not print the scale unpacking
or the quant order; those follow the GGML layout (parity unpinned by the
pages) and are pinned here by hand-worked bytes and by a reduction to the
already pinned Q4_0 decoder."""
import math
import struct

import numpy as np
import pytest

import oracle
import synthetic as syn

Q4_K, Q4_0 = oracle.Q4_K, oracle.Q4_0


def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def test_block_size_and_row_bytes_from_the_page():
    assert oracle.block_bytes(Q4_K) == 144
    assert oracle.block_elems(Q4_K) == 256
    assert oracle.row_bytes(Q4_K, 4096) == 16 * 144 == oracle.row_bytes(Q4_0, 4096)
    assert oracle.row_bytes(Q4_K, 4096 + 32) == 0        # not a whole super-block
    assert syn.row_bytes(Q4_K, 2048) == oracle.row_bytes(Q4_K, 2048)


def _lines(golden_dir, kind):
    for line in (golden_dir / "q4k.txt").read_text().splitlines():
        if line.startswith(kind + " |"):
            yield [p.strip() for p in line.split("|")[1:]]


def test_scale_unpacking_hand_table(golden_dir):
    n = 0
    for hexbytes, expect in _lines(golden_dir, "scales"):
        b = np.array([int(h, 16) for h in hexbytes.split()], dtype=np.uint8)
        for item in expect.split():
            j, v = item.split("=")
            sc, m = (int(t) for t in v.split(","))
            assert oracle.q4k_scale_min(b, int(j)) == (sc, m), (hexbytes, j)
        n += 1
    assert n == 3


def hand_block(golden_dir):
    """The worked block of the golden file: (144 raw bytes, 256 expected floats)."""
    (head, quants, expect), = list(_lines(golden_dir, "block"))
    blk = np.zeros(144, dtype=np.uint8)
    hb = [int(h, 16) for h in head.split()]
    blk[:len(hb)] = hb
    for item in quants.split():
        i, v = item.split(":")
        blk[16 + int(i)] = int(v, 16)
    want = [None] * 256
    for item in expect.split():
        rng, v = item.split("=")
        fv = 0.0 if v == "zero" else float.fromhex(v)
        a, _, b = rng.partition("-")
        for e in range(int(a), int(b or a) + 1):
            want[e] = fv
    assert None not in want
    return blk, want


def test_hand_block_bit_exact(golden_dir):
    blk, want = hand_block(golden_dir)
    got = oracle.dequantize(Q4_K, blk, 1)
    assert [f32_bits(float(g)) for g in got] == [f32_bits(w) for w in want]


def test_reduces_to_q4_0():
    """With every sub-block's scale 1 and min 8 and dmin = d, a Q4_K element is
    d*(q - 8): the Q4_0 value of the same nibble.  Written as Q4_0 blocks (in
    Q4_0's own nibble order) the same element sequence must decode to the same
    floats, which pins Q4_K's quant order against the Q4_0 decoder."""
    rng = np.random.default_rng(7)
    for d_bits in (0x3c00, 0x2e66, 0x0801):
        q = rng.integers(0, 16, size=256)                # element e's nibble
        blk = np.zeros(144, dtype=np.uint8)
        blk[0:2] = [d_bits & 0xFF, d_bits >> 8]
        blk[2:4] = [d_bits & 0xFF, d_bits >> 8]
        blk[4:8] = 1            # sc0..3 = 1 (top bits 0)
        blk[8:12] = 8           # m0..3 = 8 (top bits 0)
        blk[12:16] = 0x81       # sc4..7 = 1, m4..7 = 8
        for i in range(4):
            for l in range(32):
                blk[16 + 32 * i + l] = q[64 * i + l] | (q[64 * i + 32 + l] << 4)
        q40 = np.zeros((8, 18), dtype=np.uint8)
        for k in range(8):
            q40[k, 0:2] = [d_bits & 0xFF, d_bits >> 8]
            for j in range(16):
                q40[k, 2 + j] = q[32 * k + j] | (q[32 * k + 16 + j] << 4)
        a = oracle.dequantize(Q4_K, blk, 1)
        b = oracle.dequantize(Q4_0, q40, 8)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), hex(d_bits)


def test_scale_and_min_enter_linearly():
    """Doubling d and dmin doubles every value (exactly: a power-of-two
    scaling of exact products, rounded once)."""
    W = syn.quant_matrix(Q4_K, 1, 256, seed=9)
    W2 = W.copy()
    for off in (0, 2):
        h = np.frombuffer(W[0, off:off + 2].tobytes(), dtype="<f2")[0]
        W2[0, off:off + 2] = np.frombuffer(np.float16(2 * float(h)).tobytes(), dtype=np.uint8)
    a, b = oracle.dequantize(Q4_K, W, 1), oracle.dequantize(Q4_K, W2, 1)
    assert np.array_equal(b, 2 * a)


@pytest.mark.parametrize("rows,in_dim", [(1, 256), (4, 512), (3, 1024)])
def test_gemv_matches_bruteforce_fsum(rows, in_dim):
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=rows * 100 + in_dim)
    x = syn.normal_f32(in_dim, seed=in_dim + 1)
    y = oracle.gemv(Q4_K, W, 0, rows, in_dim, x)
    D = oracle.dequantize(Q4_K, W, rows * in_dim // 256).astype(np.float64).reshape(rows, in_dim)
    for r in range(rows):
        terms = [D[r, i] * float(x[i]) for i in range(in_dim)]
        assert abs(y[r] - math.fsum(terms)) <= 1e-12 * math.fsum(abs(t) for t in terms)


def test_gemv_one_hot_column_exact():
    rows, in_dim = 5, 512
    W = syn.quant_matrix(Q4_K, rows, in_dim, seed=3)
    D = oracle.dequantize(Q4_K, W, rows * 2).reshape(rows, in_dim)
    for i in (0, 31, 32, 63, 64, 255, 256, 511):
        x = np.zeros(in_dim, dtype=np.float32)
        x[i] = 1.0
        assert np.array_equal(oracle.gemv(Q4_K, W, 0, rows, in_dim, x), D[:, i])
