"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and lays them out as raw GGUF-style
block bytes (scale bytes first, then quant bytes); it holds none of the
method's arithmetic (no decoding, no dot products).  Both the CUDA path and
the CPU oracle consume the same bytes.

Distributions (the workloads' statement):
  Q8_0   : q uniform over the integers [-127, 127]; d = fp16(U[1e-3, 1e-2]).
  Q4_0   : each 4-bit q uniform over [0, 15] (a uniform random byte holds two
           independent uniform nibbles); d = fp16(U[1e-3, 2e-2]).
  MXFP4  : each 4-bit E2M1 code uniform over its 16 values (random bytes);
           scale exponent byte E = 127 + U{-8, ..., -2}.
  Q4_K   : 256-element super-blocks of 144 B; quant bytes and the 12 packed
           scale bytes uniform random (so every 6-bit scale and min is
           uniform over [0, 63]); d = fp16(U[1e-4, 1e-3]), dmin =
           fp16(U[1e-4, 1e-3]).
  Q6_K   : 256-element super-blocks of 210 B: the 192 quant bytes (low and
           high parts) and the 16 signed scale bytes uniform random (every
           6-bit quant uniform over [0, 63], every scale over [-128, 127]),
           then d = fp16(U[1e-4, 1e-3]) in the last two bytes.
  x      : fp32 N(0, 1); router logits fp32 N(0, 1) (or, for expert-cache
           runs, a fixed per-expert bias 0.5*N(0,1) plus N(0,1) per token).

Reproducibility: rows are generated in fixed chunks of ``CHUNK_ROWS`` rows,
each from ``numpy.random.default_rng([seed, chunk])``, so the bytes depend
only on (seed, shape) and chunks may be drawn in parallel.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np

Q4_0, Q8_0, MXFP4, Q4_K, Q6_K = 2, 8, 39, 12, 14
FMT_IDS = {"Q4_0": Q4_0, "Q8_0": Q8_0, "MXFP4": MXFP4, "Q4_K": Q4_K, "Q6_K": Q6_K}
FMT_NAMES = {v: k for k, v in FMT_IDS.items()}
# (block bytes, quant bytes after the scale, scale bytes)
# (Q6_K keeps its fp16 scale in the last two bytes; the other 208 are drawn
# uniformly.)
_LAYOUT = {Q8_0: (34, 32, 2), Q4_0: (18, 16, 2), MXFP4: (17, 16, 1), Q4_K: (144, 140, 4),
           Q6_K: (210, 208, 2)}
DEFAULT_SCALE = {Q8_0: (1e-3, 1e-2), Q4_0: (1e-3, 2e-2), MXFP4: (-8, -2), Q4_K: (1e-4, 1e-3),
                 Q6_K: (1e-4, 1e-3)}
_ELEMS = {Q8_0: 32, Q4_0: 32, MXFP4: 32, Q4_K: 256, Q6_K: 256}
CHUNK_ROWS = 1024


def block_bytes(fmt: int) -> int:
    return _LAYOUT[fmt][0]


def block_elems(fmt: int) -> int:
    return _ELEMS[fmt]


def row_bytes(fmt: int, in_dim: int) -> int:
    assert in_dim % _ELEMS[fmt] == 0
    return in_dim // _ELEMS[fmt] * _LAYOUT[fmt][0]


def _fill_rows(fmt: int, out: np.ndarray, in_dim: int, seed: int, chunk: int,
               scale_range) -> None:
    rows = out.shape[0]
    nb = in_dim // _ELEMS[fmt]
    bb, nq, ns = _LAYOUT[fmt]
    rng = np.random.default_rng([seed, chunk])
    blk = out.reshape(rows, nb, bb)
    if fmt == Q8_0:
        q = rng.integers(-127, 128, size=(rows, nb, nq), dtype=np.int8)
        blk[:, :, ns:] = q.view(np.uint8)
    elif fmt == Q6_K:
        blk[:, :, :nq] = rng.integers(0, 256, size=(rows, nb, nq), dtype=np.uint8)
        d = rng.uniform(*scale_range, size=(rows, nb)).astype("<f2")
        blk[:, :, nq:] = d.view(np.uint8).reshape(rows, nb, 2)
        return
    else:
        blk[:, :, ns:] = rng.integers(0, 256, size=(rows, nb, nq), dtype=np.uint8)
    lo, hi = scale_range
    if fmt == Q4_K:   # d and dmin, both fp16
        dd = rng.uniform(lo, hi, size=(rows, nb, 2)).astype("<f2")
        blk[:, :, 0:4] = dd.view(np.uint8).reshape(rows, nb, 4)
    elif fmt == MXFP4:
        blk[:, :, 0] = (127 + rng.integers(lo, hi + 1, size=(rows, nb))).astype(np.uint8)
    else:
        d = rng.uniform(lo, hi, size=(rows, nb)).astype("<f2")
        blk[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)


def quant_matrix(fmt: int, rows: int, in_dim: int, seed: int, out: np.ndarray | None = None,
                 scale_range=None, threads: int = 1) -> np.ndarray:
    """Raw row-major [rows][row_bytes] matrix of ``fmt`` blocks (uint8)."""
    rb = row_bytes(fmt, in_dim)
    if out is None:
        out = np.empty((rows, rb), dtype=np.uint8)
    out = out.reshape(rows, rb)
    scale_range = DEFAULT_SCALE[fmt] if scale_range is None else scale_range
    chunks = [(c, c * CHUNK_ROWS, min(rows, (c + 1) * CHUNK_ROWS))
              for c in range((rows + CHUNK_ROWS - 1) // CHUNK_ROWS)]

    def work(item):
        c, r0, r1 = item
        _fill_rows(fmt, out[r0:r1], in_dim, seed, c, scale_range)

    if threads > 1 and len(chunks) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, chunks))
    else:
        for item in chunks:
            work(item)
    return out


def stacked_experts(fmt: int, n_expert: int, out_dim: int, in_dim: int, seed: int,
                    threads: int = 1) -> np.ndarray:
    """Stacked (n_expert, out, in) tensor as [n_expert*out][row_bytes] bytes."""
    return quant_matrix(fmt, n_expert * out_dim, in_dim, seed, threads=threads)


def normal_f32(n: int, seed: int) -> np.ndarray:
    return np.random.default_rng([seed, 0x5EED]).standard_normal(n).astype(np.float32)


def router_logits(n_expert: int, seed: int) -> np.ndarray:
    return np.random.default_rng([seed, 0x1061]).standard_normal(n_expert).astype(np.float32)


def skewed_router_logits(n_expert: int, n_tokens: int, seed: int,
                         skew: float = 0.5) -> np.ndarray:
    """(n_tokens, n_expert) logits with expert popularity: a fixed per-expert
    bias skew*N(0,1) plus N(0,1) per token.  skew = 0.5 makes the most
    popular 20 % of 128 experts take about 57 % of the top-4 selections."""
    rng = np.random.default_rng([seed, 0x5e1])
    bias = skew * rng.standard_normal(n_expert)
    return (bias[None, :] + rng.standard_normal((n_tokens, n_expert))).astype(np.float32)


# ----------------------------------------------------------------- workloads
# Shapes, formats and seeds of the synthetic workloads (data only).

C1 = dict(name="q8_0_gemv_512x2048_streamed", fmt=Q8_0, out_dim=512, in_dim=2048,
          block_rows=128, depth=4, arena_bytes=256 << 20, seed=0)

C2 = dict(name="q4_0_dense_decode_layer_resident", fmt=Q4_0, d_model=4096, d_ff=11008,
          seed=1, copies=8)

C3 = dict(name="mxfp4_moe_ffn_128x2880x2880_top4", fmt=MXFP4, n_expert=128, n_ff=2880,
          n_embd=2880, top_k=4, block_rows=512, seed=2)

C4 = dict(name="q8_0_host_streamed_ffn_44x24576x6144", fmt=Q8_0, n_layer=44, d_model=6144,
          d_ff=24576, arena_bytes=256 << 20, block_rows=512, depth=4, seed=3)

SWEEP_FORMATS = (Q8_0, Q4_0, MXFP4)
SWEEP_IN = (2048, 4096, 8192)
SWEEP_OUT = (4096, 16384)
SWEEP_BLOCK_ROWS = (128, 256, 512, 1024, 0)   # 0 = whole matrix


def sweep_cells():
    """The 90 (format, in, out, block_rows) cells, format-major, seed 1000+i.
    Each cell is measured resident and host-streamed."""
    cells = []
    i = 0
    for fmt in SWEEP_FORMATS:
        for in_dim in SWEEP_IN:
            for out_dim in SWEEP_OUT:
                for br in SWEEP_BLOCK_ROWS:
                    cells.append(dict(fmt=fmt, in_dim=in_dim, out_dim=out_dim, block_rows=br,
                                      seed=1000 + i))
                    i += 1
    return cells
