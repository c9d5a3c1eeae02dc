"""CPU oracle for the row-window dequant-GEMV path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product library never links, loads or calls it, and it shares no code with
the CUDA path.  The arithmetic lives in ``rf_oracle.c`` (plain C, fp64); this
module only builds it with gcc and marshals numpy arrays through ctypes.

Every function cites the page passage it follows in ``rf_oracle.c``.  Parity
status: the MXFP4 block layout, the GELU activation of the host-streamed FFN,
Q4_K's scale packing and quant order, and the Q6_K layout are "parity
unpinned" by the pages themselves (no page prints them); they are pinned in
tests by the OCP MX format definition, the GELU identities, a reduction of
Q4_K to Q4_0 and a reduction of Q6_K to Q8_0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "rf_oracle.c"
_LIBDIR = _HERE / "_lib"
_SO = _LIBDIR / "liboracle.so"

Q4_0, Q8_0, MXFP4, Q4_K, Q6_K = 2, 8, 39, 12, 14
FORMATS = {"Q4_0": Q4_0, "Q8_0": Q8_0, "MXFP4": MXFP4, "Q4_K": Q4_K, "Q6_K": Q6_K}


def build(force: bool = False) -> Path:
    """Compile rf_oracle.c into a shared library (gcc, no CUDA)."""
    if _SO.exists() and not force and _SO.stat().st_mtime >= _SRC.stat().st_mtime:
        return _SO
    _LIBDIR.mkdir(exist_ok=True)
    tmp = _SO.with_suffix(f".{os.getpid()}.tmp")
    subprocess.run(
        ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
         "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"],
        check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(str(build()))
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def _declare(L: ctypes.CDLL) -> None:
    L.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_fp16_to_double.restype = ctypes.c_double
    L.orc_e8m0_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e8m0_to_double.restype = ctypes.c_double
    L.orc_e2m1_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_to_double.restype = ctypes.c_double
    L.orc_block_bytes.argtypes = [_I]
    L.orc_block_bytes.restype = _I64
    L.orc_row_bytes.argtypes = [_I, _I64]
    L.orc_row_bytes.restype = _I64
    L.orc_block_elems.argtypes = [_I]
    L.orc_block_elems.restype = _I64
    L.orc_q4k_scale_min.argtypes = [_P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]
    L.orc_swiglu_clamped.argtypes = [ctypes.c_double] * 4
    L.orc_swiglu_clamped.restype = ctypes.c_double
    L.orc_moe_ffn_biased.argtypes = [_I, _P, _I, _I, _P, _P, _P, _P, _P, _P, ctypes.c_double,
                                     ctypes.c_double, _I64, _I64, _P, _P, _P, _P, _P]
    L.orc_q6k_quant.argtypes = [_P, _I]
    L.orc_q6k_quant.restype = _I
    L.orc_dequant_block.argtypes = [_I, _P, _P]
    L.orc_dequantize.argtypes = [_I, _P, _I64, _P]
    L.orc_gemv.argtypes = [_I, _P, _I64, _I64, _I64, _P, _P]
    L.orc_gemv_d.argtypes = [_I, _P, _I64, _I64, _I64, _P, _P]
    L.orc_row_norms.argtypes = [_I, _P, _I64, _I64, _I64, _P]
    L.orc_plan_block_rows.argtypes = [_I64, _I64, _I64, _I, _I64]
    L.orc_plan_block_rows.restype = _I64
    L.orc_stream_linear.argtypes = [_I, _P, _I64, _I64, _I64, _I64, _I, _I64, _P, _P,
                                    _P, _P, _P]
    L.orc_silu.argtypes = [ctypes.c_double]
    L.orc_silu.restype = ctypes.c_double
    L.orc_gelu.argtypes = [ctypes.c_double]
    L.orc_gelu.restype = ctypes.c_double
    L.orc_router_topk.argtypes = [_P, _I, _I, _P, _P]
    L.orc_ffn_swiglu.argtypes = [_I, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _P, _P, _P]
    L.orc_moe_ffn.argtypes = [_I, _P, _I, _I, _P, _P, _P, _I64, _I64, _P, _P, _P, _P]


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def _u8(W) -> np.ndarray:
    return np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)


def fp16_to_double(bits: int) -> float:
    return lib().orc_fp16_to_double(bits)


def e8m0_to_double(E: int) -> float:
    return lib().orc_e8m0_to_double(E)


def e2m1_to_double(code: int) -> float:
    return lib().orc_e2m1_to_double(code)


def block_bytes(fmt: int) -> int:
    return lib().orc_block_bytes(fmt)


def row_bytes(fmt: int, in_dim: int) -> int:
    return lib().orc_row_bytes(fmt, in_dim)


def block_elems(fmt: int) -> int:
    return lib().orc_block_elems(fmt)


def q6k_quant(block, e: int) -> int:
    """Q6_K element e's 6-bit quant (0..63) from one 210-byte block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    return lib().orc_q6k_quant(_ptr(b), e)


def q4k_scale_min(scale_bytes, j: int):
    """(scale, min) of Q4_K sub-block j from its 12 scale bytes."""
    b = np.ascontiguousarray(scale_bytes, dtype=np.uint8)
    sc, m = _I(0), _I(0)
    lib().orc_q4k_scale_min(_ptr(b), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def dequantize(fmt: int, W, n_blocks: int | None = None) -> np.ndarray:
    """Dequantize consecutive blocks to float32 (exact values)."""
    Wb = _u8(W)
    if n_blocks is None:
        n_blocks = Wb.size // block_bytes(fmt)
    out = np.empty(block_elems(fmt) * n_blocks, dtype=np.float32)
    _check(lib().orc_dequantize(fmt, _ptr(Wb), n_blocks, _ptr(out)), "dequantize")
    return out


def gemv(fmt: int, W, row_start: int, row_end: int, in_dim: int, x) -> np.ndarray:
    """fp64 row-window matvec of the raw [out][in] matrix W with x."""
    Wb = _u8(W)
    y = np.empty(max(row_end - row_start, 0), dtype=np.float64)
    x = np.asarray(x)
    if x.dtype == np.float64:
        xd = np.ascontiguousarray(x)
        _check(lib().orc_gemv_d(fmt, _ptr(Wb), row_start, row_end, in_dim, _ptr(xd), _ptr(y)),
               "gemv")
    else:
        xf = np.ascontiguousarray(x, dtype=np.float32)
        _check(lib().orc_gemv(fmt, _ptr(Wb), row_start, row_end, in_dim, _ptr(xf), _ptr(y)),
               "gemv")
    return y


def row_norms(fmt: int, W, row_start: int, row_end: int, in_dim: int) -> np.ndarray:
    Wb = _u8(W)
    out = np.empty(max(row_end - row_start, 0), dtype=np.float64)
    _check(lib().orc_row_norms(fmt, _ptr(Wb), row_start, row_end, in_dim, _ptr(out)),
           "row_norms")
    return out


def plan_block_rows(row_bytes_: int, n_rows: int, block_rows: int, depth: int,
                    arena_bytes: int) -> int:
    """Effective rows per block after shrink-to-fit; -1 if nothing fits."""
    return lib().orc_plan_block_rows(row_bytes_, n_rows, block_rows, depth, arena_bytes)


def stream_linear(fmt: int, W, row_start: int, row_end: int, in_dim: int, block_rows: int,
                  depth: int, arena_bytes: int, x):
    """Emulated block streaming; returns (y, eff_rows, n_blocks, peak_bytes)."""
    Wb = _u8(W)
    xf = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(max(row_end - row_start, 0), dtype=np.float64)
    eff, nblk, peak = _I64(0), _I64(0), _I64(0)
    rc = lib().orc_stream_linear(fmt, _ptr(Wb), row_start, row_end, in_dim, block_rows, depth,
                                 arena_bytes, _ptr(xf), _ptr(y), ctypes.byref(eff),
                                 ctypes.byref(nblk), ctypes.byref(peak))
    if rc == 3:
        raise MemoryError("arena too small for depth+1 one-row blocks")
    _check(rc, "stream_linear")
    return y, eff.value, nblk.value, peak.value


def silu(z: float) -> float:
    return lib().orc_silu(z)


def gelu(z: float) -> float:
    return lib().orc_gelu(z)


def router_topk(logits, top_k: int):
    lf = np.ascontiguousarray(logits, dtype=np.float32)
    idx = np.empty(top_k, dtype=np.int32)
    w = np.empty(top_k, dtype=np.float64)
    _check(lib().orc_router_topk(_ptr(lf), lf.size, top_k, _ptr(idx), _ptr(w)), "router_topk")
    return idx, w


def ffn_swiglu(fmt: int, gate, up, down, n_ff: int, n_embd: int, x, g0: int = 0,
               u0: int = 0, d0: int = 0):
    """Two-phase SwiGLU FFN; returns (y, h) in float64."""
    g, u, d = _u8(gate), _u8(up), _u8(down)
    xf = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(n_embd, dtype=np.float64)
    h = np.empty(n_ff, dtype=np.float64)
    _check(lib().orc_ffn_swiglu(fmt, _ptr(g), g0, _ptr(u), u0, _ptr(d), d0, n_ff, n_embd,
                                _ptr(xf), _ptr(y), _ptr(h)), "ffn_swiglu")
    return y, h


def moe_ffn(fmt: int, logits, top_k: int, gate, up, down, n_ff: int, n_embd: int, x):
    """Routed MoE SwiGLU FFN; returns (y, idx, w)."""
    lf = np.ascontiguousarray(logits, dtype=np.float32)
    g, u, d = _u8(gate), _u8(up), _u8(down)
    xf = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(n_embd, dtype=np.float64)
    idx = np.empty(top_k, dtype=np.int32)
    w = np.empty(top_k, dtype=np.float64)
    _check(lib().orc_moe_ffn(fmt, _ptr(lf), lf.size, top_k, _ptr(g), _ptr(u), _ptr(d), n_ff,
                             n_embd, _ptr(xf), _ptr(y), _ptr(idx), _ptr(w)), "moe_ffn")
    return y, idx, w


def gelu_vec(z) -> np.ndarray:
    return np.array([gelu(float(v)) for v in np.asarray(z).reshape(-1)], dtype=np.float64)


def silu_vec(z) -> np.ndarray:
    return np.array([silu(float(v)) for v in np.asarray(z).reshape(-1)], dtype=np.float64)


def swiglu_clamped(g: float, u: float, alpha: float, limit: float) -> float:
    """The biased experts' clamped SwiGLU (reading in rf_oracle.c)."""
    return lib().orc_swiglu_clamped(g, u, alpha, limit)


def _opt_f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def moe_ffn_biased(fmt: int, logits, top_k: int, gate, up, down, gate_bias, up_bias, down_bias,
                   alpha: float, limit: float, n_ff: int, n_embd: int, x):
    """Routed MoE over biased experts with the clamped SwiGLU; biases are
    (n_expert, n_ff), (n_expert, n_ff), (n_expert, n_embd) arrays or None.
    Returns (y, idx, w, h) with h the selected experts' activations."""
    lf = np.ascontiguousarray(logits, dtype=np.float32)
    g, u, d = _u8(gate), _u8(up), _u8(down)
    gb, ub, db = _opt_f64(gate_bias), _opt_f64(up_bias), _opt_f64(down_bias)
    xf = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(n_embd, dtype=np.float64)
    idx = np.empty(top_k, dtype=np.int32)
    w = np.empty(top_k, dtype=np.float64)
    h = np.empty((top_k, n_ff), dtype=np.float64)
    ptr = lambda a: None if a is None else _ptr(a)   # noqa: E731
    _check(lib().orc_moe_ffn_biased(fmt, _ptr(lf), lf.size, top_k, _ptr(g), _ptr(u), _ptr(d),
                                    ptr(gb), ptr(ub), ptr(db), float(alpha), float(limit), n_ff,
                                    n_embd, _ptr(xf), _ptr(y), _ptr(idx), _ptr(w), _ptr(h)),
           "moe_ffn_biased")
    return y, idx, w, h
