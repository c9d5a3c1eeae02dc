"""Python binding of the rf C ABI (include/rf.h): argument marshalling only.

Every computation runs in the CUDA kernels of ``_lib/librf.so``; this module
turns torch tensors into pointers and stream handles, allocates outputs with
torch (device memory is plumbing), and raises ``RFError`` on any non-OK
status.  There is no CPU fallback: if the library is missing or no GPU is
present, calls fail loudly.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

PKG = Path(__file__).resolve().parent
SO = PKG / "_lib" / "librf.so"
HEADER = PKG.parent / "include" / "rf.h"

Q4_0, Q8_0, Q4_K, Q6_K, MXFP4 = 2, 8, 12, 14, 39
FORMATS = {"Q4_0": Q4_0, "Q8_0": Q8_0, "Q4_K": Q4_K, "Q6_K": Q6_K, "MXFP4": MXFP4}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q4_K: 144, Q6_K: 210, MXFP4: 17}
BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q6_K: 256, MXFP4: 32}

OK = 0
CHAIN = 1   # RF_CHAIN launch flag
STATUS = {0: "RF_OK", 1: "RF_ERR_INVALID_ARG", 2: "RF_ERR_UNSUPPORTED_FMT",
          3: "RF_ERR_NOT_PINNED", 4: "RF_ERR_ARENA_TOO_SMALL", 5: "RF_ERR_CUDA",
          6: "RF_ERR_TIMEOUT", 7: "RF_ERR_OOM", 8: "RF_ERR_MISALIGNED", 9: "RF_ERR_TOO_LARGE"}


class RFError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class Window(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("row_start", ctypes.c_int64),
                ("row_end", ctypes.c_int64), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class StreamStats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("blocks", ctypes.c_uint64),
                ("bytes_copied", ctypes.c_uint64), ("peak_bytes", ctypes.c_uint64),
                ("slot_bytes", ctypes.c_uint64), ("arena_bytes", ctypes.c_uint64),
                ("slots", ctypes.c_int32), ("last_block_rows", ctypes.c_int32)]


class ExpertCacheStats(ctypes.Structure):
    _fields_ = [("lookups", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("fills", ctypes.c_uint64), ("bypasses", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("bytes_streamed", ctypes.c_uint64),
                ("bytes_cached", ctypes.c_uint64), ("slots", ctypes.c_int32),
                ("used", ctypes.c_int32)]


_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "rf_status_str": ([_I], ctypes.c_char_p),
    "rf_version": ([], _I),
    "rf_block_bytes": ([_I], _SZ),
    "rf_row_bytes": ([_I, _I64], _SZ),
    "rf_max_in_dim": ([_I, _I], _I64),
    "rf_dequantize": ([_I, _P, _I64, _P, _P], _I),
    "rf_gemv": ([_I, _P, _I64, _I64, _I64, _P, _P, _P], _I),
    "rf_gemv_batch": ([_I, _I64, _I, ctypes.POINTER(Window), _P], _I),
    "rf_gemv_ex": ([_I, _P, _I64, _I64, _I64, _P, _P, ctypes.c_uint, _P], _I),
    "rf_gemv_batch_ex": ([_I, _I64, _I, ctypes.POINTER(Window), ctypes.c_uint, _P], _I),
    "rf_ffn_swiglu_ex": ([_I, _P, _P, _P, _I64, _I64, _P, _P, _P, ctypes.c_uint, _P], _I),
    "rf_swiglu": ([_P, _P, _P, _I64, _P], _I),
    "rf_gelu": ([_P, _P, _I64, _P], _I),
    "rf_ffn_swiglu": ([_I, _P, _P, _P, _I64, _I64, _P, _P, _P, _P], _I),
    "rf_ffn_workspace_bytes": ([_I64], _SZ),
    "rf_gemv_host": ([_I, _P, _I64, _I64, _I64, _P, _P, _P], _I),
    "rf_gemm": ([_I, _P, _I64, _I64, _I64, _I, _P, _I64, _P, _I64, _P, _SZ, _P], _I),
    "rf_gemm_workspace_bytes": ([_I, _I64, _I], _SZ),
    "rf_gemv_multi": ([_I, _P, _I64, _I64, _I64, _I, _P, _I64, _P, _I64, ctypes.c_uint, _P], _I),
    "rf_ffn_swiglu_ws": ([_I, _P, _P, _P, _I64, _I64, _P, _P, _P, _P, ctypes.c_uint, _P], _I),
    "rf_arena_create": ([_SZ, _I, ctypes.POINTER(_P)], _I),
    "rf_arena_destroy": ([_P], None),
    "rf_arena_wait": ([_P, _I], _I),
    "rf_arena_inject_fault": ([_P, _I, _I64, _I], _I),
    "rf_arena_configure": ([_P, _I, _I], _I),
    "rf_stream_plan": ([_I, _I64, _I64, _I64, _I, _SZ, ctypes.POINTER(_I64),
                        ctypes.POINTER(_I64), ctypes.POINTER(_SZ)], _I),
    "rf_stream_linear": ([_I, _P, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _P], _I),
    "rf_stream_stats": ([_P, ctypes.POINTER(StreamStats)], _I),
    "rf_moe_route": ([_P, _I, _I, _P, _P, _P], _I),
    "rf_moe_workspace_bytes": ([_I, _I64, _I64, _I64], _SZ),
    "rf_moe_ffn": ([_I, _P, _I, _I, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P], _I),
    "rf_moe_ffn_biased": ([_I, _P, _I, _I, _P, _P, _P, _P, _P, _P, ctypes.c_float,
                           ctypes.c_float, _I64, _I64, _I64, _P, _P, _P, _P], _I),
    "rf_moe_ffn_noalloc": ([_I, _P, _I, _I, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P], _I),
    "rf_moe_ffn_host": ([_I, _P, _I, _I, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P], _I),
    "rf_expert_cache_create": ([_I, _I64, _I64, _I, ctypes.POINTER(_P)], _I),
    "rf_expert_cache_destroy": ([_P], None),
    "rf_expert_cache_stats": ([_P, ctypes.POINTER(ExpertCacheStats)], _I),
    "rf_moe_ffn_streamed": ([_I, _P, _I, _I, _P, _P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P,
                             _P], _I),
    "rf_device_status": ([], _I),
    "rf_debug_arm_wait_fault": ([ctypes.c_uint32], _I),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load librf.so (built by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not SO.exists():
            raise RuntimeError(f"{SO} is missing: build it with "
                               "`python -m quantized_weight_streaming_dequant_gb300.build`")
        L = ctypes.CDLL(str(SO))
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Names of the functions include/rf.h declares."""
    return re.findall(r"^RF_API[^(]*?\b(rf_\w+)\(", HEADER.read_text(), flags=re.M)


def _check(code: int, what: str) -> None:
    if code != OK:
        raise RFError(code, what)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_ptr(t, what: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def status_str(code: int) -> str:
    return lib().rf_status_str(code).decode()


def block_bytes(fmt: int) -> int:
    return lib().rf_block_bytes(fmt)


def row_bytes(fmt: int, in_dim: int) -> int:
    return lib().rf_row_bytes(fmt, in_dim)


def max_in_dim(fmt: int, n_x: int = 1) -> int:
    return lib().rf_max_in_dim(fmt, n_x)


def dequantize(fmt: int, W, n_blocks: int | None = None, out=None, stream=None):
    import torch
    if n_blocks is None:
        n_blocks = W.numel() // BLOCK_BYTES[fmt]
    if out is None:
        out = torch.empty(BLOCK_ELEMS[fmt] * n_blocks, dtype=torch.float32, device=W.device)
    _check(lib().rf_dequantize(fmt, _dev_ptr(W, "W"), n_blocks, _dev_ptr(out, "out"),
                               _stream(stream)), "rf_dequantize")
    return out


def gemv(fmt: int, W, row_start: int, row_end: int, in_dim: int, x, y=None, stream=None,
         flags: int = 0):
    import torch
    if y is None:
        y = torch.empty(max(row_end - row_start, 0), dtype=torch.float32, device=x.device)
    _check(lib().rf_gemv_ex(fmt, _dev_ptr(W, "W"), row_start, row_end, in_dim, _dev_ptr(x, "x"),
                            _dev_ptr(y, "y") if y.numel() else 1, flags, _stream(stream)),
           "rf_gemv")
    return y


def gemv_multi(fmt: int, W, row_start: int, row_end: int, in_dim: int, X, Y=None, stream=None,
               flags: int = 0):
    """rf_gemv_multi: X is (n_tok, in_dim) float32 on the device (rows may be
    strided); returns Y (n_tok, row_end - row_start)."""
    import torch
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be 2-D with unit stride along in_dim")
    n_tok = X.shape[0]
    if Y is None:
        Y = torch.empty(n_tok, max(row_end - row_start, 0), dtype=torch.float32, device=X.device)
    if Y.dim() != 2 or Y.stride(1) != 1:
        raise ValueError("Y must be 2-D with unit stride along the rows")
    _check(lib().rf_gemv_multi(fmt, _dev_ptr(W, "W"), row_start, row_end, in_dim, n_tok,
                               X.data_ptr(), X.stride(0), Y.data_ptr(), Y.stride(0), flags,
                               _stream(stream)), "rf_gemv_multi")
    return Y


def gemm_workspace_bytes(fmt: int, in_dim: int, n_tok: int) -> int:
    return int(lib().rf_gemm_workspace_bytes(fmt, in_dim, n_tok))


def gemm(fmt: int, W, row_start: int, row_end: int, in_dim: int, X, Y=None, workspace=None,
         stream=None):
    """rf_gemm (tensor cores): X is (n_tok, in_dim) float32 on the device
    (rows may be strided); returns Y (n_tok, row_end - row_start).  The
    workspace (a uint8 device tensor) is allocated when not given."""
    import torch
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be 2-D with unit stride along in_dim")
    n_tok = X.shape[0]
    if Y is None:
        Y = torch.empty(n_tok, max(row_end - row_start, 0), dtype=torch.float32, device=X.device)
    if Y.dim() != 2 or Y.stride(1) != 1:
        raise ValueError("Y must be 2-D with unit stride along the rows")
    need = gemm_workspace_bytes(fmt, in_dim, n_tok)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    ws, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) \
        if workspace is not None else (None, 0)
    _check(lib().rf_gemm(fmt, _dev_ptr(W, "W"), row_start, row_end, in_dim, n_tok,
                         X.data_ptr(), X.stride(0), Y.data_ptr(), Y.stride(0), ws, ws_bytes,
                         _stream(stream)), "rf_gemm")
    return Y


def gemv_batch(fmt: int, in_dim: int, windows, stream=None, flags: int = 0):
    """windows: list of (W, row_start, row_end, x, y) with device tensors."""
    arr = (Window * max(len(windows), 1))()
    for i, (W, r0, r1, x, y) in enumerate(windows):
        arr[i] = Window(_dev_ptr(W, "W"), r0, r1, _dev_ptr(x, "x"), _dev_ptr(y, "y"))
    _check(lib().rf_gemv_batch_ex(fmt, in_dim, len(windows), arr, flags, _stream(stream)),
           "rf_gemv_batch")


def swiglu(g, u, h=None, stream=None):
    import torch
    h = torch.empty_like(g) if h is None else h
    _check(lib().rf_swiglu(_dev_ptr(g, "g"), _dev_ptr(u, "u"), _dev_ptr(h, "h"), g.numel(),
                           _stream(stream)), "rf_swiglu")
    return h


def gelu(z, h=None, stream=None):
    import torch
    h = torch.empty_like(z) if h is None else h
    _check(lib().rf_gelu(_dev_ptr(z, "z"), _dev_ptr(h, "h"), z.numel(), _stream(stream)),
           "rf_gelu")
    return h


def gemv_host(fmt: int, host_W, row_start: int, row_end: int, in_dim: int, x, y=None,
              stream=None):
    """rf_gemv_host: host_W is a page-locked CPU tensor (uint8) read in place."""
    import torch
    if host_W.is_cuda or not host_W.is_contiguous():
        raise ValueError("host_W must be a contiguous CPU tensor")
    if y is None:
        y = torch.empty(max(row_end - row_start, 0), dtype=torch.float32, device=x.device)
    _check(lib().rf_gemv_host(fmt, host_W.data_ptr(), row_start, row_end, in_dim,
                              _dev_ptr(x, "x"), _dev_ptr(y, "y") if y.numel() else 1,
                              _stream(stream)), "rf_gemv_host")
    return y


def ffn_workspace(n_ff: int, device):
    """Device workspace for ffn_swiglu's digit hand-off between its launches."""
    import torch
    return torch.empty(lib().rf_ffn_workspace_bytes(n_ff), dtype=torch.uint8, device=device)


def ffn_swiglu(fmt: int, gate, up, down, n_ff: int, n_embd: int, x, y=None, h=None,
               stream=None, flags: int = 0, workspace=None):
    """rf_ffn_swiglu_ws (workspace: from ffn_workspace, or None)."""
    import torch
    y = torch.empty(n_embd, dtype=torch.float32, device=x.device) if y is None else y
    h = torch.empty(n_ff, dtype=torch.float32, device=x.device) if h is None else h
    _check(lib().rf_ffn_swiglu_ws(fmt, _dev_ptr(gate, "gate"), _dev_ptr(up, "up"),
                                  _dev_ptr(down, "down"), n_ff, n_embd, _dev_ptr(x, "x"),
                                  _dev_ptr(y, "y"), _dev_ptr(h, "h"),
                                  _dev_ptr(workspace, "workspace") if workspace is not None
                                  else None, flags, _stream(stream)),
           "rf_ffn_swiglu")
    return y, h


def stream_plan(fmt: int, in_dim: int, n_rows: int, block_rows: int, depth: int,
                arena_bytes: int):
    """(effective rows per block, blocks, peak arena bytes); host only."""
    eff, nblk, peak = _I64(0), _I64(0), _SZ(0)
    _check(lib().rf_stream_plan(fmt, in_dim, n_rows, block_rows, depth, arena_bytes,
                                ctypes.byref(eff), ctypes.byref(nblk), ctypes.byref(peak)),
           "rf_stream_plan")
    return eff.value, nblk.value, peak.value


FAULT_NONE, FAULT_COPY_FAIL, FAULT_COPY_STALL = 0, 1, 2
ARENA_MERGE_RUNS, ARENA_LANES = 1, 2


class Arena:
    """Bounded device arena with its copy stream (rf_arena_create); device -1
    = the current device."""

    def __init__(self, nbytes: int, device: int = -1):
        h = _P()
        _check(lib().rf_arena_create(nbytes, device, ctypes.byref(h)), "rf_arena_create")
        self.handle = h
        self.nbytes = nbytes

    def wait(self, timeout_ms: int) -> int:
        """rf_arena_wait: the status (OK, or TIMEOUT while work is outstanding)."""
        code = lib().rf_arena_wait(self.handle, timeout_ms)
        if code not in (OK, 6):
            raise RFError(code, "rf_arena_wait")
        return code

    def configure(self, option: int, value: bool) -> None:
        """rf_arena_configure: ARENA_MERGE_RUNS / ARENA_LANES on or off."""
        _check(lib().rf_arena_configure(self.handle, option, int(bool(value))),
               "rf_arena_configure")

    def inject_fault(self, kind: int, block: int, ms: int = 0) -> None:
        """rf_arena_inject_fault (test hook)."""
        _check(lib().rf_arena_inject_fault(self.handle, kind, block, ms), "rf_arena_inject_fault")

    def close(self) -> None:
        if self.handle is not None and self.handle.value:
            lib().rf_arena_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stream_linear(self, fmt: int, host_W, in_dim: int, row_start: int, row_end: int,
                      block_rows: int, depth: int, x, y=None, stream=None):
        """host_W: page-locked CPU tensor (uint8) holding row 0 onwards."""
        import torch
        if host_W.is_cuda or not host_W.is_contiguous():
            raise ValueError("host_W must be a contiguous CPU tensor")
        if y is None:
            y = torch.empty(max(row_end - row_start, 0), dtype=torch.float32, device=x.device)
        _check(lib().rf_stream_linear(fmt, host_W.data_ptr(), in_dim, row_start, row_end,
                                      block_rows, depth, self.handle, _dev_ptr(x, "x"),
                                      _dev_ptr(y, "y") if y.numel() else 1, _stream(stream)),
               "rf_stream_linear")
        return y

    def stats(self) -> dict:
        s = StreamStats()
        _check(lib().rf_stream_stats(self.handle, ctypes.byref(s)), "rf_stream_stats")
        return {k: getattr(s, k) for k, _ in StreamStats._fields_}


class ExpertCache:
    """Device cache of whole experts (rf_expert_cache_create)."""

    def __init__(self, fmt: int, n_ff: int, n_embd: int, slots: int):
        h = _P()
        _check(lib().rf_expert_cache_create(fmt, n_ff, n_embd, slots, ctypes.byref(h)),
               "rf_expert_cache_create")
        self.handle = h

    def close(self) -> None:
        if self.handle is not None and self.handle.value:
            lib().rf_expert_cache_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self) -> dict:
        s = ExpertCacheStats()
        _check(lib().rf_expert_cache_stats(self.handle, ctypes.byref(s)),
               "rf_expert_cache_stats")
        return {k: getattr(s, k) for k, _ in ExpertCacheStats._fields_}


def moe_ffn_streamed(fmt: int, logits, top_k: int, host_gate, host_up, host_down, n_ff: int,
                     n_embd: int, block_rows: int, depth: int, arena: "Arena", x, cache=None,
                     y=None, workspace=None, stream=None):
    """rf_moe_ffn_streamed: experts in page-locked CPU tensors, one layer-wide
    prefetch plan through `arena`, an optional ExpertCache."""
    import torch
    for t, nm in ((host_gate, "host_gate"), (host_up, "host_up"), (host_down, "host_down")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous CPU tensor")
    y = torch.empty(n_embd, dtype=torch.float32, device=x.device) if y is None else y
    if workspace is None:
        workspace = moe_workspace(top_k, n_ff, n_embd, block_rows, x.device)
    _check(lib().rf_moe_ffn_streamed(fmt, _dev_ptr(logits, "logits"), logits.numel(), top_k,
                                     host_gate.data_ptr(), host_up.data_ptr(),
                                     host_down.data_ptr(), n_ff, n_embd, block_rows, depth,
                                     arena.handle, cache.handle if cache is not None else None,
                                     _dev_ptr(x, "x"), _dev_ptr(y, "y"),
                                     _dev_ptr(workspace, "workspace"), _stream(stream)),
           "rf_moe_ffn_streamed")
    return y, workspace


def moe_route(logits, top_k: int, stream=None):
    import torch
    idx = torch.empty(top_k, dtype=torch.int32, device=logits.device)
    w = torch.empty(top_k, dtype=torch.float32, device=logits.device)
    _check(lib().rf_moe_route(_dev_ptr(logits, "logits"), logits.numel(), top_k,
                              _dev_ptr(idx, "idx"), _dev_ptr(w, "w"), _stream(stream)),
           "rf_moe_route")
    return idx, w


def moe_workspace_bytes(top_k: int, n_ff: int, n_embd: int, block_rows: int) -> int:
    return lib().rf_moe_workspace_bytes(top_k, n_ff, n_embd, block_rows)


def moe_workspace(top_k: int, n_ff: int, n_embd: int, block_rows: int, device):
    import torch
    n = moe_workspace_bytes(top_k, n_ff, n_embd, block_rows)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_ffn(fmt: int, logits, top_k: int, gate, up, down, n_ff: int, n_embd: int,
            block_rows: int, x, y=None, workspace=None, stream=None):
    import torch
    y = torch.empty(n_embd, dtype=torch.float32, device=x.device) if y is None else y
    if workspace is None:
        workspace = moe_workspace(top_k, n_ff, n_embd, block_rows, x.device)
    _check(lib().rf_moe_ffn(fmt, _dev_ptr(logits, "logits"), logits.numel(), top_k,
                            _dev_ptr(gate, "gate"), _dev_ptr(up, "up"), _dev_ptr(down, "down"),
                            n_ff, n_embd, block_rows, _dev_ptr(x, "x"), _dev_ptr(y, "y"),
                            _dev_ptr(workspace, "workspace"), _stream(stream)), "rf_moe_ffn")
    return y, workspace


def moe_ffn_biased(fmt: int, logits, top_k: int, gate, up, down, gate_bias, up_bias, down_bias,
                   alpha: float, limit: float, n_ff: int, n_embd: int, block_rows: int, x,
                   y=None, workspace=None, stream=None):
    """rf_moe_ffn_biased: biases are device float32 tensors (or None)."""
    import torch
    y = torch.empty(n_embd, dtype=torch.float32, device=x.device) if y is None else y
    if workspace is None:
        workspace = moe_workspace(top_k, n_ff, n_embd, block_rows, x.device)
    opt = lambda t, nm: None if t is None else _dev_ptr(t, nm)   # noqa: E731
    _check(lib().rf_moe_ffn_biased(fmt, _dev_ptr(logits, "logits"), logits.numel(), top_k,
                                   _dev_ptr(gate, "gate"), _dev_ptr(up, "up"),
                                   _dev_ptr(down, "down"), opt(gate_bias, "gate_bias"),
                                   opt(up_bias, "up_bias"), opt(down_bias, "down_bias"),
                                   alpha, limit, n_ff, n_embd, block_rows, _dev_ptr(x, "x"),
                                   _dev_ptr(y, "y"), _dev_ptr(workspace, "workspace"),
                                   _stream(stream)), "rf_moe_ffn_biased")
    return y, workspace


def moe_ffn_noalloc(fmt: int, logits, top_k: int, gate, up, down, n_ff: int, n_embd: int,
                    block_rows: int, x, y, stream=None):
    """rf_moe_ffn_noalloc: the library's own fixed scratch instead of a
    workspace; y must be preallocated."""
    _check(lib().rf_moe_ffn_noalloc(fmt, _dev_ptr(logits, "logits"), logits.numel(), top_k,
                                    _dev_ptr(gate, "gate"), _dev_ptr(up, "up"),
                                    _dev_ptr(down, "down"), n_ff, n_embd, block_rows,
                                    _dev_ptr(x, "x"), _dev_ptr(y, "y"), _stream(stream)),
           "rf_moe_ffn_noalloc")
    return y


def moe_ffn_host(fmt: int, logits, top_k: int, gate, up, down, n_ff: int, n_embd: int,
                 block_rows: int, x, y=None, workspace=None, stream=None):
    """rf_moe_ffn_host: gate/up/down are page-locked CPU tensors read in place."""
    import torch
    for t in (gate, up, down):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("expert tensors must be contiguous CPU tensors")
    y = torch.empty(n_embd, dtype=torch.float32, device=x.device) if y is None else y
    if workspace is None:
        workspace = moe_workspace(top_k, n_ff, n_embd, block_rows, x.device)
    _check(lib().rf_moe_ffn_host(fmt, _dev_ptr(logits, "logits"), logits.numel(), top_k,
                                 gate.data_ptr(), up.data_ptr(), down.data_ptr(), n_ff, n_embd,
                                 block_rows, _dev_ptr(x, "x"), _dev_ptr(y, "y"),
                                 _dev_ptr(workspace, "workspace"), _stream(stream)),
           "rf_moe_ffn_host")
    return y, workspace


def moe_workspace_views(workspace, top_k: int, n_ff: int):
    """(idx, w, h) views into an rf_moe_ffn workspace (for inspection)."""
    import torch
    idx = workspace[:32].view(torch.int32)[:top_k]
    w = workspace[256:288].view(torch.float32)[:top_k]
    h = workspace[512:512 + 4 * top_k * n_ff].view(torch.float32).view(top_k, n_ff)
    return idx, w, h


def device_status() -> int:
    """Synchronize and return (and clear) the kernels' device status word."""
    return lib().rf_device_status()


def debug_arm_wait_fault(limit_us: int) -> None:
    """rf_debug_arm_wait_fault (test hook): the next tensor-copy GEMV launch
    withholds one stage's copy and gives up its wait after limit_us."""
    _check(lib().rf_debug_arm_wait_fault(limit_us), "rf_debug_arm_wait_fault")
