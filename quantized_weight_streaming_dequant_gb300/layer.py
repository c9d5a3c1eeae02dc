"""Compositions of the C ABI calls into the decode steps the library serves.

Nothing here computes: each function only sequences C ABI launches (through
the binding) on one stream.

DenseLayer -- one dense decode layer held resident in HBM: the Q, K and V
  projections of x in one batched launch, the O projection of the attention
  output, then the two-phase SwiGLU FFN (gate/up with the SwiGLU epilogue, then
  down).  The attention core between QKV and O is not part of this library; its
  output is an input here.
StreamedFFN -- a dense FFN whose weights stay in page-locked host memory: up
  (host-streamed), GELU, down (host-streamed), all through one arena; or the
  same FFN read in place over the host link (zero copy).
"""
from __future__ import annotations

from dataclasses import dataclass

import quantized_weight_streaming_dequant_gb300 as rf


@dataclass
class DenseLayer:
    fmt: int
    d_model: int
    d_ff: int
    wq: object
    wk: object
    wv: object
    wo: object
    w_gate: object
    w_up: object
    w_down: object

    def step(self, x, attn, x_ffn, out, stream=None, chain: bool = True):
        """out: dict of device tensors q, k, v, o, h, y (preallocated), and
        optionally hd, an ffn_workspace for h's digits.  With
        `chain`, each launch copies its (static) weights while the previous
        kernel on the stream drains (RF_CHAIN)."""
        d = self.d_model
        fl = rf.CHAIN if chain else 0
        rf.gemv_batch(self.fmt, d, [(self.wq, 0, d, x, out["q"]), (self.wk, 0, d, x, out["k"]),
                                    (self.wv, 0, d, x, out["v"])], stream=stream, flags=fl)
        rf.gemv(self.fmt, self.wo, 0, d, d, attn, out["o"], stream=stream, flags=fl)
        rf.ffn_swiglu(self.fmt, self.w_gate, self.w_up, self.w_down, self.d_ff, d, x_ffn,
                      out["y"], out["h"], stream=stream, flags=fl, workspace=out.get("hd"))

    def weight_bytes(self) -> int:
        rb_d = rf.row_bytes(self.fmt, self.d_model)
        rb_ff = rf.row_bytes(self.fmt, self.d_ff)
        return 4 * self.d_model * rb_d + 2 * self.d_ff * rb_d + self.d_model * rb_ff

    @staticmethod
    def launches_per_step() -> int:
        return 4   # QKV batch, O, gate/up+SwiGLU, down


@dataclass
class StreamedFFN:
    fmt: int
    d_model: int
    d_ff: int
    host_up: object     # page-locked [d_ff][d_model] bytes
    host_down: object   # page-locked [d_model][d_ff] bytes

    def step(self, arena, x, u, h, y, block_rows, depth, stream=None):
        arena.stream_linear(self.fmt, self.host_up, self.d_model, 0, self.d_ff, block_rows, depth,
                            x, u, stream=stream)
        rf.gelu(u, h, stream=stream)
        arena.stream_linear(self.fmt, self.host_down, self.d_ff, 0, self.d_model, block_rows,
                            depth, h, y, stream=stream)

    def step_zero_copy(self, x, u, h, y, stream=None):
        """The same FFN with both projections read in place from page-locked
        host memory (rf_gemv_host): no arena, no copy engine."""
        rf.gemv_host(self.fmt, self.host_up, 0, self.d_ff, self.d_model, x, u, stream=stream)
        rf.gelu(u, h, stream=stream)
        rf.gemv_host(self.fmt, self.host_down, 0, self.d_model, self.d_ff, h, y, stream=stream)

    def weight_bytes(self) -> int:
        return (self.d_ff * rf.row_bytes(self.fmt, self.d_model) +
                self.d_model * rf.row_bytes(self.fmt, self.d_ff))
