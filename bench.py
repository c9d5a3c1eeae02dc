"""Benchmark: effective weight GB/s of the fused dequant-GEMV path.

Headline workload (default, one line of JSON from rank 0): a dense decode
layer held resident in HBM, Q4_0 -- Q/K/V/O 4096x4096, gate/up 11008x4096,
down 4096x11008, SwiGLU between gate/up and down, batch 1, x ~ N(0,1).  One
step = one pass of the layer for one token: 4 kernel launches (QKV batched,
O, gate/up with the SwiGLU epilogue, down).  Eight distinct layer copies
(910 MB, > L2) are walked round-robin so every step reads its weights from
HBM.  value = weight bytes streamed per second (whole job over all ranks);
tokens/s equivalent = value / active bytes per token (one layer here).

Also reported (each its own sub-object): the host-streamed Q8_0 GEMV
(512x2048, 128-row blocks), the routed MXFP4 MoE FFN (128 experts, top-4,
512-row windows) resident, read in place from host memory, and streamed from
host memory through the layer-wide prefetch plan with expert caches, the same
dense layer with Q4_K weights, and the host-streamed 44-layer Q8_0 FFN
(24576x6144, 256 MiB arena, 512-row blocks, depth 4), the streamed ones
measured against the pinned host-to-device bandwidth probed in the same run.

--impl reference times the CPU oracle (plain C, fp64, one host core) on a
bounded sample of the same workload and prints the same line with
"impl": "reference".  Under torchrun (N > 1) every rank runs its own replica
(no data-path collective: the layer is replicated, not sharded); value sums
the ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synthetic as syn  # noqa: E402

METRIC = "effective weight GB/s of dequant-GEMV (% of HBM / H2D peak); tokens/s equivalent"
FALLBACK_HBM_GBS = 6800.0
REPEATS = 5   # timed repeats of each headline region; the value is their median
DTYPE = ("q4_0 weights x int16 activation digits (per 32-block, power-of-two scale), "
         "exact int32 block dot, fp32 across blocks")


# ---------------------------------------------------------------- helpers

def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Measured dense bf16 TF/s (burst), else the fallback figure."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["bf16_tflops"]), "measured"
        except Exception:
            pass
    return 1900.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("rf_gemv.cu", "rf_device.cuh", "rf_internal.h"):
        h.update((ROOT / "quantized_weight_streaming_dequant_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """Per-launch DRAM bytes of the GEMV kernel from the committed ncu summary,
    or None if the kernel source changed since it was captured."""
    p = ROOT / "profiles" / "ncu_traffic.txt"
    if not p.exists():
        return None
    cur = kernel_source_hash()
    for line in p.read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload and parts[1] == cur:
            return float(parts[2])
    return None


def reduce_time_max(torch, dist, ms: float, device) -> float:
    """The slowest rank's timed region (max over ranks); unchanged on one rank."""
    if not dist:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, ms_total: float) -> float:
    """Bytes every rank streamed (each rank runs its own replica) over the
    slowest rank's time."""
    return bytes_per_step * steps * world / (ms_total * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [v.strip() for v in ln.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def h2d_probe(torch, device, nbytes: int, reps: int = 5):
    """Pinned host->device copy bandwidth (GB/s) for transfers of nbytes."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s = torch.cuda.current_stream()
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize()
    return nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9


# ------------------------------------------------------------- workloads

def build_dense_layers(torch, rf, device, copies: int, seed: int, fmt: int = syn.Q4_0):
    from quantized_weight_streaming_dequant_gb300.layer import DenseLayer
    d, f = syn.C2["d_model"], syn.C2["d_ff"]
    layers = []
    for c in range(copies):
        s = seed * 1000 + 10 * c
        mats = [syn.quant_matrix(fmt, d, d, s + i, threads=8) for i in range(4)]
        mats += [syn.quant_matrix(fmt, f, d, s + 4, threads=8),
                 syn.quant_matrix(fmt, f, d, s + 5, threads=8),
                 syn.quant_matrix(fmt, d, f, s + 6, threads=8)]
        dev = [torch.from_numpy(m).to(device) for m in mats]
        layers.append(DenseLayer(fmt, d, f, *dev))
    return layers


def dense_outputs(torch, device):
    import quantized_weight_streaming_dequant_gb300 as rf
    d, f = syn.C2["d_model"], syn.C2["d_ff"]
    out = {k: torch.empty(n, dtype=torch.float32, device=device)
           for k, n in (("q", d), ("k", d), ("v", d), ("o", d), ("h", f), ("y", d))}
    out["hd"] = rf.ffn_workspace(f, device)   # h's digits, handed from gate/up to down
    return out


def run_dense(args, torch, rf, device, rank, world, dist):
    layers = build_dense_layers(torch, rf, device, syn.C2["copies"], syn.C2["seed"] + rank)
    d = syn.C2["d_model"]
    x = torch.from_numpy(syn.normal_f32(d, 101 + rank)).to(device)
    attn = torch.from_numpy(syn.normal_f32(d, 102 + rank)).to(device)
    x_ffn = torch.from_numpy(syn.normal_f32(d, 103 + rank)).to(device)
    out = dense_outputs(torch, device)
    wbytes = layers[0].weight_bytes()
    stream = torch.cuda.Stream(device)
    nL = len(layers)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            layers[i % nL].step(x, attn, x_ffn, out, stream=stream)
    torch.cuda.synchronize()

    # CUDA graphs (programmatic dependent launch edges kept): one graph for a
    # round of nL steps (one per layer copy) and one per single step for the
    # remainder, so the timed region runs exactly args.steps steps.
    graphs, round_graph = [], None
    use_graph = not args.no_graph
    if use_graph:
        try:
            for L in layers:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    L.step(x, attn, x_ffn, out, stream=stream)
                graphs.append(g)
            round_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(round_graph, stream=stream):
                for L in layers:
                    L.step(x, attn, x_ffn, out, stream=stream)
            with torch.cuda.stream(stream):
                for i in range(nL):
                    graphs[i].replay()
                round_graph.replay()
            torch.cuda.synchronize()
        except Exception as e:  # capture unsupported: time the eager path
            print(f"# graph capture failed ({e}); timing eager launches", file=sys.stderr)
            use_graph, graphs, round_graph = False, [], None

    def run_steps(n):
        if use_graph:
            for _ in range(n // nL):
                round_graph.replay()
            for i in range(n % nL):
                graphs[i].replay()
        else:
            for i in range(n):
                layers[i % nL].step(x, attn, x_ffn, out, stream=stream)

    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The timed region (exactly args.steps steps) runs REPEATS times; each
    # repeat is bracketed by a barrier and synchronisations and timed on the
    # launching stream; the value is the median repeat.  The clock sampler
    # (200 ms period) runs across a one-second load of the same steps just
    # before the repeats and across the repeats themselves, so that it sees
    # the clocks under this load even when a repeat lasts well under 200 ms.
    reps_ms = []
    with ClockSampler(device.index or 0) as clk:
        t_end = time.perf_counter() + args.clock_soak
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                run_steps(max(args.steps, 8 * nL))
                stream.synchronize()
        # An NVTX range marks the timed repeats, so a profiler can select
        # exactly the timed steps (ncu --nvtx --nvtx-include "rf_timed/").
        torch.cuda.nvtx.range_push("rf_timed")
        for _ in range(REPEATS):
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            with torch.cuda.stream(stream):
                e0.record(stream)
                run_steps(args.steps)
                e1.record(stream)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            reps_ms.append(reduce_time_max(torch, dist, e0.elapsed_time(e1), device))
        torch.cuda.nvtx.range_pop()
    ms = statistics.median(reps_ms)
    gbs = whole_job_gbs(wbytes, args.steps, world, ms)
    spread = {"repeats": REPEATS, "ms_per_step": [round(r / args.steps, 6) for r in reps_ms],
              "min_ms_per_step": min(reps_ms) / args.steps,
              "max_ms_per_step": max(reps_ms) / args.steps}

    # Per-phase launch durations (eager, events around each launch) for the
    # roofline breakdown.
    phases = per_phase_times(torch, rf, layers, x, attn, x_ffn, out, stream, reps=40)

    # End to end through the public API: H2D of the step's inputs from pinned
    # host memory, the 4 launches, D2H of the step's outputs, every step.
    e2e = dense_e2e(torch, layers, out, device, stream, steps=min(args.steps, 400) or 1)
    return dict(ms=ms / args.steps, gbs=gbs, wbytes=wbytes, use_graph=use_graph,
                clocks=clk.summary(), phases=phases, e2e=e2e, spread=spread)


def per_phase_times(torch, rf, layers, x, attn, x_ffn, out, stream, reps):
    """Eager launches with events around each phase: QKV (one batched launch),
    O (one launch), FFN (gate/up with SwiGLU epilogue + down: two launches)."""
    d, f, fmt = syn.C2["d_model"], syn.C2["d_ff"], syn.Q4_0
    rb_d, rb_f = rf.row_bytes(fmt, d), rf.row_bytes(fmt, f)
    nbytes = {"qkv": 3 * d * rb_d, "o": d * rb_d, "ffn": 2 * f * rb_d + d * rb_f}
    acc = {k: 0.0 for k in nbytes}
    nL = len(layers)
    with torch.cuda.stream(stream):
        for it in range(reps):
            L = layers[it % nL]
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[0].record(stream)
            rf.gemv_batch(fmt, d, [(L.wq, 0, d, x, out["q"]), (L.wk, 0, d, x, out["k"]),
                                   (L.wv, 0, d, x, out["v"])], stream=stream)
            ev[1].record(stream)
            rf.gemv(fmt, L.wo, 0, d, d, attn, out["o"], stream=stream)
            ev[2].record(stream)
            rf.ffn_swiglu(fmt, L.w_gate, L.w_up, L.w_down, f, d, x_ffn, out["y"], out["h"],
                          stream=stream, workspace=out["hd"])
            ev[3].record(stream)
            torch.cuda.synchronize()
            acc["qkv"] += ev[0].elapsed_time(ev[1])
            acc["o"] += ev[1].elapsed_time(ev[2])
            acc["ffn"] += ev[2].elapsed_time(ev[3])
    res = {}
    for k, b in nbytes.items():
        ms = acc[k] / reps
        res[k] = {"ms": ms, "bytes": b, "gbs": b / (ms * 1e-3) / 1e9}
    return res


def dense_e2e(torch, layers, out, device, stream, steps):
    """End to end through the public API, every step: H2D of the step's three
    input vectors from page-locked host memory, the four launches writing
    their outputs into one device buffer, its D2H into page-locked host
    memory, then the host waits for the step and reads its result.  Each
    layer copy's step (copies included) is captured once into a CUDA graph,
    so a step costs one graph launch and one synchronisation; the eager
    figure (every call issued from Python) is reported beside it."""
    d = syn.C2["d_model"]
    h_in = torch.from_numpy(np.concatenate([syn.normal_f32(d, s) for s in (101, 102, 103)]))
    h_in = h_in.pin_memory()
    d_in = torch.empty(3 * d, dtype=torch.float32, device=device)
    outs = ["q", "k", "v", "o", "y"]
    h_out = torch.empty(len(outs) * d, dtype=torch.float32).pin_memory()
    d_out = torch.empty(len(outs) * d, dtype=torch.float32, device=device)
    # q, k, v, o and y are views of d_out, so the step's outputs leave the
    # device in one copy; h and h's digits stay on the device.
    out = dict(out, **{k: d_out[i * d:(i + 1) * d] for i, k in enumerate(outs)})
    nL = len(layers)

    def step(L):
        d_in.copy_(h_in, non_blocking=True)
        L.step(d_in[:d], d_in[d:2 * d], d_in[2 * d:], out, stream=stream)
        h_out.copy_(d_out, non_blocking=True)

    def timed(run_one):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        checksum = 0.0
        with torch.cuda.stream(stream):
            for i in range(steps):
                run_one(i)
                stream.synchronize()
                checksum += float(h_out[0])   # the host reads the step's result
        return time.perf_counter() - t0, checksum

    dt_eager, _ = timed(lambda i: step(layers[i % nL]))
    graphs = []
    try:
        with torch.cuda.stream(stream):
            for L in layers:
                step(L)
        torch.cuda.synchronize()
        for L in layers:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(L)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
        dt, _ = timed(lambda i: graphs[i % nL].replay())
        use_graph = True
    except Exception as e:   # capture unsupported: report the eager figure
        print(f"# e2e graph capture failed ({e}); eager figure only", file=sys.stderr)
        dt, use_graph = dt_eager, False
    del graphs
    wbytes = layers[0].weight_bytes()
    return {"value": wbytes * steps / dt / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": int(h_in.numel() * 4), "d2h_bytes_per_step": int(h_out.numel() * 4),
            "ms_per_step": dt / steps * 1e3, "steps": steps, "cuda_graph": use_graph,
            "eager": {"value": wbytes * steps / dt_eager / 1e9, "ms_per_step": dt_eager / steps * 1e3}}


def run_dense_format(torch, rf, device, fmt: int, steps: int = 2000):
    """The 4096/11008 dense layer with its weights in another format (same
    layer copies > L2, same four launches, one CUDA graph per round of
    copies): whole-step weight GB/s."""
    layers = build_dense_layers(torch, rf, device, syn.C2["copies"], syn.C2["seed"], fmt)
    d = syn.C2["d_model"]
    x, attn, x_ffn = (torch.from_numpy(syn.normal_f32(d, s)).to(device) for s in (101, 102, 103))
    out = dense_outputs(torch, device)
    stream = torch.cuda.Stream(device)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for L in layers:
            L.step(x, attn, x_ffn, out, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for L in layers:
            L.step(x, attn, x_ffn, out, stream=stream)
    rounds = max(1, steps // len(layers))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0.record(stream)
        for _ in range(rounds):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (rounds * len(layers))
    wbytes = layers[0].weight_bytes()
    del g, layers
    return {"ms_per_step": ms, "weight_bytes_per_step": wbytes,
            "value": wbytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "steps": rounds * syn.C2["copies"]}


def run_multi_token(torch, rf, device, reps: int = 50):
    """Several tokens through one resident matrix per launch (rf_gemv_multi):
    the 11008x4096 Q4_0 gate projection, eight copies (203 MB, > L2) walked
    round-robin in one CUDA graph of chained launches, for 1, 2, 4 and 8
    tokens.  value = weight bytes per second; token_gbs = the same times the
    tokens (what separate launches per token would have to stream)."""
    fmt, rows, in_dim = syn.Q4_0, syn.C2["d_ff"], syn.C2["d_model"]
    Ws = [torch.from_numpy(syn.quant_matrix(fmt, rows, in_dim, 70 + c, threads=8)).to(device)
          for c in range(8)]
    nbytes = Ws[0].numel()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    out = []
    for n_tok in (1, 2, 4, 8):
        X = torch.from_numpy(np.stack([syn.normal_f32(in_dim, 900 + t) for t in range(n_tok)])).to(
            device)
        Y = torch.empty(n_tok, rows, device=device)

        def walk():
            for W in Ws:
                rf.gemv_multi(fmt, W, 0, rows, in_dim, X, Y, stream=s, flags=rf.CHAIN)
        with torch.cuda.stream(s):
            walk()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            walk()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * len(Ws))
        out.append({"tokens": n_tok, "us_per_launch": us, "value": nbytes / us / 1e3,
                    "unit": "GB/s", "token_gbs": n_tok * nbytes / us / 1e3})
        del g
    return {"matrix": f"Q4_0 {rows}x{in_dim}", "copies": len(Ws), "bytes": nbytes, "rows": out}


def run_prefill(torch, rf, device, tensor_peak: float, reps: int = 5, fmt: int = syn.Q4_0,
                tokens=(8, 64, 512, 2048), shape=None, copies: int = 8):
    """Chunks of tokens through one resident matrix per call (rf_gemm, the
    tensor-core prefill dequant-GEMM): by default the 11008x4096 gate
    projection in `fmt`, `copies` copies (> L2) walked round-robin in one
    CUDA graph, for each chunk size in `tokens`.  Each call includes its
    activation pre-pass.  value = TF/s (2 * rows * in_dim * tokens per call);
    weight_gbs = weight bytes per second; vs_gemv_multi = the same tokens
    through rf_gemv_multi in launches of eight tokens, timed the same way,
    over this call."""
    rows, in_dim = shape if shape is not None else (syn.C2["d_ff"], syn.C2["d_model"])
    Ws = [torch.from_numpy(syn.quant_matrix(fmt, rows, in_dim, 70 + c, threads=8)).to(device)
          for c in range(copies)]
    nbytes = Ws[0].numel()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())

    def timed(walk, calls):
        with torch.cuda.stream(s):
            walk()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            walk()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) * 1e3 / (reps * calls)

    out = []
    for n_tok in tokens:
        X = torch.randn(n_tok, in_dim, generator=torch.Generator(device=device).manual_seed(n_tok),
                        device=device)
        Y = torch.empty(n_tok, rows, device=device)
        ws = torch.empty(rf.gemm_workspace_bytes(fmt, in_dim, n_tok), dtype=torch.uint8,
                         device=device)

        def walk_gemm():
            for W in Ws:
                rf.gemm(fmt, W, 0, rows, in_dim, X, Y, workspace=ws, stream=s)

        def walk_multi():
            for W in Ws:
                for c in range(0, n_tok, 8):
                    rf.gemv_multi(fmt, W, 0, rows, in_dim, X[c:c + 8], Y[c:c + 8], stream=s)
        us = timed(walk_gemm, len(Ws))
        tf = 2.0 * rows * in_dim * n_tok / us / 1e6
        row = {"tokens": n_tok, "us_per_call": us, "value": tf, "unit": "TF/s",
               "frac_of_tensor_peak": tf / tensor_peak, "weight_gbs": nbytes / us / 1e3}
        if n_tok <= 64:
            row["vs_gemv_multi"] = timed(walk_multi, len(Ws)) / us
        out.append(row)
    name = next(k for k, v in rf.FORMATS.items() if v == fmt)
    return {"matrix": f"{name} {rows}x{in_dim}", "copies": len(Ws), "bytes": nbytes,
            "tensor_peak_tflops": tensor_peak, "peak_source": "measured bf16 burst (else the "
            "fallback); fp16 operands run at the same nominal rate", "rows": out}


def run_streamed_gemv(torch, rf, device, depth: int, merge: bool = True, reps: int = 50):
    """Q8_0 512x2048 streamed from pinned host memory in 128-row blocks, eager
    calls and the same calls captured into one CUDA graph.  merge: a walk
    whose 4 blocks fit the ring goes as one copy and one launch; off, every
    block is its own copy and launch (the per-block pipeline)."""
    c = syn.C1
    fmt, rows, in_dim = c["fmt"], c["out_dim"], c["in_dim"]
    W = syn.quant_matrix(fmt, rows, in_dim, c["seed"])
    host = torch.from_numpy(W).pin_memory()
    x = torch.from_numpy(syn.normal_f32(in_dim, c["seed"] + 1)).to(device)
    y = torch.empty(rows, device=device)
    arena = rf.Arena(c["arena_bytes"])
    arena.configure(rf.ARENA_MERGE_RUNS, merge)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        with torch.cuda.stream(s):
            for _ in range(5):
                arena.stream_linear(fmt, host, in_dim, 0, rows, c["block_rows"], depth, x, y, stream=s)
            s.synchronize()
            e0.record(s)
            for _ in range(reps):
                arena.stream_linear(fmt, host, in_dim, 0, rows, c["block_rows"], depth, x, y, stream=s)
            e1.record(s)
        torch.cuda.synchronize()
        eager_ms = e0.elapsed_time(e1) / reps
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                arena.stream_linear(fmt, host, in_dim, 0, rows, c["block_rows"], depth, x, y, stream=s)
        with torch.cuda.stream(s):
            g.replay()
            e0.record(s)
            for _ in range(4):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        graph_ms = e0.elapsed_time(e1) / (4 * reps)
        del g
        # zero-copy arm: the kernel reads the page-locked matrix in place
        with torch.cuda.stream(s):
            for _ in range(5):
                rf.gemv_host(fmt, host, 0, rows, in_dim, x, y, stream=s)
            e0.record(s)
            for _ in range(reps):
                rf.gemv_host(fmt, host, 0, rows, in_dim, x, y, stream=s)
            e1.record(s)
        torch.cuda.synchronize()
        zc_ms = e0.elapsed_time(e1) / reps
    finally:
        torch.cuda.synchronize()
        arena.close()
    nbytes = W.nbytes
    probe = h2d_probe(torch, device, c["block_rows"] * rf.row_bytes(fmt, in_dim), reps=200)
    ms = min(eager_ms, graph_ms)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": c["name"], "depth": depth, "merge_runs": merge,
            "ms_per_gemv": ms, "value": gbs, "unit": "GB/s",
            "eager_ms_per_gemv": eager_ms, "graph_ms_per_gemv": graph_ms,
            "zero_copy_ms_per_gemv": zc_ms, "zero_copy_value": nbytes / (zc_ms * 1e-3) / 1e9,
            "h2d_probe_block_gbs": probe, "frac_of_block_h2d": gbs / probe}


def run_moe(torch, rf, device, steps: int = 200):
    c = syn.C3
    fmt, E, n_ff, n_embd, k, br = c["fmt"], c["n_expert"], c["n_ff"], c["n_embd"], c["top_k"], \
        c["block_rows"]
    G = torch.from_numpy(syn.stacked_experts(fmt, E, n_ff, n_embd, c["seed"], threads=8)).to(device)
    U = torch.from_numpy(syn.stacked_experts(fmt, E, n_ff, n_embd, c["seed"] + 1, threads=8)).to(
        device)
    D = torch.from_numpy(syn.stacked_experts(fmt, E, n_embd, n_ff, c["seed"] + 2, threads=8)).to(
        device)
    x = torch.from_numpy(syn.normal_f32(n_embd, c["seed"] + 3)).to(device)
    # fresh router logits per token so the expert windows vary
    logits = torch.from_numpy(np.stack([syn.router_logits(E, 1000 + t) for t in range(steps)])).to(
        device)
    y = torch.empty(n_embd, device=device)
    ws = rf.moe_workspace(k, n_ff, n_embd, br, device)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for t in range(10):
            rf.moe_ffn(fmt, logits[t], k, G, U, D, n_ff, n_embd, br, x, y, ws, stream=s)
    torch.cuda.synchronize()
    # One graph holds `per_graph` tokens, each with its own logits, replayed
    # until `steps` tokens have run (three launches per token).
    per_graph = 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(per_graph):
            rf.moe_ffn(fmt, logits[t], k, G, U, D, n_ff, n_embd, br, x, y, ws, stream=s)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, steps // per_graph)
    with torch.cuda.stream(s):
        g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * per_graph)
    del g
    # Zero-copy arm: the same experts in page-locked host memory, read in place.
    hG, hU, hD = (t.cpu().pin_memory() for t in (G, U, D))
    with torch.cuda.stream(s):
        for t in range(3):
            rf.moe_ffn_host(fmt, logits[t], k, hG, hU, hD, n_ff, n_embd, br, x, y, ws, stream=s)
        e0.record(s)
        for t in range(per_graph):
            rf.moe_ffn_host(fmt, logits[t], k, hG, hU, hD, n_ff, n_embd, br, x, y, ws, stream=s)
        e1.record(s)
    torch.cuda.synchronize()
    zc_ms = e0.elapsed_time(e1) / per_graph
    active = k * 3 * n_ff * rf.row_bytes(fmt, n_embd)
    del G, U, D
    streamed = run_moe_streamed(torch, rf, device, hG, hU, hD, x, active)
    return {"workload": c["name"], "ms_per_token": ms, "active_bytes": active,
            "value": active / (ms * 1e-3) / 1e9, "unit": "GB/s", "launches_per_token": 2,
            "cuda_graph": True, "tokens_per_graph": per_graph,
            "zero_copy": {"ms_per_token": zc_ms, "value": active / (zc_ms * 1e-3) / 1e9,
                          "note": "experts in page-locked host memory, read over the link"},
            "streamed": streamed}


def run_moe_streamed(torch, rf, device, hG, hU, hD, x, active, tokens: int = 60):
    """The same MoE with its experts in page-locked host memory read through
    the layer-wide prefetch plan (rf_moe_ffn_streamed: depth 4, 256 MiB
    arena, whole windows, and 512-row blocks without a cache) with expert
    caches of 0, 16, 32 and 64 experts, on router
    logits with expert popularity (the top 20 % of experts take about 57 %
    of the selections).  Host wall time per token (each call waits for its
    routing result), after 16 warm-up tokens that fill the cache."""
    c = syn.C3
    fmt, E, n_ff, n_embd, k = c["fmt"], c["n_expert"], c["n_ff"], c["n_embd"], c["top_k"]
    warm = 16
    logits = torch.from_numpy(syn.skewed_router_logits(E, warm + tokens, 11)).to(device)
    y = torch.empty(n_embd, device=device)
    ws = rf.moe_workspace(k, n_ff, n_embd, 512, device)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    arena = rf.Arena(256 << 20)
    h2d = h2d_probe(torch, device, 256 << 20)
    per_expert = 2 * n_ff * rf.row_bytes(fmt, n_embd) + n_embd * rf.row_bytes(fmt, n_ff)
    out = {"depth": 4, "arena_bytes": 256 << 20, "tokens": tokens,
           "h2d_probe_256mib_gbs": h2d, "router_skew": 0.5, "budgets": []}
    try:
        for slots, br in ((0, 512), (0, 0), (16, 0), (32, 0), (64, 0)):
            cache = rf.ExpertCache(fmt, n_ff, n_embd, slots) if slots else None
            with torch.cuda.stream(s):
                for t in range(warm):
                    rf.moe_ffn_streamed(fmt, logits[t], k, hG, hU, hD, n_ff, n_embd, br, 4, arena,
                                        x, cache=cache, y=y, workspace=ws, stream=s)
            torch.cuda.synchronize()
            st0 = cache.stats() if cache else None
            a0 = arena.stats()["bytes_copied"]
            t0 = time.perf_counter()
            with torch.cuda.stream(s):
                for t in range(warm, warm + tokens):
                    rf.moe_ffn_streamed(fmt, logits[t], k, hG, hU, hD, n_ff, n_embd, br, 4, arena,
                                        x, cache=cache, y=y, workspace=ws, stream=s)
            torch.cuda.synchronize()
            dt = (time.perf_counter() - t0) / tokens
            arena_bytes = arena.stats()["bytes_copied"] - a0
            row = {"cache_experts": slots, "block_rows": br or "whole",
                   "cache_bytes": slots * per_expert,
                   "ms_per_token": dt * 1e3, "active_gbs": active / dt / 1e9}
            if cache:
                st = cache.stats()
                look = st["lookups"] - st0["lookups"]
                hits = st["hits"] - st0["hits"]
                streamed = st["bytes_streamed"] - st0["bytes_streamed"]
                row.update({"hit_rate": hits / look, "evictions": st["evictions"] - st0["evictions"]})
                cache.close()
            else:
                streamed = arena_bytes
                row["hit_rate"] = 0.0
            row["streamed_bytes_per_token"] = streamed / tokens
            row["streamed_gbs"] = streamed / tokens / dt / 1e9
            row["frac_of_h2d"] = row["streamed_gbs"] / h2d
            out["budgets"].append(row)
    finally:
        torch.cuda.synchronize()
        arena.close()
    return out


def run_streamed_ffn(torch, rf, device, n_layer: int):
    from quantized_weight_streaming_dequant_gb300.layer import StreamedFFN
    c = syn.C4
    fmt, d, f = c["fmt"], c["d_model"], c["d_ff"]
    layers = []
    for l in range(n_layer):
        up = torch.empty((f, rf.row_bytes(fmt, d)), dtype=torch.uint8).pin_memory()
        dn = torch.empty((d, rf.row_bytes(fmt, f)), dtype=torch.uint8).pin_memory()
        syn.quant_matrix(fmt, f, d, c["seed"] * 1000 + 2 * l, out=up.numpy(), threads=16)
        syn.quant_matrix(fmt, d, f, c["seed"] * 1000 + 2 * l + 1, out=dn.numpy(), threads=16)
        layers.append(StreamedFFN(fmt, d, f, up, dn))
    xs = [torch.from_numpy(syn.normal_f32(d, 5000 + l)).to(device) for l in range(n_layer)]
    u = torch.empty(f, device=device)
    h = torch.empty(f, device=device)
    y = torch.empty(d, device=device)
    arena = rf.Arena(c["arena_bytes"])
    s = torch.cuda.current_stream()
    try:
        for l in range(min(2, n_layer)):
            layers[l].step(arena, xs[l], u, h, y, c["block_rows"], c["depth"])
        torch.cuda.synchronize()
        blocks0 = arena.stats()["blocks"]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(s)
        for l in range(n_layer):
            layers[l].step(arena, xs[l], u, h, y, c["block_rows"], c["depth"])
        e1.record(s)
        torch.cuda.synchronize()
        host_s = time.perf_counter() - t0
        ms = e0.elapsed_time(e1)
        stats = arena.stats()
        blocks_eager = stats["blocks"] - blocks0
        # The same token captured into one CUDA graph: copies and GEMVs become
        # graph nodes, so the host issues one launch per token.
        graph_ms, graph_err, graph_runs = None, None, None
        try:
            s = torch.cuda.Stream(device)   # captures need a side stream
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for l in range(n_layer):
                    layers[l].step(arena, xs[l], u, h, y, c["block_rows"], c["depth"], stream=s)
            with torch.cuda.stream(s):
                g.replay()
            torch.cuda.synchronize()
            y_graph = y.clone()
            # REPEATS timed runs of `tokens` graph-replayed tokens each
            # (continuous streaming: the copy engine never drains between
            # tokens); the figure is the median run.
            tokens = 10
            runs = []
            for _ in range(REPEATS):
                with torch.cuda.stream(s):
                    e0.record(s)
                    for _ in range(tokens):
                        g.replay()
                    e1.record(s)
                torch.cuda.synchronize()
                runs.append(e0.elapsed_time(e1) / tokens)
            graph_ms = statistics.median(runs)
            graph_runs = {"tokens_per_run": tokens, "runs": REPEATS,
                          "ms_per_token": [round(r, 3) for r in runs]}
            # eager and graph walks of the same token give the same bits
            layers[n_layer - 1].step(arena, xs[n_layer - 1], u, h, y, c["block_rows"], c["depth"])
            torch.cuda.synchronize()
            if not torch.equal(y, y_graph):
                graph_err = "graph output differs from eager output"
            del g
        except Exception as e:  # capture refused: report the eager walk only
            graph_err = str(e).splitlines()[0]
        # Zero-copy arm: the kernels read the same page-locked bytes in place.
        zs = torch.cuda.current_stream()
        for l in range(min(2, n_layer)):
            layers[l].step_zero_copy(xs[l], u, h, y, stream=zs)
        torch.cuda.synchronize()
        e0.record(zs)
        for l in range(n_layer):
            layers[l].step_zero_copy(xs[l], u, h, y, stream=zs)
        e1.record(zs)
        torch.cuda.synchronize()
        zc_ms = e0.elapsed_time(e1)
    finally:
        torch.cuda.synchronize()
        arena.close()
    nbytes = sum(L.weight_bytes() for L in layers)
    probe_big = h2d_probe(torch, device, 256 << 20)
    probe_blk = h2d_probe(torch, device, c["block_rows"] * rf.row_bytes(fmt, f), reps=20)
    eager_gbs = nbytes / (ms * 1e-3) / 1e9
    best_ms = min(ms, graph_ms) if graph_ms else ms
    gbs = nbytes / (best_ms * 1e-3) / 1e9
    return {"workload": c["name"], "layers": n_layer, "ms_per_token": best_ms,
            "bytes_per_token": nbytes, "value": gbs, "unit": "GB/s",
            "h2d_probe_256mib_gbs": probe_big, "h2d_probe_block_gbs": probe_blk,
            "frac_of_h2d": gbs / probe_big, "tokens_per_s": 1e3 / best_ms,
            "eager": {"ms_per_token": ms, "value": eager_gbs, "host_enqueue_s": host_s},
            "graph": {"ms_per_token": graph_ms, "error": graph_err, "timing": graph_runs,
                      "value": nbytes / (graph_ms * 1e-3) / 1e9 if graph_ms else None},
            "zero_copy": {"ms_per_token": zc_ms, "value": nbytes / (zc_ms * 1e-3) / 1e9,
                          "frac_of_h2d": nbytes / (zc_ms * 1e-3) / 1e9 / probe_big},
            "arena_peak_bytes": stats["peak_bytes"],
            "blocks_per_token": blocks_eager}


def run_sweep(torch, rf, device, peak_hbm: float, reduced: bool = False):
    """The format x in_dim x out_dim x block_rows sweep, resident and
    host-streamed.  Resident: the row windows of block_rows rows (whole =
    one window) go to rf_gemv_batch (at most 64 windows per launch); copies of
    the matrix are rotated until at least 4 x L2 is read between reuses; one
    CUDA graph holds one pass over the copies.  Streamed: rf_stream_linear
    from page-locked host memory, 256 MiB arena, depth 4, calls captured into
    one CUDA graph.  Each cell has its own seeded matrix."""
    l2 = 129 << 20
    h2d = h2d_probe(torch, device, 256 << 20)
    arena = rf.Arena(256 << 20)
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cells = []

    def timed_graph(fn, units):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
        with torch.cuda.stream(s):
            g.replay()
            e0.record(s)
            reps = 0
            while True:
                g.replay()
                reps += 1
                if reps >= 3:
                    break
            e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * units)
        del g
        return ms

    try:
        for c in syn.sweep_cells():
            fmt, in_dim, out, br = c["fmt"], c["in_dim"], c["out_dim"], c["block_rows"]
            if reduced and br not in (128, 0):
                continue
            W = syn.quant_matrix(fmt, out, in_dim, c["seed"], threads=16)
            nbytes = W.nbytes
            x = torch.from_numpy(syn.normal_f32(in_dim, c["seed"] + 1)).to(device)
            y = torch.empty(out, device=device)
            w_rows = out if br == 0 else br
            wins = [(r0, min(out, r0 + w_rows)) for r0 in range(0, out, w_rows)]
            copies = max(1, min(64, -(-4 * l2 // nbytes)))
            Wd = torch.from_numpy(W).to(device)
            Ws = [Wd] + [Wd.clone() for _ in range(copies - 1)]

            def resident():
                for Wc in Ws:
                    for b in range(0, len(wins), 64):
                        rf.gemv_batch(fmt, in_dim, [(Wc, r0, r1, x, y[r0:r1]) for r0, r1 in
                                                    wins[b:b + 64]], stream=s, flags=rf.CHAIN)
            res_ms = timed_graph(resident, copies)
            del Ws, Wd
            host = torch.from_numpy(W).pin_memory()
            n_calls = max(2, min(50, -(-(64 << 20) // nbytes)))

            def streamed():
                for _ in range(n_calls):
                    arena.stream_linear(fmt, host, in_dim, 0, out, br, 4, x, y, stream=s)
            str_ms = timed_graph(streamed, n_calls)
            eff = arena.stats()["last_block_rows"]
            del host
            res_gbs = nbytes / (res_ms * 1e-3) / 1e9
            str_gbs = nbytes / (str_ms * 1e-3) / 1e9
            cells.append({"fmt": {syn.Q8_0: "Q8_0", syn.Q4_0: "Q4_0", syn.MXFP4: "MXFP4"}[fmt],
                          "in": in_dim, "out": out, "block_rows": br or "whole",
                          "bytes": nbytes, "resident_gbs": round(res_gbs, 1),
                          "resident_frac_hbm": round(res_gbs / peak_hbm, 4),
                          "streamed_gbs": round(str_gbs, 1),
                          "streamed_frac_h2d": round(str_gbs / h2d, 4),
                          "streamed_block_rows_eff": eff, "launches_per_resident_pass":
                          -(-len(wins) // 64)})
    finally:
        torch.cuda.synchronize()
        arena.close()
    rf_ = sorted(cl["resident_frac_hbm"] for cl in cells)
    sf_ = sorted(cl["streamed_frac_h2d"] for cl in cells)
    return {"h2d_probe_256mib_gbs": h2d, "cells": cells,
            "block_rows": "128 and whole only" if reduced else "all",
            "resident_frac_hbm_median": rf_[len(rf_) // 2],
            "streamed_frac_h2d_median": sf_[len(sf_) // 2]}


# ------------------------------------------------------------- reference

class OracleLayer:
    """One Q4_0 4096/11008 layer for the CPU oracle: the 7 matrices with the
    first `fraction` of their rows (1.0 = the whole layer, 113,836,032
    bytes).  A pass runs the oracle's GEMV over every row; with threads > 1
    the rows of every matrix are cut into `threads` contiguous ranges run
    concurrently (the C oracle runs outside the GIL, so the threads use as
    many host cores), the oracle's own arithmetic unchanged."""

    def __init__(self, fraction: float = 1.0):
        fmt, d, f = syn.Q4_0, syn.C2["d_model"], syn.C2["d_ff"]
        self.fmt = fmt
        self.shapes = [(d, d)] * 4 + [(f, d)] * 2 + [(d, f)]
        self.mats = [syn.quant_matrix(fmt, max(1, int(r * fraction)), c, 7 + i, threads=8)
                     for i, (r, c) in enumerate(self.shapes)]
        self.xs = {c: syn.normal_f32(c, c) for c in (d, f)}
        self.nbytes = sum(m.nbytes for m in self.mats)

    def run(self, threads: int = 1, pool=None):
        import oracle
        if threads <= 1:
            for m, (_, c) in zip(self.mats, self.shapes):
                oracle.gemv(self.fmt, m, 0, m.shape[0], c, self.xs[c])
            return
        work = []
        for m, (_, c) in zip(self.mats, self.shapes):
            n = m.shape[0]
            for t in range(threads):
                r0, r1 = n * t // threads, n * (t + 1) // threads
                if r1 > r0:
                    work.append((m, r0, r1, c))
        list(pool.map(lambda a: oracle.gemv(self.fmt, a[0], a[1], a[2], a[3], self.xs[a[3]]),
                      work))

    def timed(self, min_seconds: float, threads: int = 1):
        """(GB/s, seconds per pass): passes repeated until min_seconds."""
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=max(1, threads)) as pool:
            self.run(threads, pool)   # warm-up pass
            passes, t0 = 0, time.perf_counter()
            while True:
                self.run(threads, pool)
                passes += 1
                dt = time.perf_counter() - t0
                if dt >= min_seconds:
                    break
        return self.nbytes * passes / dt / 1e9, dt / passes


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, rank: int):
    if rank != 0:
        return 0
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    total = args.steps + args.warmup
    cores = host_cores()
    # each step: the whole layer on all host cores, or (for long runs) the
    # first rows of every matrix, sized so the run takes about a minute
    probe = OracleLayer(1 / 64)
    _, t_probe = probe.timed(0.0, cores)
    frac = max(1 / 4096, min(1.0, (60.0 / max(total, 1)) / (t_probe * 64)))
    layer = OracleLayer(frac) if frac < 1.0 else OracleLayer(1.0)
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(args.warmup):
            layer.run(cores, pool)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            layer.run(cores, pool)
        dt = time.perf_counter() - t0
    value = layer.nbytes * args.steps / dt / 1e9
    what = "every row" if frac >= 1.0 else f"the first {frac:.4%} of the rows"
    sample = (f"{what} of each of the 7 matrices of one Q4_0 4096/11008 layer "
              f"({layer.nbytes} weight bytes) per step, rows split over {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / max(args.steps, 1) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": syn.C2["name"], "d_model": 4096, "d_ff": 11008,
                       "format": "Q4_0", "batch": 1},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--ffn-layers", type=int, default=syn.C4["n_layer"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true",
                    help="run the full format x shape x block_rows sweep (several minutes) "
                         "instead of the reduced one (block_rows 128 and whole)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the sweep")
    ap.add_argument("--clock-soak", type=float, default=1.0,
                    help="seconds of the headline steps run under the clock sampler before "
                         "the timed repeats")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import quantized_weight_streaming_dequant_gb300 as rf
    from quantized_weight_streaming_dequant_gb300 import build
    build.build()
    rf.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=device)
        dist = tdist

    res = run_dense(args, torch, rf, device, rank, world, dist)
    peak, peak_kind = load_peaks()
    wbytes = res["wbytes"]
    launches = 4 * args.steps
    achieved = res["gbs"] / world    # all GEMV launches of the step: the only kernels in it
    traffic = ncu_traffic("q4_0_dense_layer_4096x11008")
    line = {"metric": METRIC, "value": res["gbs"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": syn.C2["name"], "format": "Q4_0", "d_model": 4096,
                       "d_ff": 11008, "batch": 1, "layer_copies": syn.C2["copies"],
                       "weight_bytes_per_step": wbytes, "l2": "inputs > L2 (8 layer copies, "
                       f"{8 * wbytes / 1e6:.0f} MB, round-robin)",
                       "parallelism": f"replicas x{world}", "cuda_graph": res["use_graph"]},
            "tokens_per_s_equiv": res["gbs"] / (wbytes / 1e9),
            "frac_of_hbm_peak": achieved / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "kernel": "rowwin_kernel<Q4_0> (all 4 launches of the step)",
                         "traffic": traffic,
                         "traffic_source": "profiles/ncu_traffic.txt: dram__bytes_read.sum + "
                                           "dram__bytes_write.sum of one step's launches from "
                                           "an ncu capture of this kernel source (keyed by its "
                                           "hash; null when the source changed since)"},
            "timing": res["spread"],
            "phases": res["phases"], "clocks": res["clocks"], "e2e": res["e2e"],
            "gpu_launches": launches}
    if rank == 0 and world == 1 and not args.headline_only:
        extra = {}
        try:
            extra["streamed_gemv_q8_0_512x2048"] = [
                run_streamed_gemv(torch, rf, device, dp, merge)
                for dp, merge in ((4, True), (4, False), (1, False), (8, True), (8, False))]
            extra["moe_mxfp4"] = run_moe(torch, rf, device)
            extra["multi_token_q4_0"] = run_multi_token(torch, rf, device)
            extra["prefill_q4_0"] = run_prefill(torch, rf, device, load_tensor_peak()[0])
            extra["prefill_q4_k"] = run_prefill(torch, rf, device, load_tensor_peak()[0],
                                                fmt=syn.Q4_K, tokens=(64, 512, 2048))
            # 2880-wide MXFP4 rows (1,530 bytes, read directly by the decoders),
            # one expert's gate and up rows: 5760 x 2880, 24 copies > L2.
            try:
                extra["prefill_mxfp4_2880"] = run_prefill(
                    torch, rf, device, load_tensor_peak()[0], fmt=syn.MXFP4,
                    tokens=(8, 64, 512, 2048), shape=(2 * syn.C3["n_ff"], syn.C3["n_embd"]),
                    copies=24)
            except Exception as e:  # this line never hides the ones after it
                extra["prefill_mxfp4_2880"] = {"error": repr(e)}
            for name, fmt in (("dense_layer_q4_k", syn.Q4_K), ("dense_layer_q6_k", syn.Q6_K)):
                r = run_dense_format(torch, rf, device, fmt)
                r["frac_of_hbm_peak"] = r["value"] / peak
                extra[name] = r
            if args.ffn_layers > 0:
                extra["streamed_ffn_q8_0"] = run_streamed_ffn(torch, rf, device, args.ffn_layers)
            if not args.no_sweep:
                extra["sweep"] = run_sweep(torch, rf, device, peak, reduced=not args.sweep)
        except Exception as e:  # extras never hide the headline
            extra["error"] = repr(e)
        line["extra"] = extra
        # The CPU oracle on the same workload: the whole layer (every row of
        # the 7 matrices, 113.8 MB), on one core and row-parallel over every
        # host core.
        layer = OracleLayer(1.0)
        cores = host_cores()
        gbs1, s1 = layer.timed(args.cpu_seconds, 1)
        gbsn, sn = layer.timed(args.cpu_seconds, cores)
        line["cpu_baseline"] = {
            "value": gbs1, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole layer ({layer.nbytes} weight bytes) per pass, passes "
                      f"repeated for at least {args.cpu_seconds:.0f} s on one core "
                      f"({s1:.3f} s per pass)",
            "all_cores": {"value": gbsn, "unit": "GB/s", "cores": cores,
                          "sample": f"the same passes with every matrix's rows split over "
                                    f"{cores} threads ({sn:.3f} s per pass)"}}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
