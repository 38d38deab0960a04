#!/usr/bin/env python3
"""Benchmark: effective HBM GB/s of the low-bit QMV decode path on GB300.

Workload (one "step"): the full decode sweep of a 27B-class dense layer --
7 projections (q 6144x5120, k/v 1024x5120, o 5120x6144, gate/up 17408x5120,
down 5120x17408) x M = 1..5 x {1-bit, 2-bit, 2-bit sym, t5} x group size
{64, 128}: 280 QMV calls.  Each (projection, format, group size) rotates
through 64 distinct weight sets resident in HBM (~28 GB), so every call
streams its weights from HBM, not L2.  Effective bytes per call = packed
weights + fp16 scales + fp16 biases (0 for sym and t5) + fp16 x + fp16 y.

`value` is device-resident throughput (bytes of all calls / device time);
`e2e` is the same through the same C-ABI calls with activations copied from
pinned host memory and results copied back inside the timed region; the
weights are the model's resident state.  The prefill matrix product is
timed separately in TFLOP/s: t5 (key "qmm"), 2-bit and 1-bit affine with
biases (keys "qmm_affine2", "qmm_affine1").  The speculative-decoding
verification kernel is timed in GB/s of logits read (key "spec_verify").

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "QMV effective HBM GB/s and % of GB300 peak, M=1-5, 1/2-bit & t5 ternary"
UNIT = "GB/s"
WORKLOAD = ("full decode sweep, 27B-class layer: 7 projections (q 6144x5120, k/v 1024x5120, "
            "o 5120x6144, gate/up 17408x5120, down 5120x17408) x M 1..5 x {1-bit, 2-bit, "
            "2-bit sym, t5} x group_size {64,128} = 280 QMV calls per step; 64 rotating "
            "weight sets per projection/group size, each call of a step on its own set")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

F1, F2, T5 = 1, 2, 3
VARIANTS = [("affine1", F1, False), ("affine2", F2, False), ("affine2_sym", F2, True), ("t5", T5, True)]
VARIANT_INDEX = {v[0]: i for i, v in enumerate(VARIANTS)}
GROUP_SIZES = (64, 128)
MS = (1, 2, 3, 4, 5)


def shapes():
    from bit_quantized_decode_unpack_gb300.synth import LAYER_SHAPES
    return list(LAYER_SHAPES.items())


def call_bytes(fmt, sym, M, N, K, gs):
    """Algorithmic bytes of one call (what the method must move)."""
    G = K // gs
    if fmt == F1:
        w = N * K // 8
    elif fmt == F2:
        w = N * K // 4
    else:
        w = N * G * (-(-gs // 5))
    has_bias = not sym and fmt != T5
    return w + N * G * 2 + (N * G * 2 if has_bias else 0) + M * K * 2 + M * N * 2


def page_bytes(fmt, sym, M, N, K, gs):
    """The page's byte count (weights + scales + biases + activations)."""
    return call_bytes(fmt, sym, M, N, K, gs) - M * N * 2


def sweep_calls():
    out = []
    for M in MS:
        for name, (N, K) in shapes():
            for vname, fmt, sym in VARIANTS:
                for gs in GROUP_SIZES:
                    out.append(dict(M=M, proj=name, N=N, K=K, variant=vname, fmt=fmt, sym=sym, gs=gs))
    return out


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---- clocks -------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="bqd_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in Path(self.path).read_text().splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        smax = max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


# ---- replicas: timing aggregation over ranks ----------------------------------------

def max_over_ranks(v: float, dist=None, device=None) -> float:
    """The step time every rank reports: the slowest rank's."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: bytes moved by all replicas over the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / (ms_max * 1e-3) / 1e9


# ---- our arm --------------------------------------------------------------------

class Sweep:
    """Device buffers and CUDA graphs for the decode sweep."""

    def __init__(self, dev, sets: int, seed: int = 0, quick: bool = False):
        import torch
        import bit_quantized_decode_unpack_gb300 as bqd
        from bit_quantized_decode_unpack_gb300 import synth
        self.torch, self.bqd, self.dev = torch, bqd, dev
        self.sets = sets
        self.calls = sweep_calls()
        if quick:
            self.calls = [c for c in self.calls if c["proj"] in ("k_proj", "down_proj")]
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        # weight sets per (projection, group size): codes drawn and packed on the device
        self.weights = {}
        for name, (N, K) in shapes():
            if quick and name not in ("k_proj", "down_proj"):
                continue
            for gs in GROUP_SIZES:
                G = K // gs
                lst = []
                for _ in range(sets):
                    s = synth.torch_scales(gen, N, G, dev)
                    entry = {"scales": s,
                             "b1": synth.torch_biases(gen, F1, s, dev),
                             "b2": synth.torch_biases(gen, F2, s, dev)}
                    for fmt, key in ((F1, "w1"), (F2, "w2"), (T5, "w5")):
                        codes = synth.torch_codes(gen, fmt, N, K, dev)
                        entry[key] = bqd.pack(codes, fmt, gs)
                        del codes
                    lst.append(entry)
                self.weights[(name, gs)] = lst
        # activations and outputs: one slab each, sliced per call
        self.x_off, self.y_off = [], []
        xo = yo = 0
        for c in self.calls:
            self.x_off.append(xo)
            self.y_off.append(yo)
            xo += c["M"] * c["K"] + 64  # keep 128-byte alignment between slices
            yo += c["M"] * c["N"] + 64
        self.x_all = synth.torch_activations(gen, 1, xo, dev).view(-1)
        self.y_all = torch.zeros(yo, dtype=torch.float16, device=dev)
        self.x_elems, self.y_elems = xo, yo
        self.bytes_per_step = sum(call_bytes(c["fmt"], c["sym"], c["M"], c["N"], c["K"], c["gs"])
                                  for c in self.calls)
        self.page_bytes_per_step = sum(page_bytes(c["fmt"], c["sym"], c["M"], c["N"], c["K"], c["gs"])
                                       for c in self.calls)
        self.h2d = sum(c["M"] * c["K"] * 2 for c in self.calls)
        self.d2h = sum(c["M"] * c["N"] * 2 for c in self.calls)
        torch.cuda.synchronize()

    def set_index(self, q, c):
        """Weight set of call c in graph phase q.  Each variant takes its own
        window of the rotation (offset 16 sets per variant), so within a
        step no two calls share a packed matrix or a scale or bias tensor
        (every format's weights of one set share that set's scales): every
        call streams bytes that no other call of the step has read."""
        return (5 * q + c["M"] - 1 + 16 * VARIANT_INDEX[c["variant"]]) % self.sets

    def _call(self, i, c, set_idx, stream):
        torch = self.torch
        e = self.weights[(c["proj"], c["gs"])][set_idx]
        M, N, K = c["M"], c["N"], c["K"]
        x = self.x_all[self.x_off[i]:self.x_off[i] + M * K].view(M, K)
        y = self.y_all[self.y_off[i]:self.y_off[i] + M * N].view(M, N)
        w = {F1: e["w1"], F2: e["w2"], T5: e["w5"]}[c["fmt"]]
        b = None
        if not c["sym"]:
            b = e["b1"] if c["fmt"] == F1 else e["b2"]
        self.bqd.qmv(x, w, e["scales"], b, c["fmt"], c["gs"], out=y, stream=stream)

    def capture(self, n_graphs: int):
        """One graph per step phase q (weight sets from set_index)."""
        torch = self.torch
        self.stream = torch.cuda.Stream()
        self.graphs = []
        with torch.cuda.stream(self.stream):
            for q in range(n_graphs):
                # warm (outside capture) once, then capture
                for i, c in enumerate(self.calls):
                    self._call(i, c, self.set_index(q, c), self.stream)
                self.stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    for i, c in enumerate(self.calls):
                        self._call(i, c, self.set_index(q, c), self.stream)
                self.graphs.append(g)
        torch.cuda.synchronize()

    def replay(self, step):
        self.graphs[step % len(self.graphs)].replay()


def time_steps(sweep, steps, warmup, e2e=False, barrier=None):
    torch = sweep.torch
    st = sweep.stream
    x_host = y_host = None
    if e2e:
        x_host = torch.empty(sweep.x_elems, dtype=torch.float16, pin_memory=True)
        x_host.copy_(sweep.x_all.cpu())
        y_host = torch.empty(sweep.y_elems, dtype=torch.float16, pin_memory=True)

    def one(step):
        with torch.cuda.stream(st):
            if e2e:
                sweep.x_all.copy_(x_host, non_blocking=True)
            sweep.replay(step)
            if e2e:
                y_host.copy_(sweep.y_all, non_blocking=True)

    for w in range(warmup):
        one(w)
    st.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(st)
    for s in range(steps):
        one(warmup + s)
    t1.record(st)
    t1.synchronize()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return t0.elapsed_time(t1)  # ms


def _graph_calls(sweep, calls_fn, n, st):
    """Capture n calls (calls_fn(j) enqueues call j) into CUDA graphs of at
    most 1024 calls each, after one warm pass outside capture."""
    torch = sweep.torch
    graphs = []
    with torch.cuda.stream(st):
        for j in range(n):
            calls_fn(j)
        st.synchronize()
        for j0 in range(0, n, 1024):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for j in range(j0, min(n, j0 + 1024)):
                    calls_fn(j)
            graphs.append(g)
    return graphs


def time_call(sweep, c, W, x, y, reps: int = 3):
    """µs per call of configuration c: CUDA graphs of back-to-back calls, one
    per weight set of W (enough sets that together they exceed the L2), best
    of `reps` replays of the whole rotation."""
    torch = sweep.torch
    st = sweep.stream

    def one(j):
        e = W[j]
        w = {F1: e.get("w1"), F2: e.get("w2"), T5: e.get("w5")}[c["fmt"]]
        b = None if c["sym"] else (e["b1"] if c["fmt"] == F1 else e["b2"])
        sweep.bqd.qmv(x, w, e["scales"], b, c["fmt"], c["gs"], out=y, stream=st)

    graphs = _graph_calls(sweep, one, len(W), st)
    best = None
    with torch.cuda.stream(st):
        for g in graphs:  # warm replay
            g.replay()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for g in graphs:
                g.replay()
            e1.record(st)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e3 / len(W)
            best = t if best is None else min(best, t)
    del graphs
    return best


def per_call_table(sweep, calls, weights, reps: int = 3):
    """µs per call and effective GB/s for each configuration in `calls`
    (dicts as sweep_calls() makes), each timed over the rotating weight sets
    weights[(proj, gs)]."""
    torch = sweep.torch
    rows = []
    gen = torch.Generator(device=sweep.dev)
    gen.manual_seed(99)
    from bit_quantized_decode_unpack_gb300 import synth
    for c in calls:
        M, N, K = c["M"], c["N"], c["K"]
        x = synth.torch_activations(gen, M, K, sweep.dev)
        y = torch.empty((M, N), dtype=torch.float16, device=sweep.dev)
        us = time_call(sweep, c, weights[(c["proj"], c["gs"])], x, y, reps)
        nb = call_bytes(c["fmt"], c["sym"], M, N, K, c["gs"])
        rows.append(dict(proj=c["proj"], variant=c["variant"], gs=c["gs"], M=M, N=N, K=K, bytes=nb,
                         us=round(us, 3), gbs=round(nb / (us * 1e-6) / 1e9, 1)))
        del x, y
    return rows


def aggregate(rows, key):
    """Sum of bytes over sum of time, per key(row)."""
    acc = {}
    for r in rows:
        k = key(r)
        b, t = acc.get(k, (0, 0.0))
        acc[k] = (b + r["bytes"], t + r["us"])
    return {k: {"gbs": round(b / (t * 1e-6) / 1e9, 1), "us": round(t, 2)} for k, (b, t) in acc.items()}


def make_weight_sets(sweep, name, N, K, gs, fmts, sets, seed):
    """`sets` weight sets of (N, K, gs) for the formats in `fmts` (packed on
    the device), with their scales and 1/2-bit biases."""
    torch = sweep.torch
    from bit_quantized_decode_unpack_gb300 import synth
    gen = torch.Generator(device=sweep.dev)
    gen.manual_seed(seed)
    lst = []
    for _ in range(sets):
        s_ = synth.torch_scales(gen, N, K // gs, sweep.dev)
        e = {"scales": s_}
        if F1 in fmts:
            e["b1"] = synth.torch_biases(gen, F1, s_, sweep.dev)
        if F2 in fmts:
            e["b2"] = synth.torch_biases(gen, F2, s_, sweep.dev)
        for fmt, key in ((F1, "w1"), (F2, "w2"), (T5, "w5")):
            if fmt in fmts:
                e[key] = sweep.bqd.pack(synth.torch_codes(gen, fmt, N, K, sweep.dev), fmt, gs)
        lst.append(e)
    return lst


def config_tables(sweep, sweep_rows):
    """The three single-format configurations, each as per-call rows and one
    aggregate (bytes of all its calls / time of all its calls):
      config 1: 1-bit, M=1, N=256, K=512, gs=64 (8192 rotating sets, 196 MB);
      config 2: 2-bit asym + sym, M 1..5, gs 64/128, (N,K) in {(5120,5120),
                (1024,5120), (17408,5120), (5120,17408)};
      config 3: t5, M 1..5, gs 64/128, (N,K) in {(17408,5120), (5120,17408)}.
    Shapes that the sweep already timed reuse its rows; 5120x5120 and the
    1-bit 256x512 case are timed here."""
    torch = sweep.torch
    out = {}
    # config 1
    W1 = make_weight_sets(sweep, "c1", 256, 512, 64, (F1,), 8192, seed=11)
    c1 = [dict(M=1, proj="c1_256x512", N=256, K=512, variant="affine1", fmt=F1, sym=False, gs=64)]
    r1 = per_call_table(sweep, c1, {("c1_256x512", 64): W1})
    del W1
    out["config1_affine1_256x512_m1_gs64"] = {"rows": r1, **aggregate(r1, lambda r: "all")["all"]}
    # config 2: the sweep's k/gate/down rows plus 5120x5120
    extra = {}
    for gs in GROUP_SIZES:
        extra[("sq_5120", gs)] = make_weight_sets(sweep, "sq", 5120, 5120, gs, (F2,), 64, seed=20 + gs)
    c2_new = [dict(M=M, proj="sq_5120", N=5120, K=5120, variant=v, fmt=F2, sym=sym, gs=gs)
              for M in MS for v, sym in (("affine2", False), ("affine2_sym", True)) for gs in GROUP_SIZES]
    r2 = per_call_table(sweep, c2_new, extra)
    del extra
    r2 += [r for r in sweep_rows if r["variant"] in ("affine2", "affine2_sym")
           and r["proj"] in ("k_proj", "gate_proj", "down_proj")]
    out["config2_affine2"] = {"rows": len(r2), **aggregate(r2, lambda r: "all")["all"],
                              "by_shape": aggregate(r2, lambda r: f"{r['N']}x{r['K']}"),
                              "by_m": aggregate(r2, lambda r: f"M{r['M']}")}
    r3 = [r for r in sweep_rows if r["variant"] == "t5" and r["proj"] in ("gate_proj", "down_proj")]
    out["config3_t5"] = {"rows": len(r3), **aggregate(r3, lambda r: "all")["all"],
                         "by_shape": aggregate(r3, lambda r: f"{r['N']}x{r['K']}"),
                         "by_m": aggregate(r3, lambda r: f"M{r['M']}")}
    torch.cuda.synchronize()
    return out


MID_M = (9, 12, 16)


def mid_m_table(sweep, reps: int = 3):
    """Mid-M calls, between the decode kernels' M = 2~5 (p1 §二.2) and the t5
    prefill product's M > 16 (p1 §二.3): the gate and down projections, 2-bit
    gs=64 with biases and t5 gs=128, at M = 9, 12, 16.  µs per call as the
    dispatcher runs it, and with the decode kernel (passes of 8 x rows as grid
    rows of one launch) and the prefill product forced, over the sweep's
    rotating weight sets."""
    torch = sweep.torch
    bqd = sweep.bqd
    from bit_quantized_decode_unpack_gb300 import synth
    gen = torch.Generator(device=sweep.dev)
    gen.manual_seed(7)
    rows = []
    old = bqd.get_option(bqd.OPT_KERNEL)
    try:
        for proj in ("gate_proj", "down_proj"):
            N, K = dict(shapes())[proj]
            for variant, fmt, sym, gs in (("affine2", F2, False, 64), ("t5", T5, True, 128)):
                for M in MID_M:
                    c = dict(M=M, proj=proj, N=N, K=K, variant=variant, fmt=fmt, sym=sym, gs=gs)
                    x = synth.torch_activations(gen, M, K, sweep.dev)
                    y = torch.empty((M, N), dtype=torch.float16, device=sweep.dev)
                    r = dict(proj=proj, variant=variant, gs=gs, M=M)
                    for key, kern in (("us", None), ("us_decode", "tma"), ("us_prefill", "qmm")):
                        bqd.force_kernel(kern)
                        r[key] = round(time_call(sweep, c, sweep.weights[(proj, gs)], x, y, reps), 2)
                    bqd.force_kernel(None)
                    r["gbs"] = round(call_bytes(fmt, sym, M, N, K, gs) / (r["us"] * 1e-6) / 1e9, 1)
                    rows.append(r)
                    del x, y
    finally:
        bqd.set_option(bqd.OPT_KERNEL, old)
    return rows


QMM_CASES = [(M, N, K) for M in (32, 512, 2048) for (N, K) in [(17408, 5120), (5120, 17408)]]


def time_qmm(dev, fmt: int, reps: int = 10):
    """The tcgen05 prefill matrix product of one format, gs=128: TFLOP/s per
    case (2*M*N*K flops).  The product is forced (bqd_set_option) so that each
    case times that kernel, whatever the dispatcher would pick at that M.
    Each case rotates through enough weight sets (codes, scales, biases for
    1/2-bit) to exceed the 129 MB L2."""
    import bit_quantized_decode_unpack_gb300 as bqd
    old = bqd.get_option(bqd.OPT_KERNEL)
    bqd.force_kernel("qmm")
    try:
        return _time_qmm(dev, fmt, reps)
    finally:
        bqd.set_option(bqd.OPT_KERNEL, old)


def _time_qmm(dev, fmt: int, reps: int):
    import torch
    import bit_quantized_decode_unpack_gb300 as bqd
    from bit_quantized_decode_unpack_gb300 import synth
    gen = torch.Generator(device=dev)
    gen.manual_seed(77 + fmt)
    rows, tot_flop, tot_ms = [], 0.0, 0.0
    for M, N, K in QMM_CASES:
        set_bytes = bqd.packed_bytes(fmt, N, K, 128) + N * (K // 128) * 2 * (1 if fmt == T5 else 2)
        nsets = max(2, -(-160 * 2**20 // set_bytes))
        W = []
        for _ in range(nsets):
            s_ = synth.torch_scales(gen, N, K // 128, dev)
            b_ = synth.torch_biases(gen, fmt, s_, dev)
            W.append((bqd.pack(synth.torch_codes(gen, fmt, N, K, dev), fmt, 128), s_, b_))
        x = synth.torch_activations(gen, M, K, dev)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        for i in range(3):
            w_, s_, b_ = W[i % nsets]
            bqd.qmv(x, w_, s_, b_, fmt, 128, out=y)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            w_, s_, b_ = W[i % nsets]
            bqd.qmv(x, w_, s_, b_, fmt, 128, out=y)
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1) / reps
        flop = 2.0 * M * N * K
        rows.append({"M": M, "N": N, "K": K, "us": round(ms * 1e3, 1), "tflops": round(flop / (ms * 1e-3) / 1e12, 1),
                     "weight_sets": nsets})
        tot_flop += flop
        tot_ms += ms
        del W, x, y
    return rows, tot_flop / (tot_ms * 1e-3) / 1e12


SPEC_CASE = (64, 8, 151936)  # sequences, draft tokens, vocabulary (a Qwen-sized vocabulary)


def time_spec_verify(dev, reps: int = 20):
    """Speculative-decoding verification over fp16 logits [B, D+1, V]: GB/s of
    logits read (plus drafts and results) per call.  A CUDA graph of `reps`
    calls alternating two logits sets (each larger than the L2 at the default
    size) is replayed, so that small batches time the device, not the host's
    launch path."""
    import torch
    import bit_quantized_decode_unpack_gb300 as bqd
    B, D, V = SPEC_CASE
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    sets = [torch.randn((B, D + 1, V), generator=gen, device=dev).to(torch.float16) for _ in range(2)]
    draft = torch.randint(0, V, (B, D), generator=gen, device=dev, dtype=torch.int32)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(3):
            bqd.spec_decode_verify(sets[i % 2], draft, acc, nxt, stream=stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(reps):
                bqd.spec_decode_verify(sets[i % 2], draft, acc, nxt, stream=stream)
        for _ in range(3):
            graph.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        e1.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    nbytes = B * (D + 1) * V * 2 + B * D * 4 + 2 * B * 4
    del graph, sets
    return us, nbytes / (us * 1e-6) / 1e9


def kernel_traffic_from_profiles():
    """(DRAM read + write, DRAM read) / algorithmic bytes of the QMV kernels over
    the eight calls of one sweep group, captured without cache flushes between
    them (profiles/qmv_traffic.json), or None when a kernel source changed since."""
    p = ROOT / "profiles" / "qmv_traffic.json"
    if not p.exists():
        return None
    try:
        d = json.loads(p.read_text())
        for src, digest in d["kernel_sha256"].items():
            if hashlib.sha256((ROOT / src).read_bytes()).hexdigest() != digest:
                return None
        return float(d["aggregate"]), float(d["aggregate_read"])
    except Exception:
        return None


def run_case(spec: str, sets: int, reps: int = 64, graph: bool = False):
    """--case fmt,M,N,K,gs[,sym]: one configuration over rotating weight sets
    (the command line used for single-kernel ncu captures).  With --graph the
    reps calls also run as one CUDA graph (best of 5 replays), which takes the
    host's launch time out of the per-call figure."""
    import torch
    import bit_quantized_decode_unpack_gb300 as bqd
    from bit_quantized_decode_unpack_gb300 import _build, synth
    _build.build()
    f = spec.split(",")
    fmt, M, N, K, gs = (int(v) for v in f[:5])
    sym = len(f) > 5 and f[5] == "sym"
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    W = []
    for _ in range(sets):
        s_ = synth.torch_scales(gen, N, K // gs, dev)
        b_ = None if sym else synth.torch_biases(gen, fmt, s_, dev)
        W.append((bqd.pack(synth.torch_codes(gen, fmt, N, K, dev), fmt, gs), s_, b_))
    x = synth.torch_activations(gen, M, K, dev)
    y = torch.empty(M, N, dtype=torch.float16, device=dev)
    for i in range(4):
        w, s_, b_ = W[i % sets]
        bqd.qmv(x, w, s_, b_, fmt, gs, out=y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        w, s_, b_ = W[i % sets]
        bqd.qmv(x, w, s_, b_, fmt, gs, out=y)
    e1.record()
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    nb = call_bytes(fmt, sym or fmt == T5, M, N, K, gs)
    res = {"case": spec, "us_per_call_eager": us, "gbs": nb / (us * 1e-6) / 1e9,
           "tflops": 2.0 * M * N * K / (us * 1e-6) / 1e12}
    if graph:
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(reps):
                w, s_, b_ = W[i % sets]
                bqd.qmv(x, w, s_, b_, fmt, gs, out=y)
        best = float("inf")
        with torch.cuda.stream(st):
            for r in range(8):
                e0.record(st)
                g.replay()
                e1.record(st)
                e1.synchronize()
                if r >= 3:
                    best = min(best, e0.elapsed_time(e1) * 1e3 / reps)
        res.update({"us_per_call_graph": best, "gbs_graph": nb / (best * 1e-6) / 1e9})
    print(json.dumps(res), flush=True)
    return 0


def run_group(spec: str):
    """--group M,proj: the eight calls of one (M, projection) group of the
    sweep (4 variants x 2 group sizes), in sweep order, each on tensors of its
    own, after a 512 MB read of a buffer not written since it was allocated:
    the L2 then holds only clean lines of that buffer, so no write-back of
    earlier dirty lines lands inside a captured launch.  Used for the ncu
    check that a step's calls read their weights from DRAM, not from the L2
    (with --cache-control none, DRAM bytes per launch = algorithmic bytes)."""
    import torch
    import bit_quantized_decode_unpack_gb300 as bqd
    from bit_quantized_decode_unpack_gb300 import _build, synth
    _build.build()
    M_s, proj = spec.split(",")
    M = int(M_s)
    N, K = dict(shapes())[proj]
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    calls = [c for c in sweep_calls() if c["M"] == M and c["proj"] == proj]
    data = []
    for c in calls:
        s_ = synth.torch_scales(gen, N, K // c["gs"], dev)
        b_ = None if c["sym"] else synth.torch_biases(gen, c["fmt"], s_, dev)
        w = bqd.pack(synth.torch_codes(gen, c["fmt"], N, K, dev), c["fmt"], c["gs"])
        x = synth.torch_activations(gen, M, K, dev)
        data.append((c, x, w, s_, b_, torch.empty(M, N, dtype=torch.float16, device=dev)))
    flush = torch.ones(128 * 2**20, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    rows = []
    for rep in range(3):
        flush.sum()
        torch.cuda.synchronize()
        for c, x, w, s_, b_, y in data:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            bqd.qmv(x, w, s_, b_, c["fmt"], c["gs"], out=y)
            e1.record()
            e1.synchronize()
            if rep == 2:
                nb = call_bytes(c["fmt"], c["sym"], M, N, K, c["gs"])
                rows.append({"variant": c["variant"], "gs": c["gs"], "bytes": nb,
                             "us_eager": round(e0.elapsed_time(e1) * 1e3, 2)})
    print(json.dumps({"group": spec, "calls": rows}), flush=True)
    return 0


# ---- CPU baseline / reference arm (the oracle on host cores) ----------------------

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(rows_per_call: int, calls, seed=0, threads: int = 1):
    """Time the float64 oracle on the first `rows_per_call` weight rows of each
    call (same distributions).  With threads > 1 the rows of each call are
    split into contiguous ranges, one per thread (the C oracle runs without
    the interpreter lock).  Returns (bytes, seconds)."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from bit_quantized_decode_unpack_gb300 import synth
    tot_b, tot_t = 0, 0.0
    cache = {}
    pool = ThreadPoolExecutor(threads) if threads > 1 else None
    for c in calls:
        key = (c["proj"], c["variant"], c["gs"])
        if key not in cache:
            rng = np.random.default_rng(seed + len(cache))
            R, K, gs = rows_per_call, c["K"], c["gs"]
            codes = synth.codes(rng, c["fmt"], R, K)
            s = synth.scales(rng, R, K // gs)
            b = None if c["sym"] else synth.biases(rng, c["fmt"], s)
            cache[key] = (oracle.c_pack(codes, c["fmt"], gs), s, b)
        packed, s, b = cache[key]
        x = synth.activations(np.random.default_rng(c["M"]), c["M"], c["K"])
        t = time.perf_counter()
        if pool is None:
            oracle.c_qmv_rows(x, packed, s, b, c["fmt"], c["gs"])
        else:
            edges = np.linspace(0, rows_per_call, threads + 1).astype(np.int64)
            futs = [pool.submit(oracle.c_qmv_rows, x, packed, s, b, c["fmt"], c["gs"], np.arange(lo, hi))
                    for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]
            for f in futs:
                f.result()
        tot_t += time.perf_counter() - t
        tot_b += call_bytes(c["fmt"], c["sym"], c["M"], rows_per_call, c["K"], c["gs"])
    if pool is not None:
        pool.shutdown()
    return tot_b, tot_t


def calibrate_rows(calls, seconds: float, cap: int = 256):
    """Rows per call so that one oracle pass over `calls` takes ~`seconds`."""
    b, t = oracle_sample(2, calls)
    per_row = t / 2
    return max(1, min(cap, int(seconds / max(per_row, 1e-9)))), per_row


def reference_arm(args):
    """The float64 oracle as the reference arm, on all host cores: every
    step is a bounded sample of the same workload (the first R weight rows of
    a stride-j subset of the 280 calls, the rows of each call split over the
    cores), sized so that the whole run ends within about two minutes
    (--ref-budget)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    calls = sweep_calls()
    cores = host_cores()
    budget = args.ref_budget / max(1, args.steps + args.warmup)  # seconds per step
    _, per_row = calibrate_rows(calls, 1.0)
    per_row /= cores  # rows are split over the cores
    stride = 1
    while per_row / stride > budget / 8 and stride < len(calls):
        stride *= 2
    sub = calls[::stride]
    rows = max(cores, min(64 * cores, int(budget / max(per_row * len(sub), 1e-9))))
    for _ in range(args.warmup):
        oracle_sample(rows, sub, threads=cores)
    b = t = 0.0
    for _ in range(args.steps):
        bb, tt = oracle_sample(rows, sub, threads=cores)
        b += bb
        t += tt
    value = b / t / 1e9
    sample = (f"first {rows} weight rows of " + ("each" if stride == 1 else f"every {stride}th") +
              f" of the 280 calls, per step, rows split over {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- main --------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=64)
    ap.add_argument("--quick", action="store_true", help="two projections only (development)")
    ap.add_argument("--table", type=str, default=None, help="also write the per-call table (CSV) here")
    ap.add_argument("--no-table", action="store_true", help="skip the per-call table and the config figures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-qmm", action="store_true", help="skip the prefill matrix-product timings")
    ap.add_argument("--no-spec", action="store_true", help="skip the speculative-decoding verification timing")
    ap.add_argument("--cpu-rows", type=int, default=0, help="0: sized for ~12 s of oracle work")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--case", type=str, default=None, help="fmt,M,N,K,gs[,sym]: time one configuration")
    ap.add_argument("--graph", action="store_true", help="--case: also time the calls replayed from a CUDA graph")
    ap.add_argument("--group", type=str, default=None,
                    help="M,proj: the eight calls of one sweep group on their own tensors (L2 check)")
    ap.add_argument("--spec-case", type=str, default=None,
                    help="B,D,V: time the speculative-decoding verification on fp16 logits")
    args = ap.parse_args()

    if args.case:
        return run_case(args.case, args.sets, graph=args.graph)
    if args.group:
        return run_group(args.group)
    if args.spec_case:
        import torch
        global SPEC_CASE
        SPEC_CASE = tuple(int(v) for v in args.spec_case.split(","))
        us, gbs = time_spec_verify(torch.device("cuda", 0))
        print(json.dumps({"spec_case": args.spec_case, "us_per_call": us, "gbs": gbs}), flush=True)
        return 0

    if args.impl == "reference":
        return reference_arm(args)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from bit_quantized_decode_unpack_gb300 import _build
    _build.build()

    sweep = Sweep(dev, args.sets, seed=1234 + rank, quick=args.quick)
    n_graphs = -(-args.sets // 5) + 0
    sweep.capture(n_graphs)

    def barrier():
        if dist is not None:
            dist.barrier()

    with ClockSampler(local) as clk:
        ms = time_steps(sweep, args.steps, args.warmup, barrier=barrier)
    clocks = clk.summary()
    ms_e2e = time_steps(sweep, args.steps, args.warmup, e2e=True, barrier=barrier)

    ms = max_over_ranks(ms, dist, dev)
    ms_e2e = max_over_ranks(ms_e2e, dist, dev)
    value = whole_job_gbs(sweep.bytes_per_step, args.steps, world, ms)
    value_e2e = whole_job_gbs(sweep.bytes_per_step, args.steps, world, ms_e2e)

    table = configs = mid_m = None
    if rank == 0 and not args.no_table:
        table = per_call_table(sweep, sweep.calls, sweep.weights)
        if args.table:
            with open(args.table, "w") as f:
                f.write("proj,variant,gs,M,us_per_call,gbs\n")
                for r in table:
                    f.write(f"{r['proj']},{r['variant']},{r['gs']},{r['M']},{r['us']},{r['gbs']}\n")
        if not args.quick:
            configs = config_tables(sweep, table)
            mid_m = mid_m_table(sweep)

    if rank == 0:
        peaks, src = load_peaks()
        hbm = float(peaks["hbm_gbs"])
        achieved = sweep.bytes_per_step / (ms / args.steps * 1e-3) / 1e9
        tr = kernel_traffic_from_profiles()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "calls_per_step": len(sweep.calls),
                       "bytes_per_step": sweep.bytes_per_step,
                       "page_bytes_per_step": sweep.page_bytes_per_step,
                       "weight_sets": args.sets, "l2": "inputs larger than L2 (rotating weight sets)",
                       "accumulate": "fp32", "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": src,
                         "traffic": None if tr is None else tr[0] * sweep.bytes_per_step,
                         "traffic_read": None if tr is None else tr[1] * sweep.bytes_per_step,
                         "traffic_basis": "DRAM read + write (traffic) and read (traffic_read) / algorithmic "
                                          "bytes over the eight calls of one sweep group, no cache flush between "
                                          "them (profiles/qmv_traffic.json), x bytes per step; the writes are "
                                          "write-backs of lines dirtied before the launches",
                         "kernel": "qmv (all 280 launches of a step)",
                         "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS},
            "e2e": {"value": value_e2e, "unit": UNIT, "h2d_bytes_per_step": sweep.h2d,
                    "d2h_bytes_per_step": sweep.d2h},
            "gpu_launches": len(sweep.calls) * args.steps,
            "clocks": clocks,
        }
        if table is not None:
            line["per_call"] = {
                "columns": ["proj", "variant", "gs", "M", "us", "gbs"],
                "how": "graph of back-to-back calls of one configuration over its 64 rotating weight sets; "
                       "best of 3 replays",
                "rows": [[r["proj"], r["variant"], r["gs"], r["M"], r["us"], r["gbs"]] for r in table]}
            line["per_format_m"] = aggregate(table, lambda r: f"{r['variant']}/M{r['M']}")
            line["per_format"] = aggregate(table, lambda r: r["variant"])
            line["per_projection"] = aggregate(table, lambda r: r["proj"])
        if configs is not None:
            line["configs"] = configs
        if mid_m is not None:
            line["mid_m"] = {"columns": ["proj", "variant", "gs", "M", "us", "us_decode", "us_prefill", "gbs"],
                             "rows": [[r["proj"], r["variant"], r["gs"], r["M"], r["us"], r["us_decode"],
                                       r["us_prefill"], r["gbs"]] for r in mid_m],
                             "note": "us: as dispatched; us_decode: decode kernel forced (passes of 8 x rows "
                                     "in one launch); us_prefill: prefill product forced"}
        if not args.no_qmm:
            tf_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
            for key, fmt, label in (("qmm", T5, "t5"), ("qmm_affine2", F2, "2-bit affine"),
                                    ("qmm_affine1", F1, "1-bit affine")):
                qrows, qagg = time_qmm(dev, fmt)
                line[key] = {"metric": f"{label} prefill QMM TFLOP/s (2*M*N*K), gs=128", "value": qagg,
                             "unit": "TFLOP/s", "cases": qrows,
                             "roofline": {"bound": "tensor", "achieved": qagg, "peak": tf_peak, "unit": "TFLOP/s",
                                          "frac": qagg / tf_peak,
                                          "peak_source": src + " bf16 burst (fp16 runs at the bf16 rate)"}}
        if not args.no_spec:
            us, gbs = time_spec_verify(dev)
            hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            B, D, V = SPEC_CASE
            line["spec_verify"] = {"metric": "speculative-decoding verification GB/s (fp16 logits read)",
                                   "value": gbs, "unit": "GB/s", "us_per_call": us,
                                   "config": {"sequences": B, "draft_tokens": D, "vocab": V, "dtype": "f16"},
                                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                                "frac": gbs / hbm, "peak_source": src}}
        if not args.no_cpu_baseline:
            import oracle
            oracle.build()
            rows = args.cpu_rows or calibrate_rows(sweep_calls(), 12.0)[0]
            b, t = oracle_sample(rows, sweep_calls())
            cores = host_cores()
            rows_mt = rows * cores
            b_mt, t_mt = oracle_sample(rows_mt, sweep_calls(), threads=cores)
            line["cpu_baseline"] = {"value": b_mt / t_mt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": f"first {rows_mt} weight rows of each of the 280 calls, rows split "
                                              f"over {cores} threads ({t_mt:.1f} s)",
                                    "single_thread": {"value": b / t / 1e9, "unit": UNIT, "cores": 1,
                                                      "sample": f"first {rows} weight rows of each of the 280 "
                                                                f"calls ({t:.1f} s)"},
                                    "host_cpu_count": os.cpu_count()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
