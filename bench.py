"""Benchmark of the FP8 paged-KV hot path on one GB300 (replicas across GPUs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload verify48|decode128k|serving64]
                    [--page-size 32|64] [--impl ours|reference]

A step is one pass of the whole hot path over one batch:
  verify48   (default) 48 layers [SW512 x3, G] x12, B=1, M=12, L=8192: per
             layer a 12-token E4M3 insert then paged attention (+ reduce),
             one fp8kv_append_paged_attention call;
  decode128k 12 global layers, B=1, M=1, L=131072, page 64: 1-token insert +
             split-KV attention + reduce per layer (one append call);
  serving64  8 layers G/SW512, B=64, L ~ U[1024, 32768], M=12, page 32:
             fused Q/K RMSNorm + RoPE + E4M3 insert, then attention.
Inputs are seeded synthetic tensors generated on the device; the whole step
is captured in CUDA graphs (one per cache copy) and replayed; cache copies
rotate so that the data a step reads is not in L2 (working set > 4x L2).

Prints one JSON line.  `value` is the step's algorithmic HBM bytes / step time
(GB/s); `verify_steps_per_s` is steps / time.  `--impl reference` times the
CPU oracle (float64, single thread) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from verify_attention_gb300 import bytemodel as bm  # noqa: E402
from verify_attention_gb300 import inputs as gen  # noqa: E402

METRIC = "FP8 paged attn achieved HBM GB/s (% of ~8 TB/s) and verify-steps/s at M=12"
L2_BYTES = 129 * 1024 * 1024


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# DRAM traffic of the dominant kernel per launch, from an ncu capture kept in
# profiles/: the summary names the kernel, the bytes and the SHA-256 of the
# sources it was built from; a changed source makes the figure stale (None).
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "ncu_attention_tc_verify_global.md")
KERNEL_SOURCES = ["verify_attention_gb300/csrc/attention_tc.cu", "verify_attention_gb300/csrc/attention.cuh",
                  "verify_attention_gb300/csrc/common.cuh", "verify_attention_gb300/csrc/tcgen05.cuh"]


def kernel_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(dispatch):
    """(bytes per launch, note) for the tcgen05 verifier kernel, or (None, why)."""
    if not dispatch.startswith("attention_tc"):
        return None, "no capture for this kernel"
    try:
        fields = {}
        for line in open(TRAFFIC_PROFILE):
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        if fields.get("kernel_sources_sha256") != kernel_sources_sha256():
            return None, "kernel changed since the capture"
        if fields.get("dispatch", "").split(" cluster=")[0] != dispatch.split(" cluster=")[0]:
            return None, "captured launch shape differs"
        return int(fields["dram_bytes_per_launch"]), os.path.relpath(TRAFFIC_PROFILE, ROOT)
    except (OSError, KeyError, ValueError):
        return None, "no capture"


# ------------------------------------------------------------- workloads

class Layer:
    """Device tensors of one layer (one cache copy)."""

    def __init__(self, case: gen.LayerCase, device, cache_dtype="e4m3", split_tokens=0, fused=None):
        from verify_attention_gb300 import fp8kv
        lay = case.layout
        self.case = case
        self.M = case.M
        self.page_size = lay.page_size
        self.window_left = case.window_left
        self.split_tokens = split_tokens
        self.q = case.q.to(device)
        self.k_new = case.k_new.to(device)
        self.v_new = case.v_new.to(device)
        self.slots_new = case.slots_new.to(device)
        self.bt = lay.block_table.to(device)
        self.sl = lay.seq_lens.to(device)
        self.max_seq_len = int(lay.seq_lens.max())
        self.seq_lens = lay.seq_lens.tolist()
        Hkv = self.k_new.shape[1]
        shape = (lay.num_pages, Hkv, lay.page_size, 128)
        dt = torch.uint8 if cache_dtype == "e4m3" else torch.bfloat16
        self.kc = torch.zeros(shape, dtype=dt, device=device)
        self.vc = torch.zeros(shape, dtype=dt, device=device)
        self.ks = torch.tensor([case.k_scale], dtype=torch.float32, device=device)
        self.vs = torch.tensor([case.v_scale], dtype=torch.float32, device=device)
        n = case.k_prior.shape[0]
        for i in range(0, n, 1 << 20):   # prefill the context (untimed)
            fp8kv.fp8kv_cache_insert(case.k_prior[i:i + (1 << 20)].to(device),
                                     case.v_prior[i:i + (1 << 20)].to(device),
                                     case.slots_prior[i:i + (1 << 20)].to(device), self.ks, self.vs,
                                     self.kc, self.vc)
        self.fused = fused
        if fused is not None:
            self.fq = fused.q.to(device)
            self.fk = fused.k.to(device)
            self.fv = fused.v.to(device)
            self.fpos = fused.positions.to(device)
            self.fqw = fused.q_norm_w.to(device)
            self.fkw = fused.k_norm_w.to(device)
            self.fcs = fused.cos_sin.to(device)
            self.fslots = fused.slots.to(device)
        B, M, Hq, D = self.q.shape
        self.ws_bytes = fp8kv.fp8kv_paged_attention_workspace_size(
            B, M, Hq, Hkv, D, self.page_size, self.max_seq_len, self.window_left, split_tokens)
        self.out = torch.empty_like(self.q)

    def insert(self):
        from verify_attention_gb300 import fp8kv
        if self.fused is None:
            fp8kv.fp8kv_cache_insert(self.k_new, self.v_new, self.slots_new, self.ks, self.vs, self.kc, self.vc)
        else:
            # the fused boundary writes the normed, rotated Q rows the attention reads
            fp8kv.fp8kv_qk_norm_rope_insert(self.fq, self.fk, self.fv, self.fpos, self.fqw, self.fkw,
                                            self.fused.eps, self.fcs, self.q.view(self.fq.shape),
                                            self.fslots, self.ks, self.vs, self.kc, self.vc)

    def attend(self, ws):
        from verify_attention_gb300 import fp8kv
        fp8kv.fp8kv_paged_attention(self.q, self.kc, self.vc, self.bt, self.sl, self.max_seq_len, self.ks,
                                    self.vs, self.case.sm_scale, self.window_left, self.split_tokens,
                                    workspace=ws, out=self.out)

    def prepare(self, ws):
        """The layer's step as prepared calls (arguments marshalled once)."""
        from verify_attention_gb300 import fp8kv
        B, M, Hq, D = self.q.shape
        if self.fused is None:
            self._prepared = [fp8kv.PreparedAttention(
                self.q, self.kc, self.vc, self.bt, self.sl, self.max_seq_len, self.ks, self.vs, self.case.sm_scale,
                self.window_left, self.split_tokens, workspace=ws, out=self.out, k_new=self.k_new.view(B, M, -1, D),
                v_new=self.v_new.view(B, M, -1, D))]
        else:
            self._prepared = None

    def step_prepared(self, ws):
        if getattr(self, "_prepared", None):
            for call in self._prepared:
                call()
        else:
            self.step(ws)

    def step(self, ws):
        """The layer's share of a step: the new tokens' insert, then attention.
        Plain inserts of the new rows go through the one-call append entry
        (same cache bytes and output as insert + attention); the fused
        norm/RoPE boundary is its own call."""
        from verify_attention_gb300 import fp8kv
        if self.fused is None:
            B, M, Hq, D = self.q.shape
            fp8kv.fp8kv_append_paged_attention(self.k_new.view(B, M, -1, D), self.v_new.view(B, M, -1, D),
                                               self.q, self.kc, self.vc, self.bt, self.sl, self.max_seq_len,
                                               self.ks, self.vs, self.case.sm_scale, self.window_left,
                                               self.split_tokens, workspace=ws, out=self.out)
        else:
            self.insert()
            self.attend(ws)

    def attn_bytes(self):
        B, M, Hq, D = self.q.shape
        e = 1 if self.kc.dtype == torch.uint8 else 2
        return bm.attention_bytes(self.seq_lens, M, Hq, self.k_new.shape[1], D, e, self.window_left,
                                  self.page_size)

    def insert_bytes(self):
        T, Hkv, D = self.k_new.shape
        if self.fused is None:
            return bm.insert_bytes(T, Hkv, D, 1 if self.kc.dtype == torch.uint8 else 2)
        return bm.fused_insert_bytes(T, self.fq.shape[1], Hkv, D)

    def flops(self):
        B, M, Hq, D = self.q.shape
        return bm.attention_flops(self.seq_lens, M, Hq, D, self.window_left)


class Workload:
    def __init__(self, name, layers_per_copy, description, unit_rows):
        self.name = name
        self.copies = layers_per_copy           # [copy][layer]
        self.description = description
        self.unit_rows = unit_rows
        self.inputs_sha256 = None               # of the first layer's generated inputs
        dev = layers_per_copy[0][0].q.device
        need = max(l.ws_bytes for c in layers_per_copy for l in c)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    def step(self, copy):
        for layer in self.copies[copy]:
            layer.step(self.ws)

    def bytes_per_step(self):
        return sum(l.attn_bytes() + l.insert_bytes() for l in self.copies[0])

    def flops_per_step(self):
        return sum(l.flops() for l in self.copies[0])


def case_sha256(case):
    """SHA-256 of one layer's generated inputs (queries, context and new
    K/V, slots, block table, sequence lengths): a fingerprint of the inputs."""
    import hashlib
    h = hashlib.sha256()
    try:
        for t in (case.q, case.k_prior, case.v_prior, case.k_new, case.v_new, case.slots_prior, case.slots_new,
                  case.layout.block_table, case.layout.seq_lens):
            if t is not None:
                h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    except (RuntimeError, TypeError) as e:     # a fingerprint is extra: never stop the measurement
        return f"unavailable: {str(e)[:80]}"
    return h.hexdigest()


def _free_context(cases):
    # the bf16 context was only needed to prefill the caches
    for c in cases:
        c.k_prior = c.v_prior = c.slots_prior = None
    torch.cuda.empty_cache()


def workload_page_size(name, page_size_arg):
    """The page size a workload runs at: --page-size for the verify step and
    the long-context decode, else the workload's own (verify step 32, decode
    and prefill 64, serving mix 32)."""
    if name in ("verify48", "decode128k") and page_size_arg is not None:
        return page_size_arg
    return {"verify48": 32, "decode128k": 64, "prefill16k": 64}.get(name, 32)


def workload_description(name, page_size, cache_dtype="e4m3"):
    return {
        "verify48": (f"48 layers [SW512,SW512,SW512,G]x12, B=1, M=12, Hq=72, Hkv=8, D=128, L=8192, "
                     f"page {page_size}, E4M3 cache; per layer 12-token insert + attention"),
        "decode128k": (f"12 global layers, B=1, M=1, Hq=72, Hkv=8, D=128, L=131072, page {page_size}, "
                       f"{cache_dtype} cache; per layer 1-token insert + split-KV attention + reduce"),
        "prefill16k": ("4 global layers, B=1, a prefill chunk of M=1024 tokens at the end of L=16384, Hq=72, "
                       "Hkv=8, D=128, page 64, E4M3 cache; per layer 1024-token append + causal attention in "
                       "128-row tiles"),
        "serving64": ("8 layers G/SW512 alternating, B=64, L~U[1024,32768] (seed 1005), M=12, Hq=72, Hkv=8, "
                      "D=128, page 32, E4M3 cache; per layer fused Q/K RMSNorm+RoPE+insert + attention"),
    }[name]


def _fingerprinted(w, sha):
    w.inputs_sha256 = sha
    return w


def build_workload(name, page_size, device, cache_dtype="e4m3", layers=None):
    if name == "verify48":
        n = layers or 48
        base = [gen.cfg3_case(l, page_size, device=device) for l in range(n)]
        per_copy = sum(bm.attention_bytes([8192], 12, 72, 8, 128, 1, -1, page_size) for _ in range(n))
        ncopies = max(2, math.ceil(4 * L2_BYTES / per_copy))
        copies = [[Layer(c, device) for c in base] for _ in range(ncopies)]
        fp = case_sha256(base[0])
        _free_context(base)
        return _fingerprinted(Workload(name, copies, workload_description(name, page_size), 12), fp)
    if name == "decode128k":
        copies = [[]]
        for l in range(layers or 12):
            c = gen.cfg4_case(l, device=device, page_size=page_size)
            copies[0].append(Layer(c, device, cache_dtype=cache_dtype, split_tokens=0))
            fp = case_sha256(c) if l == 0 else fp
            _free_context([c])
        return _fingerprinted(Workload(name, copies, workload_description(name, page_size, cache_dtype), 1), fp)
    if name == "prefill16k":
        copies = [[]]
        for l in range(layers or 4):
            c = gen.layer_case(1006 * 100 + l, [16384], 1024, 64, window=None, device=device)
            copies[0].append(Layer(c, device, split_tokens=0))
            fp = case_sha256(c) if l == 0 else fp
            _free_context([c])
        return _fingerprinted(Workload(name, copies, workload_description(name, 64), 1024), fp)
    if name == "serving64":
        lens = gen.cfg5_seq_lens()
        built = []
        for l in range(layers or 8):
            c = gen.cfg5_case(l, device=device, seq_lens=lens)
            f = gen.fused_case(1005 * 100 + 50 + l, c.layout, 12)
            built.append(Layer(c, device, fused=f))
            fp = case_sha256(c) if l == 0 else fp
            _free_context([c])
        return _fingerprinted(Workload(name, [built], workload_description(name, 32), 64 * 12), fp)
    raise ValueError(name)


# ------------------------------------------------------------------ timing

class ClockSampler:
    """nvidia-smi samples every 100 ms while the block runs; `load(t0, t1)`
    marks the host-time window in which the GPU ran the measured work, and the
    summary keeps the samples taken inside it (all samples when none is)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.window = None

    def load(self, t0, t1):
        self.window = (t0, t1)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        import datetime
        if not getattr(self, "lines", None):
            return None
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), float(f[4]),
                             [n for n, v in zip(names, f[6:10]) if v.lower().startswith("active")]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        use = inside or rows
        reasons = sorted({n for r in use for n in r[4]})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in rows),
                "power_w_max": max(r[3] for r in use), "reasons": reasons, "samples": len(use),
                "samples_under_load": len(inside)}


def time_graphs(graphs, steps, warmup, stream):
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def step_percentiles(graphs, n, stream):
    """Device time of each of n further replays (an event between every two),
    outside the timed region: p10, p50, p90 in ms."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(n):
            graphs[i % len(graphs)].replay()
            evs[i + 1].record(stream)
    evs[-1].synchronize()
    d = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(n))
    return {"p10": d[int(0.1 * (n - 1))], "p50": d[int(0.5 * (n - 1))], "p90": d[int(0.9 * (n - 1))],
            "steps": n}


def capture_step_graphs(w: Workload, stream):
    """One CUDA graph per cache copy; also returns the kernel launches one
    step makes (counted by the library while the first graph is captured)."""
    from verify_attention_gb300 import fp8kv
    graphs = []
    with torch.cuda.stream(stream):
        for c in range(len(w.copies)):
            w.step(c)                  # warm: attributes, tensor maps, lazy loading
    torch.cuda.synchronize()
    launches = None
    for c in range(len(w.copies)):
        g = torch.cuda.CUDAGraph()
        n0 = fp8kv.fp8kv_launch_count()
        with torch.cuda.graph(g, stream=stream):
            w.step(c)
        if launches is None:
            launches = fp8kv.fp8kv_launch_count() - n0
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs, launches


def layers_of_kind(w: Workload, window_left):
    """Every layer (all cache copies) of one kind (-1 = global)."""
    return [c[li] for c in w.copies for li, l in enumerate(w.copies[0]) if l.window_left == window_left]


def dominant_kernel(w: Workload, stream, reps=24):
    """Average device duration of the attention call (partial kernel + reduce) on
    the layer kind with the most bytes.  `reps` calls, rotating over cache copies
    and layers so the cache reads come from HBM, are captured in one CUDA graph;
    graph replays are timed with CUDA events on the launching stream, so host
    launch overhead stays outside the figure."""
    cands = [(l.attn_bytes(), li) for li, l in enumerate(w.copies[0])]
    top = max(b for b, _ in cands)
    idx = [li for b, li in cands if b == top]
    layers = [c[li] for c in w.copies for li in idx]
    secs, dispatch = time_attention_calls(layers, stream, w.ws, reps)
    return top, secs, flops_of(layers[0]), dispatch


def flops_of(layer):
    return layer.flops()


def time_attention_calls(layers, stream, ws, reps=24, step=False):
    """Median device time of one attention call (partial kernel + reduce, as
    one fp8kv_paged_attention call; with step=True the layer's whole step, new
    tokens into the cache then attention), `reps` calls rotating over `layers`
    (other cache copies, so the reads come from HBM) captured in one CUDA
    graph; also the dispatch marker of the last call."""
    from verify_attention_gb300 import fp8kv

    def call(layer):
        (layer.step if step else layer.attend)(ws)
    with torch.cuda.stream(stream):
        for i in range(3):
            call(layers[i % len(layers)])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(reps):
            call(layers[i % len(layers)])
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    per_call = []
    for _ in range(7):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        b.synchronize()
        per_call.append(a.elapsed_time(b) / reps)
    del g
    return statistics.median(per_call) / 1e3, fp8kv.fp8kv_last_dispatch()


def rotating_copies(layer, n):
    """n views of one layer that share its queries and metadata but each own a
    copy of its caches (and an output buffer), so that consecutive calls over
    them read from HBM even when one layer fits in L2."""
    import copy
    out = []
    for _ in range(n):
        c = copy.copy(layer)
        c.kc = layer.kc.clone()
        c.vc = layer.vc.clone()
        c.out = torch.empty_like(layer.out)
        out.append(c)
    return out


def call_record(layer, secs, dispatch, hbm_peak):
    b = layer.attn_bytes()
    return {"us": secs * 1e6, "algorithmic_bytes": b, "gbs": b / secs / 1e9, "frac_of_hbm": b / secs / 1e9 / hbm_peak,
            "dispatch": dispatch}


def _packed(tensors, device, align=256, pin=False):
    """One byte buffer with room for `tensors` back to back (each start
    aligned to `align` bytes) and views of it with their shapes and dtypes."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += -(-t.numel() * t.element_size() // align) * align
    buf = torch.empty(max(n, align), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views, offs


def e2e_measure(w: Workload, steps, stream, chunks=8):
    """Through the public API with host buffers: per step, every layer's new
    tokens and queries come from a pinned host buffer and every layer's
    attention output goes back into pinned host memory (the layers read and
    write views of two device staging buffers).  The copies run on a copy
    stream, overlapped with the kernels: the inputs in `chunks` copies of
    consecutive layers' inputs, each layer group starting once its chunk has
    landed, and each group's outputs copied back as soon as it finishes.  The
    step is captured once in a CUDA graph (copies included) and replayed, as a
    serving loop would run it; the same step launched eagerly from Python is
    timed too (`eager_ms_per_step`: binding and launch overhead included).
    Returns the outputs' agreement with the device-timed step's outputs (same
    inputs and cache, same kernels: bit-identical)."""
    layers = w.copies[0]
    dev = layers[0].q.device
    names = [["q", "k_new", "v_new"] if l.fused is None else ["fq", "fk", "fv", "fpos", "fslots"] for l in layers]
    saved_in = [[getattr(l, n) for n in ns] for l, ns in zip(layers, names)]
    saved_out = [l.out for l in layers]
    flat_in = [t for ts in saved_in for t in ts]
    dev_in, dviews, in_offs = _packed(flat_in, dev)
    host_in, hviews, _ = _packed(flat_in, "cpu", pin=True)
    for h, t in zip(hviews, flat_in):
        h.copy_(t)
    dev_out, oviews, out_offs = _packed(saved_out, dev)
    host_out, hoviews, _ = _packed(saved_out, "cpu", pin=True)
    h2d, d2h = host_in.numel(), host_out.numel()
    # layer groups and the byte ranges of their inputs and outputs
    n = len(layers)
    chunks = max(1, min(chunks, n))
    bounds = [round(c * n / chunks) for c in range(chunks + 1)]
    first = [0]
    for ns in names:
        first.append(first[-1] + len(ns))
    in_cut = [in_offs[first[g]] if g < n else h2d for g in bounds]
    out_cut = [out_offs[g] if g < n else d2h for g in bounds]
    cstream = torch.cuda.Stream(device=dev)
    prepared_layers = []
    eager_prepared_s = None
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in range(chunks)]
    ev_out = [torch.cuda.Event() for _ in range(chunks)]
    it = iter(dviews)
    for l, ns in zip(layers, names):
        for n in ns:
            setattr(l, n, next(it))
    for l, o in zip(layers, oviews):
        l.out = o
    torch.cuda.synchronize()

    def one():
        ev_fork.record(stream)
        cstream.wait_event(ev_fork)
        with torch.cuda.stream(cstream):
            for c in range(chunks):
                dev_in[in_cut[c]:in_cut[c + 1]].copy_(host_in[in_cut[c]:in_cut[c + 1]], non_blocking=True)
                ev_in[c].record(cstream)
        for c in range(chunks):
            stream.wait_event(ev_in[c])
            with torch.cuda.stream(stream):
                for l in layers[bounds[c]:bounds[c + 1]]:
                    if prepared_layers:
                        l.step_prepared(w.ws)
                    else:
                        l.step(w.ws)
            ev_out[c].record(stream)
            cstream.wait_event(ev_out[c])
            with torch.cuda.stream(cstream):
                host_out[out_cut[c]:out_cut[c + 1]].copy_(dev_out[out_cut[c]:out_cut[c + 1]], non_blocking=True)
        ev_join.record(cstream)
        stream.wait_event(ev_join)

    def timed(run, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            run()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / 1e3 / n

    try:
        one()
        torch.cuda.synchronize()
        match = all(torch.equal(h, o.cpu()) for h, o in zip(hoviews, saved_out))
        eager_s = timed(one, steps)
        # the same eager step with each layer's call prepared once (arguments
        # marshalled ahead, as a serving loop over fixed buffers would)
        for l in layers:
            l.prepare(w.ws)
        prepared_layers[:] = [True]
        one()
        torch.cuda.synchronize()
        eager_prepared_s = timed(one, steps)
        prepared_layers[:] = []
        mode = (f"step captured in a CUDA graph and replayed; pinned-host copies on a copy stream "
                f"overlapped with the kernels ({chunks} input chunks, outputs per layer group)")
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                one()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            torch.cuda.synchronize()

            def replay():
                with torch.cuda.stream(stream):
                    g.replay()
            graph_s = timed(replay, steps)
            del g
        except RuntimeError as e:      # a torch without host-copy capture: eager only
            torch.cuda.synchronize()
            graph_s, mode = eager_s, f"eager launches (graph capture of the copies failed: {e})"[:200]
    finally:
        for l, ns, ts in zip(layers, names, saved_in):
            for n, t in zip(ns, ts):
                setattr(l, n, t)
        for l, o in zip(layers, saved_out):
            l.out = o
            l._prepared = None
    return graph_s, eager_s, eager_prepared_s, h2d, d2h, mode, match


# ---------------------------------------------------------- CPU oracle leg

def oracle_case(name, page_size):
    """The layer the CPU oracle samples: the first global layer of the workload."""
    if name == "verify48":
        return gen.cfg3_case(3, page_size)
    if name == "decode128k":
        return gen.cfg4_case(0)
    if name == "prefill16k":
        return gen.layer_case(1006 * 100, [16384], 1024, 64, window=None)
    return gen.cfg5_case(0)


class OracleSample:
    """CPU oracle on one global layer of the workload, prefilled once
    (untimed).  A sample is the layer's E4M3 insert of its new tokens plus the
    attention of the first n query rows (b, m, h order) of sequence 0; its
    bytes are those rows' share of the layer's algorithmic bytes (KV bytes of
    their KV heads pro rata per row, plus their Q and O)."""

    def __init__(self, name, page_size):
        import oracle
        self.oracle = oracle
        case = oracle_case(name, page_size)
        lay = case.layout
        self.case = case
        self.Hkv = case.k_new.shape[1]
        self.G = case.q.shape[2] // self.Hkv
        self.kc = np.zeros((lay.num_pages, self.Hkv, lay.page_size, 128), np.uint8)
        self.vc = self.kc.copy()
        oracle.cache_insert(gen.bf16_bits(case.k_prior), gen.bf16_bits(case.v_prior),
                            case.slots_prior.numpy(), case.k_scale, case.v_scale, self.kc, self.vc)
        M, Hq = case.M, case.q.shape[2]
        self.rows_all = np.array([(0, m, h) for h in range(Hq) for m in range(M)], np.int32)
        self.q = gen.bf16_bits(case.q)
        self.bt, self.sl = lay.block_table.numpy(), lay.seq_lens.numpy()
        L = int(self.sl[0])
        per_head = bm.attention_bytes([L], M, self.G, 1, 128, 1, case.window_left, lay.page_size)
        self.bytes_per_row = per_head / (M * self.G)

    def run(self, n_rows):
        c = self.case
        o = self.oracle
        rows = self.rows_all[:n_rows]
        t0 = time.perf_counter()
        o.cache_insert(gen.bf16_bits(c.k_new), gen.bf16_bits(c.v_new), c.slots_new.numpy(), c.k_scale,
                       c.v_scale, self.kc, self.vc)
        o.paged_attention_rows(self.q, self.kc, self.vc, self.bt, self.sl, c.k_scale, c.v_scale, c.sm_scale,
                               rows, window_left=c.window_left)
        secs = time.perf_counter() - t0
        byts = n_rows * self.bytes_per_row + bm.insert_bytes(c.k_new.shape[0], self.Hkv, 128)
        return byts, secs

    def describe(self, n_rows):
        c = self.case
        L = int(self.sl[0])
        return (f"global layer of the workload (L={L}, M={c.M}): E4M3 insert of {c.k_new.shape[0]} tokens "
                f"+ float64 attention of {n_rows} query rows of sequence 0; 1 thread")


def cpu_baseline(name, page_size, target_s=12.0):
    s = OracleSample(name, page_size)
    n0 = min(s.G * s.case.M, 256)
    b, t = s.run(n0)                                      # up to one KV head's rows: calibration
    n = int(min(len(s.rows_all), max(1, n0 * target_s / max(t, 1e-3))))
    b, t = s.run(n)
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": s.describe(n) + f"; host has {os.cpu_count()} cores"}


# ------------------------------------------------ the step in one launch

def one_launch_step(w: Workload, stream, steps, warmup, per_layer_step_s, hbm_peak):
    """The workload's step through fp8kv_paged_attention_layers: every
    layer's append + attention in one persistent launch (layer order kept),
    one prepared call per cache copy, each captured in a CUDA graph; timed
    like the per-layer step (same steps, same rotation over cache copies)."""
    from verify_attention_gb300 import fp8kv
    calls = []
    for copy in w.copies:
        layers = []
        for l in copy:
            B, M, Hq, D = l.q.shape
            layers.append(dict(q=l.q, k_new=l.k_new.view(B, M, -1, D), v_new=l.v_new.view(B, M, -1, D),
                               k_cache=l.kc, v_cache=l.vc, block_table=l.bt, seq_lens=l.sl,
                               max_seq_len=l.max_seq_len, k_scale=l.ks, v_scale=l.vs, sm_scale=l.case.sm_scale,
                               window_left=l.window_left, out=l.out))
        calls.append(fp8kv.PagedAttentionLayers(layers))
    with torch.cuda.stream(stream):
        for c in calls:
            c(stream)
    torch.cuda.synchronize()
    graphs = []
    n0 = fp8kv.fp8kv_launch_count()
    for c in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            c(stream)
        graphs.append(g)
    launches = (fp8kv.fp8kv_launch_count() - n0) // len(calls)
    dispatch = fp8kv.fp8kv_last_dispatch()
    secs = time_graphs(graphs, steps, warmup, stream) / steps
    status = fp8kv.fp8kv_device_status(clear=True)
    b = w.bytes_per_step()
    return {"ms_per_step": secs * 1e3, "verify_steps_per_s": 1 / secs, "gbs": b / secs / 1e9,
            "frac_of_hbm": b / secs / 1e9 / hbm_peak, "launches_per_step": launches,
            "speedup_over_per_layer_calls": per_layer_step_s / secs, "device_status": status,
            "dispatch": dispatch,
            "entry": "fp8kv_paged_attention_layers (one persistent cooperative launch per step)"}


# ------------------------------------------------------ side measurements

def _step_time(w, stream, steps=10, warmup=3):
    graphs, launches = capture_step_graphs(w, stream)
    secs = time_graphs(graphs, steps, warmup, stream) / steps
    del graphs
    return secs, launches


def side_measurements(dev, stream, hbm_peak, bf16_peak):
    """The A/B runs and the other configurations, each under its own key of
    the one JSON line (device time, CUDA-graph replays, caches rotated or
    larger than L2):
      verify48_page64  the 48-layer step at page 64 (the page-size A/B);
      decode128k       12 long-context decode layers, E4M3 and BF16 cache at
                       page 64, E4M3 at page 32;
      prefill16k       a prefill chunk on the tensor cores;
      serving64        the batched serving mix, per layer kind, and its layers'
                       append + attention per layer and in one launch;
      cfg1, cfg2       the single-layer configurations (rotating cache copies)."""
    out = {}
    torch.cuda.empty_cache()
    w = build_workload("verify48", 64, dev)
    s64, n64 = _step_time(w, stream, steps=20)
    b64 = w.bytes_per_step()
    calls = {}
    for kind, wl in (("sliding_512", 511), ("global", -1)):
        ls = layers_of_kind(w, wl)
        secs, disp = time_attention_calls(ls, stream, w.ws)
        calls[kind] = call_record(ls[0], secs, disp, hbm_peak)
    out["verify48_page64"] = {"ms_per_step": s64 * 1e3, "verify_steps_per_s": 1 / s64, "gbs": b64 / s64 / 1e9,
                              "frac_of_hbm": b64 / s64 / 1e9 / hbm_peak, "algorithmic_bytes_per_step": b64,
                              "launches_per_step": n64, "attention_calls": calls}
    del w
    torch.cuda.empty_cache()
    dec = {}
    for dt in ("e4m3", "bf16"):
        w = build_workload("decode128k", 64, dev, cache_dtype=dt)
        s2, _ = _step_time(w, stream, steps=5)
        b2, t2, _, d2 = dominant_kernel(w, stream, reps=12)
        dec[dt] = {"gbs_step": w.bytes_per_step() / s2 / 1e9, "ms_per_step": s2 * 1e3,
                   "attention_gbs": b2 / t2 / 1e9, "attention_frac": b2 / t2 / 1e9 / hbm_peak,
                   "attention_ms": t2 * 1e3, "attention_bytes": b2, "dispatch": d2}
        del w
        torch.cuda.empty_cache()
    w = build_workload("decode128k", 32, dev)
    s2, _ = _step_time(w, stream, steps=5)
    b2, t2, _, d2 = dominant_kernel(w, stream, reps=12)
    dec["e4m3_page32"] = {"gbs_step": w.bytes_per_step() / s2 / 1e9, "ms_per_step": s2 * 1e3,
                          "attention_gbs": b2 / t2 / 1e9, "attention_frac": b2 / t2 / 1e9 / hbm_peak,
                          "attention_ms": t2 * 1e3, "attention_bytes": b2, "dispatch": d2}
    del w
    torch.cuda.empty_cache()
    out["decode128k"] = {**dec["e4m3"], "bf16": dec["bf16"], "page32": dec["e4m3_page32"],
                         "fp8_over_bf16_step_speedup": dec["bf16"]["ms_per_step"] / dec["e4m3"]["ms_per_step"],
                         "fp8_over_bf16_attention_speedup": dec["bf16"]["attention_ms"] / dec["e4m3"]["attention_ms"]}
    w = build_workload("prefill16k", 64, dev)
    s3, _ = _step_time(w, stream, steps=5)
    _, t3, f3, d3 = dominant_kernel(w, stream, reps=8)
    out["prefill16k"] = {"ms_per_step": s3 * 1e3, "tflops_step": w.flops_per_step() / s3 / 1e12,
                         "attention_ms": t3 * 1e3, "attention_tflops": f3 / t3 / 1e12,
                         "attention_frac_of_bf16_peak": f3 / t3 / 1e12 / bf16_peak, "dispatch": d3}
    del w
    torch.cuda.empty_cache()
    w = build_workload("serving64", 32, dev)
    s5, n5 = _step_time(w, stream, steps=5)
    srv = {"ms_per_step": s5 * 1e3, "gbs_step": w.bytes_per_step() / s5 / 1e9,
           "frac_of_hbm_step": w.bytes_per_step() / s5 / 1e9 / hbm_peak, "launches_per_step": n5}
    for kind, wl in (("global", -1), ("sliding_512", 511)):
        ls = layers_of_kind(w, wl)
        secs, disp = time_attention_calls(ls, stream, w.ws, reps=8)
        srv[kind] = call_record(ls[0], secs, disp, hbm_peak)
    # the 8 layers' append + attention (plain insert of the new tokens, no
    # norm/RoPE) as per-layer calls and as one persistent launch
    fused = [l.fused for c in w.copies for l in c]
    for c in w.copies:
        for l in c:
            l.fused = None
    s_app, _ = _step_time(w, stream, steps=5)
    srv["append_step_ms"] = s_app * 1e3
    srv["one_launch"] = one_launch_step(w, stream, 5, 2, s_app, hbm_peak)
    it = iter(fused)
    for c in w.copies:
        for l in c:
            l.fused = next(it)
    out["serving64"] = srv
    del w
    torch.cuda.empty_cache()
    small = {}
    for name, case, copies in (("cfg1_tiny_decode", gen.cfg1_case(device=dev), 256),
                               ("cfg2_verify_global", gen.cfg2_case(None, device=dev), 40),
                               ("cfg2_verify_sliding_512", gen.cfg2_case(512, device=dev), 40)):
        base = Layer(case, dev)
        ws = torch.empty(max(base.ws_bytes, 16), dtype=torch.uint8, device=dev)
        ls = rotating_copies(base, copies)
        secs, disp = time_attention_calls(ls, stream, ws, reps=48)
        rec = call_record(base, secs, disp, hbm_peak)
        ssecs, _ = time_attention_calls(ls, stream, ws, reps=48, step=True)
        rec["step_us"] = ssecs * 1e6
        rec["step"] = "append of the new tokens + attention (one fp8kv_append_paged_attention call)"
        small[name] = rec
        del ls, base, ws
    out.update(small)
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------------- main

def dist_setup():
    """One process per GPU (torchrun env); NCCL on GPUs, gloo without one
    (the host-side logic is the same; the CPU tests use gloo)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(ws, bytes_per_rank_step, step_s):
    """Replicas: every rank runs the same step; the job moves ws times one
    rank's bytes in the slowest rank's time."""
    return ws * bytes_per_rank_step / step_s / 1e9


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    ps = workload_page_size(args.workload, args.page_size)
    sample = OracleSample(args.workload, ps)
    _, t1 = sample.run(1)
    budget = 150.0 / (args.warmup + args.steps)          # seconds of oracle work per step
    n = int(min(len(sample.rows_all), max(1, budget / max(t1, 1e-4))))
    byts = secs = 0.0
    for i in range(args.warmup + args.steps):
        b, s = sample.run(n)
        if i >= args.warmup:
            byts += b
            secs += s
    gbs = byts / secs / 1e9
    desc = sample.describe(n)
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload,
                                            "description": workload_description(args.workload, ps),
                                            "page_size": ps},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc + f"; host has {os.cpu_count()} cores"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="verify48", choices=["verify48", "decode128k", "serving64",
                                                                  "prefill16k"])
    ap.add_argument("--page-size", type=int, default=None, choices=[32, 64])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the side measurements (page-64 step, decode, prefill, serving mix, single layers)")
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (small profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_setup()
    from verify_attention_gb300 import build, fp8kv
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, bf16_peak, peak_src = peaks()

    ps = workload_page_size(args.workload, args.page_size)
    w = build_workload(args.workload, ps, dev, layers=args.layers)
    graphs, launches_per_step = capture_step_graphs(w, stream)
    fp8kv.fp8kv_device_status(clear=True)

    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_load = time.time()
        secs = time_graphs(graphs, args.steps, args.warmup, stream)
        # the same replays continue untimed until the load has lasted 1 s, so
        # that the 100 ms clock samples see it even when the timed steps are few
        n_soak = 0
        while time.time() - t_load < 1.0 and n_soak < 100000:
            with torch.cuda.stream(stream):
                for g in graphs:
                    g.replay()
            n_soak += len(graphs)
            torch.cuda.synchronize()
        clk.load(t_load, time.time())
    barrier(ws)
    torch.cuda.synchronize()
    secs = max_over_ranks(secs, ws)
    status = fp8kv.fp8kv_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed region")

    try:
        pct = step_percentiles(graphs, max(10, min(args.steps, 200)), stream)
    except Exception as e:                       # a distribution is extra; the timed mean stands
        pct = {"error": str(e)[:120]}
    step_bytes = w.bytes_per_step()
    step_s = secs / args.steps
    value = whole_job_gbs(ws, step_bytes, step_s)

    dom_bytes, dom_s, dom_flops, dispatch = dominant_kernel(w, stream)
    achieved = dom_bytes / dom_s / 1e9
    traffic, traffic_note = measured_traffic(dispatch)
    e2e_s, e2e_eager_s, e2e_prep_s, h2d, d2h, e2e_mode, e2e_match = e2e_measure(w, max(3, min(args.steps, 20)),
                                                                                 stream)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "step_ms_percentiles": pct,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 cache, f16/fp32 math", "data": "synthetic",
        "config": {"workload": args.workload, "description": w.description, "page_size": ps,
                   "cache_copies": len(w.copies), "l2": "inputs larger than L2: cache copies rotate",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "first_layer_inputs_sha256": w.inputs_sha256},
        "verify_steps_per_s": ws / step_s,
        "pct_of_hbm_roofline": value / ws / hbm_peak,
        "algorithmic_bytes_per_step": step_bytes,
        "useful_flops_per_step": w.flops_per_step(),
        "gpu_launches": args.steps * launches_per_step,
        "gpu_launches_per_step": launches_per_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": "fp8kv_paged_attention (partial + reduce) on the largest layer",
                     "launch_ms": dom_s * 1e3, "bytes_per_launch": dom_bytes,
                     "tflops": dom_flops / dom_s / 1e12, "dispatch": dispatch,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)"},
        "e2e": {"value": ws * step_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "mode": e2e_mode,
                "eager_ms_per_step": e2e_eager_s * 1e3,
                "eager_prepared_calls_ms_per_step": e2e_prep_s * 1e3 if e2e_prep_s else None,
                "outputs_match_device_step": e2e_match},
        "clocks": clk.summary(),
    }
    if args.workload == "prefill16k":
        # a prefill chunk is bound by the tensor cores: useful FLOPs against the
        # measured dense bf16 peak (P.V runs in f16, Q.K^T as two E4M3 terms)
        tf = dom_flops / dom_s / 1e12
        line["roofline"].update({"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                                 "frac": tf / bf16_peak, "traffic": None,
                                 "traffic_source": "no capture for this kernel and workload",
                                 "gbs": achieved,
                                 "peak_source": f"{peak_src} bf16_tflops (MEASURED_PEAKS.json)"})
    if args.workload == "verify48":
        # the step's two attention-call kinds, each against HBM, and the
        # step's own append + attention calls of each kind
        line["attention_calls"] = {}
        for kind, wl in (("sliding_512", 511), ("global", -1)):
            ls = layers_of_kind(w, wl)
            secs, disp = time_attention_calls(ls, stream, w.ws)
            line["attention_calls"][kind] = call_record(ls[0], secs, disp, hbm_peak)
            ssecs, _ = time_attention_calls(ls, stream, w.ws, step=True)
            line["attention_calls"][kind]["append_call_us"] = ssecs * 1e6
    if args.workload == "verify48":
        line["one_launch"] = one_launch_step(w, stream, args.steps, args.warmup, step_s, hbm_peak)
    if rank == 0 and args.workload == "verify48" and not args.no_extra:
        del graphs
        line.update(side_measurements(dev, stream, hbm_peak, bf16_peak))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, ps)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
