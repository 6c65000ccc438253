#!/usr/bin/env python3
"""Benchmark of the quantized paged KV-cache hot path on GB300.

One step = one layer's serving decode step over a resident paged cache: the
step's new K/V rows go into the cache and every sequence is decoded.  When the
step brings one token per sequence, both happen in one call,
kvq_decode_attention_append (--unfused: kvq_append then kvq_decode_attention);
a prefill chunk (the Llama-3-70B workload) is kvq_append followed by
kvq_decode_attention.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     # the CPU oracle, timed on host cores
  python bench.py --prefill [--workload llama3-70b] [--chunk N]   # chunked prefill

The default workload is the Llama-3-70B decode batch (256 sequences of 32768
tokens, 64/8 heads, E4M3, plus a 2048-token chunk appended per sequence), the
largest single-GPU batch of the target list.  In the same run (N=1) the other
target decode batches -- Llama-2-7B E4M3, Llama-3-8B E5M2 and Llama-2-13B
INT8 -- are measured each in its own timed region and reported under
``per_config`` (step and stream-kernel GB/s, roofline fractions, bulk append
GB/s, tokens/s, clocks).

Prints ONE JSON line (rank 0).  ``value`` is decode KV-read GB/s: the
algorithmic bytes of the decode calls (every cached K/V byte of every context
once, INT8 / INT4 scales, q, out, block tables) over the step time, summed over
ranks (each rank runs its own copy of the workload: weak scaling, no
collective on the data path).  Workloads whose decode reads more than the L2
size run K steps back to back between two events; smaller ones (a small
--batch, or the tiny workload) write a buffer of twice the L2 size before
every step and time each step alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention: KV-read GB/s and % of GB300 HBM peak; tokens/s"
# The largest single-GPU decode batch of the target list is the headline; the
# other decode batches of that list are measured in the same run (per_config).
DEFAULT_WORKLOAD = "llama3-70b"
PER_CONFIG = ("llama2-7b", "llama3-8b", "llama2-13b-int8")
PER_CONFIG_STEPS = {"llama2-7b": 3000, "llama3-8b": 3000, "llama2-13b-int8": 400}
L2_BYTES = 129 * 1024 * 1024
DEFAULT_STEPS = {"tiny": 2000, "llama2-7b": 10000, "llama3-8b": 10000, "llama2-13b-int8": 1000,
                 "llama2-13b-int4": 2000,
                 "llama2-13b-int4-g32": 2000,
                 "llama3-70b": 300, "llama3-70b-int8-g32": 200, "llama3-70b-int4-g32": 300}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: workload default)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the batch (small profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="append one-token steps with a separate kvq_append launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other target decode batches (measured after the headline at N=1)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU-baseline sample time")
    ap.add_argument("--prefill", action="store_true",
                    help="time a chunked-prefill step (append of the chunk + causal attention of its queries)")
    ap.add_argument("--chunk", type=int, default=0, help="prefill chunk per sequence (0: the workload's, else 2048)")
    return ap.parse_args()


# ------------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms: float, local_units: float, world: int, group=None):
    """Whole-job numbers: the slowest rank's time and the units of all ranks."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples: $KVQ_CLOCKS_DIR if set, else the system temporary directory
        self.path = os.path.join(os.environ.get("KVQ_CLOCKS_DIR") or tempfile.gettempdir(),
                                 f"kvq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers --

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_tensor_peak(sustained: bool = False):
    """Dense bf16 TFLOP/s (the fp16 tensor rate is the same): the measured burst
    figure for a kernel timed alone, the measured sustained one (seconds of
    back-to-back GEMMs under the power cap) for a kernel timed inside a long
    step; else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        if sustained and "bf16_tflops_sustained" in p:
            return float(p["bf16_tflops_sustained"]), "measured sustained"
        return float(p["bf16_tflops"]), "measured burst"
    except Exception:
        return (1700.0, "fallback sustained") if sustained else (1900.0, "fallback burst")


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty lines
    (string and character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        ch = src[i]
        if ch in "\"'":
            j = i + 1
            while j < n and src[j] != ch:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """Hash of the decode kernel's sources with comments and blank lines
    removed: a change to the code (not to its comments) invalidates the
    recorded traffic."""
    h = hashlib.sha256()
    for name in ("kvq_decode.cu", "kvq_device.cuh", "kvq_launch.h"):
        with open(os.path.join(ROOT, "fp8_int8_quantized_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
            h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes of the decode split kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        for line in open(path):
            line = line.split("#", 1)[0].split()
            if len(line) >= 3 and line[0] == workload and line[1] == kernel_source_hash():
                return float(line[2])
    except OSError:
        pass
    return None


class Setup:
    """A workload's resident cache plus the step's inputs, all on the device."""

    def __init__(self, wl, device, partition, unfused=False):
        import torch

        import fp8_int8_quantized_gb300 as kvq
        from fp8_int8_quantized_gb300 import workloads as W
        self.wl, self.device = wl, device
        self.lay = W.Layout(wl)
        ctx_max = self.lay.max_context_len
        step_tok = wl.append_chunk if wl.append_chunk else 1
        self.cache = kvq.KVCache(self.lay.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.fmt, device,
                                 group_size=wl.quant_group)
        windows = W.chunk_positions(wl, 1 << 19)
        k0, v0 = W.kv_tokens(wl, *windows[0], device=device)
        sv = W.calibration_scale(wl, k0, v0)
        del k0, v0
        self.scale_value = sv
        self.scale = None if sv is None else torch.tensor([sv], dtype=torch.float32, device=device)
        # every position before the step's own tokens, untimed
        cl = self.lay.context_lens
        for p0, p1 in windows:
            k, v = W.kv_tokens(wl, p0, p1, device)
            slots = self.lay.slots(p0, p1)
            pos = torch.arange(p0, p1).repeat(wl.batch)
            keep = pos < (cl.repeat_interleave(p1 - p0) - step_tok)
            slots = torch.where(keep, slots, torch.full_like(slots, -1)).to(device)
            kvq.append(k, v, self.cache, slots, self.scale)
            del k, v
        # the step's tokens: positions [ctx - step_tok, ctx) of every sequence
        ks, vs, ss = [], [], []
        for b in range(wl.batch):
            n = int(cl[b])
            p0 = max(0, n - step_tok)
            k, v = W.kv_tokens(wl, p0, n, device, seqs=[b]) if n > 0 else (None, None)
            if k is not None:
                ks.append(k)
                vs.append(v)
                ss.append(self.lay.slots(p0, n, seqs=[b]))
        self.k_step = torch.cat(ks)
        self.v_step = torch.cat(vs)
        self.slots_step = torch.cat(ss).to(device)
        self.q = W.query(wl, device)
        self.bt = self.lay.block_tables.to(device)
        self.cl = cl.to(device)
        self.out = torch.empty_like(self.q)
        self.partition = partition
        need = kvq.workspace_size(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, ctx_max, partition)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.num_parts = 1 if need == 0 else None
        self.dec_bytes = W.decode_bytes(wl, cl)
        self.app_bytes = W.append_bytes(wl, self.slots_step.numel())
        # one new token per sequence: the decode launch appends it (unless --unfused)
        self.fused = (not unfused and step_tok == 1 and self.slots_step.numel() == wl.batch
                      and bool((cl >= 1).all()))
        if self.fused:
            self.k_step = self.k_step.view(wl.batch, wl.num_kv_heads, wl.head_dim)
            self.v_step = self.v_step.view(wl.batch, wl.num_kv_heads, wl.head_dim)
        torch.cuda.synchronize()

    def append(self):
        import fp8_int8_quantized_gb300 as kvq
        kvq.append(self.k_step, self.v_step, self.cache, self.slots_step, self.scale)

    def decode(self):
        import fp8_int8_quantized_gb300 as kvq
        kvq.decode_attention(self.q, self.cache, self.bt, self.cl, self.lay.max_context_len, self.scale,
                             out=self.out, workspace=self.ws, partition_size=self.partition)

    def decode_step(self, q=None, k=None, v=None, bt=None, cl=None, out=None):
        """The decode call of one step: with the step's new rows appended in the
        same launch when the step is one token per sequence (fused), else the
        plain decode (the append is a separate call)."""
        import fp8_int8_quantized_gb300 as kvq
        q = self.q if q is None else q
        bt = self.bt if bt is None else bt
        cl = self.cl if cl is None else cl
        out = self.out if out is None else out
        if self.fused:
            k = self.k_step if k is None else k
            v = self.v_step if v is None else v
            kvq.decode_attention_append(q, k, v, self.cache, bt, cl, self.lay.max_context_len, self.scale,
                                        out=out, workspace=self.ws, partition_size=self.partition)
        else:
            kvq.decode_attention(q, self.cache, bt, cl, self.lay.max_context_len, self.scale, out=out,
                                 workspace=self.ws, partition_size=self.partition)

    def step(self):
        if not self.fused:
            self.append()
        self.decode_step()


# ---------------------------------------------------------------- kvq arm --

def cpu_baseline(wl, target_s: float, scale_value):
    """The oracle, as it stands, on a bounded sample of the same workload: the
    decode of a few whole sequences (all their q-heads, full context) plus the
    append of their step tokens, on a cache the oracle itself filled (untimed)
    with the GPU arm's per-tensor scale.  The sample size is chosen so that the
    untimed fill and the timed work together take about ``target_s``."""
    import numpy as np
    import torch

    import oracle
    from fp8_int8_quantized_gb300 import workloads as W
    lay = W.Layout(wl)
    fmt = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2, "int8": oracle.INT8,
           "int4": oracle.INT4}[wl.fmt]
    order = list(range(wl.batch))

    def run(seqs):
        bs = wl.block_size
        nblk = [(int(lay.context_lens[b]) + bs - 1) // bs for b in seqs]
        cache = oracle.Cache(sum(nblk), wl.num_kv_heads, bs, wl.head_dim, fmt, group=wl.quant_group)
        bt = np.zeros((len(seqs), max(nblk)), np.int32)
        at = 0
        for i, n in enumerate(nblk):
            bt[i, :n] = np.arange(at, at + n)
            at += n
        cl = lay.context_lens[seqs].numpy().astype(np.int32)
        t_fill = time.perf_counter()
        # fill (untimed): the oracle's own append of every position
        for i, b in enumerate(seqs):
            n = int(cl[i])
            k, v = W.kv_tokens(wl, 0, n, "cpu", seqs=[b])
            pos = np.arange(n)
            slots = (bt[i][pos // bs].astype(np.int64) * bs + pos % bs)
            oracle.append(k.numpy(), v.numpy(), slots, cache, scale_value)
        q = W.query(wl, "cpu")[seqs].numpy()
        step_tok = wl.append_chunk if wl.append_chunk else 1
        ks, vs, ss = [], [], []
        for i, b in enumerate(seqs):
            n = int(cl[i])
            p0 = max(0, n - step_tok)
            k, v = W.kv_tokens(wl, p0, n, "cpu", seqs=[b])
            pos = np.arange(p0, n)
            ks.append(k.numpy())
            vs.append(v.numpy())
            ss.append(bt[i][pos // bs].astype(np.int64) * bs + pos % bs)
        k, v, s = np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)
        t_fill = time.perf_counter() - t_fill
        t0 = time.perf_counter()
        oracle.append(k, v, s, cache, scale_value)
        oracle.decode_attention(q, cache, bt, cl, scale_value)
        dt = time.perf_counter() - t0
        return dt, t_fill, W.decode_bytes(wl, torch.from_numpy(cl))

    dt, fill, by = run(order[:1])
    n = max(1, min(wl.batch, int(target_s / max(dt + fill, 1e-3))))
    if n > 1:
        dt, fill, by = run(order[:n])
    return {"value": by["total"] / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {wl.batch} sequences (all {wl.num_q_heads} q-heads, full context, "
                      f"{by['tokens']} cached tokens) decoded plus their step tokens appended, "
                      f"{dt:.2f} s timed (cache filled by the oracle beforehand, {fill:.1f} s untimed), "
                      f"per-tensor scale {scale_value if scale_value is not None else 'none (1.0 / row scales)'}"}


def e2e_latency(S, K, flush):
    """End-to-end steps for inputs smaller than L2, one at a time: before each
    step an untimed write of ``flush`` (twice the L2 size) evicts the cache from
    L2; the step -- the packed pinned upload, append and decode, the download of
    the output to pinned memory -- runs on one stream between two events.
    Returns (ms per step, H2D bytes per step, D2H bytes per step, steps)."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    parts = [S.q, S.k_step, S.v_step, S.slots_step, S.bt, S.cl]
    offs, at = [], 0
    for t in parts:
        offs.append(at)
        at += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(at, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.reshape(-1).view(torch.uint8).cpu())
    d_in = torch.empty(at, dtype=torch.uint8, device=S.q.device)
    q, k, v, slots, bt, cl = [d_in[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                              for t, o in zip(parts, offs)]
    out = torch.empty_like(S.q)
    h_out = torch.empty(S.q.shape, dtype=S.q.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    Ke = max(3, min(K, 2000))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke + 3)]
    for i, (a, b) in enumerate(ev):
        flush.fill_(i)
        a.record(stream)
        d_in.copy_(h_in, non_blocking=True)
        if slots.numel() and not S.fused:
            kvq.append(k, v, S.cache, slots, S.scale)
        S.decode_step(q, k, v, bt, cl, out)
        h_out.copy_(out, non_blocking=True)
        b.record(stream)
    torch.cuda.synchronize()
    if not torch.equal(h_out.to(S.out.device), S.out):
        raise RuntimeError("end-to-end output differs from the device-resident step's")
    ms = sum(a.elapsed_time(b) for a, b in ev[3:]) / Ke
    return ms, at, h_out.numel() * h_out.element_size(), Ke


def e2e_pipeline(S, K):
    """End-to-end steps as a serving loop issues them, through the public API.

    Every step uploads its own inputs -- queries, the new K/V rows, their
    slots, the block tables and the context lengths -- from pinned host memory
    as one packed buffer on an upload stream; the compute stream waits for that
    upload, appends and decodes; a download stream copies the step's output
    back to pinned host memory.  Two device input/output sets alternate, so
    step i+1's upload overlaps step i's kernels and step i's download overlaps
    step i+1's.  Times min(K, 2000) steps (3 untimed first) between two events
    on the compute stream, the last one after the final download.  Returns
    (ms per step, H2D bytes per step, D2H bytes per step, steps)."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    parts = [S.q, S.k_step, S.v_step, S.slots_step, S.bt, S.cl]
    offs, at = [], 0
    for t in parts:
        offs.append(at)
        at += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(at, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.reshape(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(at, dtype=torch.uint8, device=S.q.device) for _ in range(2)]

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]

    sets = [views(b) for b in d_in]
    outs = [torch.empty_like(S.q) for _ in range(2)]
    h_out = [torch.empty(S.q.shape, dtype=S.q.dtype).pin_memory() for _ in range(2)]
    cs, us, ds = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    torch.cuda.synchronize()

    def step(i):
        j = i & 1
        q, k, v, slots, bt, cl = sets[j]
        if used[j]:
            us.wait_event(consumed[j])  # step i-2 has finished reading set j
            cs.wait_event(read[j])      # ... and its output has been read back
        with torch.cuda.stream(us):
            d_in[j].copy_(h_in, non_blocking=True)
            uploaded[j].record(us)
        cs.wait_event(uploaded[j])
        with torch.cuda.stream(cs):
            if slots.numel() and not S.fused:
                kvq.append(k, v, S.cache, slots, S.scale)
            S.decode_step(q, k, v, bt, cl, outs[j])
            consumed[j].record(cs)
        ds.wait_event(consumed[j])
        with torch.cuda.stream(ds):
            h_out[j].copy_(outs[j], non_blocking=True)
            read[j].record(ds)
        used[j] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    Ke = max(3, min(K, 2000))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cs)
    for i in range(Ke):
        step(3 + i)
    cs.wait_stream(ds)
    b.record(cs)
    b.synchronize()
    if not torch.equal(h_out[(3 + Ke - 1) & 1].to(S.out.device), S.out):
        raise RuntimeError("end-to-end output differs from the device-resident step's")
    return a.elapsed_time(b) / Ke, at, h_out[0].numel() * h_out[0].element_size(), Ke


def time_steps(S, K, stream, flush, gpu_index):
    """K decode steps of a resident workload.

    The timed region is exactly K steps with events only at its two ends (or,
    when the step's inputs fit in L2, each step timed alone after an L2 flush).
    A second, instrumented pass over min(K, 2000) steps times each part of the
    step: append start / decode start / decode end, and -- recorded by the
    library on the same stream -- the decode stream kernel's own start and end.
    Events between kernels serialise them, so that pass feeds only the
    per-kernel figures and the roofline, never the step value."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps_ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
                if flush is not None else None)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        if flush is None:
            start.record(stream)
            for _ in range(K):
                S.step()
            end.record(stream)
        else:
            for i, (a, b) in enumerate(steps_ev):
                flush.fill_(i)
                a.record(stream)
                S.step()
                b.record(stream)
        torch.cuda.synchronize()
    Ki = min(K, 2000)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(Ki)]
    for e in ev:  # materialise the event handles
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(Ki):
        e = ev[i]
        if flush is not None:
            flush.fill_(i)
        e[0].record(stream)
        if not S.fused:
            S.append()
        e[1].record(stream)
        kvq.set_decode_timing_events(e[3], e[4])
        S.decode_step()
        e[2].record(stream)
    torch.cuda.synchronize()
    kvq.set_decode_timing_events()
    total_ms = (start.elapsed_time(end) if flush is None else sum(a.elapsed_time(b) for a, b in steps_ev))
    return {"ms_step": total_ms / K, "instrumented": Ki,
            "app_ms": sum(e[0].elapsed_time(e[1]) for e in ev) / Ki,
            "dec_ms": sum(e[1].elapsed_time(e[2]) for e in ev) / Ki,
            "kern_ms": sum(e[3].elapsed_time(e[4]) for e in ev) / Ki,
            "clocks": clk.summary()}


def bulk_append_gbs(S, stream, reps=5):
    """Quantize-on-write throughput of the workload's format on a bulk append:
    kvq_append of the rows of the first fill window again (the same values
    into the same slots, so the cache is unchanged), CUDA events around each of
    ``reps`` calls.  Returns (GB/s, rows per call, ms per call)."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    from fp8_int8_quantized_gb300 import workloads as W
    wl = S.wl
    p0, p1 = W.chunk_positions(wl, 1 << 19)[0]
    k, v = W.kv_tokens(wl, p0, p1, S.device)
    slots = S.lay.slots(p0, p1).to(S.device)
    cl = S.lay.context_lens.to(S.device)
    step_tok = wl.append_chunk if wl.append_chunk else 1
    pos = torch.arange(p0, p1, device=S.device).repeat(wl.batch)
    keep = pos < (cl.repeat_interleave(p1 - p0) - step_tok)  # the rows the fill wrote
    k, v, slots = k[keep].contiguous(), v[keep].contiguous(), slots[keep].contiguous()
    kvq.append(k, v, S.cache, slots, S.scale)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        kvq.append(k, v, S.cache, slots, S.scale)
        b.record(stream)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / reps
    return W.append_bytes(wl, slots.numel()) / (ms * 1e-3) / 1e9, slots.numel(), ms


def per_config_entry(name, dev, args, local, peak):
    """One target decode batch measured in the headline's run: step GB/s, the
    decode stream kernel's GB/s and roofline fractions, the bulk append rate,
    tokens/s and the clocks seen during its timed region."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    from fp8_int8_quantized_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    S = Setup(wl, dev, 0, args.unfused)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        S.step()
    torch.cuda.synchronize()
    st, detail = kvq.device_error_check()
    if st != 0:
        raise RuntimeError(f"{name}: device error {st} ({detail})")
    K = PER_CONFIG_STEPS.get(name, 200)
    flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
             if S.dec_bytes["total"] <= L2_BYTES else None)
    r = time_steps(S, K, stream, flush, local)
    kern_bytes = S.dec_bytes["total"] + (S.app_bytes if S.fused else 0)
    achieved = kern_bytes / (r["kern_ms"] * 1e-3) / 1e9
    app_gbs, app_rows, app_ms = bulk_append_gbs(S, stream)
    out = {"workload": name, "description": wl.description, "steps": K, "warmup": max(3, args.warmup),
           "decode_bytes": S.dec_bytes["total"],
           "ms_per_step": round(r["ms_step"], 5),
           "value": round(S.dec_bytes["total"] / (r["ms_step"] * 1e-3) / 1e9, 2), "unit": "GB/s",
           "tokens_per_s": round(wl.batch / (r["ms_step"] * 1e-3), 1),
           "step": f"append {S.slots_step.numel()} tokens + decode {wl.batch} sequences"
                   + (" (the append fused into the decode launch)" if S.fused else ""),
           "decode_kernel_ms": round(r["kern_ms"], 5),
           "decode_kernel_gbs": round(achieved, 1),
           "frac": round(achieved / peak, 4), "frac_of_nominal_8TBps": round(achieved / 8000.0, 4),
           "traffic": recorded_traffic(name),
           "append_gbs": round(app_gbs, 2),
           "append": f"kvq_append of {app_rows} (token, all kv-heads) rows of the workload's first fill "
                     f"window, {app_ms:.4f} ms per call",
           "clocks": r["clocks"]}
    del S
    torch.cuda.empty_cache()
    return out


def run_kvq(args):
    import torch

    import fp8_int8_quantized_gb300 as kvq
    from fp8_int8_quantized_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.lib()
    kvq.set_decode_kernel({"auto": 0, "simt": 1, "mma": 2}[args.kernel])
    wl = W.WORKLOADS[args.workload]
    if args.batch:
        import dataclasses
        wl = dataclasses.replace(wl, batch=args.batch)
    K = args.steps or DEFAULT_STEPS.get(wl.name, 100)
    Wm = max(3, args.warmup)
    S = Setup(wl, dev, args.partition, args.unfused)
    stream = torch.cuda.current_stream()

    for _ in range(Wm):
        S.step()
    torch.cuda.synchronize()
    st, detail = kvq.device_error_check()
    if st != 0:
        raise RuntimeError(f"device error {st} ({detail})")

    # Inputs that fit in L2 (small batches) would be read from L2 by every step
    # after the first: such runs write a buffer of twice the L2 size before
    # each step and time each step alone between two events.
    flush = None
    if S.dec_bytes["total"] <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    if world > 1:
        torch.distributed.barrier()
    r = time_steps(S, K, stream, flush, local)
    if world > 1:
        torch.distributed.barrier()
    Ki, app_ms, dec_ms, kern_ms = r["instrumented"], r["app_ms"], r["dec_ms"], r["kern_ms"]
    ms_step = r["ms_step"]
    max_ms, units = aggregate(ms_step, float(S.dec_bytes["total"]), world)
    _, seqs = aggregate(ms_step, float(wl.batch), world)
    value = units / (max_ms * 1e-3) / 1e9
    launches_per_step = (1 if S.slots_step.numel() and not S.fused else 0) + 2  # [append], stream, reduce

    # end to end through the public API: pinned host inputs in, result out
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h, Ke = e2e_pipeline(S, K) if flush is None else e2e_latency(S, K, flush)
        e_max, e_units = aggregate(e_ms, float(S.dec_bytes["total"]), world)
        e2e = {"value": round(e_units / (e_max * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e_max, 4), "steps": Ke,
               "pipeline": ("one packed pinned upload per step on a copy stream, double-buffered device "
                            "inputs and outputs, output read back to pinned memory every step"
                            if flush is None else
                            "one step at a time after an L2 flush: packed pinned upload, kernels and the "
                            "output's read back to pinned memory on one stream between two events")}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    # the stream kernel's algorithmic bytes (with the new rows when it appends them)
    kern_bytes = S.dec_bytes["total"] + (S.app_bytes if S.fused else 0)
    achieved = kern_bytes / (kern_ms * 1e-3) / 1e9
    # the recorded figures are for the workload's own batch
    traffic = recorded_traffic(wl.name) if wl.batch == W.WORKLOADS[wl.name].batch else None
    scale_value = S.scale_value
    step_desc = (f"append {S.slots_step.numel()} tokens + decode {wl.batch} sequences"
                 + (" (the append fused into the decode launch)" if S.fused else ""))
    in_l2 = flush is not None
    # the step's own append (the 70B workload's 2048-token chunks), when it is
    # a separate kvq_append launch
    append_gbs = round(S.app_bytes / (app_ms * 1e-3) / 1e9, 2) if app_ms > 0 and not S.fused else None
    del S
    torch.cuda.empty_cache()
    # the other target decode batches, each in its own timed region (N=1 only)
    per_config = None
    if (world == 1 and not args.no_per_config and args.workload == DEFAULT_WORKLOAD and not args.batch
            and not args.partition):
        per_config = {n: per_config_entry(n, dev, args, local, peak) for n in PER_CONFIG}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, args.cpu_seconds, scale_value)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(max_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"e4m3": "fp8-e4m3 storage, f16xf16->f32 compute", "e5m2": "fp8-e5m2 storage, f16xf16->f32 compute",
                  "int8": "int8 storage, f16xf16->f32 compute",
                  "int4": "int4 storage (two codes per byte), f16xf16->f32 compute"}[wl.fmt]
                 + (f", one scale per {wl.quant_group} channels" if wl.quant_group else ""),
        "data": "synthetic (seeded N(0,1) fp16 K/V/Q, shuffled block tables)",
        "config": {"workload": wl.name, "description": wl.description, "batch": wl.batch,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "format": wl.fmt,
                   "context": wl.ctx if isinstance(wl.ctx, int) else list(wl.ctx),
                   "step": step_desc,
                   "l2": (f"inputs larger than L2 ({units / world / 1e6:.0f} MB read per decode > 129 MB)"
                          if not in_l2 else
                          f"inputs smaller than L2: a {2 * L2_BYTES / 1e6:.0f} MB buffer written before every "
                          "step, each step timed alone between two events"),
                   "kernel": args.kernel, "partition": args.partition or "auto",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(seqs / (max_ms * 1e-3), 1),
        "instrumented_steps": Ki,
        "decode_ms": round(dec_ms, 5),
        "append_ms": round(app_ms, 5),
        "append_gbs": append_gbs,
        "decode_bytes": int(units / world),
        "decode_kernel_ms": round(kern_ms, 5),
        "roofline": {"bound": "hbm", "kernel": "decode_stream_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8TBps": round(achieved / 8000.0, 4), "traffic": traffic},
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": r["clocks"],
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------- prefill arm --

class PrefillSetup:
    """A workload's cache filled up to each sequence's chunk, plus the chunk:
    its K/V rows, slots and queries (on the device) -- one chunked-prefill step."""

    def __init__(self, wl, device, chunk):
        import torch

        import fp8_int8_quantized_gb300 as kvq
        from fp8_int8_quantized_gb300 import workloads as W
        self.wl = wl
        self.lay = W.Layout(wl)
        cl = self.lay.context_lens
        self.n = W.prefill_chunks(wl, cl, chunk)
        self.cache = kvq.KVCache(self.lay.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.fmt, device,
                                 group_size=wl.quant_group)
        windows = W.chunk_positions(wl, 1 << 19)
        k0, v0 = W.kv_tokens(wl, *windows[0], device=device)
        sv = W.calibration_scale(wl, k0, v0)
        del k0, v0
        self.scale_value = sv
        self.scale = None if sv is None else torch.tensor([sv], dtype=torch.float32, device=device)
        first = (cl - self.n).to(torch.int64)           # the chunk's first position per sequence
        for p0, p1 in windows:                           # every earlier position, untimed
            k, v = W.kv_tokens(wl, p0, p1, device)
            slots = self.lay.slots(p0, p1)
            pos = torch.arange(p0, p1).repeat(wl.batch)
            keep = pos < first.repeat_interleave(p1 - p0)
            kvq.append(k, v, self.cache, torch.where(keep, slots, torch.full_like(slots, -1)).to(device),
                       self.scale)
            del k, v
        ks, vs, ss = [], [], []
        for b in range(wl.batch):
            c, f = int(cl[b]), int(first[b])
            if c > f:
                k, v = W.kv_tokens(wl, f, c, device, seqs=[b])
                ks.append(k)
                vs.append(v)
                ss.append(self.lay.slots(f, c, seqs=[b]))
        self.k_step, self.v_step = torch.cat(ks), torch.cat(vs)
        self.slots = torch.cat(ss).to(device)
        self.q, qs = W.prefill_queries(wl, self.n, device)
        self.qs = qs.to(device)
        self.max_n = int(self.n.max())
        self.bt = self.lay.block_tables.to(device)
        self.cl = cl.to(device)
        self.out = torch.empty_like(self.q)
        self.flops = W.prefill_flops(wl, cl, self.n)
        self.app_bytes = W.append_bytes(wl, self.slots.numel())
        torch.cuda.synchronize()

    def attend(self, q=None, out=None):
        import fp8_int8_quantized_gb300 as kvq
        kvq.prefill_attention(self.q if q is None else q, self.cache, self.bt, self.cl, self.qs, self.max_n,
                              self.scale, out=self.out if out is None else out)

    def step(self, k=None, v=None, slots=None, q=None, out=None):
        import fp8_int8_quantized_gb300 as kvq
        kvq.append(self.k_step if k is None else k, self.v_step if v is None else v, self.cache,
                   self.slots if slots is None else slots, self.scale)
        self.attend(q, out)


def prefill_cpu_baseline(wl, n_chunk: int, target_s: float):
    """The oracle, as it stands, on a bounded sample of the prefill step: the
    last m queries of sequence 0's chunk (all q-heads, causal over the cache
    the oracle itself filled) plus the append of those m tokens."""
    import numpy as np
    import torch

    import oracle
    from fp8_int8_quantized_gb300 import workloads as W
    lay = W.Layout(wl)
    fmt = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2, "int8": oracle.INT8,
           "int4": oracle.INT4}[wl.fmt]
    bs, c = wl.block_size, int(lay.context_lens[0])
    nb = (c + bs - 1) // bs
    cache = oracle.Cache(nb, wl.num_kv_heads, bs, wl.head_dim, fmt, group=wl.quant_group)
    bt = np.arange(nb, dtype=np.int32)[None]
    k, v = W.kv_tokens(wl, 0, c, "cpu", seqs=[0])
    pos = np.arange(c)
    slots = (pos // bs) * bs + pos % bs
    oracle.append(k.numpy(), v.numpy(), slots, cache, None)
    q, _ = W.prefill_queries(wl, torch.tensor([min(n_chunk, c)], dtype=torch.int32), "cpu")
    q = q.numpy()

    def run(m):
        qs = np.array([0, m], np.int32)
        t0 = time.perf_counter()
        oracle.append(k.numpy()[c - m:], v.numpy()[c - m:], slots[c - m:], cache, None)
        oracle.prefill_attention(q[-m:], cache, bt, np.array([c], np.int32), qs, None)
        dt = time.perf_counter() - t0
        one = W.Workload(wl.name, 1, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, bs, wl.fmt, c, wl.scale_rule)
        return dt, W.prefill_flops(one, torch.tensor([c]), torch.tensor([m]))

    dt, fl = run(1)
    m = max(1, min(q.shape[0], int(target_s / max(dt, 1e-3))))
    if m > 1:
        dt, fl = run(m)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the last {m} queries of sequence 0's {q.shape[0]}-query chunk (all {wl.num_q_heads} "
                      f"q-heads, context {c}) plus the append of their K/V, {dt:.2f} s"}


def run_prefill_bench(args):
    """Chunked-prefill step: kvq_append of each sequence's chunk of K/V, then
    kvq_prefill_attention of the chunk's queries over the whole cache.
    value = attention TFLOP/s of the step (4 * head_dim flops per attended
    (query, q-head, token)); the roofline is the prefill kernel's own time
    against the measured dense bf16 rate (the fp16 tensor rate)."""
    import torch

    import fp8_int8_quantized_gb300 as kvq
    from fp8_int8_quantized_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvq.lib()
    wl = W.WORKLOADS[args.workload]
    if args.batch:
        import dataclasses
        wl = dataclasses.replace(wl, batch=args.batch)
    chunk = args.chunk or wl.append_chunk or 2048
    K = args.steps or 5
    Wm = max(3, args.warmup)
    S = PrefillSetup(wl, dev, chunk)
    stream = torch.cuda.current_stream()
    for _ in range(Wm):
        S.step()
    torch.cuda.synchronize()
    st, detail = kvq.device_error_check()
    if st != 0:
        raise RuntimeError(f"device error {st} ({detail})")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(K):
            S.step()
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # instrumented pass: append and attention timed apart
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for e in ev:
        e[0].record(stream)
        kvq.append(S.k_step, S.v_step, S.cache, S.slots, S.scale)
        e[1].record(stream)
        S.attend()
        e[2].record(stream)
    torch.cuda.synchronize()
    ms_step = start.elapsed_time(end) / K
    app_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    att_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    max_ms, flops = aggregate(ms_step, float(S.flops), world)
    value = flops / (max_ms * 1e-3) / 1e12

    # end to end through the public API: the chunk's K/V, slots and queries
    # uploaded from pinned host memory every step, the output read back
    e2e = None
    if not args.no_e2e:
        parts = [S.k_step, S.v_step, S.slots, S.q]
        host = [t.cpu().pin_memory() for t in parts]
        dev_in = [torch.empty_like(t) for t in parts]
        h_out = torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory()
        Ke = max(3, min(K, 20))
        for i in range(Ke + 1):
            if i == 1:
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
            for d, h in zip(dev_in, host):
                d.copy_(h, non_blocking=True)
            S.step(*dev_in, out=S.out)
            h_out.copy_(S.out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        e_ms = a.elapsed_time(b) / Ke
        e_max, e_fl = aggregate(e_ms, float(S.flops), world)
        e2e = {"value": round(e_fl / (e_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in parts),
               "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "ms_per_step": round(e_max, 3),
               "steps": Ke}
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    # a timed region of more than a second of back-to-back prefill runs under
    # the power cap: the sustained peak is its denominator
    peak, peak_kind = measured_tensor_peak(sustained=K * att_ms > 1000.0)
    burst, _ = measured_tensor_peak()
    achieved = S.flops / (att_ms * 1e-3) / 1e12
    # tensor work executed per algorithmic flop: PV twice (fp16 hi + residual
    # weights); with group scales also S twice and PV three times
    executed = 2.5 if wl.quant_group else 1.5
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = prefill_cpu_baseline(wl, chunk, args.cpu_seconds)
    line = {
        "metric": "quantized-KV chunked-prefill attention: TFLOP/s (causal attention of each chunk over the cache)",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(max_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"e4m3": "fp8-e4m3 storage, f16xf16->f32 compute", "e5m2": "fp8-e5m2 storage, f16xf16->f32 compute",
                  "int8": "int8 storage, f16xf16->f32 compute",
                  "int4": "int4 storage (two codes per byte), f16xf16->f32 compute"}[wl.fmt]
                 + (f", one scale per {wl.quant_group} channels" if wl.quant_group else ""),
        "data": "synthetic (seeded N(0,1) fp16 K/V/Q, shuffled block tables)",
        "config": {"workload": wl.name + "-prefill", "description": wl.description, "batch": wl.batch,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "format": wl.fmt,
                   "context": wl.ctx if isinstance(wl.ctx, int) else list(wl.ctx),
                   "chunk": chunk, "queries": int(S.n.sum()),
                   "step": f"append {S.slots.numel()} tokens + causal attention of their queries over the cache",
                   "l2": "inputs larger than L2 (cache and queries)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "attention_flops_per_step": S.flops,
        "tokens_per_s": round(float(S.n.sum()) * world / (max_ms * 1e-3), 1),
        "append_ms": round(app_ms, 4),
        "append_gbs": round(S.app_bytes / (app_ms * 1e-3) / 1e9, 2),
        "prefill_kernel_ms": round(att_ms, 4),
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_burst": round(achieved / burst, 4),
                     "executed_tensor_tflops": round(executed * achieved, 1),
                     "note": "achieved counts the algorithmic QK^T and PV flops; the kernel executes PV twice "
                             "(fp16 hi + residual weights), 1.5x the algorithmic tensor work"
                             + ("; with group scales S twice and PV three times, 2.5x" if wl.quant_group else ""),
                     "traffic": None},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------- reference arm --

def run_reference(args):
    """The CPU oracle timed as the reference arm: each step decodes one whole
    sequence of the workload (all its q-heads, full context) and appends its
    step tokens, on host cores.  Ranks other than 0 exit without work."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from fp8_int8_quantized_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    lay = W.Layout(wl)
    fmt = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2, "int8": oracle.INT8,
           "int4": oracle.INT4}[wl.fmt]
    bs = wl.block_size
    step_tok = wl.append_chunk if wl.append_chunk else 1
    K = args.steps or 5
    Wm = max(3, args.warmup)
    nseq = min(wl.batch, 4)
    kv = [W.kv_tokens(wl, 0, int(lay.context_lens[b]), "cpu", seqs=[b]) for b in range(nseq)]
    # the per-tensor scale by the workloads' calibration rule (amax / format
    # max), taken over the sampled sequences' K and V
    scale = None
    if wl.scale_rule == "amax":
        scale = W.calibration_scale(wl, torch.cat([k for k, _ in kv]), torch.cat([v for _, v in kv]))
    caches = []
    for b in range(nseq):
        n = int(lay.context_lens[b])
        nb = (n + bs - 1) // bs
        cache = oracle.Cache(nb, wl.num_kv_heads, bs, wl.head_dim, fmt, group=wl.quant_group)
        bt = np.arange(nb, dtype=np.int32)[None]
        k, v = kv[b]
        pos = np.arange(n)
        oracle.append(k.numpy(), v.numpy(), (pos // bs) * bs + pos % bs, cache, scale)
        q = W.query(wl, "cpu")[b:b + 1].numpy()
        p0 = max(0, n - step_tok)
        sk, sv = k[p0:].numpy(), v[p0:].numpy()
        caches.append((cache, bt, np.array([n], np.int32), q, sk, sv, np.arange(p0, n, dtype=np.int64)))
    del kv

    def step(i):
        cache, bt, cl, q, sk, sv, slots = caches[i % nseq]
        oracle.append(sk, sv, slots, cache, scale)
        oracle.decode_attention(q, cache, bt, cl, scale)

    for i in range(Wm):
        step(i)
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    dt = (time.perf_counter() - t0) / K
    # bytes of the decode of one whole sequence: the unit of one step
    ctx_mean = sum(int(lay.context_lens[i]) for i in range(nseq)) / nseq
    one = W.Workload(wl.name, 1, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.fmt,
                     int(ctx_mean), wl.scale_rule)
    value = W.decode_bytes(one, torch.tensor([int(ctx_mean)]))["total"] / dt / 1e9
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": Wm, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": wl.name, "description": wl.description},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: one sequence of {wl.name} (all {wl.num_q_heads} q-heads, "
                                       f"context {int(lay.context_lens[0])}) decoded + {step_tok} tokens appended"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill:
        run_prefill_bench(args)
    else:
        run_kvq(args)


if __name__ == "__main__":
    main()
