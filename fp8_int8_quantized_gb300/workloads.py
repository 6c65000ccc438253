"""Seeded synthetic inputs for the quantized paged KV cache.

This module draws inputs only: fp16 K/V/Q, paged block tables, context lengths,
slot mappings and the per-tensor calibration scale that a checkpoint would
carry.  It holds none of the quantization or attention arithmetic, so both the
CUDA path and the CPU oracle can consume what it produces.

Shapes follow the decode batches of 7B-70B models (Llama-2-7B MHA, Llama-3-8B
GQA, Llama-2-13B INT8, Llama-3-70B long context).  Value recipe: K, V and Q are
N(0, 1) in fp32 rounded to fp16; where a workload has outliers, a seeded 1% of
the (kv-head, channel) pairs of K and of V are multiplied by 20 for every
token.  Block tables are a seeded random permutation of the physical blocks,
handed out to sequences in order.  The FP8 per-tensor scale for "amax" workloads
is the calibration stand-in for a checkpoint's ``kv_scale``: the largest |K| or
|V| over the first generated chunk, divided by the format's largest finite
value, in fp32.
"""
from __future__ import annotations

import dataclasses
import math

import torch

FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    fmt: str                       # "e4m3" | "e5m2" | "int8" | "int4"
    ctx: int | tuple[int, int]     # fixed length, or inclusive uniform range
    scale_rule: str                # "amax" | "one" | "row" (INT8 / INT4: per (token, kv-head))
    outliers: bool = False
    append_chunk: int = 0          # prefill chunk appended per sequence inside a step
    seed: int = 0
    description: str = ""
    quant_group: int = 0           # INT8 / INT4: channels per scale (0 = one scale per row)

    @property
    def scales_per_row(self) -> int:
        return self.head_dim // self.quant_group if self.quant_group else 1

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 4, 64, 16, "e4m3", 128, "amax", seed=0,
                     description="1 seq, 4/4 heads, head_dim 64, ctx 128, block 16, E4M3 amax/448"),
    "llama2-7b": Workload("llama2-7b", 32, 32, 32, 128, 16, "e4m3", 2048, "amax", seed=1001,
                          description="Llama-2-7B decode: MHA 32x128, batch 32, ctx 2048, "
                                      "block 16, shuffled blocks, E4M3 amax/448"),
    "llama3-8b": Workload("llama3-8b", 64, 32, 8, 128, 16, "e5m2", (512, 8192), "one",
                          outliers=True, seed=1002,
                          description="Llama-3-8B GQA decode: 32/8 heads x128, batch 64, "
                                      "ctx U[512,8192], block 16, E5M2 scale 1.0, 1% outliers x20"),
    "llama2-13b-int8": Workload("llama2-13b-int8", 128, 40, 40, 128, 64, "int8", 4096, "row",
                                seed=1003,
                                description="Llama-2-13B INT8 decode: 40x128, batch 128, ctx 4096, "
                                            "block 64, online INT8 per (token, kv-head)"),
    "llama2-13b-int4": Workload("llama2-13b-int4", 128, 40, 40, 128, 64, "int4", 4096, "row",
                                seed=1005,
                                description="Llama-2-13B INT4 shapes: 40x128, batch 128, ctx 4096, "
                                            "block 64, online INT4 per (token, kv-head)"),
    "llama2-13b-int4-g32": Workload("llama2-13b-int4-g32", 128, 40, 40, 128, 64, "int4", 4096, "row",
                                    seed=1006, quant_group=32,
                                    description="Llama-2-13B INT4 shapes with group quantization: "
                                                "40x128, batch 128, ctx 4096, block 64, online INT4 "
                                                "with one scale per 32 channels"),
    "llama3-70b-int8-g32": Workload("llama3-70b-int8-g32", 256, 64, 8, 128, 16, "int8", 32768, "row",
                                    outliers=True, seed=1007, quant_group=32,
                                    description="Llama-3-70B shapes with group-quantized INT8: 64/8 heads "
                                                "x128, batch 256, ctx 32768, block 16, online INT8 with one "
                                                "scale per 32 channels, 1% outliers x20"),
    "llama3-70b-int4-g32": Workload("llama3-70b-int4-g32", 256, 64, 8, 128, 16, "int4", 32768, "row",
                                    outliers=True, seed=1008, quant_group=32,
                                    description="Llama-3-70B shapes with group-quantized INT4: 64/8 heads "
                                                "x128, batch 256, ctx 32768, block 16, online INT4 with one "
                                                "scale per 32 channels, 1% outliers x20"),
    "llama3-70b": Workload("llama3-70b", 256, 64, 8, 128, 16, "e4m3", 32768, "amax",
                           outliers=True, append_chunk=2048, seed=1004,
                           description="Llama-3-70B long context: 64/8 heads x128, batch 256, "
                                       "ctx 32768, block 16, E4M3 amax/448, 1% outliers x20, "
                                       "append of a 2048-token prefill chunk per sequence"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def context_lens(wl: Workload) -> torch.Tensor:
    """int32 [batch] context lengths (CPU)."""
    if isinstance(wl.ctx, int):
        return torch.full((wl.batch,), wl.ctx, dtype=torch.int32)
    lo, hi = wl.ctx
    g = _gen(wl.seed + 2000, "cpu")
    return torch.randint(lo, hi + 1, (wl.batch,), generator=g, dtype=torch.int32)


class Layout:
    """Paged layout of one workload: block tables and the slot of every position."""

    def __init__(self, wl: Workload, ctx: torch.Tensor | None = None, spare_blocks: int = 0):
        self.wl = wl
        self.context_lens = context_lens(wl) if ctx is None else ctx.to(torch.int32)
        bs = wl.block_size
        nblk = [(int(c) + bs - 1) // bs for c in self.context_lens]
        self.max_context_len = int(self.context_lens.max()) if wl.batch else 0
        self.max_blocks_per_seq = max(1, (self.max_context_len + bs - 1) // bs)
        self.num_blocks = sum(nblk) + spare_blocks
        g = _gen(wl.seed + 1000, "cpu")
        perm = torch.randperm(max(self.num_blocks, 1), generator=g).to(torch.int32)
        bt = torch.zeros((wl.batch, self.max_blocks_per_seq), dtype=torch.int32)
        at = 0
        for b, n in enumerate(nblk):
            bt[b, :n] = perm[at:at + n]
            at += n
        self.block_tables = bt

    def slots(self, pos0: int, pos1: int, seqs=None) -> torch.Tensor:
        """int64 [len(seqs) * (pos1 - pos0)] slots of positions [pos0, pos1) of each
        sequence, sequence-major; positions at or past a sequence's length are -1."""
        bs = self.wl.block_size
        seqs = range(self.wl.batch) if seqs is None else seqs
        pos = torch.arange(pos0, pos1, dtype=torch.int64)
        out = []
        for b in seqs:
            n = int(self.context_lens[b])
            blk = self.block_tables[b].to(torch.int64)[torch.clamp(pos // bs, max=self.max_blocks_per_seq - 1)]
            s = blk * bs + pos % bs
            out.append(torch.where(pos < n, s, torch.full_like(s, -1)))
        return torch.cat(out) if out else torch.zeros(0, dtype=torch.int64)


def _outlier_gain(wl: Workload, which: int, device) -> torch.Tensor | None:
    """fp32 [Hkv, D] per-channel multiplier (1 or 20) for K (which=0) or V (1)."""
    if not wl.outliers:
        return None
    n = wl.num_kv_heads * wl.head_dim
    k = max(1, round(0.01 * n))
    g = _gen(wl.seed + 4000 + which, "cpu")
    idx = torch.randperm(n, generator=g)[:k]
    gain = torch.ones(n, dtype=torch.float32)
    gain[idx] = 20.0
    return gain.view(wl.num_kv_heads, wl.head_dim).to(device)


def kv_tokens(wl: Workload, pos0: int, pos1: int, device="cpu", seqs=None):
    """fp16 K, V [len(seqs) * (pos1 - pos0)][Hkv][D] for positions [pos0, pos1) of
    each sequence (sequence-major, same order as ``Layout.slots``).  The values of
    a (sequence, position) depend only on the seed, the sequence and the position
    window start, so chunks generated separately are reproducible."""
    seqs = list(range(wl.batch)) if seqs is None else list(seqs)
    n = pos1 - pos0
    shape = (n, wl.num_kv_heads, wl.head_dim)
    ks, vs = [], []
    gk, gv = _outlier_gain(wl, 0, device), _outlier_gain(wl, 1, device)
    for b in seqs:
        g = _gen(wl.seed * 1_000_003 + b * 65_537 + pos0, device)
        k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if gk is not None:
            k = k * gk
            v = v * gv
        ks.append(k.to(torch.float16))
        vs.append(v.to(torch.float16))
    if not ks:
        e = torch.zeros((0,) + shape[1:], dtype=torch.float16, device=device)
        return e, e.clone()
    return torch.cat(ks), torch.cat(vs)


def query(wl: Workload, device="cpu", step: int = 0) -> torch.Tensor:
    """fp16 Q [batch][Hq][D] ~ N(0, 1)."""
    g = _gen(wl.seed + 5000 + 7919 * step, device)
    q = torch.randn((wl.batch, wl.num_q_heads, wl.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch.float16)


def calibration_scale(wl: Workload, k: torch.Tensor, v: torch.Tensor) -> float | None:
    """Per-tensor fp32 scale handed to both sides: None (= the 1.0 default) for
    "one" and INT8, else max(|K|, |V|) over the calibration sample / format max."""
    if wl.scale_rule != "amax":
        return None
    amax = torch.maximum(k.abs().max(), v.abs().max()).to(torch.float32)
    s = amax / torch.tensor(FP8_MAX[wl.fmt], dtype=torch.float32, device=amax.device)
    return float(s.cpu())


def chunk_positions(wl: Workload, max_tokens: int):
    """Split positions [0, max_ctx) into windows so that one window across the
    whole batch holds at most ``max_tokens`` tokens."""
    lay_max = wl.ctx if isinstance(wl.ctx, int) else wl.ctx[1]
    step = max(wl.block_size, (max_tokens // max(wl.batch, 1)) // wl.block_size * wl.block_size)
    return [(p, min(p + step, lay_max)) for p in range(0, lay_max, step)]


def decode_bytes(wl: Workload, ctx: torch.Tensor) -> dict:
    """Algorithmic HBM bytes of one decode call: every cached K/V byte of every
    (sequence, kv-head) once, the INT8 / INT4 row scales, q, out, block tables and
    lengths."""
    tok = int(ctx.to(torch.int64).sum())
    kv = 2 * tok * wl.num_kv_heads * (wl.head_dim // 2 if wl.fmt == "int4" else wl.head_dim)
    scales = 2 * tok * wl.num_kv_heads * 4 * wl.scales_per_row if wl.fmt in ("int8", "int4") else 0
    qo = 2 * wl.batch * wl.num_q_heads * wl.head_dim * 2
    bt = sum(math.ceil(int(c) / wl.block_size) for c in ctx) * 4 + wl.batch * 4
    return {"kv": kv, "scales": scales, "q_out": qo, "tables": bt,
            "total": kv + scales + qo + bt, "tokens": tok}


def append_bytes(wl: Workload, num_tokens: int) -> int:
    """Algorithmic HBM bytes of appending ``num_tokens`` tokens: fp16 K+V read,
    codes written, slots read, INT8 / INT4 row scales written."""
    e = num_tokens * wl.num_kv_heads * wl.head_dim
    b = 2 * e * 2 + (e if wl.fmt == "int4" else 2 * e) + num_tokens * 8
    if wl.fmt in ("int8", "int4"):
        b += 2 * num_tokens * wl.num_kv_heads * 4 * wl.scales_per_row
    return b


def prefill_chunks(wl: Workload, ctx: torch.Tensor, chunk: int | None = None) -> torch.Tensor:
    """int32 [batch] new-query counts of a chunked-prefill step: ``chunk`` (default
    the workload's append chunk) clipped to each sequence's context."""
    n = wl.append_chunk if chunk is None else chunk
    return torch.clamp(ctx.to(torch.int32), max=n)


def prefill_queries(wl: Workload, chunk_lens: torch.Tensor, device="cpu", step: int = 0):
    """fp16 Q [sum(chunk_lens)][Hq][D] ~ N(0, 1) and int32 query_start [batch + 1]
    for chunks of ``chunk_lens`` new queries per sequence."""
    qs = torch.zeros(chunk_lens.shape[0] + 1, dtype=torch.int32)
    qs[1:] = torch.cumsum(chunk_lens.to(torch.int64), 0).to(torch.int32)
    g = _gen(wl.seed + 6000 + 7919 * step, device)
    q = torch.randn((int(qs[-1]), wl.num_q_heads, wl.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return q.to(torch.float16), qs


def prefill_flops(wl: Workload, ctx: torch.Tensor, chunk_lens: torch.Tensor) -> int:
    """Algorithmic flops of causal chunk attention: query i of an n-query chunk at
    position ctx - n + i takes 2 * 2 * head_dim flops (QK^T and PV) per attended
    token and q-head."""
    tot = 0
    for c, n in zip(ctx.tolist(), chunk_lens.tolist()):
        tot += n * (c - n) + n * (n + 1) // 2
    return 4 * wl.num_q_heads * wl.head_dim * tot
