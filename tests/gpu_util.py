"""Helpers shared by the GPU parity tests: build a workload's paged cache on the
device through kvq_append, copy sampled sequences' blocks to the host as an
oracle cache, and compare decode outputs with the tolerance the tests use."""
from __future__ import annotations

import numpy as np
import torch

import fp8_int8_quantized_gb300 as kvq
import oracle
from fp8_int8_quantized_gb300 import workloads as W

ORACLE_FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2, "int8": oracle.INT8, "int4": oracle.INT4}

# Attention tolerance: |o_gpu - o_ref| <= 2e-3 * max(1, |o_ref|) per element,
# o_ref the fp64 oracle on the same dequantized cache.  fp16 output rounding
# alone costs up to 2^-11 relative (4.9e-4); P rounded to fp16 for PV costs about
# 2^-12 relative per weight; the rest is fp32 accumulation order.
ATOL_REL = 2e-3


def rel_err(out_gpu: np.ndarray, ref: np.ndarray) -> float:
    if out_gpu.size == 0:
        return 0.0
    return float((np.abs(out_gpu.astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref))).max())


class DeviceWorkload:
    """A workload's cache filled on the GPU with kvq_append, chunk by chunk."""

    def __init__(self, wl: W.Workload, fill_to: int | None = None, chunk_tokens: int = 1 << 19,
                 device="cuda", ctx: torch.Tensor | None = None, sentinel: int | None = 0xA5):
        self.wl, self.device = wl, device
        self.lay = W.Layout(wl, ctx)
        self.cache = kvq.KVCache(self.lay.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.fmt,
                                 device, fill=sentinel, group_size=wl.quant_group)
        self.windows = W.chunk_positions(wl, chunk_tokens)
        k0, v0 = W.kv_tokens(wl, *self.windows[0], device=device)
        self.scale_value = W.calibration_scale(wl, k0, v0)
        self.scale = (None if self.scale_value is None else
                      torch.tensor([self.scale_value], dtype=torch.float32, device=device))
        del k0, v0
        limit = self.lay.max_context_len if fill_to is None else fill_to
        for p0, p1 in self.windows:
            if p0 >= limit:
                break
            p1 = min(p1, limit)
            self.append_window(p0, p1)
        torch.cuda.synchronize()
        self.q = W.query(wl, device)
        self.block_tables = self.lay.block_tables.to(device)
        self.context_lens = self.lay.context_lens.to(device)

    def window_of(self, pos: int):
        for p0, p1 in self.windows:
            if p0 <= pos < p1:
                return p0, p1
        raise ValueError(pos)

    def append_window(self, p0, p1, seqs=None):
        k, v = W.kv_tokens(self.wl, p0, p1, self.device, seqs)
        slots = self.lay.slots(p0, p1, seqs).to(self.device)
        kvq.append(k, v, self.cache, slots, self.scale)
        return k, v, slots

    def decode(self, partition_size=0, out=None):
        return kvq.decode_attention(self.q, self.cache, self.block_tables, self.context_lens,
                                    self.lay.max_context_len, self.scale, out=out,
                                    partition_size=partition_size)

    def oracle_cache_for(self, seqs):
        """Host oracle cache holding only the blocks of ``seqs`` (renumbered), plus
        the matching block tables and lengths."""
        wl, lay = self.wl, self.lay
        bs = wl.block_size
        blocks, tables = [], []
        for b in seqs:
            n = (int(lay.context_lens[b]) + bs - 1) // bs
            ids = lay.block_tables[b, :n].to(torch.int64)
            tables.append(list(range(len(blocks), len(blocks) + n)))
            blocks.extend(ids.tolist())
        idx = torch.tensor(blocks, dtype=torch.int64, device=self.device)
        kc = self.cache.k_codes.index_select(0, idx).cpu().numpy()
        vc = self.cache.v_codes.index_select(0, idx).cpu().numpy()
        ks = vs = None
        if wl.fmt in ("int8", "int4"):
            ks = self.cache.k_scales.index_select(0, idx).cpu().numpy()
            vs = self.cache.v_scales.index_select(0, idx).cpu().numpy()
        oc = oracle.Cache(len(blocks), wl.num_kv_heads, bs, wl.head_dim, ORACLE_FMT[wl.fmt],
                          k_codes=np.ascontiguousarray(kc), v_codes=np.ascontiguousarray(vc),
                          k_scales=ks, v_scales=vs, group=wl.quant_group)
        mb = max(1, max(len(t) for t in tables))
        bt = np.zeros((len(seqs), mb), np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        cl = lay.context_lens[list(seqs)].numpy().astype(np.int32)
        return oc, bt, cl

    def oracle_decode(self, seqs):
        oc, bt, cl = self.oracle_cache_for(seqs)
        q = self.q[list(seqs)].cpu().numpy()
        return oracle.decode_attention(q, oc, bt, cl, self.scale_value)
