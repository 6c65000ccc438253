"""Attention error of each cache format against the unquantized fp16 cache.

For one workload's shapes and value distribution (outlier channels included),
the same fp16 K/V rows go into a cache of every format through ``kvq_append``
and every sequence is decoded through ``kvq_decode_attention``; each output is
compared with attention over the fp16 K/V themselves, softmax(sm_scale q K^T) V
per sequence and q-head, computed here with plain fp32 torch operations.

What this measures is the error the cache format itself introduces -- the
accuracy question of "Accelerating Inference with FP8 KV Cache" ("FP8 E4M3 KV
Cache": with a calibrated scale or the 1.0 default) and of "[Feature] TurboMind
support W8A8 or FP8 KV Cache" (online INT8, and INT4), and of group quantization
for a 4-bit cache ("[QST] Scale factors and benchmarks", the QQQ page) -- not the
kernels' rounding, which the parity tests bound far below it.

    python -m fp8_int8_quantized_gb300.quant_error [--workload NAME] [--batch B] [--json]
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math

import torch

import fp8_int8_quantized_gb300 as kvq
from fp8_int8_quantized_gb300 import workloads as W

# (format, scale rule): E4M3 / E5M2 with the amax/max calibration scale or
# the 1.0 default, INT8 and INT4 with their own scale per (token, kv-head) row
# "gN": INT8 / INT4 with one scale per group of N channels of a row
VARIANTS = [("e4m3", "amax"), ("e4m3", "one"), ("e5m2", "amax"), ("e5m2", "one"), ("int8", "row"),
            ("int4", "row"), ("int8", "g32"), ("int4", "g32"), ("int4", "g64")]


def variant(base: W.Workload, fmt: str, rule: str) -> W.Workload | None:
    """The workload of one variant (None where it does not apply)."""
    if rule.startswith("g"):
        group = int(rule[1:])
        if base.head_dim % group:
            return None
        return dataclasses.replace(base, fmt=fmt, scale_rule="row", quant_group=group)
    return dataclasses.replace(base, fmt=fmt, scale_rule=rule, quant_group=0)


def supported_variants(name: str) -> list[tuple[str, str]]:
    return [v for v in VARIANTS if variant(W.WORKLOADS[name], *v) is not None]


WINDOW_TOKENS = 1 << 19  # generation windows (values depend on the window start)


def _reference(wl: W.Workload, lay: W.Layout, q: torch.Tensor, device) -> torch.Tensor:
    """fp32 attention over the unquantized fp16 K/V, [B][Hq][D]."""
    sm = 1.0 / math.sqrt(wl.head_dim)
    out = torch.zeros((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=device)
    for b in range(wl.batch):
        n = int(lay.context_lens[b])
        if n == 0:
            continue
        ks, vs = [], []
        for p0, p1 in W.chunk_positions(wl, WINDOW_TOKENS):  # the quantized path's windows: same values
            if p0 >= n:
                break
            k, v = W.kv_tokens(wl, p0, p1, device, seqs=[b])
            ks.append(k[: n - p0])
            vs.append(v[: n - p0])
        k = torch.cat(ks).float()  # [n][Hkv][D]
        v = torch.cat(vs).float()
        kh = k.permute(1, 0, 2).repeat_interleave(wl.group, 0)  # [Hq][n][D]
        vh = v.permute(1, 0, 2).repeat_interleave(wl.group, 0)
        s = torch.einsum("hd,hnd->hn", q[b].float(), kh) * sm
        p = torch.softmax(s, dim=-1)
        out[b] = torch.einsum("hn,hnd->hd", p, vh)
    return out


def _quantized(wl: W.Workload, lay: W.Layout, q: torch.Tensor, device):
    """Output of the quantized path and the per-tensor scale it used."""
    cache = kvq.KVCache(lay.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.fmt, device,
                        group_size=wl.quant_group)
    windows = W.chunk_positions(wl, WINDOW_TOKENS)
    k0, v0 = W.kv_tokens(wl, *windows[0], device=device)
    sv = W.calibration_scale(wl, k0, v0)
    scale = None if sv is None else torch.tensor([sv], dtype=torch.float32, device=device)
    for p0, p1 in windows:
        k, v = W.kv_tokens(wl, p0, p1, device)
        kvq.append(k, v, cache, lay.slots(p0, p1).to(device), scale)
    out = kvq.decode_attention(q, cache, lay.block_tables.to(device), lay.context_lens.to(device),
                               lay.max_context_len, scale)
    return out.float(), sv


def report(name: str = "llama3-8b", batch: int = 8, device="cuda") -> list[dict]:
    """One row per format variant: relative RMS and max-abs error of the decode
    output against the fp16-cache attention, and the smallest cosine
    similarity over (sequence, q-head)."""
    base = W.WORKLOADS[name]
    base = dataclasses.replace(base, batch=min(batch, base.batch))
    lay = W.Layout(base)
    q = W.query(base, device)
    ref = _reference(base, lay, q, device)
    rows = []
    for fmt, rule in VARIANTS:
        wl = variant(base, fmt, rule)
        if wl is None:
            continue
        out, sv = _quantized(wl, lay, q, device)
        d = out - ref
        cos = torch.nn.functional.cosine_similarity(out.flatten(0, 1), ref.flatten(0, 1), dim=-1)
        rows.append({"workload": name, "batch": base.batch, "format": fmt, "scale": rule,
                     "scale_value": sv, "rel_rms": float(d.pow(2).mean().sqrt() / ref.pow(2).mean().sqrt()),
                     "max_abs": float(d.abs().max()), "ref_max_abs": float(ref.abs().max()),
                     "min_cos": float(cos.min())})
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3-8b")
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--json", action="store_true")
    args = ap.parse_args()
    kvq.lib()
    rows = report(args.workload, args.batch)
    if args.json:
        for r in rows:
            print(json.dumps(r))
        return
    print(f"| format | scale | rel. RMS error | max abs error (max abs output {rows[0]['ref_max_abs']:.3g}) "
          f"| min cosine |")
    print("|---|---|---|---|---|")
    for r in rows:
        sc = r["scale"] if r["scale_value"] is None else f"{r['scale']} ({r['scale_value']:.4g})"
        print(f"| {r['format']} | {sc} | {r['rel_rms']:.3e} | {r['max_abs']:.3e} | {r['min_cos']:.6f} |")


if __name__ == "__main__":
    main()
