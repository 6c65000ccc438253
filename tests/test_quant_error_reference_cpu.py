"""Pin of the quantization-error report's yardstick: ``quant_error._reference``
(plain fp32 attention over the unquantized fp16 K/V) against fp64
``scaled_dot_product_attention`` on the same rows, reached by another route.

The independent side follows the data path the quantized arm of the report
uses: every generation window's K/V rows of every sequence are scattered by the
layout's slot mapping into a dense fp16 paged store ([slot][kv-head][head_dim]),
and each sequence's rows are gathered back through its block table, position
by position; q-head h reads kv-head h // (Hq / Hkv) (the contiguous GQA groups
of the "which kv-head" reading), softmax scale 1/sqrt(head_dim).  The windows
are made small so that contexts cross several of them.  A planted head-mapping
or window mistake in the reference moves its output far outside the bound
(checked below on the independent side), so the pin would catch either.
"""
import math

import numpy as np
import pytest
import torch

from fp8_int8_quantized_gb300 import quant_error
from fp8_int8_quantized_gb300 import workloads as W

TOL = 1e-5   # fp32 softmax and sums against fp64: a few fp32 ulps of the logits


def paged_store(wl, lay, window):
    """fp16 [num_blocks * block_size][Hkv][D]: every window's rows at their slots."""
    store = torch.full((lay.num_blocks * wl.block_size, wl.num_kv_heads, wl.head_dim), float("nan"),
                       dtype=torch.float16)
    vstore = store.clone()
    for p0, p1 in W.chunk_positions(wl, window):
        k, v = W.kv_tokens(wl, p0, p1, "cpu")
        slots = lay.slots(p0, p1)
        keep = slots >= 0
        store[slots[keep]] = k[keep]
        vstore[slots[keep]] = v[keep]
    return store, vstore


def sdpa_fp64(wl, lay, q, kstore, vstore, head_map=None, shift=0):
    """fp64 attention per sequence over rows gathered through the block table.
    head_map / shift plant mistakes (a wrong q-head -> kv-head map, positions
    read one window slot off) for the sensitivity checks."""
    G = wl.num_q_heads // wl.num_kv_heads
    hm = head_map or (lambda h: h // G)
    out = torch.zeros((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float64)
    bs = wl.block_size
    for b in range(wl.batch):
        n = int(lay.context_lens[b])
        if n == 0:
            continue
        pos = torch.clamp(torch.arange(n) + shift, 0, n - 1)
        slot = lay.block_tables[b].to(torch.int64)[pos // bs] * bs + pos % bs
        k = kstore[slot].double()           # [n][Hkv][D]
        v = vstore[slot].double()
        idx = torch.tensor([hm(h) for h in range(wl.num_q_heads)])
        kh = k[:, idx].permute(1, 0, 2)     # [Hq][n][D]
        vh = v[:, idx].permute(1, 0, 2)
        qh = q[b].double()[:, None, :]      # [Hq][1][D]
        out[b] = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, scale=1.0 / math.sqrt(wl.head_dim))[:, 0]
    return out


@pytest.mark.parametrize("outliers", [False, True])
def test_reference_matches_fp64_sdpa_over_paged_rows(monkeypatch, outliers):
    window = 3 * 32                    # windows of 32 positions for a batch of 3
    monkeypatch.setattr(quant_error, "WINDOW_TOKENS", window)
    wl = W.Workload("qe-pin", 3, 6, 2, 64, 16, "e4m3", 200, "amax", outliers=outliers, seed=11)
    lay = W.Layout(wl, torch.tensor([200, 77, 0], dtype=torch.int32))
    assert len(W.chunk_positions(wl, window)) > 4       # contexts cross several windows
    q = W.query(wl, "cpu")
    ref = quant_error._reference(wl, lay, q, "cpu")
    ks, vs = paged_store(wl, lay, window)
    exp = sdpa_fp64(wl, lay, q, ks, vs)
    err = ((ref.double() - exp).abs() / exp.abs().clamp(min=1.0)).max().item()
    assert err <= TOL, err
    assert not ref[2].any()                              # context 0: zeros
    # the case separates the plausible mistakes by far more than the bound
    G = wl.num_q_heads // wl.num_kv_heads
    wrong_map = sdpa_fp64(wl, lay, q, ks, vs, head_map=lambda h: h % wl.num_kv_heads)
    assert (wrong_map - exp).abs().max().item() > 1e-2
    wrong_pos = sdpa_fp64(wl, lay, q, ks, vs, shift=1)
    assert (wrong_pos - exp).abs().max().item() > 1e-2
    assert G == 3


def test_reference_single_token_is_the_v_row(monkeypatch):
    """Context 1: softmax over one token is 1, so the output is that token's
    fp16 V row exactly (closed form)."""
    monkeypatch.setattr(quant_error, "WINDOW_TOKENS", 64)
    wl = W.Workload("qe-one", 2, 4, 4, 128, 16, "e5m2", 1, "one", seed=3)
    lay = W.Layout(wl, torch.tensor([1, 1], dtype=torch.int32))
    q = W.query(wl, "cpu")
    ref = quant_error._reference(wl, lay, q, "cpu")
    _, v = W.kv_tokens(wl, 0, 1, "cpu")
    assert np.array_equal(ref.numpy(), v.float().numpy().reshape(2, 4, 128))
