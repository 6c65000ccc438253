"""The seeded synthetic inputs (fp8_int8_quantized_gb300/workloads.py) on CPU:
shapes and byte counts of the workloads, the paged layout (block tables are a
permutation of the cache's blocks, slots follow the tables), reproducible
generation, and the outlier channels."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from fp8_int8_quantized_gb300 import workloads as W


def test_decode_bytes_of_the_fixed_context_workloads():
    # every cached K/V byte once, scales, q and out, block-table entries and lengths
    want = {
        "llama2-7b": 536_870_912 + 2 * 262_144 + 32 * 128 * 4 + 32 * 4,
        "llama2-13b-int8": 5_368_709_120 + 167_772_160 + 2 * 1_310_720 + 128 * 64 * 4 + 128 * 4,
        "llama2-13b-int4": 2_684_354_560 + 167_772_160 + 2 * 1_310_720 + 128 * 64 * 4 + 128 * 4,
        "llama2-13b-int4-g32": 2_684_354_560 + 4 * 167_772_160 + 2 * 1_310_720 + 128 * 64 * 4 + 128 * 4,
        "llama3-70b": 17_179_869_184 + 2 * 4_194_304 + 256 * 2048 * 4 + 256 * 4,
        # four fp32 scales per (token, kv-head) row of K and of V
        "llama3-70b-int8-g32": 17_179_869_184 + 2 * 256 * 32768 * 8 * 4 * 4 + 2 * 4_194_304 + 256 * 2048 * 4
                               + 256 * 4,
        "llama3-70b-int4-g32": 8_589_934_592 + 2 * 256 * 32768 * 8 * 4 * 4 + 2 * 4_194_304 + 256 * 2048 * 4
                               + 256 * 4,
    }
    for name, total in want.items():
        wl = W.WORKLOADS[name]
        assert W.decode_bytes(wl, W.context_lens(wl))["total"] == total, name


def test_ragged_contexts_are_seeded_and_in_range():
    wl = W.WORKLOADS["llama3-8b"]
    a, b = W.context_lens(wl), W.context_lens(wl)
    assert torch.equal(a, b)
    lo, hi = wl.ctx
    assert int(a.min()) >= lo and int(a.max()) <= hi
    assert len(set(a.tolist())) > wl.batch // 2          # lengths really vary


@pytest.mark.parametrize("name", ["tiny", "llama2-7b", "llama3-8b", "llama2-13b-int8"])
def test_block_tables_are_a_permutation_and_slots_follow_them(name):
    wl = W.WORKLOADS[name]
    lay = W.Layout(wl)
    bs = wl.block_size
    used = []
    for b in range(wl.batch):
        n = math.ceil(int(lay.context_lens[b]) / bs)
        used.extend(lay.block_tables[b, :n].tolist())
    assert sorted(used) == list(range(lay.num_blocks))    # every block once, none shared
    if wl.batch > 1 and lay.num_blocks > 8:
        assert used != sorted(used)                       # shuffled
    seqs = [0, wl.batch - 1]
    p1 = min(40, lay.max_context_len)
    slots = lay.slots(0, p1, seqs).view(len(seqs), p1)
    for i, b in enumerate(seqs):
        for t in range(p1):
            if t < int(lay.context_lens[b]):
                assert int(slots[i, t]) == int(lay.block_tables[b, t // bs]) * bs + t % bs
            else:
                assert int(slots[i, t]) == -1


def test_kv_tokens_are_reproducible_per_window():
    wl = W.WORKLOADS["tiny"]
    k1, v1 = W.kv_tokens(wl, 0, 64)
    k2, v2 = W.kv_tokens(wl, 0, 64)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert k1.shape == (64, wl.num_kv_heads, wl.head_dim) and k1.dtype == torch.float16
    assert not torch.equal(k1, v1)
    k3, _ = W.kv_tokens(wl, 64, 128)
    assert not torch.equal(k1, k3)                         # another window, other values


def test_outlier_channels_are_one_percent_at_20x():
    wl = W.WORKLOADS["llama3-8b"]
    assert wl.outliers
    k, v = W.kv_tokens(wl, 0, 512, seqs=[0])
    for x in (k, v):
        rms = x.float().pow(2).mean(0).sqrt().numpy()     # [Hkv][D] per channel
        big = rms > 5.0
        n = wl.num_kv_heads * wl.head_dim
        assert big.sum() == max(1, round(0.01 * n))
        assert np.all(np.abs(rms[big] / 20.0 - 1.0) < 0.2)
        assert np.all(np.abs(rms[~big] - 1.0) < 0.2)


def test_chunk_windows_cover_the_context():
    for name in ("llama2-7b", "llama3-70b"):
        wl = W.WORKLOADS[name]
        win = W.chunk_positions(wl, 1 << 19)
        assert win[0][0] == 0 and win[-1][1] == (wl.ctx if isinstance(wl.ctx, int) else wl.ctx[1])
        assert all(a[1] == b[0] for a, b in zip(win, win[1:]))
        assert all((p1 - p0) * wl.batch <= max(1 << 19, wl.block_size * wl.batch) for p0, p1 in win)


def test_quant_error_variants():
    from fp8_int8_quantized_gb300 import quant_error as Q
    base = W.WORKLOADS["llama2-7b"]
    v = Q.variant(base, "int4", "g32")
    assert (v.fmt, v.scale_rule, v.quant_group, v.scales_per_row) == ("int4", "row", 32, 4)
    v = Q.variant(base, "e5m2", "one")
    assert (v.fmt, v.scale_rule, v.quant_group) == ("e5m2", "one", 0)
    assert Q.variant(dataclasses.replace(base, head_dim=64), "int4", "g48") is None   # 48 does not divide 64
    assert set(Q.supported_variants("llama2-7b")) == set(Q.VARIANTS)
