"""Pins for the oracle's causal attention of a chunk of new queries over the cache.

  * torch's scaled_dot_product_attention in fp64 (a library routine sharing
    nothing with the oracle) with an explicit boolean mask -- query i of an
    n-query chunk sits at position ctx - n + i and sees t <= that position --
    on K/V dequantized by torch's own float8 conversion (or code * row scale)
    and gathered through the block table with torch indexing;
  * closed form: a chunk that starts at position 0 gives its first query
    exactly the dequantized V row 0;
  * invariants: the last query of every chunk equals single-token decode
    attention over the whole context, and a one-query chunk equals decode;
  * argument checks: a chunk longer than its context is rejected.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_attention import make_case, torch_dequant


def torch_prefill_reference(q, cache, bt, ctx, qs, scale, sm_scale=None):
    kk, vv = torch_dequant(cache, scale)
    Tq, Hq, D = q.shape
    G = Hq // cache.num_kv_heads
    BS = cache.block_size
    out = torch.zeros((Tq, Hq, D), dtype=torch.float64)
    sc = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    for b in range(len(ctx)):
        n, c = int(qs[b + 1] - qs[b]), int(ctx[b])
        if n == 0:
            continue
        t = torch.arange(c)
        blk = torch.from_numpy(bt[b]).long()[t // BS]
        K = kk[blk, :, t % BS, :].permute(1, 0, 2).repeat_interleave(G, dim=0)[None]   # [1, Hq, c, D]
        V = vv[blk, :, t % BS, :].permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        Q = torch.from_numpy(q[qs[b]:qs[b + 1]].astype(np.float64)).permute(1, 0, 2)[None]  # [1, Hq, n, D]
        pos = torch.arange(c - n, c)[:, None]
        mask = torch.arange(c)[None, :] <= pos                                            # [n, c]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=sc)
        out[qs[b]:qs[b + 1]] = o[0].permute(1, 0, 2)
    return out.numpy()


def chunked_case(rng, Hq, Hkv, D, BS, fmt, ctx, chunk, scale=None, outliers=False, group=0):
    q1, cache, bt, ctx, scale, k, v, slots = make_case(rng, len(ctx), Hq, Hkv, D, BS, fmt, ctx,
                                                       scale=scale, outliers=outliers, group=group)
    qs = np.zeros(len(ctx) + 1, np.int32)
    qs[1:] = np.cumsum(chunk)
    q = rng.standard_normal((int(qs[-1]), Hq, D)).astype(np.float16)
    return q, cache, bt, ctx, qs, scale


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("Hq,Hkv,D,BS", [(4, 4, 64, 16), (8, 2, 64, 32), (8, 1, 128, 64)])
def test_matches_masked_sdpa(fmt, Hq, Hkv, D, BS):
    rng = np.random.default_rng(100 * fmt + Hq + D + BS)
    ctx = [37, BS + 5, 70, 9]
    chunk = [37, 3, 1, 0]            # whole context, ragged chunk, one query, no query
    q, cache, bt, ctx, qs, scale = chunked_case(rng, Hq, Hkv, D, BS, fmt, ctx, chunk,
                                                scale=("amax" if fmt == oracle.E4M3 else None),
                                                outliers=(fmt == oracle.E5M2))
    got = oracle.prefill_attention(q, cache, bt, ctx, qs, scale)
    want = torch_prefill_reference(q, cache, bt, ctx, qs, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_custom_softmax_scale_matches_sdpa():
    rng = np.random.default_rng(7)
    q, cache, bt, ctx, qs, scale = chunked_case(rng, 4, 2, 64, 16, oracle.E4M3, [50, 20], [17, 20])
    got = oracle.prefill_attention(q, cache, bt, ctx, qs, scale, sm_scale=0.37)
    want = torch_prefill_reference(q, cache, bt, ctx, qs, scale, sm_scale=0.37)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.INT8])
def test_first_position_is_v0(fmt):
    rng = np.random.default_rng(11 + fmt)
    q, cache, bt, ctx, qs, scale = chunked_case(rng, 4, 2, 64, 16, fmt, [20, 33], [20, 33])
    out = oracle.prefill_attention(q, cache, bt, ctx, qs, scale)
    G = 2
    for b in range(2):
        slot = np.array([int(bt[b, 0]) * 16], np.int64)
        _, v0 = oracle.dequant(cache, slot, scale)
        for h in range(4):
            assert np.array_equal(out[qs[b], h], v0[0, h // G].astype(np.float64))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.INT8])
def test_last_query_equals_decode(fmt):
    rng = np.random.default_rng(21 + fmt)
    ctx = [64, 41, 100]
    chunk = [16, 41, 1]
    q, cache, bt, ctx, qs, scale = chunked_case(rng, 8, 2, 128, 16, fmt, ctx, chunk,
                                                scale=("amax" if fmt != oracle.INT8 else None))
    out = oracle.prefill_attention(q, cache, bt, ctx, qs, scale)
    last = np.stack([q[qs[b + 1] - 1] for b in range(3)])
    dec = oracle.decode_attention(last, cache, bt, ctx, scale)
    for b in range(3):
        np.testing.assert_allclose(out[qs[b + 1] - 1], dec[b], rtol=1e-13, atol=1e-13)
    # a query in the middle of a chunk equals decode with its own prefix only
    mid = qs[1] + 5                      # sequence 1, position 5
    dmid = oracle.decode_attention(q[mid][None], cache, bt[1:2], np.array([6], np.int32), scale)
    np.testing.assert_allclose(out[mid], dmid[0], rtol=1e-13, atol=1e-13)


def test_chunk_longer_than_context_rejected():
    rng = np.random.default_rng(3)
    q, cache, bt, ctx, qs, scale = chunked_case(rng, 4, 4, 64, 16, oracle.E4M3, [10], [10])
    qs_bad = np.array([0, 10], np.int32)
    with pytest.raises(IndexError):
        oracle.prefill_attention(q, cache, bt, np.array([9], np.int32), qs_bad, scale)
