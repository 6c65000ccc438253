"""Pins for the oracle's append, dequant and decode attention.

  * append: every token lands at block slot // BS, row slot % BS of the
    [num_blocks][kv_heads][block][head_dim] layout, as the pinned encoder's code of
    x / scale; slot -1 and untouched slots keep the sentinel;
  * attention: torch's scaled_dot_product_attention in fp64 (a library routine
    sharing nothing with the oracle) on K/V dequantized by torch's own float8
    conversion and gathered through the block table with torch indexing;
  * closed forms and invariants: a hand-computed 2-token case, softmax weights sum
    to 1, context 1 returns V[0], q = 0 returns the mean of V, a dominant logit
    returns its V row, context 0 returns zeros, relabelling physical blocks
    changes nothing.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import golden

TORCH_DT = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def make_case(rng, B, Hq, Hkv, D, BS, fmt, ctx, scale=None, outliers=False, group=0):
    ctx = np.asarray(ctx, np.int32)
    nblk = [(int(c) + BS - 1) // BS for c in ctx]
    NB = sum(nblk) + 3
    maxb = max(1, max(nblk))
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((B, maxb), -7, np.int32)      # unused entries hold junk on purpose
    at = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[at:at + n]
        at += n
    cache = oracle.Cache(NB, Hkv, BS, D, fmt, group=group)
    slots = []
    for b in range(B):
        for t in range(int(ctx[b])):
            slots.append(int(bt[b, t // BS]) * BS + t % BS)
    T = len(slots)
    k = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    if outliers:
        k[:, 0, 3] *= 20
        v[:, -1, 5] *= 20
    k, v = k.astype(np.float16), v.astype(np.float16)
    if scale == "amax":
        scale = float(np.float32(max(np.abs(k).max(), np.abs(v).max())) / np.float32(448.0))
    oracle.append(k, v, np.array(slots, np.int64), cache, scale)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    return q, cache, bt, ctx, scale, k, v, np.array(slots, np.int64)


def torch_dequant(cache, scale):
    def per_channel(sc):      # row scales broadcast, or group scales repeated over their channels
        t = torch.from_numpy(sc)
        return t.repeat_interleave(cache.group, dim=-1) if getattr(cache, "group", 0) else t[..., None]
    if cache.fmt == oracle.INT4:
        def nibbles(codes):   # channel 2i = low nibble; (n ^ 8) - 8 sign-extends 4 bits
            t = torch.from_numpy(codes.astype(np.int32))
            both = torch.stack([t & 15, t >> 4], dim=-1).flatten(-2)
            return ((both ^ 8) - 8).to(torch.float32)
        kk = nibbles(cache.k_codes) * per_channel(cache.k_scales)
        vv = nibbles(cache.v_codes) * per_channel(cache.v_scales)
    elif cache.fmt == oracle.INT8:
        kk = torch.from_numpy(cache.k_codes.view(np.int8)).to(torch.float32) * per_channel(cache.k_scales)
        vv = torch.from_numpy(cache.v_codes.view(np.int8)).to(torch.float32) * per_channel(cache.v_scales)
    else:
        s = torch.tensor(1.0 if scale is None else scale, dtype=torch.float32)
        kk = torch.from_numpy(cache.k_codes).view(TORCH_DT[cache.fmt]).to(torch.float32) * s
        vv = torch.from_numpy(cache.v_codes).view(TORCH_DT[cache.fmt]).to(torch.float32) * s
    return kk.double(), vv.double()


def torch_reference(q, cache, bt, ctx, scale, sm_scale=None):
    kk, vv = torch_dequant(cache, scale)
    B, Hq, D = q.shape
    G = Hq // cache.num_kv_heads
    BS = cache.block_size
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        n = int(ctx[b])
        if n == 0:
            continue
        t = torch.arange(n)
        blk = torch.from_numpy(bt[b]).long()[t // BS]
        K = kk[blk, :, t % BS, :].permute(1, 0, 2)          # [Hkv, n, D]
        V = vv[blk, :, t % BS, :].permute(1, 0, 2)
        K = K.repeat_interleave(G, dim=0)[None]
        V = V.repeat_interleave(G, dim=0)[None]
        Q = torch.from_numpy(q[b].astype(np.float64))[None, :, None, :]
        sc = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
        out[b] = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=sc)[0, :, 0, :]
    return out.numpy()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("BS", [16, 64])
def test_append_layout(fmt, BS):
    rng = np.random.default_rng(fmt * 10 + BS)
    q, cache, bt, ctx, scale, k, v, slots = make_case(
        rng, 3, 4, 2, 64, BS, fmt, [5, BS + 3, 0], scale=("amax" if fmt == oracle.E4M3 else None))
    written = np.zeros(cache.k_codes.shape[:3], bool)
    for t, slot in enumerate(slots):
        blk, off = slot // BS, slot % BS
        for h in range(cache.num_kv_heads):
            written[blk, h, off] = True
            for src, codes, sc in ((k, cache.k_codes, cache.k_scales), (v, cache.v_codes, cache.v_scales)):
                x = src[t, h].astype(np.float32)
                if fmt == oracle.INT8:
                    qq, s = oracle.int8_quant_row(x)
                    assert np.array_equal(codes[blk, h, off].view(np.int8), qq)
                    assert sc[blk, h, off] == s
                elif fmt == oracle.INT4:
                    qq, s = oracle.int4_quant_row(x)
                    assert np.array_equal(codes[blk, h, off], qq)
                    assert sc[blk, h, off] == s
                else:
                    s = np.float32(1.0 if scale is None else scale)
                    assert np.array_equal(codes[blk, h, off], oracle.fp8_encode(fmt, x / s))
    assert (cache.k_codes[~written] == 0xA5).all() and (cache.v_codes[~written] == 0xA5).all()


def test_append_skips_minus_one_and_default_scale():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((4, 2, 64)).astype(np.float16)
    v = rng.standard_normal((4, 2, 64)).astype(np.float16)
    a = oracle.Cache(2, 2, 16, 64, oracle.E4M3)
    b = oracle.Cache(2, 2, 16, 64, oracle.E4M3)
    slots = np.array([0, -1, 17, -1], np.int64)
    oracle.append(k, v, slots, a, None)
    oracle.append(k, v, slots, b, 1.0)
    assert np.array_equal(a.k_codes, b.k_codes) and np.array_equal(a.v_codes, b.v_codes)
    assert (a.k_codes[0, :, 1:] == 0xA5).all() and (a.k_codes[1, :, 0] == 0xA5).all()
    with pytest.raises(IndexError):
        oracle.append(k, v, np.array([0, 1, 2, 32], np.int64), a, None)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.INT8, oracle.INT4])
def test_dequant_matches_torch(fmt):
    rng = np.random.default_rng(11 + fmt)
    q, cache, bt, ctx, scale, k, v, slots = make_case(rng, 2, 4, 2, 64, 16, fmt, [20, 9], scale=0.75)
    ok, ov = oracle.dequant(cache, slots, scale)
    kk, vv = torch_dequant(cache, scale)
    blk, off = slots // 16, slots % 16
    assert np.array_equal(ok, kk[blk, :, off, :].float().numpy())
    assert np.array_equal(ov, vv[blk, :, off, :].float().numpy())


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2, oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("shape", [(2, 4, 4, 64, 16), (3, 8, 2, 128, 16), (2, 8, 1, 64, 32), (1, 16, 2, 128, 64)])
def test_attention_matches_torch_sdpa(fmt, shape):
    B, Hq, Hkv, D, BS = shape
    rng = np.random.default_rng(hash((fmt,) + shape) % 2**32)
    ctx = rng.integers(1, 3 * BS + 5, size=B)
    ctx[0] = 1
    q, cache, bt, ctx, scale, *_ = make_case(rng, B, Hq, Hkv, D, BS, fmt, ctx,
                                             scale=("amax" if fmt == oracle.E4M3 else None),
                                             outliers=True)
    out = oracle.decode_attention(q, cache, bt, ctx, scale)
    ref = torch_reference(q, cache, bt, ctx, scale)
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_attention_custom_sm_scale():
    rng = np.random.default_rng(5)
    q, cache, bt, ctx, scale, *_ = make_case(rng, 2, 4, 2, 64, 16, oracle.E5M2, [17, 40])
    out = oracle.decode_attention(q, cache, bt, ctx, scale, sm_scale=0.3)
    ref = torch_reference(q, cache, bt, ctx, scale, sm_scale=0.3)
    assert np.max(np.abs(out - ref)) <= 1e-12


def test_hand_two_token_case():
    g = {r[0]: float(r[1]) for r in golden("attention_2tok.txt")}
    cache = oracle.Cache(1, 1, 2, 2, oracle.E4M3, fill=0)
    cache.k_codes[0, 0] = [[0x38, 0x00], [0x40, 0x00]]
    cache.v_codes[0, 0] = [[0x38, 0x00], [0x00, 0x38]]
    q = np.array([[[1.0, 0.0]]], np.float16)
    out, w = oracle.decode_attention(q, cache, np.array([[0]], np.int32), np.array([2], np.int32),
                                     1.0, sm_scale=1.0, return_weights=True)
    assert abs(w[0, 0, 0] - g["w0"]) < 1e-15 and abs(w[0, 0, 1] - g["w1"]) < 1e-15
    assert abs(out[0, 0, 0] - g["out0"]) < 1e-15 and abs(out[0, 0, 1] - g["out1"]) < 1e-15


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.INT8, oracle.INT4])
def test_invariants(fmt):
    rng = np.random.default_rng(99 + fmt)
    B, Hq, Hkv, D, BS = 4, 8, 2, 64, 16
    ctx = np.array([1, 37, 0, 64], np.int32)
    q, cache, bt, ctx, scale, *_ = make_case(rng, B, Hq, Hkv, D, BS, fmt, ctx, scale=0.5)
    out, w = oracle.decode_attention(q, cache, bt, ctx, scale, return_weights=True)
    kk, vv = torch_dequant(cache, scale)
    G = Hq // Hkv
    for b in range(B):
        n = int(ctx[b])
        if n == 0:
            assert not out[b].any()
            continue
        assert np.allclose(w[b, :, :n].sum(-1), 1.0, rtol=0, atol=1e-12)
        assert (w[b, :, :n] > 0).all()
        if n == 1:
            blk = bt[b, 0]
            for h in range(Hq):
                assert np.array_equal(out[b, h], vv[blk, h // G, 0].numpy())
    # q = 0: every weight is 1/n, out is the mean of V
    q0 = np.zeros_like(q)
    out0 = oracle.decode_attention(q0, cache, bt, ctx, scale)
    b, n = 1, int(ctx[1])
    t = np.arange(n)
    V = vv[torch.from_numpy(bt[b][t // BS]).long(), :, torch.from_numpy(t % BS).long(), :].numpy()
    for h in range(Hq):
        assert np.allclose(out0[b, h], V[:, h // G].mean(0), rtol=0, atol=1e-13)


def test_dominant_logit_and_block_relabel():
    rng = np.random.default_rng(1234)
    B, Hq, Hkv, D, BS = 1, 2, 1, 64, 16
    q, cache, bt, ctx, scale, *_ = make_case(rng, B, Hq, Hkv, D, BS, oracle.E4M3, [45], scale=1.0)
    # make token 30 dominate: K row = q direction * large, E4M3 codes set directly
    q[:] = 0
    q[0, :, 0] = 1.0
    blk, off = bt[0, 30 // BS], 30 % BS
    cache.k_codes[:, 0, :, 0] = 0x00
    cache.k_codes[blk, 0, off, 0] = 0x7E        # 448 * 1/sqrt(64) = 56 logit gap
    out = oracle.decode_attention(q, cache, bt, ctx, scale)
    vrow = np.array([oracle.fp8_decode(oracle.E4M3, c) for c in cache.v_codes[blk, 0, off]])
    # the other 44 weights are each about e^-56, so they move out by < 1e-18
    assert np.allclose(out[0, 0], vrow, rtol=0, atol=1e-18)
    # relabel physical blocks: permute the cache's blocks and the table together
    perm = rng.permutation(cache.num_blocks)
    inv = np.argsort(perm)
    c2 = oracle.Cache(cache.num_blocks, Hkv, BS, D, cache.fmt,
                      k_codes=np.ascontiguousarray(cache.k_codes[perm]),
                      v_codes=np.ascontiguousarray(cache.v_codes[perm]))
    bt2 = np.where(bt >= 0, inv[np.clip(bt, 0, None)], bt).astype(np.int32)
    out2 = oracle.decode_attention(q, c2, bt2, ctx, scale)
    assert np.array_equal(out, out2)
