"""Pins for the oracle's online INT4 row quantizer: the INT8 row reading of
"[Feature] TurboMind support W8A8 or FP8 KV Cache" (lmdeploy issue 1463) with 4
bits -- one fp32 scale amax / 7 per (token, kv-head) row, codes in [-7, 7], two
per byte with channel 2i in the low nibble."""
import numpy as np
import torch

import oracle
from tests.conftest import golden


def test_hand_row_and_packing():
    rows = golden("int4_row.txt")
    x = np.array([float(r[0]) for r in rows], np.float32)
    packed, s = oracle.int4_quant_row(x)
    assert s == np.float32(0.25)
    assert list(oracle.int4_unpack(packed)) == [int(r[1]) for r in rows]
    assert list(packed) == [0xC7, 0x01, 0x90, 0x42]


def test_zero_row():
    packed, s = oracle.int4_quant_row(np.zeros(64, np.float32))
    assert s == 0 and not packed.any()


def test_unpack_is_signed_nibbles():
    every = np.arange(256, dtype=np.uint8)[None]
    codes = oracle.int4_unpack(every)[0].reshape(256, 2)
    for b in range(256):
        lo, hi = b & 0xF, b >> 4
        assert codes[b, 0] == (lo - 16 if lo >= 8 else lo)
        assert codes[b, 1] == (hi - 16 if hi >= 8 else hi)


def test_properties_random_rows():
    rng = np.random.default_rng(17)
    for i in range(2000):
        d = 128 if i % 2 else 64
        x = (rng.standard_normal(d) * rng.choice([1e-4, 1.0, 20.0, 3000.0])).astype(np.float16)
        x32 = x.astype(np.float32)
        packed, s = oracle.int4_quant_row(x32)
        q = oracle.int4_unpack(packed).astype(np.int64)
        amax = np.abs(x32).max()
        assert s > 0 and abs(float(s) * 7.0 - float(amax)) <= float(amax) * 2.0 ** -23
        assert q.min() >= -7 and q.max() <= 7          # -8 never produced
        j = int(np.argmax(np.abs(x32)))
        assert q[j] == (7 if x32[j] > 0 else -7)
        # the decision in the precision the method fixes: the fp32 quotient,
        # rounded to the nearest integer, ties to even (brute force over -7..7)
        y = (x32 / s).astype(np.float32).astype(np.float64)
        cand = np.arange(-7, 8)[None, :]
        dist = np.abs(y[:, None] - cand)
        best = dist.min(1, keepdims=True)
        tie_even = np.where(dist == best, cand, 99)
        want = np.where((dist == best).sum(1) > 1, tie_even[np.arange(d), np.argmin(np.abs(tie_even % 2), 1)],
                        cand[0, np.argmin(dist, 1)])
        assert np.array_equal(q, want)


def test_append_and_dequant_through_the_cache():
    rng = np.random.default_rng(5)
    T, Hkv, D, BS = 5, 2, 64, 16
    k = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    cache = oracle.Cache(2, Hkv, BS, D, oracle.INT4)
    assert cache.k_codes.shape == (2, Hkv, BS, D // 2)
    slots = np.array([0, 17, -1, 5, 31], np.int64)
    oracle.append(k, v, slots, cache)
    ok, ov = oracle.dequant(cache, slots[slots >= 0])
    for i, t in enumerate(np.nonzero(slots >= 0)[0]):
        blk, off = slots[t] // BS, slots[t] % BS
        for h in range(Hkv):
            for src, codes, sc, out in ((k, cache.k_codes, cache.k_scales, ok), (v, cache.v_codes, cache.v_scales, ov)):
                packed, s = oracle.int4_quant_row(src[t, h].astype(np.float32))
                assert np.array_equal(codes[blk, h, off], packed) and sc[blk, h, off] == s
                want = torch.from_numpy(oracle.int4_unpack(packed).astype(np.float32)) * torch.tensor(s)
                assert np.array_equal(out[i, h], want.numpy())
