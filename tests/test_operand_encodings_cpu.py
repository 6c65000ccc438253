"""Exhaustive host checks of the bit-level identities the decode and prefill
kernels use to turn cached integer codes into exact fp16 tensor-core operands
(no GPU needed: numpy's IEEE binary16 decodes the same bit patterns):

  * INT8: the byte b = code XOR 0x80 (code + 128 as unsigned) placed in the
    low mantissa byte of 0x6400 (1024.0) is the fp16 value 1152 + code;
  * INT4: a signed nibble n = code (two's complement) XOR 8 is code + 8 in
    0..15; as the low bits of an fp16 with a zero exponent it is the subnormal
    (code + 8) * 2^-24, and left in mantissa bits 4..7 (the high nibble of a
    byte, masked in place) it is 16x that; both exact, and so is every
    product of such an operand with an fp16 query value in fp32.
"""
import numpy as np


def f16(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def nibble(n):
    """A 4-bit two's complement code."""
    return n - 16 if n >= 8 else n


def test_int8_biased_operand_is_exact():
    codes = np.arange(-128, 128)
    b = (codes & 0xFF) ^ 0x80
    assert np.array_equal(f16(0x6400 | b), 1152.0 + codes)


def test_int4_subnormal_operands_are_exact():
    for byte in range(256):
        c_lo, c_hi = nibble(byte & 0xF), nibble(byte >> 4)
        # the low nibble masked in place (bits 0..3), offset by XOR 8
        assert f16((byte & 0x0F) ^ 0x08) == (c_lo + 8) * 2.0 ** -24
        # the high nibble masked in place (bits 4..7): 16x its subnormal
        assert f16((byte & 0xF0) ^ 0x80) == 16 * (c_hi + 8) * 2.0 ** -24


def test_int4_pair_in_one_word_masks_two_lanes():
    # one 32-bit word: bytes 0 and 2 land in the two fp16 halves of an operand
    rng = np.random.default_rng(0)
    for w in rng.integers(0, 1 << 32, 200, dtype=np.uint64):
        w = int(w)
        h0 = (w & 0x00F0000F) ^ 0x00800008           # [byte0 low nibble, 16 x byte2 high nibble]
        lo_half, hi_half = h0 & 0xFFFF, h0 >> 16
        b0, b2 = w & 0xFF, (w >> 16) & 0xFF
        assert f16(lo_half) == (nibble(b0 & 0xF) + 8) * 2.0 ** -24
        assert f16(hi_half) == 16 * (nibble(b2 >> 4) + 8) * 2.0 ** -24


def test_int4_operand_products_are_exact_in_fp32():
    # every product of an INT4 operand (k * 2^-24 or 16 k * 2^-24, k = 0..15)
    # with any finite fp16 query value is exact in fp32 (15 significant bits at
    # most) and stays in fp32's normal range, so the tensor cores' fp32 sums see
    # the same products as exact integer codes scaled by 2^-24 would give
    ops = np.array([k * 2.0 ** -24 for k in range(16)] + [16 * k * 2.0 ** -24 for k in range(16)])
    q = np.arange(0, 0x7C00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)   # finite, >= 0
    q = np.concatenate([q, [2.0 ** -24, 65504.0]])
    prod64 = ops[:, None] * q[None, :]
    prod32 = ops.astype(np.float32)[:, None] * q.astype(np.float32)[None, :]
    assert np.array_equal(prod32.astype(np.float64), prod64)
    nz = prod64[prod64 > 0]
    assert nz.min() >= np.finfo(np.float32).tiny and nz.max() < np.finfo(np.float32).max
