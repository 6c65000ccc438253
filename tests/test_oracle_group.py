"""Pins for the oracle's per-group INT8 / INT4 cache: group quantization (named
for a 4-bit KV cache on the QQQ page "[QST] Scale factors and benchmarks") read
as the online row quantizer of "[Feature] TurboMind support W8A8 or FP8 KV Cache"
(lmdeploy issue 1463) applied to every group of ``group`` consecutive channels,
one fp32 scale per group, scales stored [NB][Hkv][BS][D / group].

  * hand-derived rows (tests/golden/group_row.txt) through the oracle's append;
  * special case: group = head_dim gives the per-row format byte for byte;
  * closed-form properties of every group: its largest |x| maps to +-127 (+-7),
    its scale is fl32(amax / 127) (fl32(amax / 7)), every value is within half a
    step of its code times the scale, and an exact doubling of one group doubles
    its scale and changes no code anywhere;
  * dequant against numpy, attention against torch's scaled_dot_product_attention
    in fp64 on K/V dequantized with torch (group scales repeated over their
    channels), decode and chunked prefill;
  * a row with an outlier channel loses less to per-group INT4 than to per-row.
"""
import numpy as np
import pytest

import oracle
from tests.conftest import golden
from tests.test_oracle_attention import make_case, torch_reference
from tests.test_oracle_prefill import chunked_case, torch_prefill_reference

QMAX = {oracle.INT8: 127, oracle.INT4: 7}


def quantize_rows(x16, fmt, group):
    """Append rows x16 (fp16 [n][D]) as K and V of a one-head cache, one row per slot;
    returns (signed codes int8 [n][D], scales fp32 [n][D / group or 1])."""
    n, D = x16.shape
    cache = oracle.Cache(n, 1, 1, D, fmt, group=group)
    oracle.append(x16[:, None], x16[:, None], np.arange(n, dtype=np.int64), cache)
    codes = cache.k_codes[:, 0, 0]
    codes = oracle.int4_unpack(codes) if fmt == oracle.INT4 else codes.view(np.int8)
    assert np.array_equal(cache.k_codes, cache.v_codes)
    return codes, cache.k_scales.reshape(n, -1)


@pytest.mark.parametrize("name,fmt", [("int8", oracle.INT8), ("int4", oracle.INT4)])
def test_hand_rows(name, fmt):
    rows = [r for r in golden("group_row.txt") if r[0] == name]
    x = np.array([[float(r[1]) for r in rows]], np.float16)
    codes, scales = quantize_rows(x, fmt, 4)
    assert list(codes[0]) == [int(r[2]) for r in rows]
    assert list(scales[0]) == [1.0, 0.0625]
    if fmt == oracle.INT4:
        cache = oracle.Cache(1, 1, 1, 8, fmt, group=4)
        oracle.append(x[:, None], x[:, None], np.zeros(1, np.int64), cache)
        assert list(cache.k_codes.reshape(-1)) == [0xC7, 0x02, 0x07, 0xE3]


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("D", [64, 128])
def test_group_of_whole_row_is_per_row(fmt, D):
    rng = np.random.default_rng(D + fmt)
    x = (rng.standard_normal((300, D)) * rng.choice([1e-3, 1.0, 50.0], (300, 1))).astype(np.float16)
    x[::7, 3] *= 20
    c0, s0 = quantize_rows(x, fmt, 0)
    c1, s1 = quantize_rows(x, fmt, D)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("D,group", [(64, 16), (64, 32), (128, 32), (128, 64), (8, 2)])
def test_group_properties(fmt, D, group):
    rng = np.random.default_rng(7 * D + group + fmt)
    n = 400
    x = (rng.standard_normal((n, D)) * rng.choice([1e-4, 1.0, 20.0, 300.0], (n, 1))).astype(np.float16)
    x[::5, 1] *= 20                           # outlier channels in some rows
    x[3] = 0                                  # an all-zero row
    x[4, :group] = 0                          # an all-zero group beside non-zero ones
    codes, scales = quantize_rows(x, fmt, group)
    ng = D // group
    assert scales.shape == (n, ng)
    qmax = QMAX[fmt]
    xg = x.astype(np.float32).reshape(n, ng, group)
    cg = codes.astype(np.int32).reshape(n, ng, group)
    amax = np.abs(xg).max(-1)
    assert np.array_equal(scales, amax / np.float32(qmax))            # fl32(amax / qmax)
    assert np.abs(cg).max() <= qmax
    nz = amax > 0
    assert np.array_equal(np.abs(cg).max(-1)[nz], np.full(nz.sum(), qmax))
    assert not cg[~nz].any()
    # within half a step, plus the rounding of s and of x / s to fp32 (|x / s| <= qmax)
    err = np.abs(xg.astype(np.float64) - cg * scales[..., None].astype(np.float64))
    assert (err <= scales[..., None].astype(np.float64) * (0.5 + 2 * qmax * 2.0 ** -24)).all()
    # doubling one group exactly (fp16 * 2 stays finite at these sizes) doubles its
    # scale only; every code stays
    y = x.copy()
    y[:, group:2 * group] *= 2 if ng > 1 else 1
    if ng > 1:
        small = np.abs(x).max(1) < 1000
        c2, s2 = quantize_rows(y[small], fmt, group)
        assert np.array_equal(c2, codes[small])
        assert np.array_equal(s2[:, 1], 2 * scales[small][:, 1])
        assert np.array_equal(np.delete(s2, 1, axis=1), np.delete(scales[small], 1, axis=1))


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4])
def test_dequant_matches_numpy(fmt):
    rng = np.random.default_rng(40 + fmt)
    q, cache, bt, ctx, scale, k, v, slots = make_case(rng, 2, 4, 2, 64, 16, fmt, [40, 23], group=16)
    ok, ov = oracle.dequant(cache, slots)
    for codes, sc, got in ((cache.k_codes, cache.k_scales, ok), (cache.v_codes, cache.v_scales, ov)):
        blk, off = slots // 16, slots % 16
        c = codes[blk, :, off]
        c = oracle.int4_unpack(c) if fmt == oracle.INT4 else c.view(np.int8)
        want = c.astype(np.float32) * np.repeat(sc[blk, :, off], 16, axis=-1)
        assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4])
@pytest.mark.parametrize("Hq,Hkv,D,BS,group", [(4, 4, 64, 16, 16), (8, 2, 128, 32, 32), (2, 1, 128, 64, 64)])
def test_decode_matches_sdpa(fmt, Hq, Hkv, D, BS, group):
    rng = np.random.default_rng(fmt + Hq + D + group)
    ctx = [1, BS + 3, 70, 0]
    q, cache, bt, ctx, scale, k, v, slots = make_case(rng, 4, Hq, Hkv, D, BS, fmt, ctx, outliers=True,
                                                      group=group)
    got = oracle.decode_attention(q, cache, bt, ctx)
    want = torch_reference(q, cache, bt, ctx, None)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", [oracle.INT8, oracle.INT4])
def test_prefill_matches_masked_sdpa(fmt):
    rng = np.random.default_rng(90 + fmt)
    q, cache, bt, ctx, qs, scale = chunked_case(rng, 8, 2, 128, 16, fmt, [37, 21, 70], [37, 3, 1],
                                                outliers=True, group=32)
    got = oracle.prefill_attention(q, cache, bt, ctx, qs, scale)
    want = torch_prefill_reference(q, cache, bt, ctx, qs, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_groups_help_rows_with_an_outlier():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((500, 128)).astype(np.float32)
    x[:, 5] *= 20
    x16 = x.astype(np.float16)
    errs = []
    for group in (0, 32):
        codes, scales = quantize_rows(x16, oracle.INT4, group)
        per = scales if group == 0 else np.repeat(scales, group, axis=1)
        e = codes * per - x16.astype(np.float32)
        errs.append(np.sqrt(np.mean(e[:, 32:] ** 2)))    # the channels outside the outlier's group
    assert errs[1] < 0.25 * errs[0]


def test_bad_groups_rejected():
    with pytest.raises(ValueError):
        oracle.Cache(1, 1, 16, 64, oracle.INT8, group=24)      # does not divide head_dim
    with pytest.raises(ValueError):
        oracle.Cache(1, 1, 16, 64, oracle.E4M3, group=32)      # FP8 has one per-tensor scale
    with pytest.raises(ValueError):
        oracle.Cache(1, 1, 16, 8, oracle.INT4, group=1)        # a byte holds two channels
