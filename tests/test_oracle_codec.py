"""Pins for the oracle's FP8 codec (decode table and encoder).

What pins what:
  * hand-derived spot values from the bit layouts of "Accelerating Inference with
    FP8 KV Cache", section "FP8 Formats: E4M3 and E5M2" (tests/golden);
  * torch's own float8_e4m3fn / float8_e5m2 conversions (a library routine that
    shares nothing with the oracle), for all 256 codes and all 2^32 fp32 inputs;
  * the closed form E5M2(c) == binary16 with bits c << 8.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import golden

FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
TORCH_DT = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}
FMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0}


def test_decode_spot_values():
    for fmt, code, val in golden("fp8_decode_spot.txt"):
        got = oracle.fp8_decode(FMT[fmt], int(code, 16))
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got), (fmt, code)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, code, got)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_table_matches_torch(fmt):
    tab = oracle.fp8_decode_table(fmt)
    ref = torch.arange(256, dtype=torch.uint8).view(TORCH_DT[fmt]).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(tab[ok], ref[ok])
    assert np.array_equal(np.signbit(tab[ok]), np.signbit(ref[ok]))


def test_decode_table_structure():
    e4 = oracle.fp8_decode_table(oracle.E4M3)
    assert np.count_nonzero(np.isnan(e4)) == 2 and not np.isinf(e4).any()   # no infinities
    assert np.nanmax(e4) == 448.0 and np.nanmin(e4) == -448.0
    e5 = oracle.fp8_decode_table(oracle.E5M2)
    assert np.count_nonzero(np.isinf(e5)) == 2 and np.count_nonzero(np.isnan(e5)) == 6
    assert np.max(e5[np.isfinite(e5)]) == 57344.0
    # every finite FP8 value is exact in fp16 (compute in FP16 loses nothing)
    for tab in (e4, e5):
        f = tab[np.isfinite(tab)]
        assert np.array_equal(f.astype(np.float16).astype(np.float64), f)


def test_e5m2_is_top_byte_of_fp16():
    codes = np.arange(256, dtype=np.uint16)
    as_half = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    tab = oracle.fp8_decode_table(oracle.E5M2)
    assert np.array_equal(np.isnan(tab), np.isnan(as_half))
    ok = ~np.isnan(tab)
    assert np.array_equal(tab[ok], as_half[ok])


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_round_trip_every_finite_code(fmt):
    tab = oracle.fp8_decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(tab[c])], dtype=np.uint8)
    vals = tab[codes].astype(np.float32)
    vals = np.where(codes == 0x80, np.float32(-0.0), vals)
    assert np.array_equal(oracle.fp8_encode(fmt, vals), codes)


def test_encode_spot_values():
    for row in golden("fp8_encode_spot.txt"):
        fmt, val, code = row[0], float(row[1]), int(row[2], 16)
        got = int(oracle.fp8_encode(FMT[fmt], np.array([val], np.float32))[0])
        assert got == code, (fmt, val, hex(got), hex(code))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_nan(fmt):
    nans = np.array([np.nan, -np.nan], np.float32)
    nans[1] = np.frombuffer(np.uint32(0xFFC00001).tobytes(), np.float32)[0]
    assert list(oracle.fp8_encode(fmt, nans)) == [0x7F, 0x7F]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_all_fp32_against_torch(fmt):
    """Every one of the 2^32 fp32 bit patterns: the oracle equals torch's
    round-to-nearest-even conversion of the input clamped to +-max (clamping is
    what saturation means); NaN inputs give 0x7F."""
    chunk = 1 << 26
    m = FMAX[fmt]
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64).to(torch.int32)
        x = bits.view(torch.float32)
        want = x.clamp(-m, m).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
        got = oracle.fp8_encode(fmt, x.numpy())
        nan = torch.isnan(x).numpy()
        bad = (got != want) & ~nan
        assert not bad.any(), (start, np.flatnonzero(bad)[:5])
        assert (got[nan] == 0x7F).all()
