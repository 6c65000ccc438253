"""The quantization-error report: every format's decode output against
attention over the unquantized fp16 cache.  Checks what the formats' precision
fixes: on N(0, 1) data an E4M3 code carries 3 mantissa bits (relative
rounding error about 2^-4 / sqrt(3) RMS), E5M2 one fewer (twice the error),
and INT8 with a scale per row far less; INT4 with a scale per row has a step
of amax / 7 (about 0.4 sigma for 128 Gaussian values: error ~ 0.11 RMS, above
E4M3's); on the outlier workload the same order holds.  One INT4 scale per group
of channels lowers INT4's error, on Gaussian data (a group's amax is smaller
than the row's) and most where an outlier channel sets a row's scale."""
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
from fp8_int8_quantized_gb300 import quant_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.build()
    torch.cuda.init()


def rows_of(name, batch):
    rows = {(r["format"], r["scale"]): r for r in quant_error.report(name, batch=batch)}
    assert len(rows) == len(quant_error.supported_variants(name))
    for r in rows.values():
        assert 0.0 < r["rel_rms"] < 1.0, r
    return rows


def test_report_gaussian_data():
    rows = rows_of("llama2-7b", 2)
    e4 = rows[("e4m3", "amax")]["rel_rms"]
    e5 = rows[("e5m2", "amax")]["rel_rms"]
    i8 = rows[("int8", "row")]["rel_rms"]
    assert 0.02 < e4 < 0.06
    assert 1.5 < e5 / e4 < 2.5           # one mantissa bit fewer
    assert i8 < e4 / 2
    i4 = rows[("int4", "row")]["rel_rms"]
    assert 1.5 < i4 / e4 < 6 and i4 > e5 * 0.9
    for (fmt, _), r in rows.items():
        assert r["min_cos"] > (0.97 if fmt == "int4" else 0.99), r
    assert rows[("int4", "g32")]["rel_rms"] < 0.95 * i4
    assert rows[("int4", "g32")]["rel_rms"] < rows[("int4", "g64")]["rel_rms"] < i4
    assert rows[("int8", "g32")]["rel_rms"] < i8


def test_report_outlier_data_keeps_the_order():
    rows = rows_of("llama3-8b", 2)
    assert rows[("e4m3", "amax")]["rel_rms"] < rows[("e5m2", "amax")]["rel_rms"]
    assert rows[("int8", "row")]["rel_rms"] < rows[("e4m3", "amax")]["rel_rms"]
    assert rows[("int4", "row")]["rel_rms"] > rows[("int8", "row")]["rel_rms"]
    assert rows[("int4", "g32")]["rel_rms"] < rows[("int4", "g64")]["rel_rms"] < 0.8 * rows[("int4", "row")]["rel_rms"]
