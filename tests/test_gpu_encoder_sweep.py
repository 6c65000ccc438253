"""The FP8 encoder of the append kernels on every fp32 input.

"Accelerating Inference with FP8 KV Cache", "FP8 Formats: E4M3 and E5M2": the
cache holds E4M3 / E5M2 codes of x / scale.  kvq_append rounds fl32(x / s)
with the hardware conversion (round to nearest even, saturating to +-max);
kvq_encode_fp8 applies that same device encoder to raw fp32 values, so here it
runs on all 2^32 fp32 bit patterns (NaN, Inf, subnormals, every binade) and is
compared with the CPU oracle's encoder (a nearest-value search over the code
table) byte for byte.  NaN inputs must give a NaN code of the format (which one
is not fixed by the pages; the oracle writes 0x7F).  The append kernels
themselves are checked on all 65536 fp16 inputs at several scales in
test_gpu_append.py."""
import numpy as np
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.build()
    torch.cuda.init()


def is_nan_code(fmt, c):
    if fmt == oracle.E4M3:
        return (c & 0x7F) == 0x7F
    return (c & 0x7F) > 0x7C


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2], ids=["e4m3", "e5m2"])
def test_device_encoder_on_every_fp32_input(fmt):
    lib = kvq.lib()
    codes = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    host = torch.empty(CHUNK, dtype=torch.uint8).pin_memory()
    checked = 0
    for start in range(0, 1 << 32, CHUNK):
        x = torch.arange(start, start + CHUNK, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
        st = lib.kvq_encode_fp8(x.data_ptr(), codes.data_ptr(), CHUNK, fmt, None)
        assert st == 0
        host.copy_(codes)
        got = host.numpy()
        xh = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = oracle.fp8_encode(fmt, xh)
        nan = np.isnan(xh)
        bad = (got != want) & ~nan
        assert not bad.any(), (hex(start), np.flatnonzero(bad)[:5], got[bad][:5], want[bad][:5])
        assert is_nan_code(fmt, got[nan]).all()
        checked += CHUNK
    assert checked == 1 << 32
    assert kvq.device_error_check()[0] == 0


def test_encoder_tail_and_arguments():
    """A count that is not a multiple of 16 (the tail is encoded one value at a
    time) and the argument checks."""
    lib = kvq.lib()
    x = (torch.randn(1000, device="cuda") * 100).float()
    codes = torch.zeros(1008, dtype=torch.uint8, device="cuda")
    assert lib.kvq_encode_fp8(x.data_ptr(), codes.data_ptr(), 999, oracle.E4M3, None) == 0
    torch.cuda.synchronize()
    want = oracle.fp8_encode(oracle.E4M3, x.cpu().numpy()[:999])
    assert np.array_equal(codes.cpu().numpy()[:999], want)
    assert (codes.cpu().numpy()[999:] == 0).all()
    assert np.array_equal(kvq.encode_fp8(x[:999].contiguous(), oracle.E4M3).cpu().numpy(), want)
    assert lib.kvq_encode_fp8(x.data_ptr(), codes.data_ptr(), 16, 3, None) == 1        # INT8 is not FP8
