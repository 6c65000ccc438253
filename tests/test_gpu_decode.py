"""GPU parity of decode attention (kvq_decode_attention) against the fp64 CPU
oracle on the same cache bytes: |o_gpu - o_ref| <= 2e-3 * max(1, |o_ref|) per
element.  Small cases span several tiles, partitions and a ragged tail; the
workload-sized cases run the launch configuration the benchmark times and check
a seeded sample of sequences."""
import numpy as np
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
import oracle
from fp8_int8_quantized_gb300 import workloads as W
from tests.gpu_util import ATOL_REL, DeviceWorkload, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.build()
    torch.cuda.init()
    yield
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)


def small(fmt, B, Hq, Hkv, D, BS, ctx, seed=0, outliers=True, scale_rule=None, group=0):
    wl = W.Workload(f"t-{fmt}", B, Hq, Hkv, D, BS, fmt, max(ctx), scale_rule or
                    ("amax" if fmt == "e4m3" else ("row" if fmt in ("int8", "int4") else "one")),
                    outliers=outliers, seed=seed, quant_group=group)
    return DeviceWorkload(wl, chunk_tokens=1 << 16, ctx=torch.tensor(ctx, dtype=torch.int32))


CASES = [
    # fmt, B, Hq, Hkv, D, BS, contexts
    ("e4m3", 3, 4, 4, 64, 16, [128, 1, 77]),
    ("e4m3", 2, 8, 1, 128, 16, [300, 17]),
    ("e5m2", 3, 32, 8, 128, 16, [1000, 512, 33]),
    ("e5m2", 2, 6, 3, 64, 32, [95, 400]),
    ("int8", 2, 4, 4, 128, 64, [640, 65]),
    ("int8", 3, 8, 2, 64, 64, [129, 1, 256]),
    ("e4m3", 2, 16, 2, 128, 32, [2050, 700]),
    ("e5m2", 1, 7, 7, 128, 16, [16]),
    ("int4", 2, 4, 4, 128, 64, [640, 65]),
    ("int4", 3, 8, 2, 64, 16, [129, 1, 256]),
    ("int4", 2, 32, 8, 128, 32, [1000, 33]),
    ("int4", 2, 16, 2, 128, 16, [700, 40]),
    ("int4", 2, 8, 1, 64, 32, [333, 64]),
    ("int8", 2, 10, 2, 128, 16, [257, 96]),
    ("int8", 2, 16, 2, 128, 16, [700, 129]),     # 8-head groups: one CTA of 12 warps per SM
    ("e5m2", 3, 16, 2, 64, 32, [300, 40, 1]),
    # group quantization (last field: channels per scale): q-heads per kv-head x groups <= 8
    ("int8", 2, 4, 2, 128, 32, [500, 33], 32),
    ("int4", 2, 4, 4, 128, 64, [640, 65], 32),
    ("int4", 3, 8, 2, 64, 16, [129, 1, 256], 32),
    ("int8", 3, 8, 1, 64, 16, [300, 1, 77], 64),
    ("int8", 2, 3, 3, 64, 16, [200, 45], 16),
    ("int4", 2, 4, 1, 128, 16, [96, 1000], 64),
    # more than 8 (q-head, group) operand rows: INT8, and INT4 with groups of
    # 32 or more channels, take the grouped consumer (one pass, a scale group
    # per contraction slice and output m-tile); INT4 with 16-channel groups the
    # 16-row consumer, one pass up to 16 rows, several launches beyond
    ("int8", 2, 16, 2, 128, 32, [500, 64], 32),
    ("int8", 2, 48, 8, 64, 16, [300, 90], 32),
    ("int4", 2, 8, 1, 128, 16, [300, 33], 64),
    ("int8", 3, 8, 2, 64, 16, [200, 17, 1], 16),
    ("int8", 2, 24, 8, 128, 16, [333, 1000], 32),
    ("int4", 3, 16, 2, 128, 32, [129, 700, 2], 64),
    ("int8", 2, 64, 8, 128, 16, [1500, 40], 32),
    ("int4", 2, 32, 8, 64, 16, [600, 31], 32),
    ("int8", 2, 40, 8, 128, 64, [520, 77], 64),
    ("int4", 2, 64, 8, 128, 16, [1500, 40], 32),
    ("int4", 2, 12, 4, 128, 32, [400, 77], 32),
    ("int4", 2, 16, 2, 64, 16, [400, 77], 32),
    ("int4", 2, 8, 2, 64, 16, [300, 45], 16),
    ("int8", 2, 40, 8, 64, 32, [300, 90], 16),
]


def case_id(c):
    return f"{c[0]}-G{c[2] // c[3]}-D{c[4]}-BS{c[5]}" + (f"-g{c[7]}" if len(c) > 7 else "")


@pytest.mark.parametrize("case", CASES, ids=case_id)
@pytest.mark.parametrize("kernel", [kvq.KERNEL_MMA, kvq.KERNEL_SIMT])
@pytest.mark.parametrize("partition", [0, 64, 256])
def test_decode_small(case, kernel, partition):
    fmt, B, Hq, Hkv, D, BS, ctx = case[:7]
    group = case[7] if len(case) > 7 else 0
    if kernel == kvq.KERNEL_SIMT and (Hq // Hkv > 4 or fmt == "int4"):
        pytest.skip("CUDA-core kernel covers 8-bit codes and group size <= 4")
    dw = small(fmt, B, Hq, Hkv, D, BS, ctx, seed=len(ctx) + D, group=group)
    kvq.set_decode_kernel(kernel)
    out = dw.decode(partition_size=partition)
    torch.cuda.synchronize()
    assert kvq.device_error_check()[0] == 0
    ref = dw.oracle_decode(list(range(B)))
    e = rel_err(out.float().cpu().numpy(), ref)
    assert e <= ATOL_REL, e


SPLIT_CASES = [
    # fmt, B, Hq, Hkv, D, BS, contexts, channels per scale
    ("e4m3", 4, 8, 2, 128, 16, [3000, 1500, 64, 4097], 0),
    ("e5m2", 4, 32, 8, 128, 16, [3000, 1500, 64, 4097], 0),
    ("int8", 4, 8, 8, 128, 64, [3000, 1500, 64, 4097], 0),
    ("int8", 4, 16, 2, 128, 16, [3000, 1500, 64, 4097], 0),
    ("int8", 4, 16, 4, 128, 16, [3000, 1500, 64, 4097], 0),
    ("int4", 4, 8, 8, 128, 64, [3000, 1500, 64, 4097], 0),
    ("int4", 4, 16, 2, 128, 16, [3000, 1500, 64, 4097], 0),
    ("int8", 4, 8, 4, 128, 16, [3000, 1500, 64, 4097], 32),
    ("int4", 4, 8, 8, 128, 16, [3000, 1500, 64, 4097], 32),
    ("int8", 4, 32, 4, 128, 16, [3000, 1500, 64, 4097], 32),
    ("int8", 4, 20, 4, 128, 16, [3000, 1500, 64, 4097], 64),
    ("int4", 4, 32, 4, 128, 16, [3000, 1500, 64, 4097], 32),
    ("int8", 4, 16, 2, 64, 16, [3000, 1500, 64, 4097], 16),
]


def f16_ulp(x: torch.Tensor) -> torch.Tensor:
    """Spacing of fp16 values at |x| (2^-24 below the normal range)."""
    return torch.exp2(torch.floor(torch.log2(x.abs().clamp(min=2.0 ** -14))) - 10)


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: f"{c[0]}-G{c[2] // c[3]}-BS{c[5]}-g{c[7]}")
def test_kernels_and_partitions_agree(case):
    """Split invariance: the result does not depend on how a context is cut
    into chunks, nor on the consumer (tensor-core / CUDA-core) -- the fp32
    results agree within 1e-5 of max(1, |o|).  The library returns them
    rounded to fp16, one rounding each, and two values within d of each other
    round to fp16 values at most d + one fp16 ulp apart; so the fp16 outputs
    must agree within one ulp (of the larger) plus 1e-5 * max(1, |o|)."""
    fmt, B, Hq, Hkv, D, BS, ctx, group = case
    dw = small(fmt, B, Hq, Hkv, D, BS, ctx, seed=5, group=group)
    kernels = [kvq.KERNEL_MMA]
    if fmt != "int4" and Hq // Hkv <= 4:
        kernels.append(kvq.KERNEL_SIMT)
    outs = []
    for kernel in kernels:
        kvq.set_decode_kernel(kernel)
        for p in (0, 64, 512, 4160):
            outs.append(dw.decode(partition_size=p).float())
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)
    for o in outs[1:]:
        mag = torch.maximum(o.abs(), outs[0].abs())
        excess = (((o - outs[0]).abs() - f16_ulp(mag)) / mag.clamp(min=1.0)).max().item()
        assert excess <= 1e-5, excess


@pytest.mark.parametrize("fmt,group", [("int8", 0), ("int4", 0), ("int8", 32), ("int4", 64)])
def test_long_chunks_with_outlier_rows(fmt, group):
    """INT8 / INT4 rows holding a x20 outlier channel have scales ~19x the
    Gaussian rows': the longest chunks the library forms (one 16384-token
    chunk here, partition 16384; and the automatic choice) stay within the
    tolerance."""
    dw = small(fmt, 2, 16, 4, 128, 16, [16384, 9000], seed=21, group=group)
    ref = dw.oracle_decode([0, 1])
    for p in (0, 16384):
        out = dw.decode(partition_size=p)
        torch.cuda.synchronize()
        assert kvq.device_error_check()[0] == 0
        e = rel_err(out.float().cpu().numpy(), ref)
        assert e <= ATOL_REL, (p, e)


def test_edge_contexts_zero_one_and_max():
    dw = small("e5m2", 4, 4, 2, 128, 16, [0, 1, 8192, 15], seed=9)
    out = dw.decode().float().cpu().numpy()
    assert not out[0].any()
    ref = dw.oracle_decode([1, 2, 3])
    assert rel_err(out[1:], ref) <= ATOL_REL
    # context 1: the output is the single V row (times the scale, here 1.0)
    assert np.abs(out[1] - ref[0]).max() <= 1e-3


def test_nan_codes_past_the_context_do_not_leak():
    """Rows of the last block past the context hold NaN codes; they must not reach
    the output."""
    wl = W.Workload("nan", 2, 4, 2, 128, 16, "e4m3", 40, "amax", seed=3)
    lay = W.Layout(wl, torch.tensor([37, 40], dtype=torch.int32))
    dev = torch.device("cuda")
    cache = kvq.KVCache(lay.num_blocks, 2, 16, 128, "e4m3", dev, fill=0x7F)
    k, v = W.kv_tokens(wl, 0, 40, dev)
    slots = lay.slots(0, 40).to(dev)
    kvq.append(k, v, cache, slots)
    q = W.query(wl, dev)
    out = kvq.decode_attention(q, cache, lay.block_tables.to(dev), lay.context_lens.to(dev), 40)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    oc = oracle.Cache(lay.num_blocks, 2, 16, 128, oracle.E4M3, k_codes=cache.k_codes.cpu().numpy(),
                      v_codes=cache.v_codes.cpu().numpy())
    ref = oracle.decode_attention(q.cpu().numpy(), oc, lay.block_tables.numpy(), lay.context_lens.numpy(), None)
    assert rel_err(o, ref) <= ATOL_REL


@pytest.mark.parametrize("fmt,group,hq", [("int8", 0, 4), ("int4", 0, 4), ("int4", 32, 4), ("int8", 32, 16),
                                          ("int8", 64, 16), ("int4", 32, 16), ("int4", 64, 16)])
def test_nan_scales_past_the_context_do_not_leak(fmt, group, hq):
    """Scale slots of rows past the context that were never written hold NaN
    (the caller's memory is not cleared): the masked tokens' weights stay 0.
    Sixteen q-heads over two kv-heads with groups take the grouped consumer."""
    wl = W.Workload("nans", 3, hq, 2, 128, 16, fmt, 40, "row", seed=4, quant_group=group)
    ctx = torch.tensor([37, 40, 17], dtype=torch.int32)
    lay = W.Layout(wl, ctx)
    dev = torch.device("cuda")
    cache = kvq.KVCache(lay.num_blocks, 2, 16, 128, fmt, dev, fill=0x77, group_size=group)
    cache.k_scales.fill_(float("nan"))
    cache.v_scales.fill_(float("nan"))
    k, v = W.kv_tokens(wl, 0, 40, dev)
    slots = lay.slots(0, 40).to(dev)          # -1 past each sequence's context
    kvq.append(k, v, cache, slots)
    q = W.query(wl, dev)
    for kernel in (kvq.KERNEL_MMA, kvq.KERNEL_SIMT) if fmt == "int8" and hq <= 8 else (kvq.KERNEL_MMA,):
        kvq.set_decode_kernel(kernel)
        out = kvq.decode_attention(q, cache, lay.block_tables.to(dev), ctx.to(dev), 40)
        o = out.float().cpu().numpy()
        assert np.isfinite(o).all(), kernel
        oc = oracle.Cache(lay.num_blocks, 2, 16, 128, oracle.FORMATS[fmt], k_codes=cache.k_codes.cpu().numpy(),
                          v_codes=cache.v_codes.cpu().numpy(), k_scales=cache.k_scales.cpu().numpy(),
                          v_scales=cache.v_scales.cpu().numpy(), group=group)
        ref = oracle.decode_attention(q.cpu().numpy(), oc, lay.block_tables.numpy(), ctx.numpy(), None)
        assert rel_err(o, ref) <= ATOL_REL
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)


def test_bad_block_id_is_reported_without_fault():
    dw = small("e4m3", 2, 4, 4, 128, 16, [64, 64], seed=1)
    bt = dw.block_tables.clone()
    bt[1, 2] = 10 ** 6
    out = kvq.decode_attention(dw.q, dw.cache, bt, dw.context_lens, 64, dw.scale)
    st, detail = kvq.device_error_check()
    assert st == 4 and detail == 10 ** 6
    ref = dw.oracle_decode([0])
    assert rel_err(out[:1].float().cpu().numpy(), ref) <= ATOL_REL   # sequence 0 is untouched
    assert kvq.device_error_check()[0] == 0


def test_workspace_too_small_and_empty_batch():
    dw = small("e4m3", 2, 4, 4, 128, 16, [2000, 100], seed=2)
    need = kvq.workspace_size(2, 4, 4, 128, 2000, 256)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as ei:
        kvq.decode_attention(dw.q, dw.cache, dw.block_tables, dw.context_lens, 2000, dw.scale, workspace=ws,
                             partition_size=256)
    assert ei.value.status == 3
    q0 = dw.q[:0]
    out = kvq.decode_attention(q0, dw.cache, dw.block_tables[:0], dw.context_lens[:0], 2000, dw.scale)
    assert out.shape == (0, 4, 128)


@pytest.mark.parametrize("name,seqs", [("tiny", [0]), ("llama2-7b", [0, 13, 31]),
                                       ("llama3-8b", [0, 21, 40, 63]),
                                       ("llama2-13b-int8", [0, 77, 127]),
                                       ("llama2-13b-int4", [0, 64, 127]),
                                       ("llama2-13b-int4-g32", [0, 50, 127]),
                                       ("llama3-70b", [0, 255]),
                                       ("llama3-70b-int8-g32", [0, 131, 255]),
                                       ("llama3-70b-int4-g32", [0, 97, 255])])
def test_decode_workload_sampled(name, seqs):
    wl = W.WORKLOADS[name]
    dw = DeviceWorkload(wl)
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)
    out = dw.decode()
    torch.cuda.synchronize()
    assert kvq.device_error_check()[0] == 0
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    ref = dw.oracle_decode(seqs)
    e = rel_err(o[seqs], ref)
    assert e <= ATOL_REL, e
    # the sample covers the shortest and longest sequences of ragged workloads
    if not isinstance(wl.ctx, int):
        cl = dw.lay.context_lens
        extra = [int(torch.argmin(cl)), int(torch.argmax(cl))]
        assert rel_err(o[extra], dw.oracle_decode(extra)) <= ATOL_REL
