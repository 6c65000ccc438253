"""GPU parity of the decode step that quantizes each sequence's newest K/V row
into the cache in the same launch (kvq_decode_attention_append): cache bytes,
INT8 / INT4 row scales and outputs bit-identical to kvq_append followed by
kvq_decode_attention, and the output within the oracle tolerance on the cache
the fused call left behind."""
import numpy as np
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
from fp8_int8_quantized_gb300 import workloads as W
from tests.gpu_util import ATOL_REL, DeviceWorkload, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.build()
    torch.cuda.init()
    yield
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)


def small(fmt, B, Hq, Hkv, D, BS, ctx, seed, group=0):
    wl = W.Workload(f"f-{fmt}", B, Hq, Hkv, D, BS, fmt, max(max(ctx), 1),
                    "amax" if fmt == "e4m3" else ("row" if fmt in ("int8", "int4") else "one"), outliers=True,
                    seed=seed, quant_group=group)
    return DeviceWorkload(wl, chunk_tokens=1 << 16, ctx=torch.tensor(ctx, dtype=torch.int32))


def clone(c: kvq.KVCache) -> kvq.KVCache:
    n = kvq.KVCache(c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim, c.fmt, c.k_codes.device,
                    group_size=c.group_size)
    n.k_codes.copy_(c.k_codes)
    n.v_codes.copy_(c.v_codes)
    if c.k_scales is not None:
        n.k_scales.copy_(c.k_scales)
        n.v_scales.copy_(c.v_scales)
    return n


def newest_slots(dw, block_tables):
    bs = dw.wl.block_size
    out = []
    for b, n in enumerate(dw.lay.context_lens.tolist()):
        out.append(-1 if n == 0 else int(block_tables[b, (n - 1) // bs]) * bs + (n - 1) % bs)
    return torch.tensor(out, dtype=torch.int64)


def both_paths(dw, k_new, v_new, block_tables, partition):
    """(cache, out) of append-then-decode and of the fused call, from the same start."""
    c1, c2 = clone(dw.cache), clone(dw.cache)
    slots = newest_slots(dw, block_tables.cpu()).to(dw.device)
    kvq.append(k_new, v_new, c1, slots, dw.scale)
    o1 = kvq.decode_attention(dw.q, c1, block_tables, dw.context_lens, dw.lay.max_context_len, dw.scale,
                              partition_size=partition)
    torch.cuda.synchronize()
    st1 = kvq.device_error_check()
    o2 = kvq.decode_attention_append(dw.q, k_new, v_new, c2, block_tables, dw.context_lens,
                                     dw.lay.max_context_len, dw.scale, partition_size=partition)
    torch.cuda.synchronize()
    st2 = kvq.device_error_check()
    return (c1, o1, st1), (c2, o2, st2)


def assert_same_cache(c1, c2):
    assert torch.equal(c1.k_codes, c2.k_codes)
    assert torch.equal(c1.v_codes, c2.v_codes)
    if c1.k_scales is not None:
        assert torch.equal(c1.k_scales.view(torch.int32), c2.k_scales.view(torch.int32))
        assert torch.equal(c1.v_scales.view(torch.int32), c2.v_scales.view(torch.int32))


CASES = [
    # fmt, B, Hq, Hkv, D, BS, contexts (0, 1 and box / tile / block edges included)
    ("e4m3", 6, 4, 4, 64, 16, [128, 1, 77, 0, 16, 17]),
    ("e4m3", 4, 8, 1, 128, 16, [300, 32, 33, 2]),
    ("e5m2", 4, 32, 8, 128, 16, [1000, 512, 31, 64]),
    ("e5m2", 3, 6, 3, 64, 32, [95, 400, 15]),
    ("int8", 4, 4, 4, 128, 64, [640, 65, 1, 48]),
    ("int8", 3, 8, 2, 64, 64, [129, 0, 256]),
    ("e4m3", 2, 16, 2, 128, 32, [2050, 700]),
    ("int4", 4, 4, 4, 128, 64, [640, 65, 1, 48]),
    ("int4", 3, 8, 2, 64, 16, [129, 0, 256]),
    # group quantization (last field: channels per scale)
    ("int8", 4, 4, 2, 128, 32, [500, 33, 1, 64], 32),
    ("int4", 4, 4, 4, 128, 64, [640, 65, 1, 48], 32),
    ("int4", 3, 8, 2, 64, 16, [129, 0, 256], 32),
    ("int8", 3, 3, 3, 64, 16, [200, 45, 16], 16),
    ("int8", 3, 16, 2, 128, 32, [500, 1, 64], 32),
    ("int8", 3, 40, 8, 128, 16, [300, 1, 77], 64),
    ("int4", 2, 8, 1, 64, 16, [129, 48], 16),
    ("int4", 3, 32, 4, 128, 16, [300, 1, 77], 32),
    ("int4", 3, 16, 2, 64, 32, [129, 0, 64], 32),
]


def case_id(c):
    return f"{c[0]}-G{c[2] // c[3]}-D{c[4]}-BS{c[5]}" + (f"-g{c[7]}" if len(c) > 7 else "")


@pytest.mark.parametrize("case", CASES, ids=case_id)
@pytest.mark.parametrize("kernel", [kvq.KERNEL_MMA, kvq.KERNEL_SIMT])
@pytest.mark.parametrize("partition", [0, 64])
def test_fused_equals_append_then_decode(case, kernel, partition):
    fmt, B, Hq, Hkv, D, BS, ctx = case[:7]
    group = case[7] if len(case) > 7 else 0
    if kernel == kvq.KERNEL_SIMT and (Hq // Hkv > 4 or fmt == "int4"):
        pytest.skip("CUDA-core kernel covers 8-bit codes and group size <= 4")
    dw = small(fmt, B, Hq, Hkv, D, BS, ctx, seed=len(ctx) * 31 + D, group=group)
    kvq.set_decode_kernel(kernel)
    g = torch.Generator(device="cpu").manual_seed(B * 100 + D)
    k_new = (torch.randn((B, Hkv, D), generator=g) * 2).to(torch.float16).to(dw.device)
    v_new = (torch.randn((B, Hkv, D), generator=g) * 2).to(torch.float16).to(dw.device)
    if fmt in ("int8", "int4"):
        k_new[0, 0] = 0  # an all-zero row: scale 0, codes 0
    (c1, o1, st1), (c2, o2, st2) = both_paths(dw, k_new, v_new, dw.block_tables, partition)
    assert st1[0] == 0 and st2[0] == 0
    assert_same_cache(c1, c2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    dw.cache = c2
    ref = dw.oracle_decode(list(range(B)))
    e = rel_err(o2.float().cpu().numpy(), ref)
    assert e <= ATOL_REL, e


def test_fused_grouped_int4_large_batch():
    """INT4 with four scale groups at G = 8 runs 16-warp CTAs while their
    shared memory fits.  It grows with the batch (the context-length scan):
    a fused call over 3400 sequences takes 4-warp CTAs instead, the plain
    decode of the same batch still the 16-warp ones.  The caches are
    identical, and both outputs match the oracle on sampled sequences (the
    two grids split the contexts differently, so the outputs may differ in
    their last bits)."""
    B = 3400
    ctx = [1 + (i * 37) % 96 for i in range(B)]
    dw = small("int4", B, 8, 1, 128, 16, ctx, seed=11, group=32)
    g = torch.Generator(device="cpu").manual_seed(77)
    k_new = (torch.randn((B, 1, 128), generator=g) * 2).to(torch.float16).to(dw.device)
    v_new = (torch.randn((B, 1, 128), generator=g) * 2).to(torch.float16).to(dw.device)
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)
    (c1, o1, st1), (c2, o2, st2) = both_paths(dw, k_new, v_new, dw.block_tables, 0)
    assert st1[0] == 0 and st2[0] == 0
    assert_same_cache(c1, c2)
    dw.cache = c2
    seqs = [0, 1, 95, 1700, B - 1]
    ref = dw.oracle_decode(seqs)
    for o in (o1, o2):
        assert rel_err(o[seqs].float().cpu().numpy(), ref) <= ATOL_REL
    assert rel_err(o2.float().cpu().numpy(), o1.float().cpu().numpy().astype(np.float64)) <= ATOL_REL


@pytest.mark.parametrize("fmt,group", [("e4m3", 0), ("e5m2", 0), ("int8", 0), ("int4", 0), ("int8", 32),
                                       ("int4", 32), ("int4", 64)])
def test_fused_at_the_batch_limit(fmt, group):
    """4096 sequences (the library's batch limit) of 8 q-heads over one
    kv-head: every consumer's shared memory, which grows with the batch (the
    context-length scan), still fits or falls back to a smaller CTA; the fused
    and the two-call paths leave the same cache, and sampled sequences match
    the oracle."""
    B = 4096
    ctx = [1 + (i * 13) % 40 for i in range(B)]
    dw = small(fmt, B, 8, 1, 128, 16, ctx, seed=21, group=group)
    g = torch.Generator(device="cpu").manual_seed(5)
    k_new = (torch.randn((B, 1, 128), generator=g) * 2).to(torch.float16).to(dw.device)
    v_new = (torch.randn((B, 1, 128), generator=g) * 2).to(torch.float16).to(dw.device)
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)
    (c1, o1, st1), (c2, o2, st2) = both_paths(dw, k_new, v_new, dw.block_tables, 0)
    assert st1[0] == 0 and st2[0] == 0
    assert_same_cache(c1, c2)
    dw.cache = c2
    seqs = [0, 1, 2047, B - 1]
    ref = dw.oracle_decode(seqs)
    for o in (o1, o2):
        assert rel_err(o[seqs].float().cpu().numpy(), ref) <= ATOL_REL


def test_fused_bad_block_id_is_reported_and_not_written():
    dw = small("e4m3", 3, 4, 2, 128, 16, [40, 100, 7], seed=5)
    bt = dw.block_tables.clone()
    bt[1, 99 // 16] = 10 ** 6  # the block that would receive sequence 1's newest row
    k_new = torch.randn((3, 2, 128), device=dw.device).to(torch.float16)
    v_new = torch.randn((3, 2, 128), device=dw.device).to(torch.float16)
    (c1, o1, st1), (c2, o2, st2) = both_paths(dw, k_new, v_new, bt, 0)
    assert st1[0] == 4 and st2[0] == 4  # KVQ_ERR_OUT_OF_RANGE on both paths
    assert_same_cache(c1, c2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("name", ["llama2-7b", "llama3-8b", "llama2-13b-int8", "llama2-13b-int4",
                                  "llama2-13b-int4-g32"])
def test_fused_full_size_sampled(name):
    """The benchmark's fused step on a full decode workload: the cache it leaves
    equals kvq_append of the same rows, and sampled sequences' outputs match
    the oracle on that cache."""
    wl = W.WORKLOADS[name]
    kvq.set_decode_kernel(kvq.KERNEL_AUTO)
    dw = DeviceWorkload(wl)
    cl = dw.lay.context_lens
    k_new, v_new = [], []
    for b in range(wl.batch):
        n = int(cl[b])
        k, v = W.kv_tokens(wl, n - 1, n, dw.device, seqs=[b])
        k_new.append(k)
        v_new.append(v)
    k_new, v_new = torch.cat(k_new), torch.cat(v_new)
    expect = clone(dw.cache)
    kvq.append(k_new, v_new, expect, newest_slots(dw, dw.lay.block_tables).to(dw.device), dw.scale)
    out = kvq.decode_attention_append(dw.q, k_new, v_new, dw.cache, dw.block_tables, dw.context_lens,
                                      dw.lay.max_context_len, dw.scale)
    torch.cuda.synchronize()
    assert kvq.device_error_check()[0] == 0
    assert_same_cache(expect, dw.cache)
    del expect
    seqs = sorted({0, wl.batch - 1, wl.batch // 2, 7 % wl.batch})
    ref = dw.oracle_decode(seqs)
    e = rel_err(out[seqs].float().cpu().numpy(), ref)
    assert e <= ATOL_REL, e
