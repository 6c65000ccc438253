"""GPU parity of chunked-prefill attention (kvq_prefill_attention) against the
fp64 CPU oracle on the same cache bytes: |o_gpu - o_ref| <= 2e-3 * max(1,
|o_ref|) per element.  Small cases span several 64-token KV tiles and 128-row
query tiles (odd and even counts of them: a CTA takes two), ragged tails,
whole-context chunks, one-query and empty chunks, every q-head group size class
(1, 2, 3, 4, 8, 16), both head sizes and INT8 / INT4 scale groups; the
workload-sized cases run the launch the benchmark times and check sampled
queries, each against the oracle's decode attention over its own prefix (the
definition of causal attention for one query)."""
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


def small(fmt, B, Hq, Hkv, D, BS, ctx, seed=0, group=0):
    wl = W.Workload(f"p-{fmt}", B, Hq, Hkv, D, BS, fmt, max(ctx),
                    "amax" if fmt == "e4m3" else ("row" if fmt in ("int8", "int4") else "one"),
                    outliers=True, seed=seed, quant_group=group)
    return DeviceWorkload(wl, chunk_tokens=1 << 16, ctx=torch.tensor(ctx, dtype=torch.int32))


def run_prefill(dw, chunk, step=0):
    n = torch.tensor(chunk, dtype=torch.int32)
    q, qs = W.prefill_queries(dw.wl, n, "cuda", step)
    out = kvq.prefill_attention(q, dw.cache, dw.block_tables, dw.context_lens, qs.cuda(),
                                int(n.max()) if n.numel() else 0, dw.scale)
    torch.cuda.synchronize()
    return q, qs, out


PCASES = [
    # fmt, B, Hq, Hkv, D, BS, contexts, chunk lengths
    ("e4m3", 2, 4, 4, 64, 16, [300, 77], [300, 77]),
    ("e4m3", 2, 8, 1, 128, 16, [520, 130], [200, 3]),
    ("e5m2", 3, 32, 8, 128, 16, [700, 256, 33], [129, 256, 1]),
    ("e5m2", 2, 6, 3, 64, 32, [400, 95], [95, 0]),
    ("int8", 2, 4, 4, 128, 64, [640, 65], [300, 65]),
    ("int8", 3, 8, 2, 64, 64, [129, 1, 256], [129, 1, 17]),
    ("e4m3", 1, 48, 16, 128, 32, [390], [390]),
    ("e4m3", 2, 16, 1, 128, 16, [260, 50], [40, 50]),
    ("int4", 2, 4, 4, 128, 64, [640, 65], [300, 65]),
    ("int4", 3, 8, 2, 64, 16, [129, 1, 256], [129, 1, 17]),
    ("int4", 1, 32, 8, 128, 32, [500], [200]),
    # scale groups (last field: channels per scale)
    ("int8", 2, 4, 4, 128, 64, [640, 65], [300, 65], 32),
    ("int8", 3, 8, 2, 64, 16, [129, 1, 256], [129, 1, 17], 16),
    ("int4", 2, 16, 2, 128, 16, [700, 64], [260, 64], 64),
    ("int4", 3, 4, 4, 64, 32, [300, 77, 1], [300, 10, 1], 16),
    ("int4", 1, 32, 8, 128, 32, [500], [200], 32),
]


def case_id(c):
    return f"{c[0]}-G{c[2] // c[3]}-D{c[4]}-BS{c[5]}" + (f"-g{c[8]}" if len(c) > 8 else "")


@pytest.mark.parametrize("case", PCASES, ids=case_id)
def test_prefill_small(case):
    fmt, B, Hq, Hkv, D, BS, ctx, chunk = case[:8]
    group = case[8] if len(case) > 8 else 0
    dw = small(fmt, B, Hq, Hkv, D, BS, ctx, seed=sum(ctx) + D, group=group)
    q, qs, out = run_prefill(dw, chunk)
    assert kvq.device_error_check()[0] == 0
    oc, bt, cl = dw.oracle_cache_for(list(range(B)))
    ref = oracle.prefill_attention(q.cpu().numpy(), oc, bt, cl, qs.numpy(), dw.scale_value)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    e = rel_err(o, ref)
    assert e <= ATOL_REL, e


def test_last_query_agrees_with_decode_kernel():
    """The last query of each chunk is a decode query: two independent kernels
    (tensor-memory MMAs here, mma.sync there) agree within a few fp16 ulps."""
    dw = small("e4m3", 3, 16, 2, 128, 16, [1000, 300, 129], seed=5)
    q, qs, out = run_prefill(dw, [64, 300, 1])
    last = torch.stack([q[int(qs[b + 1]) - 1] for b in range(3)])
    dec = kvq.decode_attention(last.contiguous(), dw.cache, dw.block_tables, dw.context_lens,
                               dw.lay.max_context_len, dw.scale)
    got = torch.stack([out[int(qs[b + 1]) - 1] for b in range(3)]).float()
    diff = (got - dec.float()).abs() / torch.clamp(dec.float().abs(), min=1.0)
    assert float(diff.max()) <= 2e-3


def test_empty_and_validation():
    dw = small("e4m3", 2, 8, 2, 64, 16, [40, 20], seed=9)
    q = torch.zeros((0, 8, 64), dtype=torch.float16, device="cuda")
    qs = torch.zeros(3, dtype=torch.int32, device="cuda")
    out = kvq.prefill_attention(q, dw.cache, dw.block_tables, dw.context_lens, qs, 0, dw.scale)
    assert out.shape == (0, 8, 64)
    # group size above 128 is not built
    with pytest.raises(kvq.KvqError) as ei:
        big = torch.zeros((1, 256 * 2, 64), dtype=torch.float16, device="cuda")
        kvq.prefill_attention(big, dw.cache, dw.block_tables, dw.context_lens, qs, 1, dw.scale)
    assert ei.value.status == 2
    # fmt mismatch
    with pytest.raises(kvq.KvqError):
        d = dw.cache._cdesc()
        st = kvq.lib().kvq_prefill_attention(q.data_ptr(), kvq.ctypes.byref(d), dw.block_tables.data_ptr(), 2,
                                             dw.context_lens.data_ptr(), qs.data_ptr(), 2, 1, 8, 1, None,
                                             kvq.E5M2, 0.0, q.data_ptr(), None)
        kvq._check(st, "kvq_prefill_attention")


def test_chunk_longer_than_context_is_reported_and_others_computed():
    dw = small("e5m2", 2, 4, 4, 64, 16, [40, 30], seed=13)
    n = torch.tensor([41, 30], dtype=torch.int32)            # sequence 0 claims more queries than tokens
    q, qs = W.prefill_queries(dw.wl, n, "cuda")
    out = torch.full_like(q, float("nan"))
    kvq.prefill_attention(q, dw.cache, dw.block_tables, dw.context_lens, qs.cuda(), 41, dw.scale, out=out)
    st, detail = kvq.device_error_check()
    assert st == 4 and detail == 0
    assert torch.isnan(out[:41].float()).all()              # left unwritten
    oc, bt, cl = dw.oracle_cache_for([1])
    ref = oracle.prefill_attention(q[41:].cpu().numpy(), oc, bt, cl, np.array([0, 30], np.int32), dw.scale_value)
    assert rel_err(out[41:].float().cpu().numpy(), ref) <= ATOL_REL


def test_bad_block_id_is_reported_without_fault():
    dw = small("e4m3", 1, 4, 4, 64, 16, [100], seed=17)
    bt = dw.block_tables.clone()
    bt[0, 2] = dw.cache.num_blocks + 5
    n = torch.tensor([100], dtype=torch.int32)
    q, qs = W.prefill_queries(dw.wl, n, "cuda")
    out = kvq.prefill_attention(q, dw.cache, bt, dw.context_lens, qs.cuda(), 100, dw.scale)
    st, detail = kvq.device_error_check()
    assert st == 4 and detail == dw.cache.num_blocks + 5
    assert torch.isfinite(out.float()).all()
    # queries before the bad block see only good blocks and stay exact
    oc, obt, cl = dw.oracle_cache_for([0])
    ref = oracle.prefill_attention(q[:32].cpu().numpy(), oc, obt, np.array([32], np.int32),
                                   np.array([0, 32], np.int32), dw.scale_value)
    assert rel_err(out[:32].float().cpu().numpy(), ref) <= ATOL_REL


@pytest.mark.parametrize("name,chunk,seqs", [("llama3-70b", 2048, [0, 255]),
                                             ("llama3-8b", 1024, [0, 33]),
                                             ("llama2-13b-int8", 512, [5]),
                                             ("llama2-13b-int4", 512, [7]),
                                             ("llama2-13b-int4-g32", 512, [9]),
                                             ("llama2-7b", 2048, [31])])
def test_prefill_workload_sampled(name, chunk, seqs):
    wl = W.WORKLOADS[name]
    dw = DeviceWorkload(wl)
    n = W.prefill_chunks(wl, dw.lay.context_lens, chunk)
    q, qs, out = run_prefill(dw, n.tolist())
    assert kvq.device_error_check()[0] == 0
    for b in seqs:
        nb, cb = int(n[b]), int(dw.lay.context_lens[b])
        oc, bt, cl = dw.oracle_cache_for([b])
        for i in sorted({0, 1, nb // 2, nb - 2, nb - 1}):
            if not 0 <= i < nb:
                continue
            row = int(qs[b]) + i
            pos = cb - nb + i
            ref = oracle.decode_attention(q[row:row + 1].cpu().numpy(), oc, bt, np.array([pos + 1], np.int32),
                                          dw.scale_value)
            o = out[row:row + 1].float().cpu().numpy()
            assert np.isfinite(o).all()
            e = rel_err(o, ref)
            assert e <= ATOL_REL, (b, i, e)


@pytest.mark.parametrize("fmt,scale", [("e4m3", -0.0123), ("e5m2", 3.0)])
def test_prefill_explicit_scale(fmt, scale):
    """A scale given by the caller, negative included (dequantization multiplies
    every code by it, so K and V both change sign)."""
    wl = W.Workload(f"s-{fmt}", 2, 8, 2, 128, 16, fmt, 300, "one", outliers=False, seed=23)
    lay = W.Layout(wl, torch.tensor([300, 140], dtype=torch.int32))
    cache = kvq.KVCache(lay.num_blocks, 2, 16, 128, fmt, "cuda", fill=0xA5)
    k, v = W.kv_tokens(wl, 0, 300, "cuda")
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    kvq.append(k, v, cache, lay.slots(0, 300).cuda(), sc)
    n = torch.tensor([160, 140], dtype=torch.int32)
    q, qs = W.prefill_queries(wl, n, "cuda")
    out = kvq.prefill_attention(q, cache, lay.block_tables.cuda(), lay.context_lens.cuda(), qs.cuda(), 160, sc)
    torch.cuda.synchronize()
    assert kvq.device_error_check()[0] == 0
    oc = oracle.Cache(lay.num_blocks, 2, 16, 128, {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}[fmt],
                      k_codes=cache.k_codes.cpu().numpy(), v_codes=cache.v_codes.cpu().numpy())
    ref = oracle.prefill_attention(q.cpu().numpy(), oc, lay.block_tables.numpy(), lay.context_lens.numpy(),
                                   qs.numpy(), float(np.float32(scale)))
    assert rel_err(out.float().cpu().numpy(), ref) <= ATOL_REL
