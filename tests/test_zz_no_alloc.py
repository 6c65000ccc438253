"""The scratch-free decode entry point, for callers that cannot allocate device
memory (plugin hosts that hand an operator only its inputs and outputs, serving
loops that must not allocate once running).

kvq_decode_attention_static_scratch is called directly through the C ABI and
its output is compared with kvq_decode_attention's (caller-provided workspace)
on the same inputs, within the decode tolerance of the parity tests, on two
calls in a row.  The second call changes the layout of what goes into the
shared array -- other queries, shorter contexts, one sequence with context 0,
and a larger partition (fewer chunks, so every partial slot and the (max, sum)
pairs sit at other offsets) -- so it reads across what the first call left
there, and shows that none of it leaks into its result.
This file is collected last; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
from fp8_int8_quantized_gb300 import workloads as W
from tests.gpu_util import ATOL_REL, DeviceWorkload

pytestmark = pytest.mark.gpu


def call_static(lib, dw, q, ctx, out, partition):
    d = dw.cache.desc()
    return lib.kvq_decode_attention_static_scratch(
        q.data_ptr(), ctypes.byref(d), dw.block_tables.data_ptr(), dw.block_tables.shape[1],
        ctx.data_ptr(), q.shape[0], q.shape[1], dw.lay.max_context_len,
        None if dw.scale is None else dw.scale.data_ptr(), dw.cache.fmt, ctypes.c_float(0.0),
        out.data_ptr(), partition, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_matches_workspace_entry_point():
    kvq.build()
    lib = kvq.lib()
    assert lib.kvq_static_scratch_bytes() == 64 << 20
    wl = W.Workload("no-alloc", 8, 32, 8, 128, 16, "e4m3", (300, 6000), "amax", outliers=True, seed=77)
    dw = DeviceWorkload(wl)
    shorter = torch.clamp(dw.context_lens // 3, min=1)
    shorter[5] = 0
    # call 1: many 64-token partitions over the full contexts; call 2: other
    # queries, shorter contexts (one empty) and 512-token partitions
    calls = [(64, dw.context_lens), (512, shorter)]
    for call, (partition, ctx) in enumerate(calls):
        assert kvq.workspace_size(8, 32, 8, 128, dw.lay.max_context_len, partition) > 0
        q = W.query(wl, "cuda", step=call)
        ref = kvq.decode_attention(q, dw.cache, dw.block_tables, ctx, dw.lay.max_context_len,
                                   dw.scale, partition_size=partition)
        out = torch.full_like(q, float("nan"))
        assert call_static(lib, dw, q, ctx, out, partition) == 0
        torch.cuda.synchronize()
        a, b = out.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(a).all()
        err = (np.abs(a - b) / np.maximum(1.0, np.abs(b))).max()
        assert err <= ATOL_REL, (call, err)
    assert not out[5].any()                       # context 0: zeros, whatever the array held
    assert kvq.device_error_check()[0] == 0


def test_static_scratch_rejects_sizes_beyond_the_array():
    lib = kvq.lib()
    wl = W.Workload("no-alloc-small", 2, 4, 4, 128, 16, "e4m3", 64, "amax", seed=3)
    dw = DeviceWorkload(wl)
    out = torch.zeros_like(dw.q)
    d = dw.cache.desc()
    # 64 sequences x 32 q-heads (8 per kv-head) x 128 partitions of 64 tokens:
    # far more partials than 64 MiB; the arguments are otherwise good (the
    # block tables would span 8192 tokens), so the size limit is the answer
    need = kvq.workspace_size(64, 32, 4, 128, 8192, 64)
    assert need > lib.kvq_static_scratch_bytes()
    st = lib.kvq_decode_attention_static_scratch(
        dw.q.data_ptr(), ctypes.byref(d), dw.block_tables.data_ptr(), 8192 // 16,
        dw.context_lens.data_ptr(), 64, 32, 8192, None, dw.cache.fmt, ctypes.c_float(0.0),
        out.data_ptr(), 64, None)
    assert st == 7                    # KVQ_ERR_SCRATCH_LIMIT, nothing launched
    torch.cuda.synchronize()
    assert not out.any()
