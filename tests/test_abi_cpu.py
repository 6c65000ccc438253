"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point include/kvq.h declares, with the declared status codes."""
import os
import re

import pytest

import fp8_int8_quantized_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kvq.build()
    return kvq.lib()


def declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared() == sorted(kvq.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.kvq_abi_version() == 1
    for code in range(8):
        assert kvq.status_string(code)
    assert kvq.status_string(99) == "unknown status"


def test_status_codes_match_header():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    for code, name in kvq.STATUS.items():
        assert re.search(rf"\b{name}\s*=\s*{code}\b", src), name


def test_cache_struct_matches_header():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    body = re.search(r"typedef struct \{([^}]*)\} kvq_cache;", src).group(1)
    names = re.findall(r"\b(\w+);", body)
    assert names == [f[0] for f in kvq.KvqCacheDesc._fields_]


def test_group_sizes_checked_before_any_cuda_call(lib):
    import ctypes
    d8 = kvq.KvqCacheDesc(16, 16, 16, 16, 8, 16, 2, 128, kvq.INT8, 24)
    assert lib.kvq_append(16, 16, ctypes.byref(d8), 16, 4, None, kvq.INT8, None) == 1     # 24 does not divide
    d8.group_size = 16
    assert lib.kvq_append(16, 16, ctypes.byref(d8), 16, 4, None, kvq.INT8, None) == 1     # 8 groups
    f8 = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 128, kvq.E4M3, 32)
    assert lib.kvq_append(16, 16, ctypes.byref(f8), 16, 4, None, kvq.E4M3, None) == 1     # FP8 has no groups
    d4 = kvq.KvqCacheDesc(16, 16, 16, 16, 8, 16, 2, 128, kvq.INT4, 40)
    assert lib.kvq_decode_attention(16, ctypes.byref(d4), 16, 4, 16, 2, 8, 64, None, kvq.INT4, 0.0,
                                    16, None, 0, 0, None) == 1                             # 40 does not divide
    d4.group_size = 48
    assert lib.kvq_prefill_attention(16, ctypes.byref(d4), 16, 4, 16, 16, 2, 4, 4, 4, None, kvq.INT4,
                                     0.0, 16, None) == 1                                   # 48 does not divide


def test_decode_kernel_knob(lib):
    prev = lib.kvq_set_decode_kernel(1)
    assert lib.kvq_set_decode_kernel(prev) == 1
    assert lib.kvq_set_decode_kernel(7) == -1


def test_invalid_args_rejected_before_any_cuda_call(lib):
    import ctypes
    d = kvq.KvqCacheDesc(None, None, None, None, 8, 16, 2, 128, kvq.E4M3)
    assert lib.kvq_append(None, None, ctypes.byref(d), None, 4, None, kvq.E4M3, None) == 1
    d = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 96, kvq.E4M3)
    assert lib.kvq_append(16, 16, ctypes.byref(d), 16, 4, None, kvq.E4M3, None) == 2       # head_dim 96
    d = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 128, kvq.E4M3)
    assert lib.kvq_append(16, 16, ctypes.byref(d), 16, 4, None, kvq.E5M2, None) == 1       # fmt mismatch
    d8 = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 128, kvq.INT8)
    assert lib.kvq_append(16, 16, ctypes.byref(d8), 16, 4, None, kvq.INT8, None) == 1      # no scales
    assert lib.kvq_decode_attention(16, ctypes.byref(d), 16, 4, 16, 2, 3, 64, None, kvq.E4M3, 0.0,
                                    16, None, 0, 0, None) == 1                              # 3 % 2 != 0
    assert lib.kvq_decode_attention(16, ctypes.byref(d), 16, 4, 16, 2, 32, 64, None, kvq.E4M3, 0.0,
                                    16, None, 0, 0, None) == 2                              # group 16
    assert lib.kvq_decode_attention(16, ctypes.byref(d), 16, 2, 16, 2, 4, 64, None, kvq.E4M3, 0.0,
                                    16, None, 0, 0, None) == 1                              # table too short
    assert lib.kvq_decode_attention(16, ctypes.byref(d), 16, 4, 16, 2, 4, 64, None, kvq.E4M3, 0.0,
                                    16, None, 0, 100, None) == 1                            # partition % 64
    assert lib.kvq_dequant(ctypes.byref(d), None, 3, None, kvq.E4M3, None, None, None) == 1
    assert lib.kvq_decode_attention_append(16, None, 16, ctypes.byref(d), 16, 4, 16, 2, 4, 64, None, kvq.E4M3,
                                           0.0, 16, None, 0, 0, None) == 1                  # no k_new
    assert lib.kvq_decode_attention_append(16, 24, 16, ctypes.byref(d), 16, 4, 16, 2, 4, 64, None, kvq.E4M3,
                                           0.0, 16, None, 0, 0, None) == 1                  # misaligned k_new


def test_more_decode_checks_before_any_cuda_call(lib):
    import ctypes
    d = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 128, kvq.E4M3)

    def dec(q=16, cache=d, ctx=64, batch=2, nq=4, sm=0.0, out=16, ws=256, ws_bytes=1 << 30, part=64, fmt=kvq.E4M3):
        return lib.kvq_decode_attention(q, ctypes.byref(cache), 16, 4, 16, batch, nq, ctx, None, fmt, sm,
                                        out, ws, ws_bytes, part, None)

    assert dec(q=8) == 1                                   # q not 16-byte aligned
    assert dec(out=24) == 1                                # out not 16-byte aligned
    assert dec(sm=float("nan")) == 1
    assert dec(sm=float("inf")) == 1
    assert dec(sm=-1.0) == 1
    assert dec(batch=-1) == 1
    assert dec(ctx=-5) == 1
    assert dec(batch=5000) == 2                            # the context-length scan holds 4096
    assert dec(batch=0) == 0                               # nothing to do, nothing launched
    assert dec(ws=None) == 3                               # no workspace
    assert dec(ws=128) == 3                                # workspace not 256-byte aligned
    assert dec(ws_bytes=64) == 3                           # workspace too small
    bs8 = kvq.KvqCacheDesc(16, 16, None, None, 8, 8, 2, 128, kvq.E4M3)
    assert dec(cache=bs8) == 2                             # block size 8
    huge = kvq.KvqCacheDesc(16, 16, None, None, 1 << 27, 16, 2, 128, kvq.E4M3)
    assert dec(cache=huge) == 2                            # TMA row coordinates are 32-bit
    i4 = kvq.KvqCacheDesc(16, 16, 16, 16, 8, 16, 2, 128, kvq.INT4)
    prev = lib.kvq_set_decode_kernel(kvq.KERNEL_SIMT)
    try:
        assert dec(cache=i4, fmt=kvq.INT4) == 2            # the CUDA-core kernel takes 8-bit codes only
        assert dec(nq=10) == 2                             # ... and at most 4 q-heads per kv-head
    finally:
        lib.kvq_set_decode_kernel(prev)


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.kvq_decode_workspace_size(0, 4, 2, 128, 64, 64) == 0
    assert lib.kvq_decode_workspace_size(2, 3, 2, 128, 64, 64) == 0       # 3 % 2 != 0
    assert lib.kvq_decode_workspace_size(2, 4, 2, 128, -1, 64) == 0
    assert lib.kvq_decode_workspace_size(2, 4, 2, 128, 64, 64) > 0
    # more context, more chunks: never smaller
    assert lib.kvq_decode_workspace_size(2, 4, 2, 128, 4096, 64) >= lib.kvq_decode_workspace_size(2, 4, 2, 128, 64, 64)


def test_prefill_append_dequant_checks_before_any_cuda_call(lib):
    import ctypes
    d = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 2, 128, kvq.E4M3)
    one = kvq.KvqCacheDesc(16, 16, None, None, 8, 16, 1, 128, kvq.E4M3)

    def pre(q=16, cache=d, batch=2, ntok=8, nq=4, maxq=4, sm=0.0, out=16, qs=16):
        return lib.kvq_prefill_attention(q, ctypes.byref(cache), 16, 4, 16, qs, batch, ntok, nq, maxq, None,
                                         kvq.E4M3, sm, out, None)

    assert pre(q=8) == 1                                   # q not 16-byte aligned
    assert pre(qs=None) == 1                               # no query_start
    assert pre(qs=18) == 1                                 # query_start not 4-byte aligned
    assert pre(sm=float("nan")) == 1
    assert pre(nq=3) == 1                                  # 3 q-heads over 2 kv-heads
    assert pre(ntok=-1) == 1
    assert pre(cache=one, nq=256) == 2                     # 256 q-heads per kv-head: above the 128-row tile
    assert pre(ntok=1 << 31) == 2                          # query_start entries are int32
    assert pre(batch=0) == 0 and pre(maxq=0) == 0 and pre(ntok=0) == 0   # nothing to do
    # append: negative or zero token counts, misaligned slot mapping
    assert lib.kvq_append(16, 16, ctypes.byref(d), 16, -1, None, kvq.E4M3, None) == 1
    assert lib.kvq_append(16, 16, ctypes.byref(d), 16, 0, None, kvq.E4M3, None) == 0
    assert lib.kvq_append(16, 16, ctypes.byref(d), 12, 4, None, kvq.E4M3, None) == 1
    assert lib.kvq_append(16, 16, ctypes.byref(d), 16, 4, 2, kvq.E4M3, None) == 1      # scale not 4-byte aligned
    # dequant: negative count, missing outputs
    assert lib.kvq_dequant(ctypes.byref(d), 16, -1, None, kvq.E4M3, 16, 16, None) == 1
    assert lib.kvq_dequant(ctypes.byref(d), 16, 0, None, kvq.E4M3, 16, 16, None) == 0


def test_static_scratch_checks_arguments_before_its_size_limit(lib):
    """The no-workspace decode gives the statuses kvq_decode_attention gives for
    bad arguments (even where the sizes would also overflow its fixed array), and
    KVQ_ERR_SCRATCH_LIMIT only for good arguments that need more than the array;
    all of these before any CUDA call."""
    import ctypes
    d = kvq.KvqCacheDesc(16, 16, None, None, 1 << 16, 16, 4, 128, kvq.E4M3)
    d256 = kvq.KvqCacheDesc(16, 16, None, None, 1 << 16, 16, 4, 256, kvq.E4M3)

    def st(cache=d, batch=64, nq=32, ctx=8192, part=64, q=16):
        return lib.kvq_decode_attention_static_scratch(q, ctypes.byref(cache), 16, 1 << 12, 16, batch, nq, ctx,
                                                       None, kvq.E4M3, 0.0, 16, part, None)

    assert lib.kvq_decode_workspace_size(64, 32, 4, 128, 8192, 64) > lib.kvq_static_scratch_bytes()
    assert st() == 7                                       # good arguments, more than the array holds
    assert st(part=32) == 1                                # partition not a multiple of 64
    assert st(batch=5000) == 2                             # above the context-length scan's 4096
    assert st(cache=d256) == 2                             # head_dim 256
    assert st(q=8) == 1                                    # misaligned q
    assert st(batch=0) == 0                                # nothing to do, nothing launched


def test_encode_checks_before_any_cuda_call(lib):
    assert lib.kvq_encode_fp8(16, 16, 32, kvq.INT8, None) == 1        # not an FP8 format
    assert lib.kvq_encode_fp8(16, 16, -1, kvq.E4M3, None) == 1        # negative count
    assert lib.kvq_encode_fp8(16, 24, 32, kvq.E5M2, None) == 1        # codes not 16-byte aligned
    assert lib.kvq_encode_fp8(None, 16, 32, kvq.E4M3, None) == 1
    assert lib.kvq_encode_fp8(None, None, 0, kvq.E4M3, None) == 0     # nothing to do
