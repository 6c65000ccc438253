"""Python binding of the kvq C ABI (``include/kvq.h``): a GB300 quantized paged
KV cache -- FP8 (E4M3 / E5M2, per-tensor scale) or online INT8 / INT4
(one scale per row or per channel group) quantize-on-write -- with single-token
decode attention (optionally fused with the step's append) and chunked causal
prefill attention that dequantize on read.

This module only marshals arguments: it checks tensor dtypes, devices and
layouts, passes raw device pointers and the current CUDA stream to
``libkvq.so`` and raises on a non-OK status.  Every step of the hot path runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  There
is no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

E4M3, E5M2, INT8, INT4 = 1, 2, 3, 4
FORMATS = {"e4m3": E4M3, "fp8": E4M3, "e5m2": E5M2, "fp8_e5m2": E5M2, "int8": INT8, "int4": INT4}
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_WORKSPACE",
          4: "KVQ_ERR_OUT_OF_RANGE", 5: "KVQ_ERR_TIMEOUT", 6: "KVQ_ERR_CUDA",
          7: "KVQ_ERR_SCRATCH_LIMIT"}
KERNEL_AUTO, KERNEL_SIMT, KERNEL_MMA = 0, 1, 2
EXPORTS = ("kvq_append", "kvq_decode_workspace_size", "kvq_decode_attention", "kvq_decode_attention_append",
           "kvq_dequant",
           "kvq_set_decode_kernel", "kvq_device_error_check", "kvq_status_string", "kvq_abi_version",
           "kvq_decode_attention_static_scratch", "kvq_static_scratch_bytes", "kvq_set_decode_timing_events",
           "kvq_prefill_attention", "kvq_encode_fp8")

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")
_lib = None
_lock = threading.Lock()


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


class KvqCacheDesc(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("fmt", ctypes.c_int32), ("group_size", ctypes.c_int32)]


def build(force: bool = False) -> str:
    from . import build_lib
    return build_lib.build(force=force)


def lib():
    """The loaded ``libkvq.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run fp8_int8_quantized_gb300.build() first "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.kvq_append.restype = ctypes.c_int
        L.kvq_append.argtypes = [P, P, P, P, i64, P, i32, P]
        L.kvq_decode_workspace_size.restype = ctypes.c_size_t
        L.kvq_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.kvq_decode_attention.restype = ctypes.c_int
        L.kvq_decode_attention.argtypes = [P, P, P, i32, P, i32, i32, i32, P, i32, ctypes.c_float, P, P,
                                           ctypes.c_size_t, i32, P]
        L.kvq_decode_attention_append.restype = ctypes.c_int
        L.kvq_decode_attention_append.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, P, i32, ctypes.c_float, P,
                                                  P, ctypes.c_size_t, i32, P]
        L.kvq_decode_attention_static_scratch.restype = ctypes.c_int
        L.kvq_decode_attention_static_scratch.argtypes = [P, P, P, i32, P, i32, i32, i32, P, i32, ctypes.c_float,
                                                          P, i32, P]
        L.kvq_static_scratch_bytes.restype = ctypes.c_size_t
        L.kvq_prefill_attention.restype = ctypes.c_int
        L.kvq_prefill_attention.argtypes = [P, P, P, i32, P, P, i32, i64, i32, i32, P, i32, ctypes.c_float, P,
                                            P]
        L.kvq_encode_fp8.restype = ctypes.c_int
        L.kvq_encode_fp8.argtypes = [P, P, i64, i32, P]
        L.kvq_dequant.restype = ctypes.c_int
        L.kvq_dequant.argtypes = [P, P, i64, P, i32, P, P, P]
        L.kvq_set_decode_timing_events.restype = None
        L.kvq_set_decode_timing_events.argtypes = [P, P]
        L.kvq_set_decode_kernel.restype = i32
        L.kvq_set_decode_kernel.argtypes = [i32]
        L.kvq_device_error_check.restype = ctypes.c_int
        L.kvq_device_error_check.argtypes = [P, ctypes.POINTER(i64)]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_abi_version.restype = i32
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().kvq_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "?"


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KvqError(status, where)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _scale_ptr(scale) -> int | None:
    if scale is None:
        return None
    return _dev(scale, torch.float32, "scale")


class KVCache:
    """A paged quantized cache in device memory:
    codes uint8 [num_blocks][num_kv_heads][block_size][head_dim] for K and V
    ([..][head_dim / 2] packed codes for INT4), and for INT8 / INT4 the fp32
    scales [num_blocks][num_kv_heads][block_size] (one per row, group_size 0) or
    [num_blocks][num_kv_heads][block_size][head_dim / group_size] (one per group
    of channels; group_size head_dim / 2 or head_dim / 4)."""

    def __init__(self, num_blocks, num_kv_heads, block_size, head_dim, fmt, device="cuda", fill=None,
                 group_size=0):
        self.fmt = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
        self.num_blocks, self.num_kv_heads = int(num_blocks), int(num_kv_heads)
        self.block_size, self.head_dim = int(block_size), int(head_dim)
        self.group_size = int(group_size)
        shape = (self.num_blocks, self.num_kv_heads, self.block_size,
                 self.head_dim // 2 if self.fmt == INT4 else self.head_dim)
        mk = (lambda: torch.full(shape, fill, dtype=torch.uint8, device=device)) if fill is not None else \
            (lambda: torch.empty(shape, dtype=torch.uint8, device=device))
        self.k_codes, self.v_codes = mk(), mk()
        if self.fmt in (INT8, INT4):
            sshape = shape[:3] + ((self.head_dim // self.group_size,) if self.group_size else ())
            self.k_scales = torch.zeros(sshape, dtype=torch.float32, device=device)
            self.v_scales = torch.zeros(sshape, dtype=torch.float32, device=device)
        else:
            self.k_scales = self.v_scales = None
        self._desc = None

    def desc(self) -> KvqCacheDesc:
        """A new C descriptor of this cache."""
        return KvqCacheDesc(self.k_codes.data_ptr(), self.v_codes.data_ptr(),
                            self.k_scales.data_ptr() if self.k_scales is not None else None,
                            self.v_scales.data_ptr() if self.v_scales is not None else None,
                            self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim, self.fmt,
                            self.group_size)

    def _cdesc(self) -> KvqCacheDesc:
        # the binding's own descriptor, built once per format (the arrays never move)
        if self._desc is None or self._desc.fmt != self.fmt:
            self._desc = self.desc()
        return self._desc


def append(k: torch.Tensor, v: torch.Tensor, cache: KVCache, slot_mapping: torch.Tensor,
           scale: torch.Tensor | None = None, stream=None) -> None:
    """kvq_append: quantize fp16 K/V [T][Hkv][D] into ``cache`` at ``slot_mapping`` (int64, -1 skips)."""
    T = slot_mapping.shape[0]
    if k.shape != (T, cache.num_kv_heads, cache.head_dim) or v.shape != k.shape:
        raise ValueError("k/v must be [num_tokens][num_kv_heads][head_dim]")
    d = cache._cdesc()
    st = lib().kvq_append(_dev(k, torch.float16, "k"), _dev(v, torch.float16, "v"), ctypes.byref(d),
                          _dev(slot_mapping, torch.int64, "slot_mapping"), T, _scale_ptr(scale), cache.fmt,
                          _stream(stream))
    _check(st, "kvq_append")


def workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_context_len, partition_size=0) -> int:
    return int(lib().kvq_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                               max_context_len, partition_size))


def decode_attention(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor, context_lens: torch.Tensor,
                     max_context_len: int, scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     partition_size: int = 0, stream=None) -> torch.Tensor:
    """kvq_decode_attention: q fp16 [B][Hq][D] -> out fp16 [B][Hq][D]."""
    B, Hq, D = q.shape
    if D != cache.head_dim:
        raise ValueError("head_dim mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:  # a caller-given workspace is checked by the library
        need = workspace_size(B, Hq, cache.num_kv_heads, D, max_context_len, partition_size)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    d = cache._cdesc()
    st = lib().kvq_decode_attention(_dev(q, torch.float16, "q"), ctypes.byref(d),
                                    _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                    _dev(context_lens, torch.int32, "context_lens"), B, Hq, int(max_context_len),
                                    _scale_ptr(scale), cache.fmt, float(sm_scale),
                                    _dev(out, torch.float16, "out"), ws_ptr, ws_bytes, int(partition_size),
                                    _stream(stream))
    _check(st, "kvq_decode_attention")
    return out


def prefill_attention(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor, context_lens: torch.Tensor,
                      query_start: torch.Tensor, max_query_len: int, scale: torch.Tensor | None = None,
                      sm_scale: float = 0.0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvq_prefill_attention: causal attention of chunks of new queries over the cache.

    q fp16 [Tq][Hq][D]; sequence b owns rows query_start[b] .. query_start[b+1]-1, the last
    positions of its context_lens[b] cached tokens.  Returns out fp16 [Tq][Hq][D]."""
    Tq, Hq, D = q.shape
    if D != cache.head_dim:
        raise ValueError("head_dim mismatch")
    B = context_lens.shape[0]
    if query_start.shape[0] != B + 1:
        raise ValueError("query_start needs batch + 1 entries")
    if out is None:
        out = torch.empty_like(q)
    d = cache._cdesc()
    st = lib().kvq_prefill_attention(_dev(q, torch.float16, "q"), ctypes.byref(d),
                                     _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                     _dev(context_lens, torch.int32, "context_lens"),
                                     _dev(query_start, torch.int32, "query_start"), B, Tq, Hq,
                                     int(max_query_len),
                                     _scale_ptr(scale), cache.fmt, float(sm_scale),
                                     _dev(out, torch.float16, "out"), _stream(stream))
    _check(st, "kvq_prefill_attention")
    return out


def decode_attention_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: KVCache,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                            scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            partition_size: int = 0, stream=None) -> torch.Tensor:
    """kvq_decode_attention_append: one decode step with each sequence's newest
    K/V row (fp16 [B][Hkv][D], position context_lens[b] - 1) quantized into the
    cache in the same launch; bit-identical to ``append`` then ``decode_attention``."""
    B, Hq, D = q.shape
    if k_new.shape != (B, cache.num_kv_heads, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [batch][num_kv_heads][head_dim]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = workspace_size(B, Hq, cache.num_kv_heads, D, max_context_len, partition_size)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    d = cache._cdesc()
    st = lib().kvq_decode_attention_append(_dev(q, torch.float16, "q"), _dev(k_new, torch.float16, "k_new"),
                                           _dev(v_new, torch.float16, "v_new"), ctypes.byref(d),
                                           _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                           _dev(context_lens, torch.int32, "context_lens"), B, Hq,
                                           int(max_context_len), _scale_ptr(scale), cache.fmt, float(sm_scale),
                                           _dev(out, torch.float16, "out"), ws_ptr, ws_bytes, int(partition_size),
                                           _stream(stream))
    _check(st, "kvq_decode_attention_append")
    return out


def decode_attention_static_scratch(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor,
                                    context_lens: torch.Tensor, max_context_len: int,
                                    scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                                    out: torch.Tensor | None = None, partition_size: int = 0,
                                    stream=None) -> torch.Tensor:
    """kvq_decode_attention_static_scratch: decode attention for callers that cannot
    allocate device memory; the split workspace comes from the library's fixed
    device array.  ``out`` must be supplied by such callers."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    d = cache._cdesc()
    st = lib().kvq_decode_attention_static_scratch(
        _dev(q, torch.float16, "q"), ctypes.byref(d), _dev(block_tables, torch.int32, "block_tables"),
        block_tables.shape[1], _dev(context_lens, torch.int32, "context_lens"), B, Hq, int(max_context_len),
        _scale_ptr(scale), cache.fmt, float(sm_scale), _dev(out, torch.float16, "out"), int(partition_size),
        _stream(stream))
    _check(st, "kvq_decode_attention_static_scratch")
    return out


def dequant(cache: KVCache, slots: torch.Tensor, scale: torch.Tensor | None = None, stream=None):
    """kvq_dequant: fp32 K, V rows [n][Hkv][D] at ``slots`` (int64)."""
    n = slots.shape[0]
    ok = torch.empty((n, cache.num_kv_heads, cache.head_dim), dtype=torch.float32, device=slots.device)
    ov = torch.empty_like(ok)
    d = cache._cdesc()
    st = lib().kvq_dequant(ctypes.byref(d), _dev(slots, torch.int64, "slots"), n, _scale_ptr(scale), cache.fmt,
                           ok.data_ptr(), ov.data_ptr(), _stream(stream))
    _check(st, "kvq_dequant")
    return ok, ov


def encode_fp8(x: torch.Tensor, fmt: int, stream=None) -> torch.Tensor:
    """kvq_encode_fp8: uint8 FP8 codes (``fmt`` E4M3 or E5M2) of a flat fp32 tensor."""
    n = x.numel()
    codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = lib().kvq_encode_fp8(_dev(x, torch.float32, "x"), codes.data_ptr(), n, fmt, _stream(stream))
    _check(st, "kvq_encode_fp8")
    return codes


def set_decode_kernel(kind: int) -> int:
    prev = lib().kvq_set_decode_kernel(int(kind))
    if prev < 0:
        raise ValueError(f"unknown decode kernel kind {kind}")
    return prev


def set_decode_timing_events(begin=None, end=None) -> None:
    """kvq_set_decode_timing_events with two recorded torch.cuda.Event objects
    (enable_timing=True), or no arguments to turn the hook off."""
    if begin is None or end is None:
        lib().kvq_set_decode_timing_events(None, None)
    else:
        lib().kvq_set_decode_timing_events(begin.cuda_event, end.cuda_event)


def device_error_check(stream=None) -> tuple[int, int]:
    """(status, detail) of the device error word; synchronizes the stream and clears it."""
    detail = ctypes.c_int64(0)
    st = lib().kvq_device_error_check(_stream(stream), ctypes.byref(detail))
    return st, detail.value
