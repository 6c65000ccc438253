"""CPU oracle for the quantized paged KV cache (quantize-on-write, decode attention
and causal attention of a chunk of new queries over the cache).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports, links or calls it, and it shares no
code with the CUDA library: the arithmetic lives in ``kvq_oracle.c`` (plain C,
fp64 attention), built here with gcc, and this module only marshals numpy
arrays into it.

Sources, by page title and section:
  * "Accelerating Inference with FP8 KV Cache" (TGI docs): FP8 storage with FP16
    compute (intro); E4M3 / E5M2 bit layouts and the per-tensor fp32 scale
    ("FP8 Formats: E4M3 and E5M2"); scale 1.0 when none is given
    ("FP8 E4M3 KV Cache").
  * "[Feature] TurboMind support W8A8 or FP8 KV Cache" (lmdeploy issue 1463):
    online KV-cache INT8 (and the INT4 implementation named beside it).
  * "[QST] Scale factors and benchmarks" (QQQ issue page): group quantization
    named for a 4-bit KV cache; read here as INT8 / INT4 with one scale per
    group of ``group`` consecutive channels of a row.

Parity pins for every function here live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, E5M2, INT8, INT4 = 1, 2, 3, 4
FORMATS = {"e4m3": E4M3, "e5m2": E5M2, "int8": INT8, "int4": INT4}
ROW_SCALED = (INT8, INT4)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``kvq_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, IEEE fp)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-fno-strict-aliasing", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.oracle_fp8_decode.restype = f64
        lib.oracle_fp8_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
        lib.oracle_fp8_encode.restype = ctypes.c_uint8
        lib.oracle_fp8_encode.argtypes = [ctypes.c_int, f32]
        lib.oracle_fp8_encode_array.restype = None
        lib.oracle_fp8_encode_array.argtypes = [ctypes.c_int, P, P, i64]
        lib.oracle_int8_quant_row.restype = f32
        lib.oracle_int8_quant_row.argtypes = [P, ctypes.c_int, P]
        lib.oracle_int4_quant_row.restype = f32
        lib.oracle_int4_quant_row.argtypes = [P, ctypes.c_int, P]
        lib.oracle_half_to_double.restype = f64
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_append.restype = ctypes.c_int
        lib.oracle_append.argtypes = [P, P, i64, ctypes.c_int, ctypes.c_int, P, P, P, P, P,
                                      i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32]
        lib.oracle_dequant.restype = ctypes.c_int
        lib.oracle_dequant.argtypes = [P, P, P, P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P, i64, f32, P, P]
        lib.oracle_decode_attention.restype = ctypes.c_int
        lib.oracle_decode_attention.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                P, P, P, P, i64, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P, f32,
                                                f64, P, P, i64]
        lib.oracle_prefill_attention.restype = ctypes.c_int
        lib.oracle_prefill_attention.argtypes = [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 P, P, P, P, i64, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P, P, f32,
                                                 f64, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_init()
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _need(a, dtype, name):
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name}: expected C-contiguous {np.dtype(dtype)}, got {a.dtype}")
    return a


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (OMP_NUM_THREADS or all cores)."""
    return _load().oracle_num_threads()


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(bits)


def fp8_decode(fmt: int, code: int) -> float:
    """Value of one FP8 code, from the format's bit-field definition."""
    return _load().oracle_fp8_decode(fmt, code)


def fp8_decode_table(fmt: int) -> np.ndarray:
    """All 256 codes of ``fmt`` decoded to fp64 (NaN / Inf where the format has them)."""
    return np.array([fp8_decode(fmt, c) for c in range(256)], dtype=np.float64)


def fp8_encode(fmt: int, y) -> np.ndarray:
    """fp32 values -> FP8 codes: nearest, ties to even, saturating, NaN -> 0x7F."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    _load().oracle_fp8_encode_array(fmt, _ptr(y), _ptr(out), y.size)
    return out


def int4_quant_row(x) -> tuple[np.ndarray, np.float32]:
    """One INT4 row: returns (packed codes uint8 [D / 2], scale fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape[:-1] + (x.shape[-1] // 2,), dtype=np.uint8)
    s = _load().oracle_int4_quant_row(_ptr(x), x.size, _ptr(q))
    return q, np.float32(s)


def int4_unpack(packed: np.ndarray) -> np.ndarray:
    """Signed INT4 codes (int8 [..., 2 * n]) of packed rows uint8 [..., n]."""
    lo = (packed & 0xF).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    both = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (2 * packed.shape[-1],))
    return np.where(both >= 8, both - 16, both).astype(np.int8)


def int8_quant_row(x) -> tuple[np.ndarray, np.float32]:
    """One INT8 row: returns (codes int8 [D], scale fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.int8)
    s = _load().oracle_int8_quant_row(_ptr(x), x.size, _ptr(q))
    return q, np.float32(s)


class Cache:
    """Host copy of a paged cache: codes [NB][Hkv][BS][D] ([D / 2] packed bytes for
    INT4); INT8 / INT4 scales [NB][Hkv][BS] (one per row, group 0) or
    [NB][Hkv][BS][D / group] (one per group of ``group`` channels)."""

    def __init__(self, num_blocks, num_kv_heads, block_size, head_dim, fmt, fill=0xA5,
                 k_codes=None, v_codes=None, k_scales=None, v_scales=None, group=0):
        self.num_blocks, self.num_kv_heads = num_blocks, num_kv_heads
        self.block_size, self.head_dim, self.fmt = block_size, head_dim, fmt
        self.group = int(group)
        if self.group and (fmt not in ROW_SCALED or head_dim % self.group
                           or (fmt == INT4 and self.group % 2)):
            raise ValueError(f"group {group} not allowed for format {fmt}, head_dim {head_dim}")
        shape = (num_blocks, num_kv_heads, block_size, head_dim // 2 if fmt == INT4 else head_dim)
        self.k_codes = k_codes if k_codes is not None else np.full(shape, fill, np.uint8)
        self.v_codes = v_codes if v_codes is not None else np.full(shape, fill, np.uint8)
        if fmt in ROW_SCALED:
            sshape = (num_blocks, num_kv_heads, block_size)
            if self.group:
                sshape += (head_dim // self.group,)
            self.k_scales = k_scales if k_scales is not None else np.full(sshape, np.nan, np.float32)
            self.v_scales = v_scales if v_scales is not None else np.full(sshape, np.nan, np.float32)
        else:
            self.k_scales = self.v_scales = None
        for a, n in ((self.k_codes, "k_codes"), (self.v_codes, "v_codes")):
            _need(a, np.uint8, n)
            if a.shape != shape:
                raise ValueError(f"{n}: shape {a.shape} != {shape}")
        if fmt in ROW_SCALED:
            for a, n in ((self.k_scales, "k_scales"), (self.v_scales, "v_scales")):
                _need(a, np.float32, n)
                if a.size != int(np.prod(sshape)):
                    raise ValueError(f"{n}: {a.size} scales, expected shape {sshape}")


def append(k, v, slot_mapping, cache: Cache, scale: float | None = None) -> None:
    """Quantize-on-write of fp16 K/V [T][Hkv][D] into ``cache`` at ``slot_mapping`` (-1 skips)."""
    k = _need(np.ascontiguousarray(k), np.float16, "k")
    v = _need(np.ascontiguousarray(v), np.float16, "v")
    slots = _need(np.ascontiguousarray(slot_mapping, dtype=np.int64), np.int64, "slot_mapping")
    T = slots.shape[0]
    s = np.float32(1.0 if scale is None else scale)
    rc = _load().oracle_append(_ptr(k.view(np.uint16)), _ptr(v.view(np.uint16)), T,
                               cache.num_kv_heads, cache.head_dim, _ptr(slots),
                               _ptr(cache.k_codes), _ptr(cache.v_codes),
                               _ptr(cache.k_scales), _ptr(cache.v_scales),
                               cache.num_blocks, cache.block_size, cache.fmt, cache.group, s)
    if rc != 0:
        raise IndexError("slot_mapping holds a slot outside the cache")


def dequant(cache: Cache, slots, scale: float | None = None):
    """fp32 dequantized K, V rows [n][Hkv][D] at ``slots``."""
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    n = slots.shape[0]
    ok = np.empty((n, cache.num_kv_heads, cache.head_dim), np.float32)
    ov = np.empty_like(ok)
    s = np.float32(1.0 if scale is None else scale)
    rc = _load().oracle_dequant(_ptr(cache.k_codes), _ptr(cache.v_codes), _ptr(cache.k_scales),
                                _ptr(cache.v_scales), cache.num_blocks, cache.block_size,
                                cache.num_kv_heads, cache.head_dim, cache.fmt, cache.group, _ptr(slots), n, s,
                                _ptr(ok), _ptr(ov))
    if rc != 0:
        raise IndexError("slot outside the cache")
    return ok, ov


def default_sm_scale(head_dim: int) -> float:
    return 1.0 / np.sqrt(float(head_dim))


def decode_attention(q, cache: Cache, block_tables, context_lens, scale: float | None = None,
                     sm_scale: float | None = None, return_weights: bool = False):
    """fp64 single-token decode attention. q fp16 [B][Hq][D] -> out fp64 [B][Hq][D]."""
    q = _need(np.ascontiguousarray(q), np.float16, "q")
    B, Hq, D = q.shape
    if D != cache.head_dim or Hq % cache.num_kv_heads:
        raise ValueError("q shape does not match the cache")
    bt = _need(np.ascontiguousarray(block_tables, dtype=np.int32), np.int32, "block_tables")
    cl = _need(np.ascontiguousarray(context_lens, dtype=np.int32), np.int32, "context_lens")
    out = np.zeros((B, Hq, D), np.float64)
    wstride = max(1, int(cl.max()) if cl.size else 1)
    w = np.zeros((B, Hq, wstride), np.float64) if return_weights else None
    s = np.float32(1.0 if scale is None else scale)
    sm = default_sm_scale(D) if not sm_scale else float(sm_scale)
    rc = _load().oracle_decode_attention(_ptr(q.view(np.uint16)), B, Hq, D, _ptr(cache.k_codes),
                                         _ptr(cache.v_codes), _ptr(cache.k_scales),
                                         _ptr(cache.v_scales), cache.num_blocks, cache.block_size,
                                         cache.num_kv_heads, cache.fmt, cache.group, _ptr(bt),
                                         bt.shape[1], _ptr(cl), s, sm, _ptr(out), _ptr(w), wstride)
    if rc != 0:
        raise IndexError("block table / context length outside the cache")
    return (out, w) if return_weights else out


def prefill_attention(q, cache: Cache, block_tables, context_lens, query_start,
                      scale: float | None = None, sm_scale: float | None = None):
    """fp64 causal attention of chunks of new queries over the cache.

    q fp16 [Tq][Hq][D]; sequence b owns rows query_start[b] .. query_start[b+1]-1,
    the last n_b of its context_lens[b] cached positions (its own K/V already
    appended); query i of the chunk attends to positions 0 .. ctx - n_b + i.
    Returns out fp64 [Tq][Hq][D] (rows no chunk covers stay zero)."""
    q = _need(np.ascontiguousarray(q), np.float16, "q")
    Tq, Hq, D = q.shape
    if D != cache.head_dim or Hq % cache.num_kv_heads:
        raise ValueError("q shape does not match the cache")
    bt = _need(np.ascontiguousarray(block_tables, dtype=np.int32), np.int32, "block_tables")
    cl = _need(np.ascontiguousarray(context_lens, dtype=np.int32), np.int32, "context_lens")
    qs = _need(np.ascontiguousarray(query_start, dtype=np.int32), np.int32, "query_start")
    B = cl.shape[0]
    if qs.shape[0] != B + 1:
        raise ValueError("query_start needs batch + 1 entries")
    out = np.zeros((Tq, Hq, D), np.float64)
    s = np.float32(1.0 if scale is None else scale)
    sm = default_sm_scale(D) if not sm_scale else float(sm_scale)
    rc = _load().oracle_prefill_attention(_ptr(q.view(np.uint16)), Tq, B, Hq, D, _ptr(cache.k_codes),
                                          _ptr(cache.v_codes), _ptr(cache.k_scales),
                                          _ptr(cache.v_scales), cache.num_blocks, cache.block_size,
                                          cache.num_kv_heads, cache.fmt, cache.group, _ptr(bt),
                                          bt.shape[1], _ptr(cl), _ptr(qs), s, sm, _ptr(out))
    if rc != 0:
        raise IndexError("chunk longer than its context, or block table / context outside the cache")
    return out
