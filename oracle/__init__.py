"""The oracle: a plain single-threaded CPU statement (in C, double precision)
of the paged KV write and the PagedAttention decode step.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg import this package. The product path never does, and the two
share no code: this wrapper marshals numpy arrays into ``liboracle.so`` built
from ``oracle.c`` with gcc (no fast-math, no floating-point contraction).

Element type codes: 0 = binary32, 1 = binary16, 2 = bfloat16, 3 = OCP E4M3.
Host arrays carry 16-bit types as ``np.float16`` (binary16) or ``np.uint16``
bit patterns (bfloat16), and E4M3 as ``np.uint8`` codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16, E4M3 = 0, 1, 2, 3
_CODES = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3}

OK, BAD_ARG, BAD_SLOT, BAD_BLOCK, NOMEM = 0, 1, 2, 3, 4


def build_command() -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-o", _LIB, _SRC, "-lm"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to oracle.c (seconds)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        subprocess.run(build_command(), check=True)
    return _LIB


def _bind(path: str):
    """Load an oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P, I, I64, D, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                       ctypes.c_double, ctypes.c_float)
    lib.or_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.or_f16_to_double.restype = D
    lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.or_bf16_to_double.restype = D
    lib.or_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.or_e4m3_to_double.restype = D
    lib.or_e4m3_encode.argtypes = [F]
    lib.or_e4m3_encode.restype = ctypes.c_uint8
    lib.or_decode_array.argtypes = [P, I, I64, P]
    lib.or_decode_array.restype = None
    lib.or_e4m3_encode_array.argtypes = [P, I64, P]
    lib.or_e4m3_encode_array.restype = None
    lib.or_reshape_and_cache.argtypes = [P, P, P, P, P, I64, I, I, I, I64, I, I, F, F, P]
    lib.or_reshape_and_cache.restype = I
    lib.or_decode.argtypes = [P, P, I, P, P, I, P, P, I, P, I, I, I, I, I, I64, D, D, D]
    lib.or_decode.restype = I
    lib.or_merge.argtypes = [P, P, P, P, P, I, I, I, I, I]
    lib.or_merge.restype = I
    lib.or_decode_partitioned.argtypes = [P, P, P, P, P, I, P, P, I, P, P, I, P, I, I, I,
                                          I, I, I64, D, D, D, I, I]
    lib.or_decode_partitioned.restype = I
    lib.or_paged_prefill.argtypes = [P, P, I, P, P, P, I, P, P, I, P, I, I, I, I, I, I64, D, D, D]
    lib.or_paged_prefill.restype = I
    lib.or_copy_blocks.argtypes = [P, P, P, I64, I64, I64, I]
    lib.or_copy_blocks.restype = I
    lib.or_blocks_needed.argtypes = [I64, I]
    lib.or_blocks_needed.restype = I64
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def build_variant(src_text: str, out_path: str) -> None:
    """Compile a variant of the oracle source (used by the tests that plant a
    mistake in the oracle to show that its pins catch it)."""
    src = out_path[:-3] + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    cmd = build_command()
    cmd[cmd.index(_LIB)] = out_path
    cmd[cmd.index(_SRC)] = src
    subprocess.run(cmd, check=True)


class use_library:
    """Context manager: route this module's functions to another build of the
    oracle (a planted-mistake variant) for the duration of the block."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        with _lock:
            self.saved = _lib
            _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def code(dtype: str) -> int:
    return _CODES[dtype]


def declared_strides(num_kv_heads: int, block_size: int, head_size: int) -> np.ndarray:
    """Element strides of the [num_blocks, Hkv, B, d] layout."""
    return np.array([num_kv_heads * block_size * head_size, block_size * head_size,
                     head_size, 1], dtype=np.int64)


def f16_to_double(bits: int) -> float:
    return _load().or_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return _load().or_bf16_to_double(bits)


def e4m3_to_double(c: int) -> float:
    return _load().or_e4m3_to_double(c)


def e4m3_encode(x: float) -> int:
    return _load().or_e4m3_encode(x)


def decode_array(a: np.ndarray, dtype: str) -> np.ndarray:
    """Values of stored elements as float64."""
    a = np.ascontiguousarray(a)
    out = np.empty(a.shape, dtype=np.float64)
    _load().or_decode_array(_ptr(a), code(dtype), a.size, _ptr(out))
    return out


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().or_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def reshape_and_cache(key, value, k_cache, v_cache, slots, num_kv_heads, head_size, block_size,
                      in_dtype: str, cache_dtype: str, k_scale=1.0, v_scale=1.0,
                      strides=None) -> int:
    """Scatter key/value [T, Hkv, d] into k_cache/v_cache in place. Returns
    the oracle's status code (0 = OK)."""
    num_blocks = k_cache.shape[0]
    if strides is None:
        strides = declared_strides(num_kv_heads, block_size, head_size)
    strides = np.ascontiguousarray(strides, dtype=np.int64)
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    return _load().or_reshape_and_cache(
        _ptr(np.ascontiguousarray(key)), _ptr(np.ascontiguousarray(value)), _ptr(k_cache),
        _ptr(v_cache), _ptr(slots), slots.size, num_kv_heads, head_size, block_size, num_blocks,
        code(in_dtype), code(cache_dtype), k_scale, v_scale, _ptr(strides))


def decode(query, q_dtype: str, k_cache, v_cache, cache_dtype: str, block_tables, context_lens,
           num_kv_heads: int, block_size: int, scale: float, k_scale=1.0, v_scale=1.0,
           strides=None, head_size=None, num_blocks=None) -> np.ndarray:
    """Single-pass decode; returns out [S, Hq, d] float64."""
    S, Hq, d = query.shape
    head_size = head_size or d
    if strides is None:
        strides = declared_strides(num_kv_heads, block_size, head_size)
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    strides = np.ascontiguousarray(strides, dtype=np.int64)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((S, Hq, d), dtype=np.float64)
    rc = _load().or_decode(_ptr(out), _ptr(np.ascontiguousarray(query)), code(q_dtype),
                           _ptr(k_cache), _ptr(v_cache), code(cache_dtype), _ptr(strides),
                           _ptr(bt), bt.shape[1], _ptr(cl), S, Hq, num_kv_heads, d, block_size,
                           num_blocks, float(scale), float(k_scale), float(v_scale))
    if rc != OK:
        raise RuntimeError(f"oracle decode failed with code {rc}")
    return out


def decode_partitioned(query, q_dtype: str, k_cache, v_cache, cache_dtype: str, block_tables,
                       context_lens, num_kv_heads: int, block_size: int, scale: float,
                       partition_size: int, k_scale=1.0, v_scale=1.0, strides=None,
                       max_parts=None):
    """Partitioned decode; returns (out, part_o, part_m, part_l), all float64."""
    S, Hq, d = query.shape
    if strides is None:
        strides = declared_strides(num_kv_heads, block_size, d)
    strides = np.ascontiguousarray(strides, dtype=np.int64)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    if max_parts is None:
        max_parts = max(1, int(-(-int(cl.max(initial=0)) // partition_size)))
    out = np.empty((S, Hq, d), dtype=np.float64)
    po = np.empty((S, Hq, max_parts, d), dtype=np.float64)
    pm = np.empty((S, Hq, max_parts), dtype=np.float64)
    pl = np.empty((S, Hq, max_parts), dtype=np.float64)
    rc = _load().or_decode_partitioned(
        _ptr(out), _ptr(po), _ptr(pm), _ptr(pl), _ptr(np.ascontiguousarray(query)), code(q_dtype),
        _ptr(k_cache), _ptr(v_cache), code(cache_dtype), _ptr(strides), _ptr(bt), bt.shape[1],
        _ptr(cl), S, Hq, num_kv_heads, d, block_size, k_cache.shape[0], float(scale),
        float(k_scale), float(v_scale), partition_size, max_parts)
    if rc != OK:
        raise RuntimeError(f"oracle partitioned decode failed with code {rc}")
    return out, po, pm, pl


def merge(part_o, part_m, part_l, context_lens, partition_size: int) -> np.ndarray:
    """Merge partition partials [S, Hq, P, d] / [S, Hq, P] into out [S, Hq, d]."""
    part_o = np.ascontiguousarray(part_o, dtype=np.float64)
    part_m = np.ascontiguousarray(part_m, dtype=np.float64)
    part_l = np.ascontiguousarray(part_l, dtype=np.float64)
    S, Hq, P, d = part_o.shape
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((S, Hq, d), dtype=np.float64)
    rc = _load().or_merge(_ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(cl), S, Hq, d,
                          partition_size, P)
    if rc != OK:
        raise RuntimeError(f"oracle merge failed with code {rc}")
    return out


def blocks_needed(tokens: int, block_size: int) -> int:
    return _load().or_blocks_needed(tokens, block_size)


def copy_blocks(k_cache, v_cache, pairs) -> int:
    """Copy whole blocks (in place) for each (src, dst) row of pairs."""
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    nb = k_cache.shape[0]
    per = int(np.prod(k_cache.shape[1:]))
    return _load().or_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], nb,
                                  per, k_cache.dtype.itemsize)


def paged_prefill(query, q_dtype: str, query_start, k_cache, v_cache, cache_dtype: str,
                  block_tables, context_lens, num_kv_heads: int, block_size: int, scale: float,
                  k_scale=1.0, v_scale=1.0, strides=None) -> np.ndarray:
    """Multi-query paged attention; query [T, Hq, d] -> out [T, Hq, d] float64."""
    T, Hq, d = query.shape
    if strides is None:
        strides = declared_strides(num_kv_heads, block_size, d)
    strides = np.ascontiguousarray(strides, dtype=np.int64)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((T, Hq, d), dtype=np.float64)
    rc = _load().or_paged_prefill(_ptr(out), _ptr(np.ascontiguousarray(query)), code(q_dtype),
                                  _ptr(qs), _ptr(k_cache), _ptr(v_cache), code(cache_dtype),
                                  _ptr(strides), _ptr(bt), bt.shape[1], _ptr(cl), cl.size, Hq,
                                  num_kv_heads, d, block_size, k_cache.shape[0], float(scale),
                                  float(k_scale), float(v_scale))
    if rc != OK:
        raise RuntimeError(f"oracle paged prefill failed with code {rc}")
    return out
