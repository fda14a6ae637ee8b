"""Python binding of libpagedkv.so (the C ABI in include/pagedkv.h).

Argument marshalling only: every function passes tensor data pointers, sizes
and the current CUDA stream to the library, and raises PagedKVError when the
library returns a non-zero status. All computation happens in the library's
CUDA kernels. If the library has not been built, loading fails with an error;
there is no fallback path.

Tensors are CUDA tensors, contiguous, in the library's layouts:
  query/out        [num_seqs, num_q_heads, head_size]   float32/float16/bfloat16
  key/value        [num_tokens, num_kv_heads, head_size]
  k_cache/v_cache  [num_blocks, num_kv_heads, block_size, head_size]
                   (E4M3 caches as torch.uint8 or torch.float8_e4m3fn)
  block_tables     [num_seqs, max_blocks] int32
  context_lens     [num_seqs] int32
  slot_mapping     [num_tokens] int64
  dev_status       [1] int32 (read as uint32 bits), zeroed by the caller
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")
_lock = threading.Lock()
_lib = None

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_NO_BLOCKS = range(6)
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = range(4)
DEV_BAD_BLOCK_ID, DEV_BAD_SLOT, DEV_BAD_LEN, DEV_TIMEOUT, DEV_SLOT_MISMATCH = 1, 2, 4, 8, 16
DEV_BAD_ORDER = 32
DEV_BAD_PREFIX = 64

DEFAULT_PARTITION_SIZE = 512

_DTYPES = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16,
           torch.uint8: PA_FP8_E4M3}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = PA_FP8_E4M3


class PagedKVError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libpagedkv.so and declare its signatures (once)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it first "
                "(python -m paged_kv_cache_141_gb300.build)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, I64, F, S = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_size_t)
        L.pa_reshape_and_cache.argtypes = [P, P, P, P, P, I64, I, I, I, I64, I, I, F, F, P, P]
        L.pa_decode.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I64, I, F, I, I, F, F, P, P]
        L.pa_decode_partitioned_workspace_bytes.argtypes = [I, I, I, I, I]
        L.pa_decode_partitioned_workspace_bytes.restype = S
        L.pa_decode_workspace_layout.argtypes = [I, I, I, I, I, P, P, P, P]
        L.pa_decode_partitions.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I64, I, F, I, I, F, F,
                                           I, P, S, P, P]
        L.pa_merge.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
        L.pa_decode_partitioned.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I64, I, F, I, I,
                                            F, F, I, P, S, P, P]
        L.pa_decode_partitioned_static.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I64, I,
                                                   F, I, I, F, F, I, P, P]
        L.pa_write_decode.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, I64, I, F, I, I,
                                      F, F, P, P]
        L.pa_shared_prefix_plan.argtypes = [P, P, I, I, I, I, P, P, P, I, P, P]
        L.pa_write_decode_shared_prefix.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I,
                                                    I64, I, F, I, I, F, F, P, P, P, I, I, I, P, S,
                                                    P, P]
        L.pa_write_decode_partitioned.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I,
                                                  I64, I, F, I, I, F, F, I, P, S, P, P]
        L.pa_write_decode_partitions.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, I, I64,
                                                 I, F, I, I, F, F, I, P, S, P, P]
        L.pa_paged_prefill.argtypes = [P, P, P, I, I, P, P, P, I, P, I, I, I, I, I, I64, I, F, I,
                                       I, F, F, P, P, P]
        L.pa_paged_prefill_kernel.argtypes = [I, I, I, I, I, I64, I, I]
        L.pa_paged_prefill_kernel.restype = I
        L.pa_copy_blocks.argtypes = [P, P, P, I64, I, I, I, I64, I, P, P]
        L.pa_selftest_wait.argtypes = [I, P, P]
        L.pa_allocator_create.argtypes = [I64, I, I]
        L.pa_allocator_create.restype = P
        L.pa_allocator_destroy.argtypes = [P]
        L.pa_allocator_destroy.restype = None
        L.pa_allocator_num_free.argtypes = [P]
        L.pa_allocator_num_free.restype = I64
        L.pa_allocator_refcount.argtypes = [P, ctypes.c_int32]
        L.pa_allocator_refcount.restype = ctypes.c_int32
        L.pa_allocator_allocate.argtypes = [P, I64, P, I64, P]
        L.pa_allocator_fork.argtypes = [P, P, I64]
        L.pa_allocator_free.argtypes = [P, P, I64]
        L.pa_allocator_append_slot.argtypes = [P, P, P, I64, I64, P, P, P]
        L.pa_radix_create.argtypes = [I64, I, I]
        L.pa_radix_create.restype = P
        L.pa_radix_destroy.argtypes = [P]
        L.pa_radix_destroy.restype = None
        L.pa_radix_allocate.argtypes = [P, P, I64, I64, P, I64, P, P, P]
        L.pa_radix_free.argtypes = [P, I64, P, I64]
        for f in ("pa_radix_num_free", "pa_radix_num_cached", "pa_radix_num_evictable"):
            getattr(L, f).argtypes = [P]
            getattr(L, f).restype = I64
        L.pa_decode_choose.argtypes = [I, I, I, I, I]
        L.pa_decode_partition_size.argtypes = [I, I, I]
        L.pa_status_string.argtypes = [I]
        L.pa_status_string.restype = ctypes.c_char_p
        for name in ("pa_reshape_and_cache", "pa_decode", "pa_decode_workspace_layout",
                     "pa_decode_partitions", "pa_merge", "pa_decode_partitioned",
                     "pa_decode_partitioned_static", "pa_write_decode",
                     "pa_write_decode_partitioned", "pa_write_decode_partitions",
                     "pa_decode_choose", "pa_decode_partition_size", "pa_version",
                     "pa_shared_prefix_plan", "pa_write_decode_shared_prefix",
                     "pa_copy_blocks", "pa_selftest_wait", "pa_allocator_allocate", "pa_allocator_fork",
                     "pa_allocator_free", "pa_allocator_append_slot"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedKVError(what, status)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported tensor dtype {t.dtype}") from None


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, k_scale=1.0, v_scale=1.0,
                      dev_status=None, stream=None) -> None:
    """The KV write: scatter key/value [T, Hkv, d] into the caches at
    slot_mapping (E4M3 caches quantise with k_scale / v_scale)."""
    T, H, D = key.shape
    nb, H2, B, D2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (H, D) != (H2, D2):
        raise ValueError("inconsistent key/value/cache shapes")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check(lib().pa_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, H, D, B, nb,
        _dtype(key), _dtype(k_cache), float(k_scale), float(v_scale), _ptr(dev_status),
        _stream(stream)), "pa_reshape_and_cache")


def _decode_dims(query, k_cache, block_tables, context_lens):
    S, Hq, D = query.shape
    nb, Hkv, B, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("query and cache head sizes differ")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks], context_lens [num_seqs]")
    return S, Hq, D, nb, Hkv, B, block_tables.shape[1]


def decode(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
           k_scale=1.0, v_scale=1.0, dev_status=None, stream=None) -> None:
    """Single-pass paged decode into `out`."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _check(lib().pa_decode(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb,
        _ptr(context_lens), S, Hq, Hkv, D, B, nb, int(max_context_len), float(scale),
        _dtype(query), _dtype(k_cache), float(k_scale), float(v_scale), _ptr(dev_status),
        _stream(stream)), "pa_decode")


def paged_prefill(out, query, query_start, k_cache, v_cache, block_tables, context_lens,
                  max_queries_per_seq, max_context_len, scale, k_scale=1.0, v_scale=1.0,
                  dev_status=None, stream=None, *, seq_order=None) -> None:
    """Causal multi-query paged attention into `out` ([T, Hq, D] like `query`);
    the tokens of sequence s are rows query_start[s]..query_start[s+1]-1 and
    are the last Q_s positions of its context_lens[s] tokens. `seq_order`
    (int32 [num_seqs] on the device, optional): the order in which sequences'
    work starts, e.g. longest_first(context lengths known on the host)."""
    T, Hq, D = query.shape
    nb, Hkv, B, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("query and cache head sizes differ")
    S = context_lens.numel()
    if query_start.dtype != torch.int32 or query_start.numel() != S + 1:
        raise ValueError("query_start must be int32 [num_seqs + 1]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    if seq_order is not None and (seq_order.dtype != torch.int32 or seq_order.numel() != S):
        raise ValueError("seq_order must be int32 [num_seqs]")
    _check(lib().pa_paged_prefill(
        _ptr(out), _ptr(query), _ptr(query_start), T, int(max_queries_per_seq), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), S, Hq, Hkv,
        D, B, nb, int(max_context_len), float(scale), _dtype(query), _dtype(k_cache),
        float(k_scale), float(v_scale), _ptr(seq_order), _ptr(dev_status), _stream(stream)),
        "pa_paged_prefill")


PREFILL_KERNELS = {0: "cuda_cores", 1: "mma", 2: "mma_two_tiles", 3: "tc", 4: "tc_two_tiles"}


def prefill_kernel(max_queries_per_seq, num_q_heads, num_kv_heads, head_size, block_size,
                   num_blocks, q_dtype, cache_dtype) -> str:
    """The kernel paged_prefill selects for a shape (host only): one of
    PREFILL_KERNELS' names; dtypes as PA_* codes. Raises for a shape
    paged_prefill rejects."""
    k = lib().pa_paged_prefill_kernel(int(max_queries_per_seq), num_q_heads, num_kv_heads,
                                      head_size, block_size, int(num_blocks), int(q_dtype),
                                      int(cache_dtype))
    if k < 0:
        raise PagedKVError("pa_paged_prefill_kernel: unsupported arguments")
    return PREFILL_KERNELS[k]


def longest_first(context_lens) -> "np.ndarray":
    """The sequence order that starts the longest contexts first (stable for
    equal lengths), from lengths known on the host: int32 [num_seqs]."""
    import numpy as np
    L = np.asarray(context_lens)
    return np.argsort(-L.astype(np.int64), kind="stable").astype(np.int32)


def workspace_bytes(num_seqs, num_q_heads, head_size, max_context_len,
                    partition_size=DEFAULT_PARTITION_SIZE) -> int:
    return int(lib().pa_decode_partitioned_workspace_bytes(num_seqs, num_q_heads, head_size,
                                                           int(max_context_len), partition_size))


def max_partitions(max_context_len, partition_size=DEFAULT_PARTITION_SIZE) -> int:
    return max(1, -(-int(max_context_len) // partition_size))


def workspace_views(workspace, num_seqs, num_q_heads, head_size, max_context_len,
                    partition_size=DEFAULT_PARTITION_SIZE):
    """(tmp_out, max_logits, exp_sums) float32 views into a workspace tensor."""
    offs = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().pa_decode_workspace_layout(num_seqs, num_q_heads, head_size,
                                            int(max_context_len), partition_size,
                                            *[ctypes.byref(o) for o in offs]),
           "pa_decode_workspace_layout")
    P = max_partitions(max_context_len, partition_size)
    raw = workspace.view(torch.uint8)

    def region(off, n, shape):
        return raw[off:off + 4 * n].view(torch.float32).view(shape)

    tmp = region(offs[0].value, num_seqs * num_q_heads * P * head_size,
                 (num_seqs, num_q_heads, P, head_size))
    ml = region(offs[1].value, num_seqs * num_q_heads * P, (num_seqs, num_q_heads, P))
    es = region(offs[2].value, num_seqs * num_q_heads * P, (num_seqs, num_q_heads, P))
    return tmp, ml, es


def alloc_workspace(num_seqs, num_q_heads, head_size, max_context_len,
                    partition_size=DEFAULT_PARTITION_SIZE, device=None) -> torch.Tensor:
    n = workspace_bytes(num_seqs, num_q_heads, head_size, max_context_len, partition_size)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def decode_partitions(query, k_cache, v_cache, block_tables, context_lens, max_context_len,
                      scale, workspace, partition_size=DEFAULT_PARTITION_SIZE, k_scale=1.0,
                      v_scale=1.0, dev_status=None, stream=None) -> None:
    """The partition kernel: per-partition partials into `workspace`."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _check(lib().pa_decode_partitions(
        _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens),
        S, Hq, Hkv, D, B, nb, int(max_context_len), float(scale), _dtype(query),
        _dtype(k_cache), float(k_scale), float(v_scale), partition_size, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)),
        "pa_decode_partitions")


def merge(out, tmp_out, max_logits, exp_sums, context_lens, partition_size=DEFAULT_PARTITION_SIZE,
          dev_status=None, stream=None) -> None:
    """Merge partition partials [S, Hq, P, d] / [S, Hq, P] into `out`."""
    S, Hq, P, D = tmp_out.shape
    _check(lib().pa_merge(
        _ptr(out), _ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums), _ptr(context_lens), S, Hq, D,
        partition_size, P, _dtype(out), _ptr(dev_status), _stream(stream)), "pa_merge")


def decode_partitioned(out, query, k_cache, v_cache, block_tables, context_lens,
                       max_context_len, scale, workspace, partition_size=DEFAULT_PARTITION_SIZE,
                       k_scale=1.0, v_scale=1.0, dev_status=None, stream=None) -> None:
    """Partition kernel then merge kernel."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _check(lib().pa_decode_partitioned(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb,
        _ptr(context_lens), S, Hq, Hkv, D, B, nb, int(max_context_len), float(scale),
        _dtype(query), _dtype(k_cache), float(k_scale), float(v_scale), partition_size,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream)), "pa_decode_partitioned")


def _new_tokens(key, value, slot_mapping, query, k_cache):
    S, Hkv, D = key.shape
    if value.shape != key.shape or S != query.shape[0] or (Hkv, D) != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("key/value must be [num_seqs, num_kv_heads, head_size]")
    if key.dtype != query.dtype or value.dtype != query.dtype:
        raise ValueError("new key/value must have the query's dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != S:
        raise ValueError("slot_mapping must be int64 [num_seqs]")


def write_decode(out, query, key, value, k_cache, v_cache, slot_mapping, block_tables,
                 context_lens, max_context_len, scale, k_scale=1.0, v_scale=1.0, dev_status=None,
                 stream=None) -> None:
    """KV write of each sequence's newest token and single-pass decode, one launch."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _new_tokens(key, value, slot_mapping, query, k_cache)
    _check(lib().pa_write_decode(
        _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), S, Hq, Hkv, D, B, nb,
        int(max_context_len), float(scale), _dtype(query), _dtype(k_cache), float(k_scale),
        float(v_scale), _ptr(dev_status), _stream(stream)), "pa_write_decode")


def write_decode_partitions(query, key, value, k_cache, v_cache, slot_mapping, block_tables,
                            context_lens, max_context_len, scale, workspace,
                            partition_size=DEFAULT_PARTITION_SIZE, k_scale=1.0, v_scale=1.0,
                            dev_status=None, stream=None) -> None:
    """The partition kernel with the new tokens' KV write folded in (partials only)."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _new_tokens(key, value, slot_mapping, query, k_cache)
    _check(lib().pa_write_decode_partitions(
        _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), mb, _ptr(context_lens), S, Hq, Hkv, D, B, nb, int(max_context_len),
        float(scale), _dtype(query), _dtype(k_cache), float(k_scale), float(v_scale),
        partition_size, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)), "pa_write_decode_partitions")


def write_decode_partitioned(out, query, key, value, k_cache, v_cache, slot_mapping,
                             block_tables, context_lens, max_context_len, scale, workspace,
                             partition_size=DEFAULT_PARTITION_SIZE, k_scale=1.0, v_scale=1.0,
                             dev_status=None, stream=None) -> None:
    """KV write fused into the partition kernel, then the merge kernel."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    _new_tokens(key, value, slot_mapping, query, k_cache)
    _check(lib().pa_write_decode_partitioned(
        _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), S, Hq, Hkv, D, B, nb,
        int(max_context_len), float(scale), _dtype(query), _dtype(k_cache), float(k_scale),
        float(v_scale), partition_size, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)),
        "pa_write_decode_partitioned")


SHARED_UNIT_MEMBERS = 4


class SharedPrefixPlan:
    """pa_shared_prefix_plan's units for a batch (host arrays): which
    sequences share their leading partitions' KV blocks."""

    def __init__(self, seq_shared_parts, unit_seqs, unit_parts, max_unit_parts):
        self.seq_shared_parts = seq_shared_parts      # [S] int32
        self.unit_seqs = unit_seqs                    # [units, SHARED_UNIT_MEMBERS] int32
        self.unit_parts = unit_parts                  # [units] int32
        self.max_unit_parts = max_unit_parts

    @property
    def num_units(self) -> int:
        return int(self.unit_parts.shape[0])

    def to(self, device):
        """The plan's arrays as device tensors (seq_shared_parts, unit_seqs, unit_parts)."""
        t = lambda a: torch.from_numpy(a).to(device)
        return t(self.seq_shared_parts), t(self.unit_seqs), t(self.unit_parts)


def shared_prefix_plan(block_tables, context_lens, block_size,
                       partition_size=DEFAULT_PARTITION_SIZE) -> SharedPrefixPlan:
    """Units of sequences sharing their leading partitions, from host copies
    of block_tables [S, max_blocks] and context_lens [S] (numpy int32)."""
    import numpy as np
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, mb = bt.shape
    cap = max(1, S // 2)
    parts = np.zeros(S, np.int32)
    useqs = np.full((cap, SHARED_UNIT_MEMBERS), -1, np.int32)
    uparts = np.zeros(cap, np.int32)
    n, mx = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().pa_shared_prefix_plan(bt.ctypes.data, cl.ctypes.data, S, mb, int(block_size),
                                        int(partition_size), parts.ctypes.data, useqs.ctypes.data,
                                        uparts.ctypes.data, cap, ctypes.byref(n), ctypes.byref(mx)),
           "pa_shared_prefix_plan")
    return SharedPrefixPlan(parts, useqs[:n.value].copy(), uparts[:n.value].copy(), mx.value)


def write_decode_shared_prefix(out, query, k_cache, v_cache, block_tables, context_lens,
                               max_context_len, scale, workspace, seq_shared_parts, unit_seqs,
                               unit_parts, max_unit_parts, partition_size=DEFAULT_PARTITION_SIZE,
                               key=None, value=None, slot_mapping=None, k_scale=1.0,
                               v_scale=1.0, dev_status=None, stream=None) -> None:
    """Decode step with shared-prefix units (device tensors of a
    SharedPrefixPlan): shared-prefix kernel, partition kernel (with the KV
    write when key/value/slot_mapping are given), merge."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    if key is not None:
        _new_tokens(key, value, slot_mapping, query, k_cache)
    for t in (seq_shared_parts, unit_seqs, unit_parts):
        if t.dtype != torch.int32:
            raise ValueError("the plan's arrays must be int32")
    if seq_shared_parts.numel() != S or unit_seqs.numel() != SHARED_UNIT_MEMBERS * unit_parts.numel():
        raise ValueError("plan arrays do not match the batch")
    _check(lib().pa_write_decode_shared_prefix(
        _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), S, Hq, Hkv, D, B, nb,
        int(max_context_len), float(scale), _dtype(query), _dtype(k_cache), float(k_scale),
        float(v_scale), _ptr(seq_shared_parts), _ptr(unit_seqs), _ptr(unit_parts),
        int(unit_parts.numel()), int(max_unit_parts), partition_size, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)),
        "pa_write_decode_shared_prefix")


STATIC_WORKSPACE_BYTES = 64 * 1024 * 1024


def decode_partitioned_static(out, query, k_cache, v_cache, block_tables, context_lens,
                              max_context_len, scale, partition_size=DEFAULT_PARTITION_SIZE,
                              k_scale=1.0, v_scale=1.0, dev_status=None, stream=None) -> None:
    """The partitioned decode without a caller workspace, for callers that
    cannot allocate device memory (a serving loop whose memory all sits in a
    fixed pool, a plugin whose host program owns every allocation). The
    library uses a fixed STATIC_WORKSPACE_BYTES array of its own, shared by
    every call: calls that overlap on the GPU race. Nothing here allocates.
    Problems needing a larger workspace raise PagedKVError (workspace)."""
    S, Hq, D, nb, Hkv, B, mb = _decode_dims(query, k_cache, block_tables, context_lens)
    need = workspace_bytes(S, Hq, D, max_context_len, partition_size)
    status = lib().pa_decode_partitioned_static(
        _ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb,
        _ptr(context_lens), S, Hq, Hkv, D, B, nb, int(max_context_len), float(scale),
        _dtype(query), _dtype(k_cache), float(k_scale), float(v_scale), partition_size,
        _ptr(dev_status), _stream(stream))
    if status == PA_ERR_WORKSPACE and need > STATIC_WORKSPACE_BYTES:
        raise PagedKVError(f"pa_decode_partitioned_static: the problem needs {need} bytes of "
                           f"workspace, above the fixed {STATIC_WORKSPACE_BYTES}", status)
    _check(status, "pa_decode_partitioned_static")


def partition_size(num_seqs, num_kv_heads, max_context_len) -> int:
    """The library's partition size for this device (512, 1024 or 2048)."""
    return int(lib().pa_decode_partition_size(num_seqs, num_kv_heads, int(max_context_len)))


def choose(num_seqs, num_q_heads, num_kv_heads, max_context_len,
           partition_size=DEFAULT_PARTITION_SIZE) -> int:
    """0 = single pass, 1 = partitioned."""
    return int(lib().pa_decode_choose(num_seqs, num_q_heads, num_kv_heads, int(max_context_len),
                                      partition_size))


def decode_auto(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
                workspace=None, partition_size=DEFAULT_PARTITION_SIZE, k_scale=1.0, v_scale=1.0,
                dev_status=None, stream=None) -> int:
    """Run the form `choose` picks; returns which (0 single pass, 1 split).
    A partitioned run without a workspace allocates one with torch."""
    S, Hq, D = query.shape
    Hkv = k_cache.shape[1]
    form = choose(S, Hq, Hkv, max_context_len, partition_size)
    if form == 0:
        decode(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
               k_scale, v_scale, dev_status, stream)
    else:
        if workspace is None:
            workspace = alloc_workspace(S, Hq, D, max_context_len, partition_size, query.device)
        decode_partitioned(out, query, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale, workspace, partition_size, k_scale, v_scale,
                           dev_status, stream)
    return form


def version() -> int:
    return int(lib().pa_version())


# ----------------------------------------------------------------------------- block management

def copy_blocks(k_cache, v_cache, block_pairs, dev_status=None, stream=None) -> None:
    """Copy whole blocks for each (src, dst) row of block_pairs ([n, 2] int64,
    on the device): the copy of copy-on-write."""
    nb, H, B, D = k_cache.shape
    if block_pairs.dtype != torch.int64 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be int64 [n, 2]")
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs),
                                block_pairs.shape[0], H, D, B, nb, _dtype(k_cache),
                                _ptr(dev_status), _stream(stream)), "pa_copy_blocks")


def selftest_wait(arrive: bool, dev_status, stream=None) -> None:
    """Launch the device check of the kernels' bounded waits: with arrive
    False both waits run out (about a second each, concurrently) and set
    DEV_TIMEOUT in dev_status; with arrive True nothing is set."""
    _check(lib().pa_selftest_wait(int(bool(arrive)), _ptr(dev_status), _stream(stream)),
           "pa_selftest_wait")


class BlockAllocator:
    """The library's host-side block allocator (free list + reference
    counts). Block ids are plain Python ints / int32 numpy arrays."""

    def __init__(self, num_blocks: int, block_size: int, reserve_block0: bool = True):
        self._lib = lib()
        self._h = self._lib.pa_allocator_create(num_blocks, block_size, int(reserve_block0))
        if not self._h:
            raise ValueError("invalid allocator arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pa_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free(self) -> int:
        return int(self._lib.pa_allocator_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pa_allocator_refcount(self._h, block))

    def allocate(self, num_tokens: int):
        """ceil(num_tokens / block_size) blocks (int32 array)."""
        import numpy as np
        n = -(-num_tokens // self.block_size)
        out = np.zeros(max(1, n), dtype=np.int32)
        got = ctypes.c_int64(0)
        _check(self._lib.pa_allocator_allocate(self._h, num_tokens, out.ctypes.data, out.size,
                                               ctypes.byref(got)), "pa_allocator_allocate")
        return out[:got.value].copy()

    def fork(self, blocks) -> None:
        import numpy as np
        b = np.ascontiguousarray(blocks, dtype=np.int32)
        _check(self._lib.pa_allocator_fork(self._h, b.ctypes.data, b.size), "pa_allocator_fork")

    def free(self, blocks) -> None:
        import numpy as np
        b = np.ascontiguousarray(blocks, dtype=np.int32)
        _check(self._lib.pa_allocator_free(self._h, b.ctypes.data, b.size), "pa_allocator_free")

    def append_slot(self, table, position: int):
        """Slot of the token at `position` for a sequence whose block table is
        `table` (an int32 numpy array of capacity entries, updated in place)
        holding `len` blocks: returns (slot, new_len, copy) with copy =
        (src, dst) when copy-on-write replaced a shared block, else None.
        Pass the table as (array, length)."""
        import numpy as np
        arr, length = table
        assert arr.dtype == np.int32 and arr.flags["C_CONTIGUOUS"]
        n = ctypes.c_int64(length)
        slot = ctypes.c_int64(0)
        src = ctypes.c_int32(0)
        dst = ctypes.c_int32(0)
        _check(self._lib.pa_allocator_append_slot(self._h, arr.ctypes.data, ctypes.byref(n),
                                                  arr.size, position, ctypes.byref(slot),
                                                  ctypes.byref(src), ctypes.byref(dst)),
               "pa_allocator_append_slot")
        copy = (int(src.value), int(dst.value)) if src.value >= 0 else None
        return int(slot.value), int(n.value), copy


class RadixAllocator:
    """The library's prefix-caching block allocator (a radix trie from token
    sequences to blocks, LRU eviction of unused cached sequences)."""

    def __init__(self, num_blocks: int, block_size: int, reserve_block0: bool = True):
        self._lib = lib()
        self._h = self._lib.pa_radix_create(num_blocks, block_size, int(reserve_block0))
        if not self._h:
            raise ValueError("invalid allocator arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pa_radix_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free(self) -> int:
        return int(self._lib.pa_radix_num_free(self._h))

    @property
    def num_cached(self) -> int:
        return int(self._lib.pa_radix_num_cached(self._h))

    @property
    def num_evictable(self) -> int:
        return int(self._lib.pa_radix_num_evictable(self._h))

    def allocate(self, prompt, total_tokens: int | None = None):
        """Blocks for a request with this prompt (int32 tokens) that may grow
        to total_tokens: returns (blocks, prefix_len, allocation_id)."""
        import numpy as np
        t = np.ascontiguousarray(prompt, dtype=np.int32)
        total = t.size if total_tokens is None else int(total_tokens)
        n = -(-total // self.block_size)
        out = np.zeros(max(1, n), dtype=np.int32)
        got, plen, aid = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.pa_radix_allocate(self._h, t.ctypes.data, t.size, total, out.ctypes.data,
                                           out.size, ctypes.byref(got), ctypes.byref(plen),
                                           ctypes.byref(aid)), "pa_radix_allocate")
        return out[:got.value].copy(), int(plen.value), int(aid.value)

    def free(self, allocation_id: int, tokens) -> None:
        """End a request; `tokens` are those its blocks now hold."""
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(self._lib.pa_radix_free(self._h, int(allocation_id), t.ctypes.data, t.size),
               "pa_radix_free")
