"""The C ABI without a GPU: the library builds, loads, and exports every
entry point include/pagedkv.h declares; host-only calls behave."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_141_gb300 import build
    build.build()
    from paged_kv_cache_141_gb300 import binding
    return binding.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pa_reshape_and_cache", "pa_decode", "pa_decode_partitions", "pa_merge",
                 "pa_decode_partitioned", "pa_decode_partitioned_workspace_bytes",
                 "pa_decode_choose", "pa_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_141_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z_0-9]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_host_only_calls(lib):
    from paged_kv_cache_141_gb300 import binding as pk
    assert pk.version() == 100
    assert pk.status_string(pk.PA_ERR_WORKSPACE).startswith("workspace")
    # workspace: three 256-byte aligned float32 regions
    n = pk.workspace_bytes(256, 32, 128, 4096, 512)
    parts = 256 * 32 * 8
    assert n == parts * 128 * 4 + 2 * parts * 4
    assert pk.partition_size(256, 8, 4096) in (512, 1024, 2048)
    assert pk.partition_size(8, 8, 131072) in (2048, 4096)   # long contexts: at most 4096
    assert pk.partition_size(4, 4, 64) == 512
    assert pk.workspace_bytes(3, 5, 64, 1, 512) % 256 == 0
    assert pk.max_partitions(0) == 1 and pk.max_partitions(513) == 2
    # one partition -> single pass, whatever the device
    assert pk.choose(4, 4, 4, 64) == 0
    assert pk.choose(0, 4, 4, 64) == 0


def test_argument_errors_before_any_launch(lib):
    import ctypes
    from paged_kv_cache_141_gb300 import binding as pk
    L = pk.lib()
    # NULL pointers with work to do, negative sizes, non-integer GQA group
    assert L.pa_decode(None, None, None, None, None, 4, None, 2, 8, 8, 128, 16, 10, 64, 0.1,
                       pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_decode(None, None, None, None, None, 4, None, 2, 8, 3, 128, 16, 10, 64, 0.1,
                       pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_reshape_and_cache(None, None, None, None, None, -1, 8, 128, 16, 10, pk.PA_BF16,
                                  pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    # zero work is a no-op even with NULL data pointers
    assert L.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 128, 16, 10, pk.PA_BF16,
                                  pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_OK
    assert L.pa_decode(None, None, None, None, None, 0, None, 0, 8, 8, 128, 16, 10, 0, 0.1,
                       pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_OK
    # unsupported combinations
    assert L.pa_decode(None, None, None, None, None, 4, None, 0, 8, 8, 96, 16, 10, 0, 0.1,
                       pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_UNSUPPORTED
    assert L.pa_reshape_and_cache(None, None, None, None, None, 1, 8, 128, 16, 10, pk.PA_BF16,
                                  pk.PA_F16, 1.0, 1.0, None, None) == pk.PA_ERR_UNSUPPORTED
    # workspace missing
    assert L.pa_decode_partitions(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                  ctypes.c_void_p(16), 4, ctypes.c_void_p(16), 2, 8, 8, 128, 16,
                                  10, 64, 0.1, pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, 512, None, 0,
                                  None, None) == pk.PA_ERR_WORKSPACE


def test_paged_prefill_argument_errors(lib):
    import ctypes
    from paged_kv_cache_141_gb300 import binding as pk
    L = pk.lib()
    v = ctypes.c_void_p(256)
    # (out, query, query_start, T, maxQ, k, v, tables, max_blocks, lens, S, Hq, Hkv, d, B,
    #  num_blocks, max_len, scale, q_dtype, cache_dtype, k_scale, v_scale, seq_order, status,
    #  stream)
    def call(T=4, maxq=2, S=2, scale=0.1, d=128, q=pk.PA_BF16, c=pk.PA_BF16, out=v, qs=v,
             order=None):
        return L.pa_paged_prefill(out, v, qs, T, maxq, v, v, v, 4, v, S, 8, 2, d, 16, 10, 64,
                                  scale, q, c, 1.0, 1.0, order, None, None)
    assert call(scale=0.0) == pk.PA_ERR_INVALID_ARG          # scale must be > 0
    assert call(scale=-1.0) == pk.PA_ERR_INVALID_ARG
    assert call(T=-1) == pk.PA_ERR_INVALID_ARG
    assert call(maxq=0) == pk.PA_ERR_INVALID_ARG             # queries but no per-sequence bound
    assert call(out=None) == pk.PA_ERR_INVALID_ARG
    assert call(qs=None) == pk.PA_ERR_INVALID_ARG
    assert call(d=96) == pk.PA_ERR_UNSUPPORTED
    assert call(q=pk.PA_BF16, c=pk.PA_F16) == pk.PA_ERR_UNSUPPORTED
    # nothing to do: no launch
    assert call(T=0, out=None, qs=None) == pk.PA_OK
    assert call(S=0, T=0) == pk.PA_OK
    assert call(S=0, T=3) == pk.PA_ERR_INVALID_ARG           # tokens without sequences
    assert call(order=ctypes.c_void_p(258)) == pk.PA_ERR_INVALID_ARG   # int32 order, 4 bytes


def test_misaligned_pointers_are_rejected_before_any_launch(lib):
    import ctypes
    from paged_kv_cache_141_gb300 import binding as pk
    L = pk.lib()
    ok, odd = ctypes.c_void_p(256), ctypes.c_void_p(264)      # 8-byte but not 16-byte aligned
    # decode: query, caches 16-byte aligned
    assert L.pa_decode(ok, odd, ok, ok, ok, 4, ok, 2, 8, 8, 128, 16, 10, 64, 0.1, pk.PA_BF16,
                       pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_decode(ok, ok, odd, ok, ok, 4, ok, 2, 8, 8, 128, 16, 10, 64, 0.1, pk.PA_BF16,
                       pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    # ... and int32 tables at 4 bytes
    assert L.pa_decode(ok, ok, ok, ok, ctypes.c_void_p(258), 4, ok, 2, 8, 8, 128, 16, 10, 64, 0.1,
                       pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    # the write: key/value 16 bytes, slots 8 bytes
    assert L.pa_reshape_and_cache(odd, ok, ok, ok, ok, 4, 8, 128, 16, 10, pk.PA_BF16, pk.PA_BF16,
                                  1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_reshape_and_cache(ok, ok, ok, ok, ctypes.c_void_p(260), 4, 8, 128, 16, 10,
                                  pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None) == pk.PA_ERR_INVALID_ARG
    # copy-on-write copies
    assert L.pa_copy_blocks(odd, ok, ok, 2, 8, 128, 16, 10, pk.PA_BF16, None,
                            None) == pk.PA_ERR_INVALID_ARG
    # merge: out and partials
    assert L.pa_merge(odd, ok, ok, ok, ok, 2, 8, 128, 512, 4, pk.PA_BF16, None,
                      None) == pk.PA_ERR_INVALID_ARG
    # multi-query: out 16 bytes, query_start 4 bytes
    assert L.pa_paged_prefill(odd, ok, ok, 4, 2, ok, ok, ok, 4, ok, 2, 8, 2, 128, 16, 10, 64, 0.1,
                              pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None,
                              None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_paged_prefill(ok, ok, ctypes.c_void_p(258), 4, 2, ok, ok, ok, 4, ok, 2, 8, 2, 128,
                              16, 10, 64, 0.1, pk.PA_BF16, pk.PA_BF16, 1.0, 1.0, None, None,
                              None) == pk.PA_ERR_INVALID_ARG


def test_wait_selftest_argument_errors(lib):
    import ctypes
    from paged_kv_cache_141_gb300 import binding as pk
    L = pk.lib()
    assert L.pa_selftest_wait(0, None, None) == pk.PA_ERR_INVALID_ARG       # status required
    assert L.pa_selftest_wait(2, ctypes.c_void_p(256), None) == pk.PA_ERR_INVALID_ARG
    assert L.pa_selftest_wait(1, ctypes.c_void_p(258), None) == pk.PA_ERR_INVALID_ARG


def test_longest_first_is_a_stable_permutation():
    """The host-side order helper for pa_paged_prefill's seq_order: a
    permutation of the sequences, non-increasing lengths, ties in index order,
    int32 (the ABI's type)."""
    import numpy as np
    from paged_kv_cache_141_gb300 import binding as pk
    lens = np.array([5, 900, 12, 900, 0, 4096, 12], dtype=np.int32)
    order = pk.longest_first(lens)
    assert order.dtype == np.int32
    assert sorted(order.tolist()) == list(range(len(lens)))
    assert order.tolist() == [5, 1, 3, 2, 6, 0, 4]
    assert np.all(np.diff(lens[order]) <= 0)
    assert pk.longest_first(np.zeros(0, dtype=np.int32)).shape == (0,)


def test_paged_prefill_rejects_a_misshaped_order():
    """seq_order must be int32 [num_seqs]: the binding checks before the call."""
    import pytest
    import torch
    from paged_kv_cache_141_gb300 import binding as pk
    S, Hq, Hkv, D, B = 2, 8, 2, 128, 16
    q = torch.zeros(3, Hq, D, dtype=torch.bfloat16)
    kc = torch.zeros(4, Hkv, B, D, dtype=torch.bfloat16)
    qs = torch.tensor([0, 1, 3], dtype=torch.int32)
    bt = torch.zeros(S, 2, dtype=torch.int32)
    cl = torch.tensor([5, 9], dtype=torch.int32)
    for bad in (torch.zeros(S, dtype=torch.int64), torch.zeros(S + 1, dtype=torch.int32)):
        with pytest.raises(ValueError):
            pk.paged_prefill(q, q, qs, kc, kc, bt, cl, 2, 32, 0.1, seq_order=bad)


def test_paged_prefill_kernel_selection(lib):
    """The kernel choice of pa_paged_prefill, host only: warp-level MMA up to
    32 rows per (sequence, KV head) (16 at head size 256), one or two n-tiles
    per warp by 16 rows, except where the tcgen05 kernels take the E4M3
    products (E4M3 cache, bf16 query, head size 128: tcgen05 from 17 rows,
    the two-n-tile kernel only where tcgen05 is not eligible, e.g. block
    size 96); tcgen05 above (two query tiles per CTA at head size <= 128
    with two or more tiles); CUDA cores for the
    other types and block sizes; -1 for what the call rejects."""
    from paged_kv_cache_141_gb300 import binding as pk
    B16, F16, F32, E4 = pk.PA_BF16, pk.PA_F16, pk.PA_F32, pk.PA_FP8_E4M3
    cases = [
        # (max_queries, Hq, Hkv, d, B, q, cache) -> kernel
        ((1, 32, 8, 128, 16, B16, B16), "mma"),
        ((4, 32, 8, 128, 16, B16, B16), "mma"),
        ((5, 32, 8, 128, 16, B16, B16), "mma_two_tiles"),
        ((8, 32, 8, 128, 16, B16, B16), "mma_two_tiles"),
        ((9, 32, 8, 128, 16, B16, B16), "tc"),
        ((32, 32, 8, 128, 16, B16, B16), "tc"),
        ((33, 32, 8, 128, 16, B16, B16), "tc_two_tiles"),
        ((512, 32, 8, 128, 16, B16, B16), "tc_two_tiles"),
        ((8, 32, 8, 128, 8, B16, B16), "mma_two_tiles"),
        ((2, 64, 8, 128, 16, B16, E4), "mma"),
        ((3, 64, 8, 128, 16, B16, E4), "tc"),
        ((4, 64, 8, 128, 16, B16, E4), "tc"),
        ((4, 64, 8, 128, 96, B16, E4), "mma_two_tiles"),
        ((4, 64, 8, 128, 16, F16, E4), "mma_two_tiles"),
        ((8, 32, 8, 64, 16, B16, E4), "tc"),
        ((5, 64, 8, 128, 16, B16, E4), "tc"),
        ((16, 64, 8, 128, 16, B16, E4), "tc"),
        ((17, 64, 8, 128, 16, B16, E4), "tc_two_tiles"),
        ((512, 64, 8, 128, 16, B16, E4), "tc_two_tiles"),
        ((512, 32, 8, 64, 16, F16, E4), "tc_two_tiles"),
        ((4, 16, 4, 256, 16, F16, F16), "mma"),
        ((5, 16, 4, 256, 16, F16, F16), "tc"),
        ((200, 16, 4, 256, 16, F16, F16), "tc"),
        ((8, 16, 4, 256, 16, F16, E4), "cuda_cores"),
        ((4, 16, 4, 128, 24, B16, B16), "cuda_cores"),
        ((4, 16, 4, 128, 16, F32, F32), "cuda_cores"),
        ((32, 32, 32, 128, 16, F16, F16), "mma_two_tiles"),
        ((33, 32, 32, 128, 16, F16, F16), "tc"),
    ]
    for args, want in cases:
        assert pk.prefill_kernel(*args[:5], 1000, *args[5:]) == want, (args, want)
    L = pk.lib()
    assert L.pa_paged_prefill_kernel(0, 32, 8, 128, 16, 1000, B16, B16) == -1
    assert L.pa_paged_prefill_kernel(4, 30, 8, 128, 16, 1000, B16, B16) == -1
    assert L.pa_paged_prefill_kernel(4, 32, 8, 96, 16, 1000, B16, B16) == -1
    assert L.pa_paged_prefill_kernel(4, 32, 8, 128, 16, 1000, B16, F16) == -1


def test_static_workspace_capacity_examples():
    """The capacities pa_decode_partitioned_static's declaration quotes, and
    the exact-limit shape the GPU test runs (workspace sizing is host only)."""
    from paged_kv_cache_141_gb300 import binding as pk
    limit = pk.STATIC_WORKSPACE_BYTES
    assert limit == 64 * 1024 * 1024
    assert pk.workspace_bytes(256, 32, 128, 7680, 512) == 63_897_600 <= limit
    assert pk.workspace_bytes(256, 32, 128, 15360, 1024) <= limit
    assert pk.workspace_bytes(256, 32, 128, 8192, 512) == 68_157_440 > limit
    # 775 x 8 heads x 41 partitions at head size 64: exactly the array
    assert pk.workspace_bytes(775, 8, 64, 41 * 512, 512) == limit
    assert pk.workspace_bytes(775, 8, 64, 41 * 512 + 1, 512) > limit


def test_static_call_rejects_oversized_problem_without_a_device():
    """The size check runs before any CUDA call."""
    from paged_kv_cache_141_gb300 import binding as pk
    L = pk.lib()
    st = L.pa_decode_partitioned_static(None, None, None, None, None, 1, None, 775, 8, 2, 64, 16,
                                        64, 41 * 512 + 1, 0.125, pk.PA_BF16, pk.PA_BF16, 1.0, 1.0,
                                        512, None, None)
    assert st == pk.PA_ERR_WORKSPACE
