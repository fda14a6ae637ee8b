"""The partitioned decode that allocates nothing (pa_decode_partitioned_static),
for callers that cannot allocate device memory: a serving loop whose device
memory is all in a fixed pool, or a plugin whose host program owns every
allocation. Called through the C ABI and compared with pa_decode_partitioned
(caller workspace), which runs the same kernels with the same partition size,
so the outputs must be identical bit for bit, on two calls in a row with
different inputs (every call shares the library's fixed workspace); both are
also checked against the oracle. Collected last on purpose, so that a run
stopping at the first failure has run every other test first."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_common import DeviceCase, assert_decode_close, oracle_decode, oracle_pool, to_f64
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# A shape whose workspace is exactly the fixed array's 64 MiB: 775 sequences x
# 8 query heads x 41 partitions of 512 tokens at head size 64 (254,200
# partition rows: 65,075,200 bytes of partial outputs, 2 x 1,016,832 of maxima
# and sums). One token more of max_context_len adds a partition.
LIMIT_SHAPE = dict(num_seqs=775, num_q_heads=8, head_size=64, max_context_len=41 * 512, P=512)


def run_both(d, c, q, P, max_context_len=None):
    """(static, caller workspace) outputs for query q."""
    mcl = c.max_context_len if max_context_len is None else max_context_len
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, mcl, P)
    ws.fill_(0xFF)                          # NaN patterns: an unwritten partial shows
    ref = torch.empty_like(d.out)
    pk.decode_partitioned(ref, q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, mcl,
                          c.scale, ws, P, c.k_scale, c.v_scale, dev_status=d.status)
    got = torch.empty_like(d.out)
    pk.decode_partitioned_static(got, q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                                 mcl, c.scale, P, c.k_scale, c.v_scale, dev_status=d.status)
    torch.cuda.synchronize()
    return got, ref


def test_static_workspace_matches_caller_workspace():
    c = W.config_case(3, num_seqs=64)
    d = DeviceCase(c)
    d.write_step()
    P = 512
    assert pk.workspace_bytes(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P) \
        <= pk.STATIC_WORKSPACE_BYTES
    kc, vc = oracle_pool(c)
    queries = [(d.query, c.query),
               (torch.flip(d.query, dims=[0]).contiguous(), np.ascontiguousarray(c.query[::-1]))]
    for call, (q, q_host) in enumerate(queries):
        got, ref = run_both(d, c, q, P)
        assert d.status_bits() == 0
        assert torch.equal(got, ref), f"call {call}: static and caller workspace differ"
        want = oracle_decode(dataclasses.replace(c, query=q_host), kc, vc)
        assert_decode_close(to_f64(got), want, c, f"static workspace, call {call}")


def test_static_workspace_at_the_exact_limit():
    s = LIMIT_SHAPE
    need = pk.workspace_bytes(s["num_seqs"], s["num_q_heads"], s["head_size"],
                              s["max_context_len"], s["P"])
    assert need == pk.STATIC_WORKSPACE_BYTES
    c = W.make_case(num_seqs=s["num_seqs"], num_q_heads=s["num_q_heads"], num_kv_heads=2,
                    head_size=s["head_size"], block_size=16, q_dtype="bf16", cache_dtype="bf16",
                    lengths=("uniform", 1, 1200), seed=77)
    d = DeviceCase(c)
    d.write_step()
    got, ref = run_both(d, c, d.query, s["P"], s["max_context_len"])
    assert d.status_bits() == 0
    assert torch.equal(got, ref)
    kc, vc = oracle_pool(c)
    assert_decode_close(to_f64(got), oracle_decode(c, kc, vc), c, "static workspace at the limit")
    with pytest.raises(pk.PagedKVError) as e:              # one partition more: rejected
        pk.decode_partitioned_static(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                                     d.context_lens, s["max_context_len"] + 1, c.scale, s["P"])
    assert e.value.status == pk.PA_ERR_WORKSPACE


def test_static_workspace_length_past_the_table_reads_no_stale_partials():
    """A context length past what the block table can hold (a data error)
    is clamped to the table by the partition kernel and the merge alike: the
    merge reads only partials this call wrote, never the previous call's,
    and the output equals the caller-workspace path's (whose workspace starts
    as NaN patterns) bit for bit."""
    long = W.config_case(3, num_seqs=32)
    dl = DeviceCase(long)
    dl.write_step()
    got, ref = run_both(dl, long, dl.query, 512)          # fills the array with partials
    assert torch.equal(got, ref)
    # sequence 2 fills its 44-block table exactly (704 tokens, all written)
    c = W.make_case(num_seqs=4, num_q_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                    q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [300, 40, 704, 100]),
                    seed=78)
    d = DeviceCase(c)
    d.write_step()
    table_tokens = c.block_tables.shape[1] * c.block_size
    assert table_tokens == 704
    d.context_lens[2] = table_tokens + 600                  # past the table, within the bound
    mcl = table_tokens + 1024
    got, ref = run_both(d, c, d.query, 512, mcl)
    assert d.status_bits() & pk.DEV_BAD_LEN
    assert torch.isfinite(got.float()).all()
    assert torch.equal(got, ref)


def test_static_workspace_rejects_oversized_problem():
    c = W.config_case(3, num_seqs=4)
    d = DeviceCase(c)
    too_long = 1 << 22          # 4M-token bound: partials exceed the fixed workspace
    assert pk.workspace_bytes(4, 32, 128, too_long, 512) > pk.STATIC_WORKSPACE_BYTES
    with pytest.raises(pk.PagedKVError) as e:
        pk.decode_partitioned_static(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                                     d.context_lens, too_long, c.scale, 512)
    assert e.value.status == pk.PA_ERR_WORKSPACE
