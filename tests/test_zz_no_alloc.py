"""The partitioned decode that allocates nothing (pa_decode_partitioned_static),
for callers that cannot allocate device memory. Called through the C ABI and
compared with pa_decode_partitioned (caller workspace) on two calls in a row
with different inputs, since every call shares the library's fixed workspace.
Collected last on purpose: it holds no state the other tests depend on."""
import numpy as np
import pytest
import torch

from gpu_common import DeviceCase, TOL, rounding_allowance, to_f64
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_static_workspace_matches_caller_workspace():
    c = W.config_case(3, num_seqs=64)
    d = DeviceCase(c)
    d.write_step()
    P = 512
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    assert pk.workspace_bytes(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P) \
        <= pk.STATIC_WORKSPACE_BYTES
    queries = [d.query, torch.flip(d.query, dims=[0]).contiguous()]
    for call, q in enumerate(queries):
        ref = torch.empty_like(d.out)
        pk.decode_partitioned(ref, q, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                              c.max_context_len, c.scale, ws, P, dev_status=d.status)
        got = torch.empty_like(d.out)
        pk.decode_partitioned_static(got, q, d.k_cache, d.v_cache, d.block_tables,
                                     d.context_lens, c.max_context_len, c.scale, P,
                                     dev_status=d.status)
        torch.cuda.synchronize()
        assert d.status_bits() == 0
        a, b = to_f64(got), to_f64(ref)
        bound = TOL[c.cache_dtype] + rounding_allowance(b, c.q_dtype)
        assert np.all(np.abs(a - b) <= bound), f"call {call}: max diff {np.abs(a - b).max()}"


def test_static_workspace_rejects_oversized_problem():
    c = W.config_case(3, num_seqs=4)
    d = DeviceCase(c)
    too_long = 1 << 22          # 4M-token bound: partials exceed the fixed workspace
    assert pk.workspace_bytes(4, 32, 128, too_long, 512) > pk.STATIC_WORKSPACE_BYTES
    with pytest.raises(pk.PagedKVError) as e:
        pk.decode_partitioned_static(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                                     d.context_lens, too_long, c.scale, 512)
    assert e.value.status == pk.PA_ERR_WORKSPACE
