"""The hot path inside CUDA graphs: the library's calls are asynchronous on
the caller's stream and make no host synchronisation, so a whole decode step
(fused KV write + partition kernel + merge) and a multi-query launch can be
captured once and replayed; replays must give the eager results bit for bit."""
import numpy as np
import pytest
import torch

from gpu_common import DeviceCase, host_to_torch
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _step(dc, out, ws, P):
    c = dc.case
    pk.write_decode_partitions(dc.query, dc.new_key, dc.new_value, dc.k_cache, dc.v_cache,
                               dc.new_slots, dc.block_tables, dc.context_lens, c.max_context_len,
                               c.scale, ws, P, c.k_scale, c.v_scale, dc.status,
                               torch.cuda.current_stream())
    tmp, ml, es = pk.workspace_views(ws, c.num_seqs, c.num_q_heads, c.head_size,
                                     c.max_context_len, P)
    pk.merge(out, tmp, ml, es, dc.context_lens, P, dc.status, torch.cuda.current_stream())


@pytest.mark.parametrize("cfg", [3, 5], ids=["bf16", "e4m3"])
def test_decode_step_graph_replay(cfg):
    c = W.config_case(cfg, num_seqs=32)
    P = 512
    dc = DeviceCase(c)
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    eager = torch.empty_like(dc.out)
    _step(dc, eager, ws, P)                        # also sets the kernels' attributes
    torch.cuda.synchronize()
    assert dc.status_bits() == 0
    out = torch.full_like(dc.out, float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(dc, out, ws, P)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert dc.status_bits() == 0
        assert torch.equal(out.view(torch.uint8), eager.view(torch.uint8))


@pytest.mark.parametrize("cfg,qn,ordered", [(3, 100, False), (3, 4, False), (3, 8, True),
                                             (5, 100, False), (5, 16, True)],
                         ids=["tcgen05", "warp-mma", "warp-mma2-ordered", "tcgen05-e4m3-products",
                              "tcgen05-one-tile-e4m3-products-ordered"])
def test_multi_query_graph_replay(cfg, qn, ordered):
    c = W.config_case(cfg, num_seqs=16)
    q = W.make_queries(c, ("fixed", np.minimum(qn, c.context_lens)))
    dc = DeviceCase(c)
    dc.write_step()
    query = host_to_torch(q.query, c.q_dtype).cuda()
    qs = torch.from_numpy(q.query_start).cuda()
    order = torch.from_numpy(pk.longest_first(c.context_lens)).cuda() if ordered else None

    def run(out):
        pk.paged_prefill(out, query, qs, dc.k_cache, dc.v_cache, dc.block_tables,
                         dc.context_lens, q.max_queries, c.max_context_len, c.scale, c.k_scale,
                         c.v_scale, dc.status, torch.cuda.current_stream(), seq_order=order)

    eager = torch.empty_like(query)
    run(eager)
    torch.cuda.synchronize()
    assert dc.status_bits() == 0
    out = torch.full_like(query, float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run(out)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), eager.view(torch.uint8))
