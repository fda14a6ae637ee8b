"""The shared-prefix planner (pa_shared_prefix_plan, host only): its units
are valid (members' block tables agree over the shared partitions, which lie
wholly before each member's newest token; every sequence in at most one
unit; skip counts equal the unit's), it finds the sharing the workloads
build (the shared-prefix E4M3 pool: 32 units of 4 sharing the 1024-token
prefix), prefers the larger saving, and checks its arguments."""
import numpy as np
import pytest

from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_141_gb300 import build
    build.build()


def check_plan(bt, cl, B, P, plan):
    bpp = P // B
    seen = set()
    assert plan.unit_seqs.shape == (plan.num_units, pk.SHARED_UNIT_MEMBERS)
    for u in range(plan.num_units):
        mem = [int(s) for s in plan.unit_seqs[u] if s >= 0]
        parts = int(plan.unit_parts[u])
        assert len(mem) >= 2 and parts >= 1
        assert list(plan.unit_seqs[u][:len(mem)]) == mem          # padding at the end
        for s in mem:
            assert s not in seen
            seen.add(s)
            assert plan.seq_shared_parts[s] == parts
            assert cl[s] > parts * P                              # newest token past the prefix
            assert np.array_equal(bt[s, :parts * bpp], bt[mem[0], :parts * bpp])
        assert parts <= plan.max_unit_parts
    for s in range(len(cl)):
        if s not in seen:
            assert plan.seq_shared_parts[s] == 0
    return seen


def test_plan_of_the_shared_prefix_workload():
    c = W.config_case(5)
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, 512)
    seen = check_plan(c.block_tables, c.context_lens, c.block_size, 512, plan)
    assert plan.num_units == 32 and plan.max_unit_parts == 2 and len(seen) == 128
    assert np.all(plan.unit_parts == 2)
    # 1024-token partitions: the prefix is one partition
    plan2 = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, 1024)
    check_plan(c.block_tables, c.context_lens, c.block_size, 1024, plan2)
    assert np.all(plan2.unit_parts == 1) and plan2.num_units == 32


def test_no_sharing_gives_no_units():
    c = W.config_case(3, num_seqs=40)
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, 512)
    assert plan.num_units == 0 and plan.max_unit_parts == 0
    assert not plan.seq_shared_parts.any()


def test_random_trees_of_shared_prefixes():
    """Tables drawn as a random tree of shared block runs (a radix trie's
    picture): every plan is valid."""
    rng = np.random.default_rng(4)
    B, P = 16, 64
    for trial in range(30):
        S = int(rng.integers(2, 40))
        mb = 24
        nxt = [1]

        def fresh(n):
            out = np.arange(nxt[0], nxt[0] + n, dtype=np.int32)
            nxt[0] += n
            return out

        roots = [fresh(mb) for _ in range(int(rng.integers(1, 4)))]
        bt = np.zeros((S, mb), np.int32)
        for s in range(S):
            r = roots[int(rng.integers(len(roots)))]
            keep = int(rng.integers(0, mb + 1))
            bt[s, :keep] = r[:keep]
            bt[s, keep:] = fresh(mb - keep)
        cl = rng.integers(1, mb * B + 1, S).astype(np.int32)
        plan = pk.shared_prefix_plan(bt, cl, B, P)
        check_plan(bt, cl, B, P, plan)


def test_prefers_the_larger_saving():
    """Three sequences sharing five partitions and a fourth sharing one:
    one unit of three at five partitions (saving 2 x 5) beats four at one
    (saving 3 x 1)."""
    B, P = 16, 32
    base = np.arange(1, 13, dtype=np.int32)
    bt = np.stack([base, base, base, base]).copy()
    bt[3, 2:] = np.arange(100, 110, dtype=np.int32)       # differs after the first partition
    cl = np.full(4, 12 * B, np.int32)
    plan = pk.shared_prefix_plan(bt, cl, B, P)
    check_plan(bt, cl, B, P, plan)
    assert plan.num_units == 1 and int(plan.unit_parts[0]) == 5      # (192 - 1) // 32
    assert sorted(int(s) for s in plan.unit_seqs[0] if s >= 0) == [0, 1, 2]


def test_argument_errors():
    L = pk.lib()
    import ctypes
    n, m = ctypes.c_int(0), ctypes.c_int(0)
    bt = np.zeros((2, 4), np.int32)
    cl = np.ones(2, np.int32)
    out = np.zeros(2, np.int32)
    us = np.zeros(8, np.int32)
    up = np.zeros(2, np.int32)
    args = [bt.ctypes.data, cl.ctypes.data, 2, 4]
    tail = [out.ctypes.data, us.ctypes.data, up.ctypes.data, 2, ctypes.byref(n), ctypes.byref(m)]
    assert L.pa_shared_prefix_plan(*args, 16, 48, *tail) == pk.PA_ERR_INVALID_ARG   # not /32
    assert L.pa_shared_prefix_plan(*args, 24, 64, *tail) == pk.PA_ERR_INVALID_ARG   # B does not divide P
    assert L.pa_shared_prefix_plan(*args, 0, 64, *tail) == pk.PA_ERR_INVALID_ARG
    assert L.pa_shared_prefix_plan(*args, 16, 64, out.ctypes.data, us.ctypes.data, up.ctypes.data,
                                   2, None, ctypes.byref(m)) == pk.PA_ERR_INVALID_ARG
    assert L.pa_shared_prefix_plan(*args, 16, 64, *tail) == pk.PA_OK
