"""The shared-prefix decode step (pa_write_decode_shared_prefix) on the GPU:
units of sequences whose block tables share their leading partitions read
each shared partition once for all members. Outputs against the oracle
(two-part check) on the full shared-prefix E4M3 pool with the step's KV
write fused, on small 16-bit and E4M3 shapes, with the device checks of a
unit's rules (a member too short for its unit's partitions is computed by
the partition kernel instead; a member whose table differs is flagged), and
with no units (the partitioned step, bit for bit)."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_common import (DeviceCase, assert_decode_close, oracle_decode, oracle_decode_all,
                        oracle_pool, to_f64, torch_to_host)
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_shared(d, c, P, plan, fused=True, context_lens=None, max_context_len=None):
    sp, us, up = plan.to(d.query.device)
    mcl = c.max_context_len if max_context_len is None else max_context_len
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, mcl, P)
    ws.fill_(0xFF)                                     # NaN patterns: an unwritten partial shows
    kw = dict(key=d.new_key, value=d.new_value, slot_mapping=d.new_slots) if fused else {}
    pk.write_decode_shared_prefix(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                                  d.context_lens if context_lens is None else context_lens, mcl,
                                  c.scale, ws, sp, us, up, plan.max_unit_parts, P,
                                  k_scale=c.k_scale, v_scale=c.v_scale, dev_status=d.status, **kw)
    torch.cuda.synchronize()
    return d.out


def test_shared_prefix_pool_full_size():
    """The shared-prefix E4M3 pool (128 sequences in 4 groups of 32 sharing
    a 1024-token prefix): 32 units of 4 sharing 2 partitions, the step's KV
    write fused; caches bit for bit and every sequence against the oracle."""
    c = W.config_case(5)
    d = DeviceCase(c)
    P = 512
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, P)
    assert plan.num_units == 32
    got = to_f64(run_shared(d, c, P, plan))
    assert d.status_bits() == 0
    kc, vc = oracle_pool(c)
    assert np.array_equal(torch_to_host(d.k_cache, c.cache_dtype).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(torch_to_host(d.v_cache, c.cache_dtype).view(np.uint8), vc.view(np.uint8))
    assert_decode_close(got, oracle_decode_all(c, kc, vc), c,
                        f"full: {c.name}, shared-prefix step, all {c.num_seqs} sequences")


SHAPES = [
    # cache, q, Hq, Hkv, D, B, P, S, (groups, prefix blocks), suffix lengths
    ("bf16", "bf16", 8, 2, 128, 16, 64, 12, (3, 8), ("uniform", 1, 150)),
    ("f16", "f16", 32, 32, 128, 16, 32, 10, (2, 4), ("uniform", 1, 90)),
    ("bf16", "bf16", 16, 2, 64, 32, 128, 6, (1, 12), ("uniform", 1, 300)),
    ("e4m3", "bf16", 8, 1, 128, 16, 64, 8, (2, 16), ("uniform", 1, 200)),
    ("e4m3", "f16", 64, 8, 128, 16, 512, 16, (4, 64), ("uniform", 16, 512)),
    ("bf16", "bf16", 16, 2, 256, 16, 64, 9, (3, 8), ("uniform", 1, 100)),
    ("e4m3", "bf16", 16, 2, 256, 16, 64, 9, (3, 8), ("uniform", 1, 100)),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}-q{s[2]}-kv{s[3]}-d{s[4]}-b{s[5]}-p{s[6]}"
                                               for s in SHAPES])
def test_shared_prefix_shapes(shape):
    cache, q, Hq, Hkv, D, B, P, S, shared, lens = shape
    c = W.make_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=D, block_size=B,
                    q_dtype=q, cache_dtype=cache, lengths=lens, shared_prefix=shared, seed=S * 7 + D)
    d = DeviceCase(c)
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, B, P)
    assert plan.num_units >= 1
    got = to_f64(run_shared(d, c, P, plan))
    assert d.status_bits() == 0
    kc, vc = oracle_pool(c)
    assert_decode_close(got, oracle_decode(c, kc, vc), c, "shared-prefix step")


def small_shared_case(seed=5):
    # 4 sequences sharing 8 blocks (128 tokens: two 64-token partitions)
    return W.make_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                       q_dtype="bf16", cache_dtype="bf16", lengths=("uniform", 20, 60),
                       shared_prefix=(1, 8), seed=seed)


def test_member_too_short_is_computed_by_the_partition_kernel():
    """A member whose context ends inside its unit's shared partitions is
    left to the partition kernel (same rule on both sides), the flag is
    set, and every output still matches the oracle."""
    c = small_shared_case()
    d = DeviceCase(c)
    d.write_step()
    P = 64
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, 16, P)
    assert plan.num_units == 1 and int(plan.unit_parts[0]) == 2
    lens = c.context_lens.copy()
    lens[2] = 128                                      # exactly the shared partitions
    dl = torch.from_numpy(lens).cuda()
    got = to_f64(run_shared(d, c, P, plan, fused=False, context_lens=dl))
    assert d.status_bits() & pk.DEV_BAD_PREFIX
    c2 = dataclasses.replace(c, context_lens=lens)
    kc, vc = oracle_pool(c)
    assert_decode_close(got, oracle_decode(c2, kc, vc), c, "member too short")


def test_member_with_another_table_is_flagged():
    c = small_shared_case(6)
    d = DeviceCase(c)
    d.write_step()
    P = 64
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, 16, P)
    assert plan.num_units == 1
    bt = d.block_tables.clone()
    free = int(c.num_blocks) - 1                       # a block no sequence uses
    bt[1, 5] = free
    sp, us, up = plan.to(d.query.device)
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    pk.write_decode_shared_prefix(d.out, d.query, d.k_cache, d.v_cache, bt, d.context_lens,
                                  c.max_context_len, c.scale, ws, sp, us, up, plan.max_unit_parts,
                                  P, dev_status=d.status)
    assert d.status_bits() & pk.DEV_BAD_PREFIX


def test_no_units_is_the_partitioned_step():
    c = W.config_case(3, num_seqs=24)
    d = DeviceCase(c)
    d.write_step()
    P = 512
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, P)
    assert plan.num_units == 0
    got = run_shared(d, c, P, plan, fused=False).clone()
    ref = torch.empty_like(got)
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    pk.decode_partitioned(ref, d.query, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                          c.max_context_len, c.scale, ws, P, dev_status=d.status)
    torch.cuda.synchronize()
    assert d.status_bits() == 0
    assert torch.equal(got, ref)


def test_host_argument_errors():
    c = small_shared_case()
    d = DeviceCase(c)
    P = 64
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, 16, P)
    sp, us, up = plan.to(d.query.device)
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    args = (d.out, d.query, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
            c.max_context_len, c.scale, ws, sp, us, up)
    with pytest.raises(pk.PagedKVError) as e:           # more partitions than the contexts have
        pk.write_decode_shared_prefix(*args, 99, P)
    assert e.value.status == pk.PA_ERR_INVALID_ARG
    with pytest.raises(pk.PagedKVError) as e:           # partition size not a multiple of 32
        pk.write_decode_shared_prefix(*args, plan.max_unit_parts, 72)
    assert e.value.status == pk.PA_ERR_INVALID_ARG


def test_shared_prefix_step_replays_in_a_cuda_graph():
    """The step (partition kernel with units, merge) captured once and
    replayed gives the eager launch's bits."""
    c = W.make_case(num_seqs=16, num_q_heads=64, num_kv_heads=8, head_size=128, block_size=16,
                    q_dtype="bf16", cache_dtype="e4m3", lengths=("uniform", 16, 300),
                    shared_prefix=(4, 16), seed=91)
    d = DeviceCase(c)
    d.write_step()
    P = 128
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size, P)
    sp, us, up = plan.to(d.query.device)
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)

    def step(stream=None):
        pk.write_decode_shared_prefix(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                                      d.context_lens, c.max_context_len, c.scale, ws, sp, us, up,
                                      plan.max_unit_parts, P, k_scale=c.k_scale, v_scale=c.v_scale,
                                      dev_status=d.status, stream=stream)

    step()
    torch.cuda.synchronize()
    eager = d.out.clone()
    assert d.status_bits() == 0
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        d.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d.out, eager)
    assert d.status_bits() == 0


@pytest.mark.parametrize("seed", range(8))
def test_shared_prefix_random_cases(seed):
    """Seeded random shapes: batch size, prefix groups and lengths, suffix
    lengths, cache type (bf16, f16, E4M3), GQA group, head size, block and
    partition sizes; the step with its KV write against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    cache = ["bf16", "f16", "e4m3"][seed % 3]
    q = "f16" if cache == "f16" else ("bf16" if seed % 2 else "f16")
    if cache == "bf16":
        q = "bf16"
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 128])) if cache != "e4m3" else 128
    B = int(rng.choice([16, 32]))
    P = int(rng.choice([32, 64, 128])) * (B // 16)
    groups = int(rng.integers(1, 4))
    per = int(rng.integers(1, 7))
    prefix_blocks = int(rng.integers(1, 5)) * (P // B)
    c = W.make_case(num_seqs=groups * per, num_q_heads=G * Hkv, num_kv_heads=Hkv, head_size=D,
                    block_size=B, q_dtype=q, cache_dtype=cache,
                    lengths=("uniform", 1, int(rng.integers(2, 3 * P))),
                    shared_prefix=(groups, prefix_blocks), seed=2000 + seed)
    d = DeviceCase(c)
    plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, B, P)
    got = to_f64(run_shared(d, c, P, plan))
    assert d.status_bits() == 0
    kc, vc = oracle_pool(c)
    assert_decode_close(got, oracle_decode(c, kc, vc), c,
                        f"shared-prefix random case {seed} ({plan.num_units} units)")
