"""The fused KV write + decode (pa_write_decode, pa_write_decode_partitioned)
against the separate write and decode: caches and outputs must be identical
bit for bit, for each decode kernel family."""
import numpy as np
import pytest
import torch

from gpu_common import DeviceCase, assert_decode_close, oracle_decode, oracle_pool, to_f64, torch_to_host
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    # cache, q, Hq, Hkv, D, B, lengths           (kernel family)
    ("bf16", "bf16", 32, 8, 128, 16, [1, 40, 511, 512, 513, 1500]),   # tensor-core
    ("f16", "f16", 16, 2, 64, 32, [2, 33, 700]),                       # tensor-core
    ("e4m3", "bf16", 64, 8, 128, 16, [1, 77, 1100]),                   # tensor-core, E4M3
    ("f16", "f16", 8, 8, 128, 16, [5, 300]),                           # CUDA-core TMA
    ("f32", "f32", 4, 4, 64, 16, [1, 17, 64]),                         # CUDA-core TMA
    ("bf16", "bf16", 8, 2, 128, 1, [3, 90]),                           # bulk copy
]


def _case(params, seed=31):
    cache, q, Hq, Hkv, D, B, lens = params
    return W.make_case(num_seqs=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_size=D,
                       block_size=B, q_dtype=q, cache_dtype=cache, lengths=("fixed", lens),
                       seed=seed)


@pytest.mark.parametrize("params", CASES, ids=[f"{c[0]}-q{c[2]}-kv{c[3]}-d{c[4]}-b{c[5]}" for c in CASES])
@pytest.mark.parametrize("split", [False, True])
def test_fused_equals_separate(params, split):
    c = _case(params)
    sep = DeviceCase(c)
    sep.write_step()
    ref = sep.decode("split" if split else "single", 512).clone()
    fused = DeviceCase(c)
    out = torch.empty_like(ref)
    if split:
        ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, 512)
        pk.write_decode_partitioned(out, fused.query, fused.new_key, fused.new_value, fused.k_cache,
                                    fused.v_cache, fused.new_slots, fused.block_tables,
                                    fused.context_lens, c.max_context_len, c.scale, ws, 512,
                                    c.k_scale, c.v_scale, fused.status)
    else:
        pk.write_decode(out, fused.query, fused.new_key, fused.new_value, fused.k_cache,
                        fused.v_cache, fused.new_slots, fused.block_tables, fused.context_lens,
                        c.max_context_len, c.scale, c.k_scale, c.v_scale, fused.status)
    assert fused.status_bits() == 0
    assert torch.equal(fused.k_cache.view(torch.uint8), sep.k_cache.view(torch.uint8))
    assert torch.equal(fused.v_cache.view(torch.uint8), sep.v_cache.view(torch.uint8))
    assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    kc, vc = oracle_pool(c)
    assert_decode_close(to_f64(out), oracle_decode(c, kc, vc), c, "fused")


def test_fused_slot_checks():
    c = _case(CASES[0])
    d = DeviceCase(c)
    slots = d.new_slots.clone()
    slots[1] = slots[2]                           # not sequence 1's newest position
    out = torch.empty_like(d.out)
    pk.write_decode(out, d.query, d.new_key, d.new_value, d.k_cache, d.v_cache, slots,
                    d.block_tables, d.context_lens, c.max_context_len, c.scale,
                    dev_status=d.status)
    assert d.status_bits() & pk.DEV_SLOT_MISMATCH
    d.status.zero_()
    slots = d.new_slots.clone()
    slots[0] = -1                                 # padding: nothing stored, decode still runs
    slots[3] = c.num_blocks * c.block_size        # outside the pool
    pk.write_decode(out, d.query, d.new_key, d.new_value, d.k_cache, d.v_cache, slots,
                    d.block_tables, d.context_lens, c.max_context_len, c.scale,
                    dev_status=d.status)
    assert d.status_bits() & pk.DEV_BAD_SLOT
