"""The seeded input generator (CPU only): structure of the block pool and
tables it builds, determinism, and the poison pattern."""
import numpy as np
import pytest

from paged_kv_cache_141_gb300 import workloads as W


def _bits(a, dtype):
    return a.view({"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}[dtype])


@pytest.mark.parametrize("index", [1, 5])
def test_tables_and_pool(index):
    c = W.config_case(index)
    B = c.block_size
    used = {}
    for s in range(c.num_seqs):
        L = int(c.context_lens[s])
        n = -(-L // B)
        row = c.block_tables[s]
        assert np.all(row[:n] > 0) and np.all(row[:n] < c.num_blocks)
        assert np.all(row[n:] == 0)
        assert len(set(row[:n].tolist())) == n
        for j, p in enumerate(row[:n].tolist()):
            used.setdefault(p, set()).add((j, s))
        # the newest token's slot is position L-1 through the table
        slot = int(c.new_slots[s])
        assert slot // B == row[(L - 1) // B] and slot % B == (L - 1) % B
    # a physical block appears at one logical index only (shared by reference)
    for p, users in used.items():
        assert len({j for j, _ in users}) == 1
    assert 0 not in used


def test_config_shapes():
    c1 = W.config_case(1)
    assert (c1.num_seqs, c1.num_q_heads, c1.num_kv_heads, c1.head_size, c1.num_blocks) == (4, 4, 4, 64, 64)
    assert c1.context_lens.min() >= 1 and c1.context_lens.max() <= 64
    c5 = W.config_case(5)
    assert c5.num_seqs == 128 and c5.group == 8 and c5.cache_dtype == "e4m3"
    # 4 groups of 32 share their first 64 blocks
    for g in range(4):
        rows = c5.block_tables[g * 32:(g + 1) * 32, :64]
        assert np.all(rows == rows[0])
    assert len({tuple(c5.block_tables[g * 32, :64]) for g in range(4)}) == 4
    assert np.all(c5.context_lens >= 1024 + 16) and np.all(c5.context_lens <= 1024 + 512)
    assert 0 < c5.k_scale and 0 < c5.v_scale


def test_deterministic():
    a = W.config_case(1)
    b = W.config_case(1)
    for f in ("context_lens", "block_tables", "query", "k_cache", "v_cache", "new_key", "new_slots"):
        assert np.array_equal(getattr(a, f).view(np.uint8), getattr(b, f).view(np.uint8)), f
    c = W.config_case(1, seed=123)
    assert not np.array_equal(a.query, c.query)


def test_poison_marks_every_unowned_slot():
    c = W.config_case(1)
    B = c.block_size
    owned = np.zeros((c.num_blocks, B), bool)
    for s in range(c.num_seqs):
        L = int(c.context_lens[s])
        for pos in range(L - 1):
            owned[c.block_tables[s, pos // B], pos % B] = True
    kb = _bits(c.k_cache, "f32")
    nan = np.all(kb == np.uint32(0x7FC00000), axis=(1, 3))     # [nb, B]
    assert np.array_equal(nan, ~owned)
    assert np.isfinite(c.k_cache.transpose(0, 2, 1, 3)[owned]).all()


def test_loguniform_lengths():
    c = W.make_case(num_seqs=2000, num_q_heads=2, num_kv_heads=1, head_size=8, block_size=16,
                    q_dtype="bf16", cache_dtype="bf16", lengths=("loguniform", 512, 4096), seed=3)
    L = c.context_lens
    assert L.min() >= 512 and L.max() <= 4096
    # log-uniform: log-lengths have mean near (ln 512 + ln 4096) / 2
    assert abs(np.log(L).mean() - (np.log(512) + np.log(4096)) / 2) < 0.05


def test_make_queries_counts_and_determinism():
    from paged_kv_cache_141_gb300.workloads import make_case, make_queries
    c = make_case(num_seqs=6, num_q_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [0, 1, 5, 40, 17, 3]),
                  seed=3)
    a = make_queries(c, ("uniform", 2, 9))
    b = make_queries(c, ("uniform", 2, 9))
    assert np.array_equal(a.query, b.query) and np.array_equal(a.query_start, b.query_start)
    q = a.counts
    assert q[0] == 0 and q[1] == 1 and np.all(q <= c.context_lens) and np.all(q[2:] >= 2)
    assert a.query.shape == (int(a.query_start[-1]), 4, 64)
    assert a.max_queries == int(q.max())
    full = make_queries(c, ("all",))
    assert np.array_equal(full.counts, c.context_lens)


def test_unique_kv_bytes_counts_shared_prefix_blocks_once():
    from paged_kv_cache_141_gb300.workloads import ELEM_BYTES, make_case
    # no sharing: every context slot is distinct
    c = make_case(num_seqs=5, num_q_heads=4, num_kv_heads=2, head_size=64, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("uniform", 1, 300), seed=3)
    assert c.unique_kv_bytes() == c.kv_bytes()
    # 2 groups of 3 sequences sharing 4 blocks (64 tokens): the prefix counts
    # once per group, each private suffix once
    c = make_case(num_seqs=6, num_q_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                  q_dtype="bf16", cache_dtype="e4m3", lengths=("uniform", 1, 40), seed=4,
                  shared_prefix=(2, 4))
    prefix = c.meta["prefix_tokens"]
    tokens = 2 * prefix + int((c.context_lens.astype(np.int64) - prefix).sum())
    assert c.unique_kv_bytes() == 2 * tokens * 2 * 64 * ELEM_BYTES["e4m3"]
    assert c.unique_kv_bytes() < c.kv_bytes()
