"""The library's host-side block allocator (CPU only): block accounting,
reference counts, copy-on-write append, failure leaves state unchanged, and a
random allocate / fork / append / free stress run checked against a plain
Python model for duplicates, leaks and counts."""
import numpy as np
import pytest

from paged_kv_cache_141_gb300 import binding as pk


@pytest.fixture
def alloc():
    pk.lib()
    a = pk.BlockAllocator(33, 16)
    yield a
    a.close()


def test_accounting_and_reserved_block(alloc):
    assert alloc.num_free == 32
    seen = set()
    for tokens in (1, 16, 17, 48, 0):
        b = alloc.allocate(tokens)
        assert len(b) == -(-tokens // 16)
        assert 0 not in b
        assert not (seen & set(b.tolist()))
        seen |= set(b.tolist())
        assert all(alloc.refcount(int(x)) == 1 for x in b)
    assert alloc.num_free == 32 - len(seen)


def test_out_of_blocks_changes_nothing(alloc):
    b = alloc.allocate(16 * 30)
    with pytest.raises(pk.PagedKVError) as e:
        alloc.allocate(16 * 3)
    assert e.value.status == pk.PA_ERR_NO_BLOCKS
    assert alloc.num_free == 2
    alloc.free(b)
    assert alloc.num_free == 32


def test_fork_and_free_by_reference(alloc):
    b = alloc.allocate(40)
    alloc.fork(b)
    assert all(alloc.refcount(int(x)) == 2 for x in b)
    alloc.free(b)
    assert alloc.num_free == 32 - 3
    alloc.free(b)
    assert alloc.num_free == 32
    with pytest.raises(pk.PagedKVError):
        alloc.free(b)                       # double free
    with pytest.raises(pk.PagedKVError):
        alloc.fork(b)                       # forking free blocks


def test_append_slot_and_copy_on_write(alloc):
    cap = 8
    parent = np.zeros(cap, np.int32)
    n = 0
    slots = []
    for pos in range(20):                    # 20 tokens: blocks at 0 and 16
        slot, n, copy = alloc.append_slot((parent, n), pos)
        assert copy is None
        slots.append(slot)
    assert n == 2 and slots[0] == parent[0] * 16 and slots[19] == parent[1] * 16 + 3
    child = parent.copy()
    alloc.fork(child[:n])                    # the child shares both blocks
    slot, n2, copy = alloc.append_slot((child, n), 20)
    assert copy == (int(parent[1]), int(child[1])) and child[1] != parent[1]
    assert slot == child[1] * 16 + 4
    assert alloc.refcount(int(parent[1])) == 1 and alloc.refcount(int(child[1])) == 1
    assert alloc.refcount(int(parent[0])) == 2
    slot, n, copy = alloc.append_slot((parent, n), 20)   # parent's block is private again
    assert copy is None and slot == parent[1] * 16 + 4
    with pytest.raises(pk.PagedKVError):
        alloc.append_slot((parent, n), 40)               # skips a block


def test_random_stress_against_model():
    rng = np.random.default_rng(2024)
    N, B = 257, 8
    a = pk.BlockAllocator(N, B)
    model_refs = np.zeros(N, np.int64)
    seqs = {}            # id -> (table array, len, tokens)
    nid = 0
    for step in range(20000):
        op = rng.integers(0, 4)
        if op == 0 or not seqs:                                  # new sequence
            t = int(rng.integers(1, 60))
            need = -(-t // B)
            if need > a.num_free:
                with pytest.raises(pk.PagedKVError):
                    a.allocate(t)
                continue
            b = a.allocate(t)
            tab = np.zeros(64, np.int32)
            tab[:len(b)] = b
            model_refs[b] += 1
            seqs[nid] = (tab, len(b), t)
            nid += 1
        elif op == 1:                                            # fork
            k = list(seqs)[int(rng.integers(0, len(seqs)))]
            tab, n, t = seqs[k]
            a.fork(tab[:n])
            model_refs[tab[:n]] += 1
            seqs[nid] = (tab.copy(), n, t)
            nid += 1
        elif op == 2:                                            # append a token
            k = list(seqs)[int(rng.integers(0, len(seqs)))]
            tab, n, t = seqs[k]
            if t >= 64 * B:
                continue
            j = t // B
            needs_block = j == n or model_refs[tab[j]] > 1
            if needs_block and a.num_free == 0:
                with pytest.raises(pk.PagedKVError):
                    a.append_slot((tab, n), t)
                continue
            old = int(tab[j]) if j < n else None
            slot, n2, copy = a.append_slot((tab, n), t)
            if j == n:
                model_refs[tab[j]] += 1
                assert copy is None
            elif old is not None and copy is not None:
                assert copy[0] == old and model_refs[old] > 1
                model_refs[old] -= 1
                model_refs[tab[j]] += 1
            assert slot == int(tab[j]) * B + t % B
            seqs[k] = (tab, n2, t + 1)
        else:                                                    # finish a sequence
            k = list(seqs)[int(rng.integers(0, len(seqs)))]
            tab, n, t = seqs.pop(k)
            a.free(tab[:n])
            model_refs[tab[:n]] -= 1
        if step % 500 == 0 or step == 19999:
            held = [b for tab, n, _ in seqs.values() for b in tab[:n].tolist()]
            counts = np.bincount(np.array(held, dtype=np.int64), minlength=N) if held else np.zeros(N)
            assert np.array_equal(counts, model_refs)
            for b in range(N):
                assert a.refcount(b) == model_refs[b]
            assert a.num_free == (N - 1) - int((model_refs > 0).sum())   # no leaks, no duplicates
            assert model_refs[0] == 0
    a.close()
