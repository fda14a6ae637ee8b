"""The prefix-caching radix allocator (host only): prefix reuse at block
granularity, node splits where sequences part, LRU eviction of unused cached
sequences, protection of prefixes in use, argument checks, and a random
stress run checked by simulating the KV contents each block must hold."""
import numpy as np
import pytest

from paged_kv_cache_141_gb300 import binding as pk


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_141_gb300 import build
    build.build()


def test_reuse_whole_blocks_only():
    a = pk.RadixAllocator(64, 4)
    prompt = np.arange(10)
    blocks, plen, aid = a.allocate(prompt, 14)
    assert plen == 0 and len(blocks) == 4 and 0 not in blocks
    a.free(aid, np.arange(14))               # 3 whole blocks cached, the 4th returned
    assert a.num_cached == 3 and a.num_free == 63 - 3
    b2, plen2, aid2 = a.allocate(prompt, 12)
    assert plen2 == 8                        # the prompt covers 2 of the cached blocks
    assert list(b2[:2]) == list(blocks[:2]) and len(b2) == 3
    assert b2[2] not in blocks[:3]
    a.free(aid2, prompt)


def test_block_size_two_five_token_prompt():
    a = pk.RadixAllocator(32, 2)
    _, _, aid = a.allocate([7, 8, 9, 10, 11])
    a.free(aid, [7, 8, 9, 10, 11])
    assert a.num_cached == 2                 # [7,8] [9,10]; the lone 11 is not shared
    _, plen, aid = a.allocate([7, 8, 9, 10, 11])
    assert plen == 4
    a.free(aid, [7, 8, 9, 10, 11])


def test_partial_overlap_splits_and_both_branches_are_reused():
    a = pk.RadixAllocator(64, 2)
    A = list(range(12))
    bA, _, ida = a.allocate(A)
    a.free(ida, A)
    C = list(range(6)) + [99, 98, 97, 96]
    bC, plen, idc = a.allocate(C)
    assert plen == 6 and list(bC[:3]) == list(bA[:3])
    a.free(idc, C)
    assert a.num_cached == 6 + 2             # A's 6 blocks, C's own 2
    _, pa_, i1 = a.allocate(A)
    _, pc_, i2 = a.allocate(C)
    assert pa_ == 12 and pc_ == 10
    a.free(i1, A)
    a.free(i2, C)


def test_lru_eviction_order():
    a = pk.RadixAllocator(9, 4)              # 8 usable blocks
    X, Y = list(range(100, 108)), list(range(200, 208))
    _, _, ix = a.allocate(X)
    a.free(ix, X)                            # older
    _, _, iy = a.allocate(Y)
    a.free(iy, Y)                            # newer
    assert a.num_free == 4 and a.num_cached == 4
    big, plen, ib = a.allocate(list(range(300, 320)), 24)   # 6 blocks: evicts 2
    assert plen == 0 and len(big) == 6
    assert a.num_cached == 2
    a.free(ib, [])
    _, px, i1 = a.allocate(X)
    _, py, i2 = a.allocate(Y)
    assert px == 0 and py == 8               # X went first
    a.free(i1, X)
    a.free(i2, Y)


def test_prefix_in_use_is_not_evicted():
    a = pk.RadixAllocator(9, 4)
    X = list(range(8))
    _, _, ix = a.allocate(X)
    a.free(ix, X)
    _, plen, hold = a.allocate(X)            # holds the cached prefix
    assert plen == 8
    before = (a.num_free, a.num_cached)
    with pytest.raises(pk.PagedKVError):
        a.allocate(list(range(50, 74)), 28)  # 7 blocks: only 6 could be had
    assert (a.num_free, a.num_cached) == before
    a.free(hold, X)
    got, _, i = a.allocate(list(range(50, 82)), 32)   # now the prefix may go
    assert len(got) == 8
    a.free(i, [])


def test_argument_errors():
    a = pk.RadixAllocator(16, 4)
    _, _, aid = a.allocate(list(range(8)))
    a.free(aid, list(range(8)))
    _, plen, aid = a.allocate(list(range(8)))
    assert plen == 8
    with pytest.raises(pk.PagedKVError):
        a.free(aid, [1, 2, 3, 4, 5, 6, 7, 8])        # does not start with its prefix
    with pytest.raises(pk.PagedKVError):
        a.free(aid + 100, [])                         # unknown request
    with pytest.raises(pk.PagedKVError):
        a.allocate(list(range(8)), 4)                 # total below the prompt
    a.free(aid, list(range(8)))


def test_no_reference_leaks_through_splits():
    """A request holding a prefix node that a later request splits must
    release both halves; afterwards the whole pool can be taken."""
    a = pk.RadixAllocator(33, 2)                      # 32 usable
    A = list(range(16))
    _, _, i = a.allocate(A)
    a.free(i, A)                                      # one 8-block node
    _, p1, h1 = a.allocate(A)                         # holds the whole node
    _, p2, h2 = a.allocate(list(range(6)) + [77, 78])  # splits it after 3 blocks
    assert p1 == 16 and p2 == 6
    a.free(h1, A)
    a.free(h2, list(range(6)) + [77, 78])
    got, _, i = a.allocate(list(range(1000, 1064)), 64)
    assert len(got) == 32 and a.num_cached == 0
    a.free(i, [])


def test_random_stress_against_simulated_kv_contents():
    """Requests draw prompts from a few shared templates; the 'engine' writes
    each block's key (the token prefix it ends) when it computes the block.
    Every shared prefix block must hold exactly the key of its position, live
    requests' own blocks are unique, and blocks are conserved."""
    B, NB = 4, 257
    a = pk.RadixAllocator(NB, B)
    rng = np.random.default_rng(7)
    templates = [list(rng.integers(0, 50, size=int(rng.integers(4, 40)))) for _ in range(6)]
    content = {}
    live = {}
    for step in range(4000):
        if live and (rng.random() < 0.45 or len(live) > 12):
            aid = list(live)[int(rng.integers(len(live)))]
            blocks, plen, prompt, total = live.pop(aid)
            gen = list(rng.integers(0, 50, size=int(total - len(prompt))))
            toks = prompt + gen
            for k in range(plen // B, len(toks) // B):          # the engine wrote these
                content[int(blocks[k])] = tuple(toks[:(k + 1) * B])
            a.free(aid, toks)
        else:
            t = templates[int(rng.integers(len(templates)))]
            cut = int(rng.integers(0, len(t) + 1))
            prompt = t[:cut] + list(rng.integers(0, 50, size=int(rng.integers(0, 9))))
            total = len(prompt) + int(rng.integers(0, 9))
            try:
                blocks, plen, aid = a.allocate(prompt, total)
            except pk.PagedKVError:
                continue
            assert plen % B == 0 and plen <= len(prompt)
            for k in range(plen // B):
                assert content.get(int(blocks[k])) == tuple(prompt[:(k + 1) * B]), step
            for k in range(plen // B, len(prompt) // B):        # prefill writes
                content[int(blocks[k])] = tuple(prompt[:(k + 1) * B])
            live[aid] = (blocks, plen, prompt, total)
        owned = [int(b) for (bl, pl, _, _) in live.values() for b in bl[pl // B:]]
        assert len(owned) == len(set(owned))
        shared = {int(b) for (bl, pl, _, _) in live.values() for b in bl[:pl // B]}
        assert not shared & set(owned)
        assert 0 not in owned and 0 not in shared
        assert a.num_free + a.num_cached + len(owned) == NB - 1, step
    for aid, (blocks, plen, prompt, total) in list(live.items()):
        a.free(aid, prompt)
    assert a.num_free + a.num_cached == NB - 1
    assert a.num_evictable > 0
