"""A serving loop driving the library over many decode steps: the
reference-counted block allocator hands out each new token's slot (with
copy-on-write once forked sequences diverge), each step writes the new tokens
and decodes in one call (pa_write_decode_partitioned: the KV write folded into
the partition kernel, then the merge), and every sequence's length advances
by one per step. Each step's output is checked against the oracle run on an
oracle pool kept in step (its own write and block copy), and the pools are
compared bit for bit along the way."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TORCH, assert_decode_close, host_to_torch, to_f64, torch_to_host
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


class _Types:
    """The fields assert_decode_close reads."""

    def __init__(self, cache, q):
        self.cache_dtype, self.q_dtype, self.name = cache, q, f"serving loop {cache}"


@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
def test_serving_loop(cache):
    rng = np.random.default_rng(17)
    q = "bf16"
    Hq, Hkv, D, B, nb, cap = 16, 4, 128, 16, 160, 24        # cap: blocks per sequence
    P = 64
    scale = float(np.float32(1 / np.sqrt(D)))
    ks = vs = 1.0
    if cache == "e4m3":
        ks, vs = 4.5 / 448, 4.7 / 448
    alloc = pk.BlockAllocator(nb, B)
    store = {"bf16": np.uint16, "e4m3": np.uint8}[cache]
    kc = np.zeros((nb, Hkv, B, D), store)
    vc = np.zeros_like(kc)
    W.poison_fill(kc, cache)
    W.poison_fill(vc, cache)
    dk = host_to_torch(kc, cache).cuda()
    dv = host_to_torch(vc, cache).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    types = _Types(cache, q)

    def tokens(n):
        return (W.to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), q),
                W.to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), q))

    def write(tk, tv, slots):
        sl = np.asarray(slots, np.int64)
        assert oracle.reshape_and_cache(tk, tv, kc, vc, sl, Hkv, D, B, q, cache, ks, vs) == 0
        pk.reshape_and_cache(host_to_torch(tk, q).cuda(), host_to_torch(tv, q).cuda(), dk, dv,
                             torch.from_numpy(sl).cuda(), ks, vs, status)

    # four prompts, the first two forked into two children each: 8 sequences
    tables, lens = [], []
    for _ in range(4):
        L = int(rng.integers(100, 300))
        tab = np.zeros(cap, np.int32)
        n, slots = 0, []
        for pos in range(L):
            slot, n, copy = alloc.append_slot((tab, n), pos)
            assert copy is None
            slots.append(slot)
        write(*tokens(L), slots)
        tables.append([tab, n])
        lens.append(L)
    for parent in (0, 1):
        for _ in range(2):
            child = tables[parent][0].copy()
            alloc.fork(child[:tables[parent][1]])
            tables.append([child, tables[parent][1]])
            lens.append(lens[parent])
    prompt_lens = list(lens)
    S = len(tables)
    ws = pk.alloc_workspace(S, Hq, D, cap * B, P)
    copies = 0
    for step in range(40):
        new_slots, pairs = [], []
        for i in range(S):
            slot, tl, copy = alloc.append_slot((tables[i][0], tables[i][1]), lens[i])
            tables[i][1] = tl
            lens[i] += 1
            new_slots.append(slot)
            if copy:
                pairs.append(copy)
        if pairs:
            copies += len(pairs)
            pr = np.array(pairs, np.int64)
            assert oracle.copy_blocks(kc, vc, pr) == 0
            pk.copy_blocks(dk, dv, torch.from_numpy(pr).cuda(), status)
        nk, nv = tokens(S)
        qh = W.to_storage(rng.standard_normal((S, Hq, D)).astype(np.float32), q)
        bt = np.zeros((S, cap), np.int32)
        for i, (tab, tl) in enumerate(tables):
            bt[i, :tl] = tab[:tl]
        cl = np.array(lens, np.int32)
        sl = np.array(new_slots, np.int64)
        out = torch.empty(S, Hq, D, dtype=TORCH[q], device="cuda")
        pk.write_decode_partitioned(out, host_to_torch(qh, q).cuda(), host_to_torch(nk, q).cuda(),
                                    host_to_torch(nv, q).cuda(), dk, dv, torch.from_numpy(sl).cuda(),
                                    torch.from_numpy(bt).cuda(), torch.from_numpy(cl).cuda(),
                                    cap * B, scale, ws, P, ks, vs, status)
        assert oracle.reshape_and_cache(nk, nv, kc, vc, sl, Hkv, D, B, q, cache, ks, vs) == 0
        want = oracle.decode(qh, q, kc, vc, cache, bt, cl, Hkv, B, scale, ks, vs)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"step {step}: device status {int(status.item())}"
        assert_decode_close(to_f64(out), want, types, f"serving loop step {step}")
        if step % 10 == 9:
            assert np.array_equal(torch_to_host(dk, cache).view(np.uint8), kc.view(np.uint8))
            assert np.array_equal(torch_to_host(dv, cache).view(np.uint8), vc.view(np.uint8))
    # a forked prompt ending inside a block shares that block three ways: the
    # parent and the first child each take a copy, the last holder keeps it
    assert copies == sum(2 for i in (0, 1) if prompt_lens[i] % B)
    alloc.close()
