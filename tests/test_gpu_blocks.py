"""GPU: the copy-on-write block copy against the oracle, and a copy-on-write
decode scenario driven by the library's block allocator, run side by side on
the GPU and in the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TORCH, assert_decode_close, host_to_torch, to_f64, torch_to_host
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "e4m3"])
def test_copy_blocks_bitexact(dtype):
    rng = np.random.default_rng(5)
    nb, H, B, D = 40, 4, 16, 128
    st = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}[dtype]
    kc = rng.integers(0, np.iinfo(st).max, (nb, H, B, D), dtype=st)
    vc = rng.integers(0, np.iinfo(st).max, (nb, H, B, D), dtype=st)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:10], perm[10:20]], axis=1).astype(np.int64)
    dk, dv = torch.from_numpy(kc.view(np.uint8)).cuda(), torch.from_numpy(vc.view(np.uint8)).cuda()
    dk = dk.view(nb, H, B, D * kc.itemsize)
    dv = dv.view(nb, H, B, D * kc.itemsize)
    # view as the cache type for the binding
    tdt = TORCH[dtype] if dtype != "f32" else torch.float32
    k_t = dk.view(tdt) if dtype != "e4m3" else dk
    v_t = dv.view(tdt) if dtype != "e4m3" else dv
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.copy_blocks(k_t, v_t, torch.from_numpy(pairs).cuda(), status)
    assert oracle.copy_blocks(kc, vc, pairs) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(dk.cpu().numpy().reshape(-1), kc.view(np.uint8).reshape(-1))
    assert np.array_equal(dv.cpu().numpy().reshape(-1), vc.view(np.uint8).reshape(-1))
    bad = torch.tensor([[1, nb + 3]], dtype=torch.int64, device="cuda")
    pk.copy_blocks(k_t, v_t, bad, status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.DEV_BAD_BLOCK_ID


@pytest.mark.parametrize("cache,q", [("bf16", "bf16"), ("e4m3", "bf16")])
def test_copy_on_write_decode(cache, q):
    """A parent sequence (prompt of 37 tokens, block size 16) is forked into
    three children; every sequence then appends its own tokens. Appends into
    the shared last block trigger copy-on-write through the allocator; the GPU
    copies with pa_copy_blocks and writes with pa_reshape_and_cache, the oracle
    does the same on host arrays, and both decode all four sequences."""
    rng = np.random.default_rng(9)
    Hq, Hkv, D, B, nb = 16, 4, 128, 16, 64
    kv_dt = q
    alloc = pk.BlockAllocator(nb, B)
    store = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8}[cache]
    kc = np.zeros((nb, Hkv, B, D), store)
    vc = np.zeros_like(kc)
    W.poison_fill(kc, cache)
    W.poison_fill(vc, cache)
    dk = host_to_torch(kc, cache).cuda()
    dv = host_to_torch(vc, cache).cuda()
    ks = vs = 1.0
    if cache == "e4m3":
        ks, vs = 4.5 / 448, 4.7 / 448
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def write(tokens_k, tokens_v, slots):
        sl = np.asarray(slots, np.int64)
        assert oracle.reshape_and_cache(tokens_k, tokens_v, kc, vc, sl, Hkv, D, B, kv_dt, cache,
                                        ks, vs) == 0
        pk.reshape_and_cache(host_to_torch(tokens_k, kv_dt).cuda(),
                             host_to_torch(tokens_v, kv_dt).cuda(), dk, dv,
                             torch.from_numpy(sl).cuda(), ks, vs, status)

    def tokens(n):
        return (W.to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), kv_dt),
                W.to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), kv_dt))

    cap = 8
    tables, lens = [], []
    parent = np.zeros(cap, np.int32)
    n, slots = 0, []
    for pos in range(37):
        slot, n, copy = alloc.append_slot((parent, n), pos)
        assert copy is None
        slots.append(slot)
    tk, tv = tokens(37)
    write(tk, tv, slots)
    tables.append([parent, n])
    lens.append(37)
    for _ in range(3):                       # fork: share every block by reference
        child = parent.copy()
        alloc.fork(child[:n])
        tables.append([child, n])
        lens.append(37)
    copies = 0
    for step in range(5):                    # each sequence appends its own tokens
        new_slots, pairs = [], []
        for i, (tab, tl) in enumerate(tables):
            slot, tl, copy = alloc.append_slot((tab, tl), lens[i])
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
        tk, tv = tokens(len(tables))
        write(tk, tv, new_slots)
    assert copies == 3                       # three children left the shared last block
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(torch_to_host(dk, cache).view(np.uint8), kc.view(np.uint8))

    S = len(tables)
    bt = np.zeros((S, cap), np.int32)
    for i, (tab, tl) in enumerate(tables):
        bt[i, :tl] = tab[:tl]
    cl = np.array(lens, np.int32)
    qh = W.to_storage(rng.standard_normal((S, Hq, D)).astype(np.float32), q)
    scale = float(np.float32(1 / np.sqrt(D)))
    want = oracle.decode(qh, q, kc, vc, cache, bt, cl, Hkv, B, scale, ks, vs)
    out = torch.empty(S, Hq, D, dtype=TORCH[q], device="cuda")
    pk.decode(out, host_to_torch(qh, q).cuda(), dk, dv, torch.from_numpy(bt).cuda(),
              torch.from_numpy(cl).cuda(), int(cl.max()), scale, ks, vs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    class C:
        cache_dtype, q_dtype = cache, q
    assert_decode_close(to_f64(out), want, C, "copy-on-write decode")
    # the parent kept its own blocks; the children diverged after the prompt
    assert alloc.refcount(int(bt[0, 0])) == 4 and alloc.refcount(int(bt[0, 2])) == 1
    alloc.close()
