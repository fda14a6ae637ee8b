"""Decoding through block tables the prefix-caching radix allocator hands
out ("TGI PagedAttention deep-dive" (lpnh.cn) sec. 5.2-5.4: a later request
reuses the cached blocks of its longest block-aligned prefix, a node splits
where two requests part, least-recently-used unreferenced sequences are
evicted and their blocks handed out again).

Each token's K/V is a fixed function of (token id, position), so a cached
block is valid for any request whose prefix has the same tokens. Requests
write only the tokens past their cached prefix (pa_reshape_and_cache into
the blocks they were given) and decode through their radix tables on the GPU.
The expected output is the oracle's decode of the same request laid out in a
fresh private pool that holds the request's own tokens: a block handed to two
live requests, a shared prefix overwritten, or an evicted block still in a
live table would make the two differ."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TORCH, assert_decode_close, host_to_torch, to_f64
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu

Hq, Hkv, D, B = 8, 2, 128, 16
DT = "bf16"
SEED = 0x5EED0141


class Pool:
    """The device pool, block tables from the radix allocator, and the
    reference K/V of every (token, position)."""

    def __init__(self, num_blocks):
        self.alloc = pk.RadixAllocator(num_blocks, B)
        shape = (num_blocks, Hkv, B, D)
        kc = np.zeros(shape, np.uint16)
        vc = np.zeros(shape, np.uint16)
        W.poison_fill(kc, DT)
        W.poison_fill(vc, DT)
        self.kc, self.vc = host_to_torch(kc, DT).cuda(), host_to_torch(vc, DT).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = float(np.float32(1 / np.sqrt(D)))
        self._kv = {}

    def kv(self, token, pos):
        key = (int(token), int(pos))
        if key not in self._kv:
            rng = np.random.default_rng([SEED, key[0], key[1]])
            x = rng.standard_normal((2, Hkv, D)).astype(np.float32)
            self._kv[key] = W.to_storage(x, DT)
        return self._kv[key]

    def kv_of(self, tokens, start=0):
        kv = np.stack([self.kv(t, start + i) for i, t in enumerate(tokens)])
        return np.ascontiguousarray(kv[:, 0]), np.ascontiguousarray(kv[:, 1])

    def request(self, tokens, prompt_len):
        """Allocate for a request whose prompt is tokens[:prompt_len] and
        which holds len(tokens) tokens, and write the tokens past its cached
        prefix into its blocks."""
        blocks, plen, aid = self.alloc.allocate(np.asarray(tokens[:prompt_len]), len(tokens))
        assert plen % B == 0 and plen <= prompt_len
        pos = np.arange(plen, len(tokens))
        if pos.size:
            slots = blocks[pos // B].astype(np.int64) * B + pos % B
            k, v = self.kv_of(tokens[plen:], plen)
            pk.reshape_and_cache(host_to_torch(k, DT).cuda(), host_to_torch(v, DT).cuda(),
                                 self.kc, self.vc, torch.from_numpy(slots).cuda(),
                                 dev_status=self.status)
        return {"tokens": list(tokens), "blocks": blocks, "prefix": plen, "id": aid}

    def decode_and_check(self, reqs, what, seed=0, mode="single"):
        """Decode the requests in one launch through their radix tables and
        compare each with the oracle on a private pool of its own tokens."""
        S = len(reqs)
        lens = np.array([len(r["tokens"]) for r in reqs], np.int32)
        nb = max(len(r["blocks"]) for r in reqs)
        bt = np.zeros((S, nb), np.int32)
        for i, r in enumerate(reqs):
            bt[i, :len(r["blocks"])] = r["blocks"]
        rng = np.random.default_rng([SEED, seed])
        qh = W.to_storage(rng.standard_normal((S, Hq, D)).astype(np.float32), DT)
        out = torch.empty(S, Hq, D, dtype=TORCH[DT], device="cuda")
        args = (out, host_to_torch(qh, DT).cuda(), self.kc, self.vc, torch.from_numpy(bt).cuda(),
                torch.from_numpy(lens).cuda(), int(lens.max()), self.scale)
        if mode == "single":
            pk.decode(*args, dev_status=self.status)
        else:
            ws = pk.alloc_workspace(S, Hq, D, int(lens.max()), 32)
            pk.decode_partitioned(*args, ws, 32, dev_status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        got = to_f64(out)
        for i, r in enumerate(reqs):
            L = len(r["tokens"])
            n = -(-L // B)
            k, v = self.kv_of(r["tokens"])
            pool_k = np.zeros((n + 1, Hkv, B, D), np.uint16)
            pool_v = np.zeros((n + 1, Hkv, B, D), np.uint16)
            slots = (1 + np.arange(L) // B).astype(np.int64) * B + np.arange(L) % B
            assert oracle.reshape_and_cache(k, v, pool_k, pool_v, slots, Hkv, D, B, DT, DT) == 0
            want = oracle.decode(np.ascontiguousarray(qh[i:i + 1]), DT, pool_k, pool_v, DT,
                                 np.arange(1, n + 1, dtype=np.int32)[None, :],
                                 np.array([L], np.int32), Hkv, B, self.scale)
            assert_decode_close(got[i:i + 1], want, _Shape, f"{what}: request {i}")


class _Shape:
    """The dtype fields assert_decode_close reads."""
    cache_dtype = DT
    q_dtype = DT
    name = "radix"


def toks(rng, n, lo=0, hi=1000):
    return [int(t) for t in rng.integers(lo, hi, n)]


@pytest.mark.parametrize("mode", ["single", "split"])
def test_decode_through_radix_tables(mode):
    rng = np.random.default_rng(5)
    pool = Pool(40)                                      # 39 usable blocks
    A = toks(rng, 130)
    a = pool.request(A, 100)                             # nothing cached yet
    assert a["prefix"] == 0 and len(a["blocks"]) == 9
    pool.decode_and_check([a], "first request", 1, mode)
    pool.alloc.free(a["id"], A)                          # 8 whole blocks cached
    assert pool.alloc.num_cached == 8

    # B shares A's first 70 tokens: 4 whole blocks reused, A's node split
    Bt = A[:70] + toks(rng, 50, 1000, 2000)
    b = pool.request(Bt, 100)
    assert b["prefix"] == 64 and list(b["blocks"][:4]) == list(a["blocks"][:4])
    # C repeats A's prompt and grows past it: all 8 cached blocks reused
    Ct = A[:130] + toks(rng, 10, 2000, 3000)
    c = pool.request(Ct, 130)
    assert c["prefix"] == 128 and list(c["blocks"][:8]) == list(a["blocks"][:8])
    pool.decode_and_check([b, c], "prefix reuse and split", 2, mode)

    pool.alloc.free(b["id"], Bt)                         # B's 3 own whole blocks cached
    b_own = set(int(x) for x in b["blocks"][4:7])
    # D needs more blocks than are free: B's branch (unreferenced, least
    # recently used) is evicted and its blocks handed to D; A's prefix is
    # referenced by C and stays
    free_before = pool.alloc.num_free
    Dt = toks(rng, 448, 3000, 4000)
    need = -(-len(Dt) // B)
    assert need > free_before
    d = pool.request(Dt, 400)
    assert d["prefix"] == 0
    assert b_own & set(int(x) for x in d["blocks"]), "no evicted block was handed out again"
    assert not (set(int(x) for x in d["blocks"]) & set(int(x) for x in c["blocks"]))
    pool.decode_and_check([c, d], "after eviction", 3, mode)

    # B's prompt again: only A's 4 shared blocks remain cached for it
    pool.alloc.free(d["id"], Dt)
    pool.alloc.free(c["id"], Ct)
    e = pool.request(Bt, 100)
    assert e["prefix"] == 64 and list(e["blocks"][:4]) == list(a["blocks"][:4])
    pool.decode_and_check([e], "after the branch was evicted", 4, mode)
    pool.alloc.free(e["id"], Bt)


def test_random_requests_through_radix_tables():
    """A seeded stream of requests drawn from a few prompt families (shared
    prefixes of different lengths, random continuations) on a pool small
    enough to force evictions; every few requests, the live ones are decoded
    together and each is checked against its private-pool oracle."""
    rng = np.random.default_rng(9)
    pool = Pool(64)
    families = [toks(rng, 96, 10 * f, 10 * f + 10) for f in range(4)]
    live = []
    for step in range(24):
        if live and (len(live) >= 4 or rng.random() < 0.3):
            r = live.pop(int(rng.integers(len(live))))
            pool.alloc.free(r["id"], r["tokens"])
        fam = families[int(rng.integers(len(families)))]
        keep = int(rng.integers(8, 96))
        t = fam[:keep] + toks(rng, int(rng.integers(1, 120)), 5000, 6000)
        try:
            live.append(pool.request(t, len(t) - int(rng.integers(0, 8))))
        except pk.PagedKVError as err:
            assert err.status == pk.PA_ERR_NO_BLOCKS
            continue
        if step % 3 == 2:
            pool.decode_and_check(live, f"step {step}", 100 + step)
    assert pool.alloc.num_cached > 0
