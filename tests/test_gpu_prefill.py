"""Multi-query paged attention (chunked prefill / speculative verification)
on the GPU against the oracle: the tcgen05 path over its shapes, the
warp-level MMA path for a few query rows per sequence and KV head, the
CUDA-core path for the other types and block sizes, the decode as its
one-query case, block-size invariance, status flags, and full-size chunked
prefill and verification steps checked on every row (verification) or on
whole sequences plus every sequence's tile-edge rows (chunks)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W
from paged_kv_cache_141_gb300.workloads import config_case, make_case, make_queries

from gpu_common import (TORCH, DeviceCase, assert_decode_close, host_to_torch, oracle_pool,
                        parallel_rows, to_f64)

pytestmark = pytest.mark.gpu


class Prefill:
    """A Case written through the step (every context token in the pool) plus
    its query tokens, on the device."""

    def __init__(self, case, law, seed=None):
        self.case = case
        self.q = make_queries(case, law, seed)
        self.dc = DeviceCase(case)
        self.dc.write_step()
        dev = self.dc.k_cache.device
        self.query = host_to_torch(self.q.query, case.q_dtype).to(dev)
        self.query_start = torch.from_numpy(self.q.query_start).to(dev)
        self.out = torch.full_like(self.query, float("nan"))

    def run(self, max_queries=None):
        c, dc = self.case, self.dc
        pk.paged_prefill(self.out, self.query, self.query_start, dc.k_cache, dc.v_cache,
                         dc.block_tables, dc.context_lens,
                         self.q.max_queries if max_queries is None else max_queries,
                         c.max_context_len, c.scale, c.k_scale, c.v_scale, dc.status)
        return self.out

    def oracle(self, seqs=None):
        c, q = self.case, self.q
        kc, vc = oracle_pool(c)
        seqs = np.arange(c.num_seqs) if seqs is None else np.asarray(seqs)
        rows = np.concatenate([np.arange(q.query_start[s], q.query_start[s + 1]) for s in seqs])
        counts = q.counts[seqs]
        qs = np.zeros(len(seqs) + 1, dtype=np.int32)
        np.cumsum(counts, out=qs[1:])
        want = oracle.paged_prefill(np.ascontiguousarray(q.query[rows]), c.q_dtype, qs, kc, vc,
                                    c.cache_dtype, np.ascontiguousarray(c.block_tables[seqs]),
                                    np.ascontiguousarray(c.context_lens[seqs]), c.num_kv_heads,
                                    c.block_size, c.scale, c.k_scale, c.v_scale)
        return rows, want

    def oracle_rows(self, rows):
        """The oracle on single query rows: row t of sequence s at position
        pos sees the keys a one-query step over pos + 1 tokens sees. Slices
        of rows run on host threads."""
        c, q = self.case, self.q
        kc, vc = oracle_pool(c)

        def some(rows):
            seq = np.searchsorted(q.query_start, rows, side="right") - 1
            pos = c.context_lens[seq] - q.counts[seq] + (rows - q.query_start[seq])
            return oracle.paged_prefill(np.ascontiguousarray(q.query[rows]), c.q_dtype,
                                        np.arange(len(rows) + 1, dtype=np.int32), kc, vc,
                                        c.cache_dtype, np.ascontiguousarray(c.block_tables[seq]),
                                        (pos + 1).astype(np.int32), c.num_kv_heads,
                                        c.block_size, c.scale, c.k_scale, c.v_scale)

        return parallel_rows(some, np.asarray(rows))

    def dense_rows(self, whole=(), edges=(0, 1, 31, 32, 127, 128, -2, -1), n_random=0, seed=0):
        """Rows to check: every row of the sequences `whole`, the rows at
        the offsets `edges` (negative: from the end; the query-tile and
        n-tile edges) of every sequence, and n_random seeded random rows."""
        qs = self.q.query_start
        rows = set()
        for s_ in whole:
            rows.update(range(int(qs[s_]), int(qs[s_ + 1])))
        for s_ in range(self.case.num_seqs):
            lo, hi = int(qs[s_]), int(qs[s_ + 1])
            for e in edges:
                r = lo + e if e >= 0 else hi + e
                if lo <= r < hi:
                    rows.add(r)
        rng = np.random.default_rng(seed)
        if n_random:
            rows.update(int(r) for r in rng.integers(0, int(qs[-1]), size=n_random))
        return np.array(sorted(rows))


def mma_max_rows(case):
    """max_queries_per_seq * group up to this selects the warp-level MMA
    kernels (32 at head size <= 128, 16 at 256, and 16 where the tcgen05
    kernels take the E4M3 products: E4M3 cache, bf16 query, head size 128,
    a block size they take); a larger bound (any bound >= every Q_s is
    valid) selects the tcgen05 kernels."""
    if case.head_size > 128:
        return 16
    if (case.cache_dtype == "e4m3" and case.q_dtype == "bf16" and case.head_size == 128
            and case.block_size & (case.block_size - 1) == 0):
        return 16
    return 32


def tc_bound(p):
    """A max_queries_per_seq that sends the launch to the tcgen05 kernel."""
    return max(p.q.max_queries, mma_max_rows(p.case) // p.case.group + 1)


def check(case, law, what, seed=None, force_tc=False):
    p = Prefill(case, law, seed)
    got = to_f64(p.run(tc_bound(p) if force_tc else None))
    assert p.dc.status_bits() == 0
    rows, want = p.oracle()
    return assert_decode_close(got[rows], want, case, what)


# tensor-core shapes: head sizes, groups (incl. one that does not divide the
# 128-row tile), block sizes below, at and above the 128-key tile, ragged
# query counts spanning several query tiles and key tiles
TC_SWEEP = [
    # S, Hq, Hkv, d, B, dtype, lengths, queries
    (5, 8, 2, 128, 16, "bf16", ("uniform", 1, 700), ("uniform", 1, 80)),
    (4, 4, 4, 64, 8, "f16", ("uniform", 100, 400), ("uniform", 50, 300)),
    (3, 16, 2, 256, 32, "bf16", ("uniform", 64, 500), ("uniform", 1, 40)),
    (4, 12, 2, 128, 16, "bf16", ("uniform", 30, 600), ("uniform", 20, 70)),
    (3, 32, 2, 128, 256, "f16", ("uniform", 200, 1000), ("uniform", 1, 33)),
    (6, 8, 4, 128, 64, "f16", ("fixed", [1, 2, 127, 128, 129, 300]), ("all",)),
    (2, 128, 1, 64, 16, "bf16", ("uniform", 10, 300), ("uniform", 1, 5)),
    (8, 32, 8, 128, 16, "bf16", ("loguniform", 64, 2048), ("uniform", 1, 8)),
    # one query tile per sequence (the compact 64-key kernel): a full
    # 128-row tile at G=1, block sizes below, at and above 64 keys, a group
    # that does not divide 128, lengths around the key tile
    (5, 4, 4, 64, 8, "f16", ("uniform", 1, 500), ("uniform", 1, 128)),
    (4, 6, 2, 128, 256, "bf16", ("fixed", [63, 64, 65, 700]), ("uniform", 1, 14)),
    (4, 16, 2, 64, 64, "bf16", ("uniform", 1, 300), ("uniform", 1, 16)),
    (3, 8, 8, 128, 32, "f16", ("fixed", [1, 128, 129]), ("all",)),
    # binary16 weights as one term: every row of a short causal prefix sees
    # 1..24 keys, where single weights dominate the output
    (48, 8, 2, 128, 16, "f16", ("uniform", 2, 24), ("all",)),
    (32, 4, 4, 64, 8, "f16", ("uniform", 1, 12), ("all",)),
]


@pytest.mark.parametrize("i", range(len(TC_SWEEP)))
def test_prefill_tensor_core_sweep(i):
    S, Hq, Hkv, d, B, dt, lens, ql = TC_SWEEP[i]
    c = make_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=d, block_size=B,
                  q_dtype=dt, cache_dtype=dt, lengths=lens, seed=900 + i)
    check(c, ql, f"tc sweep {i}", force_tc=True)


# CUDA-core shapes: binary32, block size 1 (16-bit and E4M3), E4M3 at head
# size 256
SIMT_SWEEP = [
    (4, 4, 4, 64, 16, "f32", "f32", ("uniform", 1, 64), ("uniform", 1, 20)),
    (3, 8, 2, 128, 1, "bf16", "bf16", ("uniform", 5, 90), ("uniform", 1, 12)),
    (2, 8, 2, 128, 1, "bf16", "e4m3", ("uniform", 20, 150), ("uniform", 1, 9)),
    (2, 8, 2, 256, 16, "f16", "e4m3", ("uniform", 20, 150), ("uniform", 1, 9)),
    # block sizes that are not powers of two
    (3, 8, 2, 128, 24, "bf16", "bf16", ("uniform", 20, 200), ("uniform", 1, 12)),
    (2, 8, 4, 64, 96, "f16", "f16", ("fixed", [95, 250]), ("uniform", 1, 9)),
]

# E4M3 caches on the tensor cores (K/V widened to binary16 in shared memory;
# with a bf16 query at head size 128, the E4M3 products): one query tile per
# sequence (the one-tile kernel) and two or more (the two-tile kernel, odd
# tile counts leaving a single last tile), block sizes 8..256, groups that do
# not divide the 128-row tile
E4M3_TC_SWEEP = [
    (3, 8, 1, 128, 16, "bf16", ("uniform", 20, 300), ("uniform", 1, 40)),
    (2, 6, 2, 64, 32, "f16", ("uniform", 40, 200), ("all",)),
    (4, 32, 8, 128, 16, "bf16", ("uniform", 100, 700), ("uniform", 100, 300)),
    (3, 16, 2, 128, 256, "f16", ("uniform", 200, 600), ("uniform", 1, 12)),
    (3, 16, 2, 128, 256, "f16", ("uniform", 200, 600), ("uniform", 20, 60)),
    (4, 12, 4, 64, 8, "bf16", ("fixed", [1, 2, 129, 400]), ("all",)),
    (3, 24, 8, 128, 64, "bf16", ("fixed", [300, 511, 1000]), ("fixed", [300, 170, 257])),
    # bf16 query, head size 128, two or more tiles: the E4M3 products, with
    # 8-row and 64-row (block size 256, capped) boxes
    (3, 16, 2, 128, 8, "bf16", ("uniform", 100, 400), ("uniform", 20, 60)),
    (3, 16, 2, 128, 256, "bf16", ("uniform", 200, 700), ("uniform", 20, 90)),
    # the same on one query tile (the one-tile kernel): G = 8 with up to 16
    # tokens (128 rows), 8-, 16- and 64-row boxes; G = 3 with up to 42 tokens
    # (two padding rows)
    (4, 32, 4, 128, 16, "bf16", ("uniform", 20, 700), ("uniform", 1, 16)),
    (3, 16, 2, 128, 8, "bf16", ("uniform", 100, 400), ("uniform", 1, 16)),
    (3, 16, 2, 128, 256, "bf16", ("uniform", 200, 700), ("uniform", 1, 16)),
    (3, 12, 4, 128, 64, "bf16", ("fixed", [42, 129, 500]), ("uniform", 1, 42)),
]


@pytest.mark.parametrize("i", range(len(E4M3_TC_SWEEP)))
def test_prefill_e4m3_tensor_core_sweep(i):
    S, Hq, Hkv, d, B, qt, lens, ql = E4M3_TC_SWEEP[i]
    c = make_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=d, block_size=B,
                  q_dtype=qt, cache_dtype="e4m3", kv_dtype=qt, lengths=lens, seed=960 + i)
    check(c, ql, f"e4m3 tc sweep {i}", force_tc=True)


@pytest.mark.parametrize("tiles", ["one", "two"])
@pytest.mark.parametrize("qt", ["bf16", "f16"])
def test_e4m3_scores_query_magnitudes(qt, tiles):
    """Both tcgen05 kernels on an E4M3 cache at head size 128. A bf16 query
    takes the E4M3 products: each row goes to the tensor cores as two E4M3
    terms of the row times a power of two. An f16 query (11 significant bits,
    more than two E4M3 terms hold) keeps the widened K. Rows scaled by powers
    of two over a wide range, all-zero rows, and rows of one large element
    beside tiny ones (the E4M3 subnormal range) must all stay within the
    E4M3 tolerance of the oracle."""
    c = make_case(num_seqs=3, num_q_heads=16, num_kv_heads=2, head_size=128, block_size=16,
                  q_dtype=qt, cache_dtype="e4m3", kv_dtype=qt, lengths=("uniform", 200, 500),
                  seed=981)
    p = Prefill(c, ("uniform", 1, 16) if tiles == "one" else ("uniform", 40, 80))
    rows = p.q.query.reshape(-1, 128)
    x = oracle.decode_array(rows, qt)
    rng = np.random.default_rng(982)
    span = 12 if qt == "bf16" else 5                         # f16 keeps |x| 2^span within range
    x *= np.exp2(rng.integers(-span, span + 1, size=(len(x), 1)))
    x[rng.random(len(x)) < 0.05] = 0.0
    spike = np.flatnonzero(rng.random(len(x)) < 0.05)
    x[spike] *= 2.0 ** -10
    x[spike, rng.integers(0, 128, size=len(spike))] = 64.0
    p.q.query = W.to_storage(x.astype(np.float32), qt).reshape(p.q.query.shape)
    p.query = host_to_torch(p.q.query, qt).to(p.query.device)
    assert pk.prefill_kernel(tc_bound(p), c.num_q_heads, c.num_kv_heads, 128, 16, c.num_blocks,
                             pk.PA_BF16 if qt == "bf16" else pk.PA_F16,
                             pk.PA_FP8_E4M3) == ("tc" if tiles == "one" else "tc_two_tiles")
    got = to_f64(p.run(tc_bound(p)))
    assert p.dc.status_bits() == 0
    idx, want = p.oracle()
    assert_decode_close(got[idx], want, c, f"e4m3 scores, {qt} query magnitudes")


# warp-level MMA shapes: one and two 8-row n-tiles (up to 16 rows), four
# n-tiles two per warp (17..32 rows, head size <= 128, 16-bit and E4M3),
# padding rows (G = 3), one token of a 16-head group, head sizes 64/128/256,
# block sizes 8..256, whole prefills of short sequences, E4M3 caches at head
# size 128 and 256
MMA_SWEEP = [
    (6, 32, 8, 128, 16, "bf16", "bf16", ("loguniform", 1, 900), ("uniform", 1, 8)),
    (4, 16, 2, 64, 8, "f16", "f16", ("uniform", 1, 300), ("uniform", 1, 4)),
    (3, 6, 2, 128, 256, "bf16", "bf16", ("fixed", [31, 32, 600]), ("uniform", 6, 10)),
    (24, 8, 8, 128, 32, "f16", "f16", ("uniform", 1, 28), ("all",)),
    (4, 8, 2, 64, 64, "bf16", "bf16", ("uniform", 100, 400), ("fixed", [8, 5, 7, 6])),
    # (bf16 query, E4M3 cache, 17-32 rows: the two-n-tile kernel where the
    # tcgen05 one is not eligible, block sizes that are not powers of two)
    (4, 32, 8, 128, 96, "bf16", "e4m3", ("loguniform", 1, 900), ("uniform", 1, 8)),
    (3, 16, 2, 128, 32, "f16", "e4m3", ("uniform", 20, 500), ("uniform", 3, 4)),
    (4, 12, 4, 128, 160, "bf16", "e4m3", ("fixed", [9, 33, 64, 700]), ("uniform", 6, 10)),
    # S, Hq, Hkv, d, B, query dtype, cache dtype, lengths, queries
    (6, 32, 8, 128, 16, "bf16", "bf16", ("uniform", 1, 700), ("uniform", 1, 4)),
    (5, 8, 2, 64, 8, "f16", "f16", ("uniform", 1, 300), ("uniform", 1, 4)),
    (4, 4, 4, 256, 32, "bf16", "bf16", ("uniform", 40, 500), ("uniform", 1, 8)),
    (4, 16, 2, 128, 64, "f16", "f16", ("fixed", [1, 2, 33, 300]), ("uniform", 1, 2)),
    (3, 6, 2, 128, 256, "bf16", "bf16", ("fixed", [31, 32, 600]), ("uniform", 1, 5)),
    (32, 8, 8, 128, 16, "f16", "f16", ("uniform", 1, 12), ("all",)),
    (4, 12, 4, 64, 128, "bf16", "bf16", ("uniform", 1, 200), ("uniform", 1, 5)),
    (3, 32, 2, 128, 16, "bf16", "bf16", ("uniform", 1, 900), ("fixed", [1, 1, 1])),
    (4, 32, 8, 128, 16, "bf16", "e4m3", ("uniform", 1, 700), ("uniform", 1, 4)),
    (3, 8, 2, 256, 32, "f16", "e4m3", ("uniform", 20, 400), ("uniform", 1, 4)),
    (5, 8, 4, 128, 8, "f16", "e4m3", ("uniform", 1, 100), ("uniform", 1, 3)),
]


@pytest.mark.parametrize("i", range(len(MMA_SWEEP)))
def test_prefill_warp_mma_sweep(i):
    S, Hq, Hkv, d, B, qt, ct, lens, ql = MMA_SWEEP[i]
    c = make_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=d, block_size=B,
                  q_dtype=qt, cache_dtype=ct, kv_dtype=qt, lengths=lens, seed=1000 + i)
    p = Prefill(c, ql)
    assert p.q.max_queries * c.group <= mma_max_rows(c)
    got = to_f64(p.run())
    assert p.dc.status_bits() == 0
    rows, want = p.oracle()
    assert_decode_close(got[rows], want, c, f"mma sweep {i}")


@pytest.mark.parametrize("i", range(len(SIMT_SWEEP)))
def test_prefill_cuda_core_sweep(i):
    S, Hq, Hkv, d, B, qt, ct, lens, ql = SIMT_SWEEP[i]
    c = make_case(num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_size=d, block_size=B,
                  q_dtype=qt, cache_dtype=ct, lengths=lens, seed=950 + i)
    check(c, ql, f"simt sweep {i}")


@pytest.mark.parametrize("force_tc", [False, True], ids=["warp-mma", "tcgen05"])
def test_length_one_e4m3_tensor_core_returns_v_exactly(force_tc):
    """E4M3 cache, one key and one query per sequence, on both tensor-core
    kernels: the output is the stored code's value times v_scale, rounded
    once -- pins the widening of the tiles (in shared memory for tcgen05, in
    registers for the warp-level MMA) and the folded scale."""
    c = make_case(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  q_dtype="bf16", cache_dtype="e4m3", kv_dtype="bf16", lengths=("fixed", [1] * 4),
                  seed=977)
    p = Prefill(c, ("fixed", [1] * 4))
    out = p.run(tc_bound(p) if force_tc else None).cpu()
    assert p.dc.status_bits() == 0
    B = c.block_size
    slots = torch.from_numpy(c.new_slots)
    codes = p.dc.v_cache.cpu()[slots // B, :, slots % B, :]
    want = (codes.view(torch.float8_e4m3fn).float()
            * torch.tensor(c.v_scale, dtype=torch.float32)).to(torch.bfloat16)
    G = c.group
    for h in range(c.num_q_heads):
        assert torch.equal(out[:, h].view(torch.int16), want[:, h // G].view(torch.int16))


def test_one_query_per_sequence_is_the_decode():
    c = make_case(num_seqs=16, num_q_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("uniform", 1, 900), seed=971)
    p = Prefill(c, ("fixed", [1] * 16))
    # the decode of the same queries (the query tokens of a one-token step)
    dc = p.dc
    dq = p.query.clone()
    out_d = torch.empty_like(dq)
    pk.decode(out_d, dq, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens,
              c.max_context_len, c.scale, 1.0, 1.0, dc.status)
    got = to_f64(p.run())
    assert dc.status_bits() == 0
    dec = to_f64(out_d)
    # both paths round an fp32 result to bf16: where the two fp32 values lie
    # on either side of a rounding boundary they differ by one bf16 ulp
    mag = np.maximum(np.abs(dec), 2.0 ** -126)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    assert np.all(np.abs(got - dec) <= np.maximum(1e-3, ulp))
    rows, want = p.oracle()
    assert_decode_close(got[rows], want, c, "one query")


@pytest.mark.parametrize("qmax", [40, 4, 8], ids=["tcgen05", "warp-mma", "warp-mma2"])
def test_block_size_invariance_on_the_tensor_cores(qmax):
    """Same logical K/V, pools paged with B in {8, 16, 32, 128, 256}: the key
    tiles (stages) hold the same keys, so the outputs are bit-identical; 40
    query tokens (160 rows) run the tcgen05 kernel, 4 (16 rows) and 8 (32
    rows) the warp-level MMA kernels."""
    lens = [300, 77, 513]
    outs = []
    for B in (8, 16, 32, 128, 256):
        c = make_case(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=B,
                      q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", lens), seed=972)
        # re-page one logical K/V stream: gather it from the first pool layout
        outs.append(_run_with_logical_kv(c, lens, qmax))
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def _run_with_logical_kv(c, lens, qmax):
    """Fill the case's pool so that token t of head h of sequence s holds a
    value that depends only on (s, h, t), then run the multi-query kernel."""
    rng = np.random.default_rng(5)
    Hkv, d = c.num_kv_heads, c.head_size
    p = Prefill(c, ("fixed", [min(qmax, L) for L in lens]))
    k = p.dc.k_cache.clone()
    v = p.dc.v_cache.clone()
    for s, L in enumerate(lens):
        kl = torch.from_numpy(rng.standard_normal((L, Hkv, d), dtype=np.float32))
        vl = torch.from_numpy(rng.standard_normal((L, Hkv, d), dtype=np.float32))
        pos = torch.arange(L)
        blk = torch.from_numpy(c.block_tables[s]).long()[pos // c.block_size]
        off = pos % c.block_size
        k[blk.cuda(), :, off.cuda(), :] = kl.to(k.dtype).cuda()
        v[blk.cuda(), :, off.cuda(), :] = vl.to(v.dtype).cuda()
    p.dc.k_cache.copy_(k)
    p.dc.v_cache.copy_(v)
    out = p.run()
    assert p.dc.status_bits() == 0
    return out.clone()


@pytest.mark.parametrize("qs", [[0, 7, 0, 0, 9], [0, 3, 0, 0, 4], [0, 7, 0, 0, 8]],
                         ids=["tcgen05", "warp-mma", "warp-mma2"])
def test_empty_sequences_and_zero_queries(qs):
    c = make_case(num_seqs=5, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [0, 50, 0, 200, 9]),
                  seed=973)
    p = Prefill(c, ("fixed", qs))
    got = to_f64(p.run())
    assert p.dc.status_bits() == 0
    rows, want = p.oracle()
    assert_decode_close(got[rows], want, c, "empty sequences")
    # no queries at all: nothing launches
    pk.paged_prefill(p.out[:0], p.query[:0], torch.zeros(6, dtype=torch.int32, device="cuda"),
                     p.dc.k_cache, p.dc.v_cache, p.dc.block_tables, p.dc.context_lens, 0,
                     c.max_context_len, c.scale)


@pytest.mark.parametrize("qmax", [3, 7, 9], ids=["warp-mma", "warp-mma2", "tcgen05"])
def test_status_flags(qmax):
    c = make_case(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [40, 60, 80]), seed=974)
    p = Prefill(c, ("fixed", [3, 3, 3]))
    # more queries than context tokens for sequence 0
    bad = p.dc.context_lens.clone()
    bad[0] = 2
    pk.paged_prefill(p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache,
                     p.dc.block_tables, bad, qmax, c.max_context_len, c.scale, 1.0, 1.0,
                     p.dc.status)
    assert p.dc.status_bits() & pk.DEV_BAD_LEN
    # more queries than the host's bound for every sequence
    p.dc.status.zero_()
    pk.paged_prefill(p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache,
                     p.dc.block_tables, p.dc.context_lens, 2, c.max_context_len, c.scale, 1.0,
                     1.0, p.dc.status)
    assert p.dc.status_bits() & pk.DEV_BAD_LEN
    # a block id outside the pool: the copy is skipped and flagged
    p.dc.status.zero_()
    tables = p.dc.block_tables.clone()
    tables[1, 0] = c.num_blocks + 5
    pk.paged_prefill(p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache, tables,
                     p.dc.context_lens, qmax, c.max_context_len, c.scale, 1.0, 1.0, p.dc.status)
    assert p.dc.status_bits() & pk.DEV_BAD_BLOCK_ID
    # the other sequences are still right
    p.dc.status.zero_()
    got = to_f64(p.run(qmax))
    rows, want = p.oracle()
    assert_decode_close(got[rows], want, c, "after flags")


def test_host_argument_errors():
    c = make_case(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                  q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [40, 60]), seed=975)
    p = Prefill(c, ("fixed", [3, 4]))
    args = (p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache, p.dc.block_tables,
            p.dc.context_lens, 4, c.max_context_len)
    with pytest.raises(pk.PagedKVError):
        pk.paged_prefill(*args, -0.1)
    with pytest.raises(pk.PagedKVError):
        pk.paged_prefill(*args[:7], 0, c.max_context_len, c.scale)


@pytest.mark.parametrize("law,force_tc", [(("fixed", None), False), (("uniform", 1, 8), False),
                                          (("uniform", 1, 8), True), (("uniform", 1, 4), False)],
                         ids=["chunk512", "spec8", "spec8-tcgen05", "spec4"])
def test_full_size_llama3_8b(law, force_tc):
    """Llama-3-8B GQA shape at full size (256 sequences, contexts 512..4096):
    a 512-token prefill chunk per sequence (capped at L_s), an 8-draft
    speculative verification step (warp-level MMA with two n-tiles per warp,
    and forced onto the tcgen05 kernel), and a 4-draft one. Verification
    steps: every row against the oracle. Chunks: every row of eight whole
    sequences (the shortest, the longest and six random ones) and the
    query-tile edge rows of every sequence."""
    c = config_case(3)
    if law[0] == "fixed":
        law = ("fixed", np.minimum(512, c.context_lens))
    p = Prefill(c, law)
    got = to_f64(p.run(tc_bound(p) if force_tc else None))
    assert p.dc.status_bits() == 0
    L = c.context_lens
    if law[0] == "fixed":
        rng = np.random.default_rng(11)
        whole = {int(np.argmin(L)), int(np.argmax(L))} | set(
            int(x) for x in rng.choice(c.num_seqs, 6, replace=False))
        rows = p.dense_rows(whole=sorted(whole))
    else:
        rows = np.arange(int(p.q.query_start[-1]))
    want = p.oracle_rows(rows)
    assert_decode_close(got[rows], want, c, f"full: llama3-8b {p.q.max_queries}-query law, "
                                            f"{len(rows)} of {int(p.q.query_start[-1])} rows")


@pytest.mark.parametrize("law,force_tc", [(("uniform", 1, 4), False), (("uniform", 1, 8), False),
                                          (("uniform", 1, 8), True), (("uniform", 200, 600), False)],
                         ids=["spec4-warp-mma", "spec8-warp-mma2", "spec8-tcgen05", "chunk"])
def test_repeated_launches_are_bit_identical(law, force_tc):
    """The same launch three times gives the same bits (no race between the
    warps that share a row or a stage, the producers and the MMA issuer)."""
    c = config_case(3, num_seqs=64)
    p = Prefill(c, law)
    bound = tc_bound(p) if force_tc else None
    first = p.run(bound).clone()
    assert p.dc.status_bits() == 0
    for _ in range(2):
        p.out.fill_(float("nan"))
        assert torch.equal(p.run(bound), first)


def test_full_size_shared_prefix_e4m3():
    """The shared-prefix E4M3 pool (128 sequences, 64 query heads / 8 KV
    heads, a 1024-token prefix shared by 32 sequences each): a 256-token chunk
    per sequence on the tensor cores; every row of one sequence per prefix
    group, the tile-edge rows of every sequence and random rows against the
    oracle."""
    c = config_case(5)
    p = Prefill(c, ("fixed", np.minimum(256, c.context_lens)))
    got = to_f64(p.run())
    assert p.dc.status_bits() == 0
    # every row of one sequence per prefix group, the tile-edge rows of every
    # sequence, random rows
    rows = p.dense_rows(whole=[0, 32, 64, 96], n_random=64, seed=12)
    want = p.oracle_rows(rows)
    assert_decode_close(got[rows], want, c, f"full: shared-prefix e4m3 256-token chunks, "
                                            f"{len(rows)} of {int(p.q.query_start[-1])} rows")


@pytest.mark.parametrize("draft", [4, 8])
def test_full_size_shared_prefix_e4m3_draft_tokens(draft):
    """The shared-prefix E4M3 pool with 4 and 8 draft tokens per sequence on
    the one-tile tcgen05 kernel (the E4M3 products; 32 and 64 of a tile's 128
    rows at G = 8; the library's own choice at both): every row against the
    oracle."""
    c = config_case(5)
    p = Prefill(c, ("fixed", np.minimum(draft, c.context_lens)))
    assert tc_bound(p) == p.q.max_queries
    assert pk.prefill_kernel(tc_bound(p), c.num_q_heads, c.num_kv_heads, c.head_size,
                             c.block_size, c.num_blocks, pk.PA_BF16, pk.PA_FP8_E4M3) == "tc"
    got = to_f64(p.run(tc_bound(p)))
    assert p.dc.status_bits() == 0
    rows = np.arange(int(p.q.query_start[-1]))
    want = p.oracle_rows(rows)
    assert_decode_close(got[rows], want, c, f"full: shared-prefix e4m3 {draft} draft tokens, "
                                            f"{len(rows)} rows")


def test_full_size_llama7b_mha_f16():
    """The LLaMA-7B fp16 MHA pool (64 sequences, 32 heads, contexts up to
    2016): a 512-token chunk per sequence on the two-tile kernel with single
    binary16 weights and its deeper V ring; every row of four sequences, the
    tile-edge rows of every sequence and random rows against the oracle."""
    c = config_case(2)
    p = Prefill(c, ("fixed", np.minimum(512, c.context_lens)))
    got = to_f64(p.run())
    assert p.dc.status_bits() == 0
    L = c.context_lens
    rows = p.dense_rows(whole=[int(np.argmin(L)), int(np.argmax(L)), 5, 40], n_random=64,
                        seed=21)
    want = p.oracle_rows(rows)
    assert_decode_close(got[rows], want, c, f"full: llama-7b mha f16 512-token chunks, "
                                            f"{len(rows)} of {int(p.q.query_start[-1])} rows")


def test_full_size_long_context_chunk():
    """The long-context pool (8 sequences of 32k..131k tokens): a 512-token
    chunk at the end of each context, about a thousand key tiles per unit;
    the tile-edge rows (first, last, tile boundaries) of every sequence and
    random rows against the oracle."""
    c = config_case(4)
    p = Prefill(c, ("fixed", np.minimum(512, c.context_lens)))
    got = to_f64(p.run())
    assert p.dc.status_bits() == 0
    rows = p.dense_rows(n_random=32, seed=31)
    want = p.oracle_rows(rows)
    assert_decode_close(got[rows], want, c, f"full: long-context 512-token chunks, "
                                            f"{len(rows)} of {int(p.q.query_start[-1])} rows")


@pytest.mark.parametrize("law,force_tc", [(("uniform", 1, 4), False), (("uniform", 1, 8), False),
                                          (("uniform", 1, 8), True), (("uniform", 200, 600), False)],
                         ids=["warp-mma", "warp-mma2", "tcgen05-one-tile", "tcgen05-two-tile"])
def test_sequence_order_does_not_change_outputs(law, force_tc):
    """seq_order only changes when each sequence's work starts: longest
    first and a random permutation give the natural order's bits; an entry
    outside [0, S) raises DEV_BAD_ORDER and the launch still returns."""
    c = config_case(3, num_seqs=48)
    p = Prefill(c, law)
    bound = tc_bound(p) if force_tc else p.q.max_queries
    natural = p.run(bound).clone()
    assert p.dc.status_bits() == 0
    dev = p.out.device
    orders = [pk.longest_first(c.context_lens),
              np.random.default_rng(17).permutation(c.num_seqs).astype(np.int32)]
    for order in orders:
        p.out.fill_(float("nan"))
        pk.paged_prefill(p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache,
                         p.dc.block_tables, p.dc.context_lens, bound,
                         c.max_context_len, c.scale, c.k_scale, c.v_scale, p.dc.status,
                         seq_order=torch.from_numpy(order).to(dev))
        assert p.dc.status_bits() == 0
        assert torch.equal(p.out, natural)
    bad = torch.from_numpy(orders[0].copy()).to(dev)
    bad[5] = c.num_seqs
    pk.paged_prefill(p.out, p.query, p.query_start, p.dc.k_cache, p.dc.v_cache,
                     p.dc.block_tables, p.dc.context_lens, bound, c.max_context_len,
                     c.scale, c.k_scale, c.v_scale, p.dc.status, seq_order=bad)
    assert p.dc.status_bits() & pk.DEV_BAD_ORDER
