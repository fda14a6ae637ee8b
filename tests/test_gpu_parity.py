"""GPU parity: the library's kernels (through the C ABI) against the oracle on
the same seeded inputs. Writes must be bit-exact; decode outputs must be
within the cache type's tolerance, elements that miss it through the output
rounding alone counted and held to one ulp of the rounded oracle
(oracle.compare)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from gpu_common import (TORCH, DeviceCase, assert_decode_close, oracle_decode, oracle_pool,
                        to_f64, torch_to_host)
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def small_case(cache, q, Hq, Hkv, D, B, lens, seed=11, shared=None, **kw):
    return W.make_case(num_seqs=len(lens) if shared is None else len(lens), num_q_heads=Hq,
                       num_kv_heads=Hkv, head_size=D, block_size=B, q_dtype=q,
                       cache_dtype=cache, lengths=("fixed", list(lens)), seed=seed,
                       shared_prefix=shared, **kw)


# --------------------------------------------------------------------- write

@pytest.mark.parametrize("cache,kv", [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"),
                                      ("e4m3", "bf16"), ("e4m3", "f16")])
@pytest.mark.parametrize("B", [1, 8, 16, 32, 256])
def test_write_bitexact_small(cache, kv, B):
    q = kv
    c = small_case(cache, q, 4, 2, 128, B, [1, 17, 300, 64, 33], kv_dtype=kv)
    d = DeviceCase(c)
    d.write_step()
    kc, vc = oracle_pool(c)
    assert d.status_bits() == 0
    assert np.array_equal(torch_to_host(d.k_cache, cache).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(torch_to_host(d.v_cache, cache).view(np.uint8), vc.view(np.uint8))


def test_write_padding_and_bad_slot():
    c = small_case("bf16", "bf16", 2, 2, 64, 16, [5, 9])
    d = DeviceCase(c)
    before = d.k_cache.clone()
    slots = d.new_slots.clone()
    slots[0] = -1                                             # padding token: skipped
    slots[1] = c.num_blocks * c.block_size + 3                # outside the pool: flagged
    pk.reshape_and_cache(d.new_key, d.new_value, d.k_cache, d.v_cache, slots, 1.0, 1.0, d.status)
    assert d.status_bits() & pk.DEV_BAD_SLOT
    assert torch.equal(before.view(torch.int16), d.k_cache.view(torch.int16))


def test_write_e4m3_encoder_structured():
    """E4M3 write with scale 1 over structured binary32 patterns: every
    exponent, both signs, every top-8-bit mantissa with sticky variants."""
    exps = np.arange(256, dtype=np.uint32)
    tops = np.arange(256, dtype=np.uint32)
    lows = np.array([0, 1, 0x4000, 0x7FFF], dtype=np.uint32)
    sign = np.array([0, 1], dtype=np.uint32)
    bits = (sign[:, None, None, None] << 31 | exps[None, :, None, None] << 23
            | tops[None, None, :, None] << 15 | lows[None, None, None, :]).reshape(-1)
    rng = np.random.default_rng(5)
    bits = np.concatenate([bits, rng.integers(0, 2**32, 300000, dtype=np.uint64).astype(np.uint32)])
    H, D = 8, 128
    per = H * D
    n_tok = -(-bits.size // per)
    x = np.zeros(n_tok * per, dtype=np.uint32)
    x[:bits.size] = bits
    xf = x.view(np.float32).reshape(n_tok, H, D)
    B = 16
    nb = -(-n_tok // B)
    key = torch.from_numpy(xf).cuda()
    kc = torch.zeros(nb, H, B, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.arange(n_tok, dtype=torch.int64, device="cuda")
    pk.reshape_and_cache(key, key, kc, vc, slots, 1.0, 1.0)
    got = kc.cpu().numpy().transpose(0, 2, 1, 3).reshape(-1, H, D)[:n_tok].reshape(-1)
    want = oracle.e4m3_encode_array(x.view(np.float32))
    nan_in = np.isnan(x.view(np.float32))
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all((got[nan_in] & 0x7F) == 0x7F)


# --------------------------------------------------------------------- decode sweep

SWEEP = [
    # cache, q, Hq, Hkv, D, B, lengths
    ("f32", "f32", 4, 4, 64, 16, [1, 15, 16, 17, 64]),
    ("f16", "f16", 8, 8, 128, 16, [1, 31, 32, 33, 200, 513]),
    ("bf16", "bf16", 32, 8, 128, 16, [1, 100, 511, 512, 513, 1200]),
    ("bf16", "bf16", 16, 2, 128, 1, [1, 2, 33, 70]),
    ("bf16", "bf16", 8, 4, 64, 8, [3, 40, 129]),
    ("bf16", "bf16", 8, 1, 256, 32, [31, 32, 95, 700]),
    ("f16", "f16", 16, 1, 128, 256, [1, 255, 256, 257, 600]),
    ("bf16", "bf16", 12, 4, 128, 64, [10, 64, 65, 300]),              # group of 3
    ("bf16", "bf16", 32, 2, 128, 16, [1, 50, 600]),                    # group of 16
    ("bf16", "bf16", 128, 1, 128, 16, [1, 300, 700]),                  # group of 128
    ("e4m3", "f16", 128, 2, 64, 16, [3, 257]),                         # group of 64
    ("e4m3", "bf16", 64, 8, 128, 16, [1, 20, 512, 777]),
    ("e4m3", "f16", 8, 2, 64, 16, [5, 48, 160]),
    ("e4m3", "bf16", 8, 8, 256, 8, [9, 130]),
    ("e4m3", "bf16", 16, 4, 256, 16, [1, 33, 400]),
    ("e4m3", "f16", 8, 4, 128, 32, [2, 64, 65, 513]),
    # shapes outside the tensor-TMA kernel (block sizes below 8, 64-byte E4M3
    # rows, 1 KB float32 rows) run the bulk-copy kernel
    ("bf16", "bf16", 32, 8, 128, 4, [1, 100, 511, 512, 513, 1200]),
    # block sizes that are not powers of two: a multiple of 32 (tensor TMA,
    # a 32-token stage inside a block) and others (bulk copies); the largest
    # block size the library accepts
    ("bf16", "bf16", 32, 8, 128, 96, [1, 95, 96, 97, 400]),
    ("e4m3", "bf16", 16, 4, 128, 96, [2, 96, 193]),
    ("f16", "f16", 8, 2, 64, 24, [1, 23, 24, 25, 300]),
    ("bf16", "bf16", 8, 8, 128, 48, [47, 48, 49, 150]),
    ("bf16", "bf16", 16, 4, 128, 1024, [1, 1023, 1024, 1025, 2500]),
    ("f16", "f16", 8, 2, 128, 2, [3, 77, 640]),
    ("f32", "f32", 4, 2, 256, 16, [1, 40, 300]),
    ("e4m3", "bf16", 16, 2, 64, 16, [7, 300]),
]


def _sweep_id(p):
    return f"{p[0]}-q{p[2]}-kv{p[3]}-d{p[4]}-b{p[5]}"


@pytest.mark.parametrize("params", SWEEP, ids=[_sweep_id(p) for p in SWEEP])
@pytest.mark.parametrize("mode,P", [("single", 512), ("split", 512), ("split", 64), ("split", 32)])
def test_decode_sweep(params, mode, P):
    cache, q, Hq, Hkv, D, B, lens = params
    c = small_case(cache, q, Hq, Hkv, D, B, lens)
    d = DeviceCase(c)
    d.write_step()
    d.decode(mode, P)
    kc, vc = oracle_pool(c)
    want = oracle_decode(c, kc, vc)
    got = to_f64(d.out)
    assert d.status_bits() == 0
    assert_decode_close(got, want, c, f"{mode}/{P}")


def test_split_agrees_with_single():
    c = W.config_case(3, num_seqs=24)
    d = DeviceCase(c)
    d.write_step()
    single = to_f64(d.decode("single").clone())
    split = to_f64(d.decode("split", 512).clone())
    assert np.abs(single - split).max() <= 1e-3


def test_partials_match_oracle():
    """The partition kernel's per-partition (max, sum, output) against the
    oracle's partials, one partition at a time."""
    c = small_case("bf16", "bf16", 8, 2, 128, 16, [40, 512, 1100, 1536])
    d = DeviceCase(c)
    d.write_step()
    P = 512
    ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P)
    pk.decode_partitions(d.query, d.k_cache, d.v_cache, d.block_tables, d.context_lens,
                         c.max_context_len, c.scale, ws, P)
    tmp, ml, es = pk.workspace_views(ws, c.num_seqs, c.num_q_heads, c.head_size,
                                     c.max_context_len, P)
    kc, vc = oracle_pool(c)
    _, po, pm, pl = oracle.decode_partitioned(c.query, c.q_dtype, kc, vc, c.cache_dtype,
                                              c.block_tables, c.context_lens, c.num_kv_heads,
                                              c.block_size, c.scale, P, max_parts=tmp.shape[2])
    tmp, ml, es = to_f64(tmp), to_f64(ml), to_f64(es)
    for s in range(c.num_seqs):
        n = -(-int(c.context_lens[s]) // P)
        assert np.abs(tmp[s, :, :n] - po[s, :, :n]).max() <= 2e-3
        assert np.abs(ml[s, :, :n] - pm[s, :, :n]).max() <= 1e-4 * max(1, np.abs(pm[s, :, :n]).max())
        assert np.all(np.abs(es[s, :, :n] / pl[s, :, :n] - 1) <= 1e-4)


@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_merge_matches_oracle(out_dtype):
    rng = np.random.default_rng(3)
    S, Hq, D, P = 5, 4, 128, 64
    lens = np.array([0, 1, 64, 65, 64 * 40 + 7], dtype=np.int32)
    mp = int(-(-lens.max() // P))
    po = rng.standard_normal((S, Hq, mp, D)).astype(np.float32)
    pm = (rng.standard_normal((S, Hq, mp)) * 8).astype(np.float32)
    pl = rng.uniform(0.5, 60, (S, Hq, mp)).astype(np.float32)
    out = torch.empty(S, Hq, D, dtype=TORCH[out_dtype], device="cuda")
    pk.merge(out, torch.from_numpy(po).cuda(), torch.from_numpy(pm).cuda(),
             torch.from_numpy(pl).cuda(), torch.from_numpy(lens).cuda(), P)
    want = oracle.merge(po.astype(np.float64), pm.astype(np.float64), pl.astype(np.float64),
                        lens, P)
    got = to_f64(out)
    r = compare.check(got, want, 1e-5 * max(1.0, float(np.abs(want).max())), out_dtype)
    assert r.ok, r.summary()


# --------------------------------------------------------------------- special cases

@pytest.mark.parametrize("cache", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("mode", ["single", "split"])
def test_length_one_returns_v_exactly(cache, mode):
    c = small_case(cache, cache, 8, 2, 128, 16, [1, 1, 1])
    d = DeviceCase(c)
    d.write_step()
    out = d.decode(mode, 512)
    got = torch_to_host(out, cache)
    G = c.group
    for s in range(c.num_seqs):
        for h in range(c.num_q_heads):
            assert np.array_equal(got[s, h].view(np.uint8), c.new_value[s, h // G].view(np.uint8))


def _e4m3_token_values(d, c):
    """Each sequence's only stored V token: its E4M3 codes decoded by torch's
    float8_e4m3fn, times v_scale in float32, rounded to the output type."""
    B = c.block_size
    slots = torch.from_numpy(c.new_slots)
    codes = d.v_cache.cpu()[slots // B, :, slots % B, :]            # [S, Hkv, d] uint8
    vals = codes.view(torch.float8_e4m3fn).float() * torch.tensor(c.v_scale, dtype=torch.float32)
    return vals.to(TORCH[c.q_dtype])


@pytest.mark.parametrize("mode", ["single", "split"])
def test_length_one_e4m3_returns_v_exactly(mode):
    """One key per sequence: the weight is exactly 1, so the output is the
    stored code's value times v_scale, rounded once -- bit for bit. Pins the
    in-register widening of the codes (sign, exponent, subnormals) and the
    scale it folds in."""
    c = small_case("e4m3", "bf16", 8, 2, 128, 16, [1, 1, 1, 1])
    d = DeviceCase(c)
    d.write_step()
    out = d.decode(mode, 512).cpu()
    assert d.status_bits() == 0
    want = _e4m3_token_values(d, c)
    G = c.group
    for h in range(c.num_q_heads):
        assert torch.equal(out[:, h].view(torch.int16), want[:, h // G].view(torch.int16))


def test_empty_context_and_empty_batch():
    c = small_case("bf16", "bf16", 4, 2, 128, 16, [0, 7])
    d = DeviceCase(c)
    d.new_slots[0] = -1
    d.write_step()
    d.out.fill_(1.0)
    d.decode("single")
    assert torch.all(d.out[0] == 0)
    d.out.fill_(1.0)
    d.decode("split", 64)
    assert torch.all(d.out[0] == 0)
    kc, vc = oracle_pool(c)
    assert_decode_close(to_f64(d.out)[1:], oracle_decode(c, kc, vc)[1:], c)
    # zero sequences / zero tokens: nothing launched, no error
    e = torch.empty(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    pk.decode(e, e, d.k_cache, d.v_cache, d.block_tables[:0], d.context_lens[:0], 0, 0.1)
    pk.reshape_and_cache(d.new_key[:0], d.new_value[:0], d.k_cache, d.v_cache, d.new_slots[:0])


def test_maximum_number_of_sequences():
    """65,535 sequences (the most one call takes) of 1..40 tokens: the write,
    the single pass and the partitioned form (up to two 32-token partitions),
    all against the oracle."""
    c = W.make_case(num_seqs=65535, num_q_heads=2, num_kv_heads=1, head_size=64, block_size=16,
                    q_dtype="bf16", cache_dtype="bf16", lengths=("uniform", 1, 40), seed=91)
    d = DeviceCase(c)
    d.write_step()
    kc, vc = oracle_pool(c)
    want = oracle_decode(c, kc, vc)
    d.decode("single")
    assert d.status_bits() == 0
    assert_decode_close(to_f64(d.out), want, c, "65535 sequences, single pass")
    d.out.fill_(float("nan"))
    d.decode("split", 32)
    assert d.status_bits() == 0
    assert_decode_close(to_f64(d.out), want, c, "65535 sequences, 32-token partitions")


def test_shared_prefix_matches_copies():
    """Sequences that share prefix blocks by reference decode exactly like
    sequences holding private copies of those blocks."""
    shared = W.config_case(5, num_seqs=16, shared_prefix=(2, 8), lengths=("uniform", 16, 100))
    d = DeviceCase(shared)
    d.write_step()
    ref = d.decode("split", 128).clone()
    # copy every shared block into a private block per sequence
    kc, vc, bt = d.k_cache, d.v_cache, d.block_tables.clone()
    n_extra = 16 * 8
    kc2 = torch.cat([kc, torch.empty((n_extra,) + kc.shape[1:], dtype=kc.dtype, device="cuda")])
    vc2 = torch.cat([vc, torch.empty((n_extra,) + vc.shape[1:], dtype=vc.dtype, device="cuda")])
    nxt = kc.shape[0]
    for s in range(16):
        for j in range(8):
            kc2[nxt] = kc[bt[s, j]]
            vc2[nxt] = vc[bt[s, j]]
            bt[s, j] = nxt
            nxt += 1
    out2 = torch.empty_like(ref)
    ws = pk.alloc_workspace(16, shared.num_q_heads, 128, shared.max_context_len, 128)
    pk.decode_partitioned(out2, d.query, kc2, vc2, bt, d.context_lens, shared.max_context_len,
                          shared.scale, ws, 128, shared.k_scale, shared.v_scale)
    assert torch.equal(ref, out2)


def test_block_size_does_not_change_result():
    """The same logical K/V paged with block sizes 8, 16 and 256 gives
    bit-identical outputs (one kernel; its arithmetic follows token order, not
    the placement); block size 1 runs the bulk-copy kernel and agrees within
    tolerance."""
    outs = []
    for B in (8, 16, 256, 1):
        c = small_case("bf16", "bf16", 8, 2, 128, B, [300, 45, 1000], seed=21)
        # same logical values for every B: rebuild the pool from one logical draw
        rng = np.random.default_rng(4)
        kd = {}
        for s in range(c.num_seqs):
            L = int(c.context_lens[s])
            k = rng.standard_normal((L, 2, 128)).astype(np.float32)
            v = rng.standard_normal((L, 2, 128)).astype(np.float32)
            kd[s] = (W.to_storage(k, "bf16"), W.to_storage(v, "bf16"))
            for pos in range(L):
                p, i = c.block_tables[s, pos // B], pos % B
                c.k_cache[p, :, i, :] = kd[s][0][pos]
                c.v_cache[p, :, i, :] = kd[s][1][pos]
            c.new_slots[s] = -1
        d = DeviceCase(c)
        d.write_step()
        outs.append(d.decode("split", 512).clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    a, b = to_f64(outs[0]), to_f64(outs[3])
    r = compare.check(b, a, 2e-3, "bf16")
    assert r.ok, r.summary()


# --------------------------------------------------------------------- errors

def test_device_status_flags():
    c = small_case("bf16", "bf16", 4, 2, 128, 16, [40, 70])
    d = DeviceCase(c)
    bt = d.block_tables.clone()
    bt[1, 2] = c.num_blocks + 5                               # outside the pool
    pk.decode(d.out, d.query, d.k_cache, d.v_cache, bt, d.context_lens, c.max_context_len,
              c.scale, dev_status=d.status)
    assert d.status_bits() & pk.DEV_BAD_BLOCK_ID
    d.status.zero_()
    cl = d.context_lens.clone()
    cl[0] = 10**6                                             # longer than the table allows
    pk.decode(d.out, d.query, d.k_cache, d.v_cache, d.block_tables, cl, c.max_context_len,
              c.scale, dev_status=d.status)
    assert d.status_bits() & pk.DEV_BAD_LEN
    d.status.zero_()
    cl[0] = -3
    ws = pk.alloc_workspace(2, 4, 128, c.max_context_len, 64)
    pk.decode_partitioned(d.out, d.query, d.k_cache, d.v_cache, d.block_tables, cl,
                          c.max_context_len, c.scale, ws, 64, dev_status=d.status)
    assert d.status_bits() & pk.DEV_BAD_LEN
    assert d.status_bits() & pk.DEV_TIMEOUT == 0


def test_host_argument_errors():
    c = small_case("bf16", "bf16", 4, 2, 128, 16, [10])
    d = DeviceCase(c)
    with pytest.raises(pk.PagedKVError) as e:          # unsupported head size
        q = torch.zeros(1, 4, 96, dtype=torch.bfloat16, device="cuda")
        kc = torch.zeros(4, 2, 16, 96, dtype=torch.bfloat16, device="cuda")
        pk.decode(q, q, kc, kc, d.block_tables, d.context_lens, 10, 0.1)
    assert e.value.status == pk.PA_ERR_UNSUPPORTED
    with pytest.raises(pk.PagedKVError) as e:          # workspace too small
        ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        pk.decode_partitioned(d.out, d.query, d.k_cache, d.v_cache, d.block_tables,
                              d.context_lens, c.max_context_len, c.scale, ws, 512)
    assert e.value.status == pk.PA_ERR_WORKSPACE
    with pytest.raises(pk.PagedKVError) as e:          # partition size not a multiple of 32
        ws = pk.alloc_workspace(1, 4, 128, 10, 48)
        pk.decode_partitions(d.query, d.k_cache, d.v_cache, d.block_tables, d.context_lens, 10,
                             c.scale, ws, 48)
    assert e.value.status == pk.PA_ERR_INVALID_ARG
    with pytest.raises(pk.PagedKVError) as e:          # E4M3 scale must be positive
        kc8 = torch.zeros(4, 2, 16, 128, dtype=torch.uint8, device="cuda")
        pk.reshape_and_cache(d.new_key, d.new_value, kc8, kc8.clone(), d.new_slots, 0.0, 1.0)
    assert e.value.status == pk.PA_ERR_INVALID_ARG
    with pytest.raises(pk.PagedKVError) as e:          # f32 query with an E4M3 cache
        q = torch.zeros(1, 4, 128, dtype=torch.float32, device="cuda")
        kc8 = torch.zeros(4, 2, 16, 128, dtype=torch.uint8, device="cuda")
        pk.decode(q, q, kc8, kc8, d.block_tables, d.context_lens, 10, 0.1)
    assert e.value.status == pk.PA_ERR_UNSUPPORTED

