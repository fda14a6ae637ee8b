"""Checks that pin the oracle to something other than itself.

Each check raises AssertionError on failure. They run against whichever build
of the oracle the ``oracle`` module is bound to, so the same checks serve the
oracle's own tests and the tests that plant a mistake in a copy of the oracle
and expect some check to fail.

What each check compares against:
  * format tables: numpy's binary16, torch's bfloat16 and float8_e4m3fn, and
    the OCP OFP8 reference points in golden/e4m3_ocp.txt;
  * decode: torch's scaled_dot_product_attention in float64 on the logical
    (unpaged) sequence, closed forms, brute force over small integer inputs,
    and invariances (physical placement, block size, cache layout, shared
    blocks vs copies, token order, adding a constant to V);
  * write: the cache read back through a different layout, padding slots,
    the E4M3 quantiser applied to numpy's float32 quotient;
  * merge: single-pass equality and a two-partition closed form.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers

def storage_to_f64(a: np.ndarray, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Decode stored bits with numpy/torch (independently of the oracle)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "e4m3":
        t = torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn)
        return t.to(torch.float64).numpy() * scale
    raise ValueError(dtype)


def f64_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "e4m3":
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
        return t.view(torch.uint8).numpy()
    raise ValueError(dtype)


def random_values(rng, shape, dtype, lo=None):
    x = rng.standard_normal(shape).astype(np.float32)
    if dtype == "e4m3":
        x = np.clip(x * 40.0, -440, 440)
    return f64_to_storage(x, dtype)


def page(seqs_k, seqs_v, block_size, rng, dtype, num_kv_heads, head_size, layout="declared",
         extra_blocks=3, shared=None):
    """Place logical sequences ([L, Hkv, d] storage arrays) into a pool of
    physical blocks at random, block 0 left unused and NaN-filled, unowned
    slots NaN-filled. Returns (k_cache, v_cache, tables, lens, strides).
    layout "declared": [nb, Hkv, B, d]; "pages": [nb, Hkv, d, B].
    shared: optional dict seq -> (other_seq, nblocks) making seq reference the
      first nblocks physical blocks of other_seq instead of its own copies."""
    B, H, d = block_size, num_kv_heads, head_size
    S = len(seqs_k)
    lens = np.array([k.shape[0] for k in seqs_k], dtype=np.int32)
    nblk = [(int(L) + B - 1) // B for L in lens]
    shared = shared or {}
    own = [nblk[s] - (shared[s][1] if s in shared else 0) for s in range(S)]
    num_blocks = 1 + sum(own) + extra_blocks
    perm = rng.permutation(np.arange(1, num_blocks))
    tables = np.zeros((S, max(1, max(nblk))), dtype=np.int32)
    cur = 0
    for s in range(S):
        start = 0
        if s in shared:
            other, nb = shared[s]
            tables[s, :nb] = tables[other, :nb]
            start = nb
        for j in range(start, nblk[s]):
            tables[s, j] = perm[cur]
            cur += 1
    st_dtype = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8}[dtype]
    nan = {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0),
           "e4m3": np.uint8(0x7F)}[dtype]
    if layout == "declared":
        shape = (num_blocks, H, B, d)
        strides = np.array([H * B * d, B * d, d, 1], dtype=np.int64)
    else:
        shape = (num_blocks, H, d, B)
        strides = np.array([H * d * B, d * B, 1, B], dtype=np.int64)
    kc = np.full(shape, nan, dtype=st_dtype)
    vc = np.full(shape, nan, dtype=st_dtype)
    for s in range(S):
        for pos in range(int(lens[s])):
            p, i = tables[s, pos // B], pos % B
            if layout == "declared":
                kc[p, :, i, :] = seqs_k[s][pos]
                vc[p, :, i, :] = seqs_v[s][pos]
            else:
                kc[p, :, :, i] = seqs_k[s][pos]
                vc[p, :, :, i] = seqs_v[s][pos]
    return kc, vc, tables, lens, strides


def dense_reference(q, K, V, scale):
    """torch SDPA in float64 on one sequence. q [Hq, d]; K, V [L, Hkv, d]
    (float64). Query head h reads KV head h // (Hq/Hkv)."""
    Hq, d = q.shape
    L, Hkv, _ = K.shape
    if L == 0:
        return np.zeros((Hq, d))
    G = Hq // Hkv
    Kr = np.repeat(K, G, axis=1).transpose(1, 0, 2)[None]   # [1, Hq, L, d]
    Vr = np.repeat(V, G, axis=1).transpose(1, 0, 2)[None]
    qt = torch.from_numpy(np.ascontiguousarray(q[None, :, None, :]))
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, torch.from_numpy(np.ascontiguousarray(Kr)), torch.from_numpy(np.ascontiguousarray(Vr)),
        scale=scale)
    return out[0, :, 0, :].numpy()


def _random_problem(rng, S, Hq, Hkv, d, dtype, q_dtype, lens):
    ks = [random_values(rng, (int(L), Hkv, d), dtype) for L in lens]
    vs = [random_values(rng, (int(L), Hkv, d), dtype) for L in lens]
    q = random_values(rng, (S, Hq, d), q_dtype)
    return q, ks, vs


# ----------------------------------------------------------------- formats

def check_f16_table():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(bits.view(np.float16), "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def check_bf16_table():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def load_e4m3_golden():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_ocp.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def check_e4m3_table():
    for c, v in load_e4m3_golden():
        got = oracle.e4m3_to_double(c)
        if math.isnan(v):
            assert math.isnan(got), hex(c)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(c), got, v)
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_array(codes, "e4m3")
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0), "non-negative codes must increase"
    assert np.array_equal(got[0x80:0xFF], -got[0x00:0x7F])


def check_e4m3_encode():
    # every finite code round-trips
    for c in list(range(0x00, 0x7F)) + list(range(0x80, 0xFF)):
        v = oracle.e4m3_to_double(c)
        assert oracle.e4m3_encode(np.float32(v)) == c, hex(c)
    # midpoints between neighbours go to the even code; just above/below go the near way
    for c in range(0x00, 0x7E):
        lo, hi = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(np.inf))) == c + 1
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(-np.inf))) == c
        assert oracle.e4m3_encode(-mid) == 0x80 | even
    # saturation, NaN, signed zero
    for x in (448.0, 449.0, 464.0, 480.0, 1e30, np.inf):
        assert oracle.e4m3_encode(np.float32(x)) == 0x7E
        assert oracle.e4m3_encode(np.float32(-x)) == 0xFE
    assert oracle.e4m3_encode(np.float32(np.nan)) & 0x7F == 0x7F
    assert oracle.e4m3_encode(np.float32(-0.0)) == 0x80
    assert oracle.e4m3_encode(np.float32(2.0 ** -11)) == 0x00
    assert oracle.e4m3_encode(np.float32(-(2.0 ** -11))) == 0x80
    # agree with torch's round-to-nearest-even conversion inside the finite range
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-448, 448, 200000).astype(np.float32),
        (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 8, 200000))).astype(np.float32),
    ])
    x = x[np.abs(x) <= 448]
    got = oracle.e4m3_encode_array(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- decode

def check_dense_equivalence(seed=1):
    rng = np.random.default_rng(seed)
    cases = [
        # S, Hq, Hkv, d, B, cache dtype, q dtype, lengths
        (3, 4, 4, 8, 16, "f32", "f32", [1, 17, 40]),
        (2, 8, 2, 16, 8, "bf16", "bf16", [33, 9]),
        (2, 8, 1, 8, 1, "f16", "f16", [5, 12]),
        (2, 16, 2, 8, 32, "e4m3", "bf16", [70, 31]),
        (1, 4, 4, 16, 256, "f32", "f32", [300]),
    ]
    for S, Hq, Hkv, d, B, cdt, qdt, lens in cases:
        q, ks, vs = _random_problem(rng, S, Hq, Hkv, d, cdt, qdt, lens)
        kc, vc, tables, cl, st = page(ks, vs, B, rng, cdt, Hkv, d)
        scale = 1.0 / math.sqrt(d)
        k_scale, v_scale = (0.03125, 0.0625) if cdt == "e4m3" else (1.0, 1.0)
        got = oracle.decode(q, qdt, kc, vc, cdt, tables, cl, Hkv, B, scale, k_scale, v_scale)
        qf = storage_to_f64(q, qdt)
        for s in range(S):
            K = storage_to_f64(ks[s], cdt, k_scale)
            V = storage_to_f64(vs[s], cdt, v_scale)
            want = dense_reference(qf[s], K, V, scale)
            err = np.abs(got[s] - want).max()
            assert err <= 1e-12 * max(1.0, np.abs(want).max()), (cdt, B, s, err)


def check_figure_mapping():
    """The lecture's figure: logical blocks 0,1,2 in physical blocks 7,3,9."""
    rows = []
    with open(os.path.join(GOLDEN, "block_table_figure.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(tuple(int(x) for x in line.split()))
    phys = [p for _, p in sorted(rows)]
    B, H, d, Hq = 4, 2, 8, 4
    L = 3 * B - 1
    rng = np.random.default_rng(3)
    K = rng.standard_normal((L, H, d)).astype(np.float32)
    V = rng.standard_normal((L, H, d)).astype(np.float32)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    nb = 10
    kc = np.full((nb, H, B, d), np.nan, dtype=np.float32)
    vc = np.full((nb, H, B, d), np.nan, dtype=np.float32)
    for pos in range(L):
        kc[phys[pos // B], :, pos % B, :] = K[pos]
        vc[phys[pos // B], :, pos % B, :] = V[pos]
    tables = np.array([phys], dtype=np.int32)
    got = oracle.decode(q, "f32", kc, vc, "f32", tables, np.array([L], np.int32), H, B, 0.5)
    want = dense_reference(q[0].astype(np.float64), K.astype(np.float64), V.astype(np.float64), 0.5)
    assert np.abs(got[0] - want).max() <= 1e-12


def check_placement_and_block_size_invariance(seed=2):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, d = 3, 8, 2, 16
    lens = [1, 45, 130]
    q, ks, vs = _random_problem(rng, S, Hq, Hkv, d, "bf16", "bf16", lens)
    results = []
    for B in (1, 8, 16, 32, 64, 256):
        for trial in range(2):
            kc, vc, tables, cl, st = page(ks, vs, B, rng, "bf16", Hkv, d, extra_blocks=5 + trial)
            results.append(oracle.decode(q, "bf16", kc, vc, "bf16", tables, cl, Hkv, B, 0.25))
    for r in results[1:]:
        assert np.array_equal(r, results[0])


def check_layout_invariance(seed=3):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, d, B = 2, 4, 2, 8, 16
    q, ks, vs = _random_problem(rng, S, Hq, Hkv, d, "f32", "f32", [20, 37])
    a = page(ks, vs, B, np.random.default_rng(9), "f32", Hkv, d, layout="declared")
    b = page(ks, vs, B, np.random.default_rng(9), "f32", Hkv, d, layout="pages")
    ra = oracle.decode(q, "f32", a[0], a[1], "f32", a[2], a[3], Hkv, B, 0.3, strides=a[4])
    rb = oracle.decode(q, "f32", b[0], b[1], "f32", b[2], b[3], Hkv, B, 0.3, strides=b[4])
    assert np.array_equal(ra, rb)
    assert np.isfinite(ra).all()


def check_length_one(seed=4):
    rng = np.random.default_rng(seed)
    for dt in ("f32", "f16", "bf16"):
        q, ks, vs = _random_problem(rng, 2, 4, 2, 8, dt, dt, [1, 1])
        kc, vc, tables, cl, st = page(ks, vs, 16, rng, dt, 2, 8)
        got = oracle.decode(q, dt, kc, vc, dt, tables, cl, 2, 16, 0.7)
        for s in range(2):
            V = storage_to_f64(vs[s], dt)
            for h in range(4):
                assert np.array_equal(got[s, h], V[0, h // 2])


def check_empty_context():
    kc = np.zeros((2, 1, 4, 8), np.float32)
    q = np.ones((1, 2, 8), np.float32)
    got = oracle.decode(q, "f32", kc, kc.copy(), "f32", np.zeros((1, 1), np.int32),
                        np.array([0], np.int32), 1, 4, 1.0)
    assert np.array_equal(got, np.zeros_like(got))


def _two_token(q, k1, k2, v1, v2, scale):
    K = np.array([[k1], [k2]], dtype=np.float32)   # [2, 1, d]
    V = np.array([[v1], [v2]], dtype=np.float32)
    kc = np.full((3, 1, 2, len(q)), np.nan, np.float32)
    vc = np.full((3, 1, 2, len(q)), np.nan, np.float32)
    kc[2, 0, :2] = K[:, 0]
    vc[2, 0, :2] = V[:, 0]
    out = oracle.decode(np.array([[q]], np.float32), "f32", kc, vc, "f32",
                        np.array([[2]], np.int32), np.array([2], np.int32), 1, 2, scale)
    return out[0, 0]


def check_closed_forms():
    # equal scores -> the mean of the two values
    out = _two_token([1.0, 2.0], [0.5, 0.5], [0.5, 0.5], [1.0, -3.0], [2.0, 5.0], 1.0)
    assert np.array_equal(out, np.array([1.5, 1.0]))
    # scores 0 and ln 3 -> weights 1/4 and 3/4
    ln3 = float(np.float32(math.log(3.0)))
    out = _two_token([1.0, 0.0], [0.0, 0.0], [ln3, 0.0], [4.0, 0.0], [0.0, 8.0], 1.0)
    w2 = math.exp(ln3) / (1 + math.exp(ln3))
    assert abs(out[0] - 4.0 * (1 - w2)) <= 1e-15 and abs(out[1] - 8.0 * w2) <= 1e-14
    assert abs(w2 - 0.75) < 1e-7
    # a gap of 100 -> the larger-score value, to within e^-100
    out = _two_token([1.0, 0.0], [0.0, 0.0], [100.0, 0.0], [1.0, 1.0], [2.0, -2.0], 1.0)
    assert np.abs(out - np.array([2.0, -2.0])).max() <= 1e-40
    # brute force over small integers: out = v1*sigma(s1-s2) + v2*sigma(s2-s1)
    vals = (-2.0, -1.0, 0.0, 1.0, 2.0)
    for q0 in vals:
        for q1 in (-1.0, 2.0):
            for a in vals:
                for b in vals:
                    for c in (-2.0, 1.0):
                        q, k1, k2 = [q0, q1], [a, b], [b, c]
                        v1, v2 = [a, 1.0], [c, -b]
                        sc = 0.5
                        s1 = sc * (q0 * a + q1 * b)
                        s2 = sc * (q0 * b + q1 * c)
                        sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
                        want = np.array(v1) * sig + np.array(v2) * (1.0 - sig)
                        got = _two_token(q, k1, k2, v1, v2, sc)
                        assert np.abs(got - want).max() <= 1e-14, (q, k1, k2, got, want)


def check_shared_prefix_by_reference(seed=5):
    rng = np.random.default_rng(seed)
    B, Hkv, d, Hq = 8, 2, 8, 8
    pre_k = random_values(rng, (3 * B, Hkv, d), "bf16")
    pre_v = random_values(rng, (3 * B, Hkv, d), "bf16")
    ks, vs = [], []
    for L_suf in (5, 13, 1):
        ks.append(np.concatenate([pre_k, random_values(rng, (L_suf, Hkv, d), "bf16")]))
        vs.append(np.concatenate([pre_v, random_values(rng, (L_suf, Hkv, d), "bf16")]))
    q = random_values(rng, (3, Hq, d), "bf16")
    copied = page(ks, vs, B, np.random.default_rng(1), "bf16", Hkv, d)
    shared = page(ks, vs, B, np.random.default_rng(1), "bf16", Hkv, d,
                  shared={1: (0, 3), 2: (0, 3)})
    assert shared[0].shape[0] < copied[0].shape[0]
    assert np.array_equal(shared[2][1, :3], shared[2][0, :3])
    ra = oracle.decode(q, "bf16", copied[0], copied[1], "bf16", copied[2], copied[3], Hkv, B, 0.4)
    rb = oracle.decode(q, "bf16", shared[0], shared[1], "bf16", shared[2], shared[3], Hkv, B, 0.4)
    assert np.array_equal(ra, rb)


def check_block_accounting():
    for B in (1, 8, 16, 32, 256):
        for L in range(1, 4 * B + 1):
            touched = len({p // B for p in range(L)})
            assert oracle.blocks_needed(L, B) == touched


def check_token_permutation_and_v_shift(seed=6):
    rng = np.random.default_rng(seed)
    L, Hkv, d, Hq, B = 50, 2, 16, 4, 16
    K = rng.standard_normal((L, Hkv, d)).astype(np.float32)
    # values on a 2^-10 grid, so that V + 3 is exact in float32
    V = (np.rint(rng.standard_normal((L, Hkv, d)) * 1024) / 1024).astype(np.float32)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    perm = rng.permutation(L)

    def run(Kx, Vx):
        kc, vc, t, cl, st = page([Kx], [Vx], B, np.random.default_rng(2), "f32", Hkv, d)
        return oracle.decode(q, "f32", kc, vc, "f32", t, cl, Hkv, B, 0.25)

    base = run(K, V)
    assert np.abs(run(K[perm], V[perm]) - base).max() <= 1e-12
    shifted = run(K, V + np.float32(3.0))
    assert np.abs(shifted - (base + 3.0)).max() <= 1e-12
    same_k = np.repeat(K[:1], L, axis=0)
    out = run(same_k, V)
    mean = V.astype(np.float64).mean(axis=0)
    for h in range(Hq):
        assert np.abs(out[0, h] - mean[h // 2]).max() <= 1e-12


def check_merge_identity(seed=8):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, d = 3, 4, 2, 8
    q, ks, vs = _random_problem(rng, S, Hq, Hkv, d, "f32", "f32", [1, 100, 257])
    kc, vc, tables, cl, st = page(ks, vs, 16, rng, "f32", Hkv, d)
    single = oracle.decode(q, "f32", kc, vc, "f32", tables, cl, Hkv, 16, 0.3)
    for P in (16, 32, 64, 512):
        out, po, pm, pl = oracle.decode_partitioned(q, "f32", kc, vc, "f32", tables, cl, Hkv, 16,
                                                    0.3, P)
        assert np.abs(out - single).max() <= 1e-12, P
        # partition p's partials equal a single-pass decode of just its tokens
        s = 2
        for p in range(-(-int(cl[s]) // P)):
            t0, t1 = p * P, min((p + 1) * P, int(cl[s]))
            sub_k, sub_v = ks[s][t0:t1], vs[s][t0:t1]
            kc2, vc2, t2, cl2, _ = page([sub_k], [sub_v], 16, rng, "f32", Hkv, d)
            o2 = oracle.decode(q[s:s + 1], "f32", kc2, vc2, "f32", t2, cl2, Hkv, 16, 0.3)
            assert np.abs(po[s, :, p] - o2[0]).max() <= 1e-12


def check_merge_closed_form():
    # two partitions: (m=0, l=1, o=a) and (m=ln 3, l=1, o=b) -> weights 1/4, 3/4
    a = np.array([4.0, 0.0])
    b = np.array([0.0, 8.0])
    po = np.zeros((1, 1, 2, 2))
    po[0, 0, 0], po[0, 0, 1] = a, b
    pm = np.array([[[0.0, math.log(3.0)]]])
    pl = np.array([[[1.0, 1.0]]])
    out = oracle.merge(po, pm, pl, np.array([20], np.int32), 10)
    assert np.abs(out[0, 0] - (0.25 * a + 0.75 * b)).max() <= 1e-15
    # a partition whose sum is twice as large counts twice
    pm = np.array([[[0.0, 0.0]]])
    pl = np.array([[[2.0, 1.0]]])
    out = oracle.merge(po, pm, pl, np.array([20], np.int32), 10)
    assert np.abs(out[0, 0] - (2 * a + b) / 3).max() <= 1e-15
    # maxima 1600 apart: the merge subtracts the largest maximum, so nothing
    # overflows and the dominant partition's output comes back
    for order in ((-800.0, 800.0), (800.0, -800.0)):
        pm = np.array([[order]])
        pl = np.array([[[1.0, 1.0]]])
        out = oracle.merge(po, pm, pl, np.array([20], np.int32), 10)
        want = b if order[1] > order[0] else a
        assert np.array_equal(out[0, 0], want)


# ----------------------------------------------------------------- write

def check_write_scatter(seed=9):
    rng = np.random.default_rng(seed)
    T, H, d, B, nb = 12, 2, 8, 4, 9
    for dt in ("f32", "f16", "bf16"):
        key = random_values(rng, (T, H, d), dt)
        val = random_values(rng, (T, H, d), dt)
        slots = rng.permutation(nb * B)[:T].astype(np.int64)
        slots[3] = -1
        # write into both layouts, then compare element by element by meaning
        a_k = np.zeros((nb, H, B, d), key.dtype); a_v = np.zeros_like(a_k)
        b_k = np.zeros((nb, H, d, B), key.dtype); b_v = np.zeros_like(b_k)
        assert oracle.reshape_and_cache(key, val, a_k, a_v, slots, H, d, B, dt, dt) == 0
        assert oracle.reshape_and_cache(key, val, b_k, b_v, slots, H, d, B, dt, dt,
                                        strides=np.array([H * d * B, d * B, 1, B])) == 0
        assert np.array_equal(a_k.view(np.uint8), b_k.transpose(0, 1, 3, 2).copy().view(np.uint8))
        # each written token is found at its slot; the padding token is nowhere
        written = np.zeros((nb, B), bool)
        for t in range(T):
            if slots[t] < 0:
                continue
            blk, off = divmod(int(slots[t]), B)
            written[blk, off] = True
            assert np.array_equal(a_k[blk, :, off, :].view(np.uint8), key[t].view(np.uint8))
            assert np.array_equal(a_v[blk, :, off, :].view(np.uint8), val[t].view(np.uint8))
        untouched = a_k.transpose(0, 2, 1, 3)[~written]
        assert not np.any(untouched.view(np.uint8))
    # out-of-range slot is an error
    key = np.zeros((1, 1, 8), np.float32)
    kc = np.zeros((2, 1, 4, 8), np.float32)
    assert oracle.reshape_and_cache(key, key, kc, kc.copy(), np.array([8]), 1, 8, 4, "f32",
                                    "f32") == oracle.BAD_SLOT


def check_write_e4m3(seed=10):
    rng = np.random.default_rng(seed)
    T, H, d, B, nb = 16, 2, 16, 8, 5
    for dt in ("f16", "bf16", "f32"):
        key = random_values(rng, (T, H, d), dt)
        val = random_values(rng, (T, H, d), dt)
        slots = rng.permutation(nb * B)[:T].astype(np.int64)
        ks, vs = 0.0123, 0.0071
        kc = np.zeros((nb, H, B, d), np.uint8); vc = np.zeros_like(kc)
        assert oracle.reshape_and_cache(key, val, kc, vc, slots, H, d, B, dt, "e4m3", ks, vs) == 0
        xk = storage_to_f64(key, dt).astype(np.float32) / np.float32(ks)
        xv = storage_to_f64(val, dt).astype(np.float32) / np.float32(vs)
        want_k = torch.from_numpy(np.clip(xk, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        want_v = torch.from_numpy(np.clip(xv, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        for t in range(T):
            blk, off = divmod(int(slots[t]), B)
            assert np.array_equal(kc[blk, :, off, :], want_k[t])
            assert np.array_equal(vc[blk, :, off, :], want_v[t])


ALL = [
    check_f16_table, check_bf16_table, check_e4m3_table, check_e4m3_encode,
    check_dense_equivalence, check_figure_mapping, check_placement_and_block_size_invariance,
    check_layout_invariance, check_length_one, check_empty_context, check_closed_forms,
    check_shared_prefix_by_reference, check_block_accounting,
    check_token_permutation_and_v_shift, check_merge_identity, check_merge_closed_form,
    check_write_scatter, check_write_e4m3,
]


def check_copy_blocks():
    """The block copy: block dst equals block src afterwards, others untouched."""
    rng = np.random.default_rng(12)
    kc = rng.integers(0, 255, (6, 2, 4, 8), dtype=np.uint8)
    vc = rng.integers(0, 255, (6, 2, 4, 8), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.copy_blocks(kc, vc, [[1, 4], [2, 5]]) == 0
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[5], v0[2])
    assert np.array_equal(kc[:4], k0[:4]) and np.array_equal(vc[:4], v0[:4])
    assert oracle.copy_blocks(kc, vc, [[1, 6]]) == oracle.BAD_BLOCK


ALL.append(check_copy_blocks)


def check_prefill_reduces_to_decode_and_dense(seed=13):
    """Multi-query paged attention: one query per sequence is the decode; and
    every query equals a dense causal attention (torch SDPA with an explicit
    mask) on the unpaged sequence."""
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, d, B = 3, 8, 2, 16, 8
    lens = [5, 40, 19]
    q_counts = [5, 7, 1]
    ks = [random_values(rng, (L, Hkv, d), "bf16") for L in lens]
    vs = [random_values(rng, (L, Hkv, d), "bf16") for L in lens]
    kc, vc, tables, cl, st = page(ks, vs, B, rng, "bf16", Hkv, d)
    qstart = np.concatenate([[0], np.cumsum(q_counts)]).astype(np.int32)
    q = random_values(rng, (int(qstart[-1]), Hq, d), "bf16")
    got = oracle.paged_prefill(q, "bf16", qstart, kc, vc, "bf16", tables, cl, Hkv, B, 0.3)
    # single query per sequence: the decode of the last position
    last = qstart[1:] - 1
    dec = oracle.decode(np.ascontiguousarray(q[last]), "bf16", kc, vc, "bf16", tables, cl, Hkv, B, 0.3)
    assert np.abs(got[last] - dec).max() <= 1e-12
    # dense causal reference per sequence
    qf = storage_to_f64(q, "bf16")
    G = Hq // Hkv
    for s in range(S):
        L, Q = lens[s], q_counts[s]
        K = torch.from_numpy(np.repeat(storage_to_f64(ks[s], "bf16"), G, axis=1).transpose(1, 0, 2)[None].copy())
        V = torch.from_numpy(np.repeat(storage_to_f64(vs[s], "bf16"), G, axis=1).transpose(1, 0, 2)[None].copy())
        Qs = torch.from_numpy(qf[qstart[s]:qstart[s + 1]].transpose(1, 0, 2)[None].copy())
        pos = torch.arange(L - Q, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                        # [Q, L]
        ref = torch.nn.functional.scaled_dot_product_attention(Qs, K, V, attn_mask=mask, scale=0.3)
        want = ref[0].permute(1, 0, 2).numpy()
        assert np.abs(got[qstart[s]:qstart[s + 1]] - want).max() <= 1e-12


ALL.append(check_prefill_reduces_to_decode_and_dense)
