"""Seeded synthetic inputs for the paged KV write and the paged decode.

This module only makes inputs: context lengths, a block pool with a random
physical placement, block tables, slot mappings, and N(0,1) query / key /
value data. It holds none of the operations' arithmetic; the CUDA library and
the oracle both consume what it produces, and nothing else is shared between
them.

Host storage types: binary32 -> ``np.float32``, binary16 -> ``np.float16``,
bfloat16 -> ``np.uint16`` bit patterns, OCP E4M3 -> ``np.uint8`` codes.

Recipe (one seed per case):
  * context lengths from the case's length law;
  * the pool holds one reserved block 0, the blocks the sequences need, and a
    free margin (10% by default); sequences take physical blocks in the order
    of a seeded random permutation of 1..num_blocks-1, so logically adjacent
    blocks are physically scattered (the block-table figure of "Lecture 3:
    PagedAttention and vLLM": logical 0,1,2 -> physical 7,3,9);
  * shared-prefix cases hand each group's prefix blocks to all its members by
    reference, as fork does in "Continuous Batching and PagedAttention"
    sec. 3.2;
  * every slot that no sequence owns holds a NaN pattern (block 0, free
    blocks, the tail of each last block, and -- until the step writes it -- the
    slot of each sequence's newest token), so that any read past a sequence's
    context shows up as NaN;
  * query/key/value values are N(0,1) drawn in float32 and rounded to the
    storage type; each tensor has its own random stream keyed by (seed,
    stream id, chunk index), so the bits do not depend on the thread count.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}
NAN_PATTERN = {"f32": np.uint32(0x7FC00000), "f16": np.uint16(0x7E00),
               "bf16": np.uint16(0x7FC0), "e4m3": np.uint8(0x7F)}
_BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8}

_CHUNK = 1 << 22
_STREAM_Q, _STREAM_K, _STREAM_V, _STREAM_NEWK, _STREAM_NEWV = 1, 2, 3, 4, 5
_STREAM_MQ, _STREAM_QCOUNT = 6, 7


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normal float32 values from the (seed, stream) stream."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, i])))
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage type (round to nearest even)."""
    if dtype == "f32":
        return x.astype(np.float32, copy=False)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(f"no direct N(0,1) storage for {dtype}")


def normal(seed: int, stream: int, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    return to_storage(normal_f32(seed, stream, n), dtype).reshape(shape)


def poison_fill(arr: np.ndarray, dtype: str, index=slice(None)) -> None:
    arr.view(_BITS[dtype])[index] = NAN_PATTERN[dtype]


@dataclass
class Case:
    """One paged-decode problem plus the step's KV write."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    q_dtype: str
    cache_dtype: str
    kv_dtype: str                     # dtype of the new key/value tokens
    context_lens: np.ndarray          # [S] int32
    block_tables: np.ndarray          # [S, max_blocks] int32
    query: np.ndarray                 # [S, Hq, d]
    k_cache: np.ndarray               # [num_blocks, Hkv, B, d] (pre-step)
    v_cache: np.ndarray
    new_key: np.ndarray               # [S, Hkv, d]: each sequence's newest token
    new_value: np.ndarray
    new_slots: np.ndarray             # [S] int64
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    prefill_key: np.ndarray | None = None    # E4M3 caches: tokens written before the step
    prefill_value: np.ndarray | None = None
    prefill_slots: np.ndarray | None = None
    partition_size: int = 512
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max(initial=0))

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    def kv_bytes(self) -> int:
        """Logical K+V bytes one decode reads (every sequence's context, all KV heads)."""
        return (2 * self.total_tokens * self.num_kv_heads * self.head_size
                * ELEM_BYTES[self.cache_dtype])

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct cache slots the decode reads: a block
        shared by several sequences' tables counts once (equals kv_bytes()
        when no block is shared)."""
        B = self.block_size
        slots = [self.block_tables[s, np.arange(L) // B].astype(np.int64) * B + np.arange(L) % B
                 for s, L in enumerate(self.context_lens.astype(np.int64)) if L > 0]
        n = int(np.unique(np.concatenate(slots)).size) if slots else 0
        return 2 * n * self.num_kv_heads * self.head_size * ELEM_BYTES[self.cache_dtype]

    def qo_bytes(self) -> int:
        return 2 * self.num_seqs * self.num_q_heads * self.head_size * ELEM_BYTES[self.q_dtype]

    def write_bytes(self, num_tokens: int | None = None) -> int:
        """Bytes one KV write of `num_tokens` tokens moves: inputs read,
        cache written, and the 8-byte slot per token."""
        t = self.num_seqs if num_tokens is None else num_tokens
        per = self.num_kv_heads * self.head_size * 2
        return t * (per * (ELEM_BYTES[self.kv_dtype] + ELEM_BYTES[self.cache_dtype]) + 8)


def _draw_lengths(rng: np.random.Generator, law, n: int) -> np.ndarray:
    kind = law[0]
    if kind == "uniform":
        lo, hi = law[1], law[2]
        return rng.integers(lo, hi + 1, size=n).astype(np.int32)
    if kind == "loguniform":
        lo, hi = law[1], law[2]
        u = rng.uniform(math.log(lo), math.log(hi), size=n)
        return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int32)
    if kind == "fixed":
        return np.asarray(law[1], dtype=np.int32).reshape(n)
    raise ValueError(law)


def make_case(*, name="case", num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
              q_dtype, cache_dtype, kv_dtype=None, lengths, seed, num_blocks=None,
              free_frac=0.1, shared_prefix=None, partition_size=512, scale=None) -> Case:
    """Build a Case.

    lengths: ("uniform", lo, hi) | ("loguniform", lo, hi) | ("fixed", [L...]).
    shared_prefix: None or (groups, prefix_blocks): num_seqs is split into
      `groups` equal groups whose members share `prefix_blocks` physical
      blocks; `lengths` then draws each member's private suffix length.
    """
    if kv_dtype is None:
        kv_dtype = q_dtype if cache_dtype == "e4m3" else cache_dtype
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    S, Hkv, B, d = num_seqs, num_kv_heads, block_size, head_size

    # context lengths
    if shared_prefix is None:
        lens = _draw_lengths(rng, lengths, S)
        prefix_tokens = 0
    else:
        groups, prefix_blocks = shared_prefix
        assert S % groups == 0
        prefix_tokens = prefix_blocks * B
        lens = (prefix_tokens + _draw_lengths(rng, lengths, S)).astype(np.int32)
    nblk = [(int(L) + B - 1) // B for L in lens]

    # pool size and the physical placement
    if shared_prefix is None:
        used = sum(nblk)
    else:
        groups, prefix_blocks = shared_prefix
        used = groups * prefix_blocks + sum(n - prefix_blocks for n in nblk)
    if num_blocks is None:
        num_blocks = 1 + used + int(math.ceil(free_frac * used))
    assert num_blocks >= 1 + used, "pool too small"
    perm = rng.permutation(np.arange(1, num_blocks, dtype=np.int64))
    max_blocks = max(1, max(nblk) if nblk else 1)
    tables = np.zeros((S, max_blocks), dtype=np.int32)      # padding entries -> block 0
    owned = np.zeros(num_blocks, dtype=bool)
    cur = 0
    if shared_prefix is None:
        for s in range(S):
            tables[s, :nblk[s]] = perm[cur:cur + nblk[s]]
            cur += nblk[s]
    else:
        groups, prefix_blocks = shared_prefix
        per_group = S // groups
        for g in range(groups):
            prefix = perm[cur:cur + prefix_blocks]
            cur += prefix_blocks
            for s in range(g * per_group, (g + 1) * per_group):
                tables[s, :prefix_blocks] = prefix
                k = nblk[s] - prefix_blocks
                tables[s, prefix_blocks:nblk[s]] = perm[cur:cur + k]
                cur += k
    for s in range(S):
        owned[tables[s, :nblk[s]]] = True

    # slots of each sequence's newest token (position L-1)
    new_slots = np.full(S, -1, dtype=np.int64)
    for s in range(S):
        L = int(lens[s])
        if L > 0:
            new_slots[s] = int(tables[s, (L - 1) // B]) * B + (L - 1) % B

    query = normal(seed, _STREAM_Q, (S, num_q_heads, d), q_dtype)
    new_key = normal(seed, _STREAM_NEWK, (S, Hkv, d), kv_dtype)
    new_value = normal(seed, _STREAM_NEWV, (S, Hkv, d), kv_dtype)
    shape = (num_blocks, Hkv, B, d)

    case = Case(name=name, num_seqs=S, num_q_heads=num_q_heads, num_kv_heads=Hkv, head_size=d,
                block_size=B, num_blocks=num_blocks, q_dtype=q_dtype, cache_dtype=cache_dtype,
                kv_dtype=kv_dtype, context_lens=lens, block_tables=tables, query=query,
                k_cache=None, v_cache=None, new_key=new_key, new_value=new_value,
                new_slots=new_slots, scale=0.0, partition_size=partition_size, seed=seed)
    case.scale = float(np.float32(1.0 / math.sqrt(d))) if scale is None else float(scale)

    # which slots hold a token before the step: positions < L-1 of every sequence
    valid = np.zeros((num_blocks, B), dtype=bool)
    for s in range(S):
        L = int(lens[s])
        for j in range(nblk[s]):
            lo = j * B
            n_in = min(B, max(0, (L - 1) - lo))
            valid[tables[s, j], :n_in] = True

    if cache_dtype != "e4m3":
        k_cache = normal(seed, _STREAM_K, shape, cache_dtype)
        v_cache = normal(seed, _STREAM_V, shape, cache_dtype)
        blk_idx, pos_idx = np.nonzero(~valid)
        for arr in (k_cache, v_cache):
            bits = arr.view(_BITS[cache_dtype])
            bits[blk_idx, :, pos_idx, :] = NAN_PATTERN[cache_dtype]
        case.k_cache, case.v_cache = k_cache, v_cache
    else:
        # E4M3 pool: every slot starts as the NaN code; the tokens before the
        # step are written by the KV write itself (a prefill), from kv_dtype.
        case.k_cache = np.full(shape, NAN_PATTERN["e4m3"], dtype=np.uint8)
        case.v_cache = np.full(shape, NAN_PATTERN["e4m3"], dtype=np.uint8)
        blk_idx, pos_idx = np.nonzero(valid)
        pre_slots = (blk_idx.astype(np.int64) * B + pos_idx).astype(np.int64)
        T = pre_slots.size
        case.prefill_slots = pre_slots
        case.prefill_key = normal(seed, _STREAM_K, (T, Hkv, d), kv_dtype)
        case.prefill_value = normal(seed, _STREAM_V, (T, Hkv, d), kv_dtype)
        case.k_scale = _amax_scale(case.prefill_key, new_key, kv_dtype)
        case.v_scale = _amax_scale(case.prefill_value, new_value, kv_dtype)
    case.meta = {"owned_blocks": int(owned.sum()), "prefix_tokens": prefix_tokens}
    return case


@dataclass
class Queries:
    """Query tokens of a multi-query attention step over a Case's sequences."""
    query: np.ndarray          # [T, Hq, d], the Case's query type
    query_start: np.ndarray    # [S + 1] int32; sequence s owns rows query_start[s]..[s+1]-1
    max_queries: int           # max over s of Q_s

    @property
    def counts(self) -> np.ndarray:
        return np.diff(self.query_start)


def make_queries(case: Case, law, seed: int | None = None) -> Queries:
    """Q_s query tokens per sequence, the last Q_s positions of its context.

    law: ("uniform", lo, hi) draws Q_s, clipped to [min(1, L_s), L_s];
    ("fixed", [Q...]) gives them, clipped to [0, L_s]; ("all",) takes
    Q_s = L_s (a whole prefill).
    Query values are N(0,1) in the Case's query type, on their own stream.
    """
    seed = case.seed if seed is None else seed
    S = case.num_seqs
    L = case.context_lens.astype(np.int64)
    if law[0] == "all":
        q = L.copy()
    elif law[0] == "fixed":
        q = np.asarray(law[1], dtype=np.int64).reshape(S)
    elif law[0] == "uniform":
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM_QCOUNT])))
        q = rng.integers(law[1], law[2] + 1, size=S).astype(np.int64)
    else:
        raise ValueError(law)
    q = np.minimum(np.maximum(q, 0 if law[0] == "fixed" else np.minimum(1, L)), L)
    start = np.zeros(S + 1, dtype=np.int64)
    np.cumsum(q, out=start[1:])
    assert start[-1] < 2 ** 31
    T = int(start[-1])
    query = normal(seed, _STREAM_MQ, (T, case.num_q_heads, case.head_size), case.q_dtype)
    return Queries(query=query, query_start=start.astype(np.int32),
                   max_queries=int(q.max(initial=0)))


def _amax_scale(a: np.ndarray, b: np.ndarray, dtype: str) -> float:
    """Per-tensor E4M3 scale: max |x| over every value written, over 448 (the
    largest finite E4M3 magnitude), in float32."""
    def amax(x):
        if dtype == "bf16":
            bits = (x.astype(np.uint32) << 16).view(np.float32)
            return float(np.abs(bits).max(initial=0.0))
        return float(np.abs(x.astype(np.float32)).max(initial=0.0))
    m = np.float32(max(amax(a), amax(b)))
    return float(m / np.float32(448.0)) if m > 0 else 1.0


# The five workloads, by index. Seed = 0x5EED0000 + index.
CONFIGS = {
    1: dict(name="tiny-fp32", num_seqs=4, num_q_heads=4, num_kv_heads=4, head_size=64,
            block_size=16, q_dtype="f32", cache_dtype="f32", lengths=("uniform", 1, 64),
            num_blocks=64),
    2: dict(name="llama7b-mha-fp16", num_seqs=64, num_q_heads=32, num_kv_heads=32, head_size=128,
            block_size=16, q_dtype="f16", cache_dtype="f16", lengths=("uniform", 128, 2048)),
    3: dict(name="llama3-8b-gqa-bf16", num_seqs=256, num_q_heads=32, num_kv_heads=8,
            head_size=128, block_size=16, q_dtype="bf16", cache_dtype="bf16",
            lengths=("loguniform", 512, 4096)),
    4: dict(name="long-context-splitk-bf16", num_seqs=8, num_q_heads=32, num_kv_heads=8,
            head_size=128, block_size=16, q_dtype="bf16", cache_dtype="bf16",
            lengths=("uniform", 32768, 131072)),
    5: dict(name="shared-prefix-fp8-70b", num_seqs=128, num_q_heads=64, num_kv_heads=8,
            head_size=128, block_size=16, q_dtype="bf16", cache_dtype="e4m3", kv_dtype="bf16",
            lengths=("uniform", 16, 512), shared_prefix=(4, 64)),
}


def config_seed(index: int) -> int:
    return 0x5EED0000 + index


def config_case(index: int, **overrides) -> Case:
    spec = dict(CONFIGS[index])
    spec.update(overrides)
    seed = spec.pop("seed", config_seed(index))
    return make_case(seed=seed, **spec)
