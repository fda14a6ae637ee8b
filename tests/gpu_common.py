"""Helpers for the GPU parity tests: move a workload to the device, run the
library's path through the binding, run the oracle on the same host inputs,
and compare."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from oracle import compare
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300.workloads import Case

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8}

# Decode tolerances (max-abs, unit-variance inputs): 2e-3 for 16-bit caches
# and 3e-2 for E4M3 caches; binary32 end to end is held to 1e-4 (float32
# accumulation and ex2.approx weights are accurate to ~1e-6 here).
TOL = {"f32": 1e-4, "f16": 2e-3, "bf16": 2e-3, "e4m3": 3e-2}


def host_to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def torch_to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class DeviceCase:
    """A Case's tensors on the GPU (the pool before the step's write)."""

    def __init__(self, case: Case, device="cuda"):
        self.case = case
        c = case
        dev = torch.device(device)
        self.query = host_to_torch(c.query, c.q_dtype).to(dev)
        self.k_cache = host_to_torch(c.k_cache, c.cache_dtype).to(dev)
        self.v_cache = host_to_torch(c.v_cache, c.cache_dtype).to(dev)
        self.block_tables = torch.from_numpy(c.block_tables).to(dev)
        self.context_lens = torch.from_numpy(c.context_lens).to(dev)
        self.new_key = host_to_torch(c.new_key, c.kv_dtype).to(dev)
        self.new_value = host_to_torch(c.new_value, c.kv_dtype).to(dev)
        self.new_slots = torch.from_numpy(c.new_slots).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty(c.num_seqs, c.num_q_heads, c.head_size, dtype=TORCH[c.q_dtype],
                               device=dev)
        if c.prefill_key is not None:
            pk_ = host_to_torch(c.prefill_key, c.kv_dtype).to(dev)
            pv_ = host_to_torch(c.prefill_value, c.kv_dtype).to(dev)
            ps_ = torch.from_numpy(c.prefill_slots).to(dev)
            pk.reshape_and_cache(pk_, pv_, self.k_cache, self.v_cache, ps_, c.k_scale, c.v_scale,
                                 self.status)
            del pk_, pv_, ps_

    def write_step(self):
        c = self.case
        pk.reshape_and_cache(self.new_key, self.new_value, self.k_cache, self.v_cache,
                             self.new_slots, c.k_scale, c.v_scale, self.status)

    def decode(self, mode="auto", partition_size=None):
        c = self.case
        P = partition_size or c.partition_size
        args = (self.out, self.query, self.k_cache, self.v_cache, self.block_tables,
                self.context_lens, c.max_context_len, c.scale)
        if mode == "single":
            pk.decode(*args, c.k_scale, c.v_scale, self.status)
        elif mode == "split":
            ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len, P,
                                    self.query.device)
            pk.decode_partitioned(*args, ws, P, c.k_scale, c.v_scale, self.status)
        else:
            pk.decode_auto(*args, None, P, c.k_scale, c.v_scale, self.status)
        return self.out

    def status_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.status.item()) & 0xFFFFFFFF


def oracle_pool(case: Case):
    """The oracle's pool after the prefill (E4M3 caches) and the step's write."""
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    c = case
    if c.prefill_key is not None:
        rc = oracle.reshape_and_cache(c.prefill_key, c.prefill_value, kc, vc, c.prefill_slots,
                                      c.num_kv_heads, c.head_size, c.block_size, c.kv_dtype,
                                      c.cache_dtype, c.k_scale, c.v_scale)
        assert rc == 0
    rc = oracle.reshape_and_cache(c.new_key, c.new_value, kc, vc, c.new_slots, c.num_kv_heads,
                                  c.head_size, c.block_size, c.kv_dtype, c.cache_dtype,
                                  c.k_scale, c.v_scale)
    assert rc == 0
    return kc, vc


def parallel_rows(fn, items: np.ndarray, workers: int | None = None) -> np.ndarray:
    """fn over consecutive slices of `items` on host threads, results
    concatenated in order. Each call is the single-threaded oracle on its
    slice (the oracle keeps no shared state; ctypes releases the GIL)."""
    items = np.asarray(items)
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(items, max(1, min(len(items), 4 * workers))) if len(c)]
    with ThreadPoolExecutor(workers) as ex:
        return np.concatenate(list(ex.map(fn, chunks)))


def oracle_decode_all(case: Case, kc, vc) -> np.ndarray:
    """The oracle's decode of every sequence of the case."""
    return parallel_rows(lambda seqs: oracle_decode(case, kc, vc, seqs), np.arange(case.num_seqs))


def oracle_decode(case: Case, kc, vc, seqs=None):
    c = case
    seqs = np.arange(c.num_seqs) if seqs is None else np.asarray(seqs)
    return oracle.decode(np.ascontiguousarray(c.query[seqs]), c.q_dtype, kc, vc, c.cache_dtype,
                         np.ascontiguousarray(c.block_tables[seqs]),
                         np.ascontiguousarray(c.context_lens[seqs]), c.num_kv_heads,
                         c.block_size, c.scale, c.k_scale, c.v_scale)


# Every decode-type comparison made by the tests, for the run's summary:
# (label, cache type, oracle.compare.Parity).
PARITY_LOG: list = []


def assert_decode_close(got: np.ndarray, want: np.ndarray, case: Case, what=""):
    """The two-part check of oracle.compare: |gpu - oracle| <= tol(cache type)
    for every element, except elements that miss it through the output
    rounding alone (within one ulp of the oracle rounded to the output type),
    which are counted and reported."""
    r = compare.check(got, want, TOL[case.cache_dtype], case.q_dtype)
    PARITY_LOG.append((what or case.name, case.cache_dtype, r))
    if not r.ok:
        w = r.worst
        raise AssertionError(
            f"{what}: {r.n_bad} elements beyond tol and beyond one ulp of the rounded oracle; "
            f"worst at {w}: got {got[w]}, want {want[w]}; {r.summary()}")
    return r.max_err


def sample_seqs(case: Case, n: int, seed: int = 0) -> np.ndarray:
    L = case.context_lens
    picks = {int(np.argmin(L)), int(np.argmax(L))}
    rng = np.random.default_rng(seed)
    for s in rng.permutation(case.num_seqs):
        if len(picks) >= n:
            break
        picks.add(int(s))
    return np.array(sorted(picks))
