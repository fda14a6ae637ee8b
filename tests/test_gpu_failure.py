"""Failure detection on the device without a GPU fault. Every wait inside the
library's kernels is bounded: a self-test kernel makes both kinds of wait
(the TMA pipelines' and the tensor-core pipelines') run out on purpose, on an
mbarrier that nothing completes. They must report DEV_TIMEOUT through the
status word and return. The context must stay usable: a decode right after
still matches the oracle. With the arrival made, nothing is reported."""
import time

import pytest
import torch

from gpu_common import DeviceCase, assert_decode_close, oracle_decode, oracle_pool, to_f64
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_bounded_wait_returns_once_the_barrier_completes():
    st = _status()
    pk.selftest_wait(True, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable():
    st = _status()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pk.selftest_wait(False, st)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    bits = int(st.item())
    assert bits & pk.DEV_TIMEOUT
    assert not bits & pk.DEV_BAD_LEN                 # no wait returned without an arrival
    # the limit is about a second of SM clocks: the waits did wait
    assert 0.2 < waited < 30.0
    # the same context runs the hot path correctly afterwards
    c = W.make_case(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                    q_dtype="bf16", cache_dtype="bf16", lengths=("fixed", [5, 300, 1100]),
                    seed=77)
    d = DeviceCase(c)
    d.write_step()
    d.decode("split", 512)
    assert d.status_bits() == 0
    kc, vc = oracle_pool(c)
    assert_decode_close(to_f64(d.out), oracle_decode(c, kc, vc), c, "decode after a timeout")
