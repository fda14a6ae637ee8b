"""GPU parity on the five full-size workloads, in the launch configuration
the benchmark times: the step's KV write compared bit for bit over the whole
pool, then the decode of every sequence compared with the oracle under the
two-part check (max-abs tol of the cache type; elements missing it through
the output rounding alone counted and held to one ulp of the rounded
oracle). Also at the configured 512-token partitions where the library's
own choice differs, and (long-context workload) through the single pass."""
import numpy as np
import pytest

from gpu_common import (DeviceCase, assert_decode_close, oracle_decode_all, oracle_pool, to_f64,
                        torch_to_host)
from paged_kv_cache_141_gb300 import binding as pk
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu

_ORACLE = {}


def oracle_outputs(index):
    """The oracle's pool and every sequence's decode, once per workload."""
    if index not in _ORACLE:
        c = W.config_case(index)
        kc, vc = oracle_pool(c)
        _ORACLE[index] = (c, kc, vc, oracle_decode_all(c, kc, vc))
    return _ORACLE[index]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_full_config(index):
    c, kc, vc, want = oracle_outputs(index)
    d = DeviceCase(c)
    d.write_step()
    assert np.array_equal(torch_to_host(d.k_cache, c.cache_dtype).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(torch_to_host(d.v_cache, c.cache_dtype).view(np.uint8), vc.view(np.uint8))
    P = pk.partition_size(c.num_seqs, c.num_kv_heads, c.max_context_len)
    d.decode("auto", P)
    got = to_f64(d.out)
    assert d.status_bits() == 0
    assert_decode_close(got, want, c, f"full: {c.name}, all {c.num_seqs} sequences, P={P}")


@pytest.mark.parametrize("index", [3, 4])
def test_full_config_configured_partitions(index):
    """The configured 512-token partitions with the merge (the library's
    own choice is 1024 or 2048 on these pools)."""
    c, kc, vc, want = oracle_outputs(index)
    d = DeviceCase(c)
    d.write_step()
    d.decode("split", 512)
    got = to_f64(d.out)
    assert d.status_bits() == 0
    assert_decode_close(got, want, c, f"full: {c.name}, all {c.num_seqs} sequences, P=512")
