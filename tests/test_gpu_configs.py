"""GPU parity on the five full-size workloads, in the launch configuration
the benchmark times: the step's KV write compared bit for bit over the whole
pool, then the decode compared with the oracle on sampled sequences (always
including the shortest and the longest)."""
import numpy as np
import pytest

from gpu_common import (DeviceCase, assert_decode_close, oracle_decode, oracle_pool, sample_seqs,
                        to_f64, torch_to_host)
from paged_kv_cache_141_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SAMPLES = {1: 4, 2: 6, 3: 8, 4: 3, 5: 8}


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_full_config(index):
    c = W.config_case(index)
    d = DeviceCase(c)
    d.write_step()
    kc, vc = oracle_pool(c)
    assert np.array_equal(torch_to_host(d.k_cache, c.cache_dtype).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(torch_to_host(d.v_cache, c.cache_dtype).view(np.uint8), vc.view(np.uint8))
    d.decode("auto")
    got = to_f64(d.out)
    assert np.isfinite(got).all()
    assert d.status_bits() == 0
    seqs = sample_seqs(c, SAMPLES[index], seed=index)
    want = oracle_decode(c, kc, vc, seqs)
    err = assert_decode_close(got[seqs], want, c, c.name)
    print(f"{c.name}: max err {err:.3e} over sequences {seqs.tolist()}, "
          f"max |out| {np.abs(want).max():.3f}")
