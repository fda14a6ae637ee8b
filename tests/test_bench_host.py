"""Host-side arithmetic of bench.py on the CPU: the algorithmic work of a
multi-query step against a brute-force count, the multi-query query laws,
the rule that attaches recorded DRAM traffic to a bench line, and the kernel
name taken from the library's own selection."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_141_gb300.workloads import config_case, make_case, make_queries  # noqa: E402


def test_prefill_work_matches_a_brute_force_count():
    """FLOPs: 4 d per (query head, key a query token sees); bytes: K and V of
    every context once, the query rows read and the output rows written."""
    c = make_case(num_seqs=5, num_q_heads=8, num_kv_heads=2, head_size=64, block_size=16,
                  q_dtype="bf16", cache_dtype="e4m3", kv_dtype="bf16",
                  lengths=("fixed", [1, 7, 40, 300, 33]), seed=3)
    q = make_queries(c, ("fixed", [1, 3, 40, 12, 0]))
    flops, nbytes = bench.prefill_work(c, q.query_start)
    want_flops = 0
    tokens = 0
    for s in range(c.num_seqs):
        L = int(c.context_lens[s])
        Q = int(q.query_start[s + 1] - q.query_start[s])
        for i in range(Q):
            want_flops += 4 * c.head_size * c.num_q_heads * (L - Q + i + 1)
        tokens += Q
    kv = 2 * int(c.context_lens.sum()) * c.num_kv_heads * c.head_size * 1      # E4M3: 1 byte
    qo = 2 * tokens * c.num_q_heads * c.head_size * 2                            # bf16 rows
    assert flops == want_flops
    assert nbytes == kv + qo
    # a subset of sequences counts only theirs
    f2, b2 = bench.prefill_work(c, q.query_start, np.array([2]))
    assert f2 == sum(4 * 64 * 8 * (40 - 40 + i + 1) for i in range(40))
    assert b2 == 2 * 40 * 2 * 64 + 2 * 40 * 8 * 64 * 2


def test_prefill_query_laws():
    c = config_case(3, num_seqs=16)
    L = c.context_lens
    for kind, n in (("spec8", 8), ("spec4", 4), ("spec2", 2), ("chunk512", 512)):
        law = bench.prefill_queries(c, kind)
        assert law[0] == "fixed"
        assert np.array_equal(np.asarray(law[1]), np.minimum(n, L))


def test_recorded_traffic_only_for_its_own_workload():
    """The committed DRAM bytes are reported only for the kernel source, the
    configuration, partition size and write form they were captured on."""
    got = bench.recorded_traffic(3, 1024, "fused", True)
    with open(bench.TRAFFIC_FILE) as f:
        text = f.read()
    fields = dict(line.split(":", 1) for line in text.splitlines()
                  if ":" in line and not line.startswith("#"))
    if fields["kernel_source_sha256"].strip() == bench.kernel_source_hash():
        assert got == float(fields["dram_bytes_per_launch"])
        assert got >= float(fields["algorithmic_bytes_per_launch"]) * 0.99
    else:
        assert got is None
    assert bench.recorded_traffic(5, 1024, "fused", True) is None
    assert bench.recorded_traffic(3, 512, "fused", True) is None
    assert bench.recorded_traffic(3, 1024, "separate", True) is None
    assert bench.recorded_traffic(3, 1024, "fused", False) is None


def test_prefill_kernel_names_follow_the_library():
    c3 = config_case(3, num_seqs=4)
    assert bench.prefill_kernel_name(c3, 4).startswith("paged_prefill_mma_kernel")
    assert bench.prefill_kernel_name(c3, 8).startswith("paged_prefill_mma2_kernel")
    assert bench.prefill_kernel_name(c3, 16).startswith("paged_prefill_tc_kernel")
    assert bench.prefill_kernel_name(c3, 512).startswith("paged_prefill_tc2_kernel")
    c5 = config_case(5, num_seqs=8)
    assert "E4M3" in bench.prefill_kernel_name(c5, 2)
    assert bench.prefill_kernel_name(c5, 16).startswith("paged_prefill_tc_kernel")
    assert "E4M3 products" in bench.prefill_kernel_name(c5, 16)
    assert bench.prefill_kernel_name(c5, 256).startswith("paged_prefill_tc2_kernel")
    assert "E4M3 products" in bench.prefill_kernel_name(c5, 256)
