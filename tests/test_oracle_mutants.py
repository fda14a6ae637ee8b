"""Plant one plausible mistake at a time in a copy of the oracle (CPU only)
and check that the pins catch it: each mutant must fail at least one pin.
The product is not involved; mistakes are planted in the oracle only."""
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "gqa_modulo": ("h / G", "h % num_kv_heads"),
    "scale_dropped": ("scores[t - t0] = scale * dot;", "scores[t - t0] = dot;"),
    "softmax_sign": ("exp(scores[t - t0] - m)", "exp(m - scores[t - t0])"),
    "tail_overread": ("if (pos >= L)\n                break;", "if (pos > L)\n                break;"),
    "layout_transposed": ("i * st[2] + e * st[3]", "e * st[2] + i * st[3]"),
    "merge_drops_sum": ("double w = part_l[sh * max_parts + p] * exp(", "double w = 1.0 * exp("),
    "e4m3_ties_odd": ("((lo + 1) & 1) == 0", "((lo + 1) & 1) == 1"),
    "e4m3_subnormal_exp": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_no_saturation": ("if (a >= 448.0)\n        return (uint8_t)(sign | 0x7e);",
                           "if (a >= 480.0)\n        return (uint8_t)(sign | 0x7f);"),
    "write_offset": ("int64_t off = slot % block_size;", "int64_t off = (slot + 1) % block_size;"),
    "write_no_scale": ("float qk = xk / k_scale;", "float qk = xk;"),
    "prefill_causal_off_by_one": ("0, pos + 1, h / G, num_kv_heads", "0, pos, h / G, num_kv_heads"),
    "prefill_wrong_position": ("int pos = L - Q + i;", "int pos = L - 1 - i;"),
    "copy_wrong_target": ("((char*)k_cache)[dst * block_elems", "((char*)k_cache)[src * block_elems"),
    "fp8_dequant_no_scale": ("double ks = cache_dtype == OR_E4M3 ? k_scale : 1.0;", "double ks = 1.0;"),
    "bf16_exponent": ("v = ldexp((double)(128 + m), e - 134);", "v = ldexp((double)(128 + m), e - 133);"),
    "f16_subnormal": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -23);"),
    "gather_wrong_block": ("int64_t p = table[j];", "int64_t p = table[j > 0 ? j - 1 : 0];"),
    "partition_bounds": ("int t1 = t0 + partition_size < L ? t0 + partition_size : L;",
                         "int t1 = t0 + partition_size < L ? t0 + partition_size - 1 : L;"),
    "merge_max_first_only": ("if (part_m[sh * max_parts + p] > M)\n                    M = part_m[sh * max_parts + p];",
                             "if (p == 0)\n                    M = part_m[sh * max_parts + p];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutant = text.replace(old, new)
    lib = str(tmp_path / f"liboracle_{name}.so")
    oracle.build_variant(mutant, lib)
    # A mutant may index out of bounds and crash, so its pins run in a child
    # process; the child exits 0 only if every pin passed.
    runner = (
        "import sys, oracle, pins\n"
        "failed = []\n"
        "with oracle.use_library(sys.argv[1]):\n"
        "    for check in pins.ALL:\n"
        "        try:\n"
        "            check()\n"
        "        except (AssertionError, RuntimeError):\n"
        "            failed.append(check.__name__)\n"
        "print('failed:', failed)\n"
        "sys.exit(1 if failed else 0)\n"
    )
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([here, os.path.dirname(here)]))
    proc = subprocess.run([sys.executable, "-c", runner, lib], env=env, capture_output=True,
                          text=True, timeout=300)
    assert proc.returncode != 0, f"no pin caught the planted mistake {name}: {proc.stdout}"
