import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_terminal_summary(terminalreporter):
    """Parity report of the decode-type comparisons this run made (see
    gpu_common.assert_decode_close): one line per full-size check, and per
    cache type the number of comparisons, the worst error against its bound
    and the elements passed by the output-rounding clause."""
    gc = sys.modules.get("gpu_common")
    log = getattr(gc, "PARITY_LOG", None) if gc else None
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the oracle (two-part check)")
    for what, _, r in log:
        if what.startswith("full: "):
            tr.write_line(f"{what[6:]}: {r.summary()}")
    per = {}
    for _, cache, r in log:
        a = per.setdefault(cache, [0, 0, 0.0, 0, 0.0, 0.0])
        a[0] += 1
        a[1] += r.n
        if r.max_err / r.tol > a[2]:
            a[2], a[4] = r.max_err / r.tol, r.max_err
        a[3] += r.n_rounding
        a[5] = max(a[5], r.max_rounding_ulps)
    for cache, (checks, n, ratio, n_round, worst, ulps) in sorted(per.items()):
        tr.write_line(f"{cache} caches: {checks} checks, {n} elements, worst err {worst:.3e} "
                      f"({ratio:.2f} of tol), rounding exceptions {n_round}"
                      + (f" (max {ulps:.2f} ulp of the rounded oracle)" if n_round else ""))
