import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly (not skip) when asked for and no GPU is present."""
    return


def pytest_terminal_summary(terminalreporter):
    """GPU-vs-oracle parity counts of the session: per test, then the totals
    (lane-steps compared, near-tie divergences of the kept sets and of the
    budgets, lane-steps left uncompared after one, the largest errors)."""
    mod = sys.modules.get("tests.parity")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.section("CONF-KV parity vs the oracle")
    per = {}
    for tid, r in recs:
        a = per.setdefault(tid, [0, 0, 0, 0, 0, 0.0, 0.0])
        a[0] += r.compared
        a[1] += r.total
        a[2] += r.kept_div
        a[3] += r.budget_div
        a[4] += r.uncompared
        a[5] = max(a[5], r.max_out_err)
        a[6] = max(a[6], r.max_c_err)
    if tr.config.getoption("verbose") > 0 or os.environ.get("CONFKV_PARITY_DETAIL"):
        for tid, a in per.items():
            tr.write_line(f"{tid.split('::', 1)[-1][:60]:60s} {a[0]}/{a[1]} kept_div={a[2]} "
                          f"budget_div={a[3]} uncompared={a[4]} out={a[5]:.1e} c={a[6]:.1e}")
    tot = [sum(a[i] for a in per.values()) for i in range(5)]
    tr.write_line(f"parity runs={len(recs)} tests={len(per)} lane-steps compared={tot[0]}/{tot[1]} "
                  f"kept_div={tot[2]} budget_div={tot[3]} uncompared={tot[4]} "
                  f"max_out_err={max(a[5] for a in per.values()):.2e} (tol 1e-3) "
                  f"max_c_err={max(a[6] for a in per.values()):.2e} (tol 1e-5)")
