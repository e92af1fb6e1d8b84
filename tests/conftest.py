import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running statistical test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle._load()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-config parity table of the GPU tests: rows checked against the
    oracle, rows exempted as near-ties (top-two oracle scores closer than
    1e-5), and their fraction."""
    mod = sys.modules.get("tests.gpu_util")
    table = getattr(mod, "PARITY", None) if mod else None
    if not table:
        return
    tr = terminalreporter
    tr.section("parity against the oracle, per configuration")
    tr.write_line("%-34s %9s %7s %10s %10s" % ("config", "rows", "near", "fraction",
                                              "near-miss"))
    for name in sorted(table):
        t = table[name]
        tr.write_line("%-34s %9d %7d %10.2e %10d" % (name, t.rows, t.near, t.near_fraction,
                                                    t.near_mismatch))
    path = os.environ.get("GSAMPLE_PARITY_TABLE")
    if path:
        import json

        with open(path, "w") as f:
            json.dump({k: {"rows": v.rows, "near": v.near, "near_fraction": v.near_fraction,
                           "near_mismatch": v.near_mismatch} for k, v in table.items()}, f,
                      indent=1, sort_keys=True)
