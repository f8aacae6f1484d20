import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden_lines(name):
    """Non-comment lines of tests/golden/<name>, split at '->'."""
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            yield lhs.split(), rhs.strip()


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """How the layer-input comparisons met their tolerance (GPU runs): the
    elements beyond 2 ulp at |ref| that passed only through the
    cancellation floor, per test that needed it, and over all comparisons."""
    mod = sys.modules.get("gpu_harness")
    reports = getattr(mod, "REPORTS", None)
    if not reports:
        return
    tr = terminalreporter
    total = sum(r["layer_input_elements"] for _, r in reports)
    only = sum(r["layer_input_floor_only"] for _, r in reports)
    tr.write_sep("-", "layer input: elements passing only through the cancellation floor")
    for name, r in reports:
        if r["layer_input_floor_only"] or "large_mxfp8" in name or "glm_style" in name:
            tr.write_line(f"{name}: {r['layer_input_floor_only']} of {r['layer_input_elements']} "
                          f"(max {r['layer_input_floor_only_max_ulp']} ulp, worst T/|ref| "
                          f"{r['layer_input_floor_only_worst_t_over_ref']:.3g}; max ulp overall "
                          f"{r['layer_input_max_ulp']})")
    tr.write_line(f"all {len(reports)} comparisons: {only} of {total} elements "
                  f"({only / max(total, 1):.2e})")
