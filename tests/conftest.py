import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


@pytest.fixture(scope="session")
def gbn():
    """The ctypes binding, building the shared library first if needed."""
    from bwd_bn_pass_gb300 import build, gbnorm
    if not os.path.exists(gbnorm.library_path()):
        build.build_library()
    return gbnorm


def pytest_terminal_summary(terminalreporter):
    """How many bf16 elements were checked against the floor tau rather than
    their own magnitude (the bf16 tolerance reading), per check and in total."""
    from tests import tolerances as tol
    if not tol.TAU_FLOOR_LOG:
        return
    floor = sum(n for _, n, _ in tol.TAU_FLOOR_LOG)
    total = sum(m for _, _, m in tol.TAU_FLOOR_LOG)
    tr = terminalreporter
    tr.section("bf16 tolerance floor (tau) use")
    tr.write_line(f"{floor} of {total} bf16 elements checked ({100.0 * floor / max(total, 1):.4f} %) "
                  f"fell below tau and were bounded by 2 ulp(tau), over "
                  f"{len(tol.TAU_FLOOR_LOG)} comparisons")
    worst = sorted(tol.TAU_FLOOR_LOG, key=lambda t: -t[1] / max(t[2], 1))[:8]
    for name, n, m in worst:
        if n:
            tr.write_line(f"  {name}: {n} / {m}")
