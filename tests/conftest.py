"""Shared pytest set-up: the ``gpu`` marker and on-demand builds.

``-m "not gpu"`` tests run on any machine (CPU oracle, host-side checks of the
C ABI, multi-process host logic). ``-m gpu`` tests need a CUDA device and the
sm_103a library.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


# Worst errors the GPU tests observed, by quantity (printed at the end of the
# run): the tolerances' margins, as measured.
WORST_ERRORS: dict = {}


def record_error(what: str, value: float) -> None:
    if value > WORST_ERRORS.get(what, -1.0):
        WORST_ERRORS[what] = float(value)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if WORST_ERRORS:
        terminalreporter.write_sep("-", "worst observed errors")
        for k in sorted(WORST_ERRORS):
            terminalreporter.write_line(f"{k}: {WORST_ERRORS[k]:.3e}")
