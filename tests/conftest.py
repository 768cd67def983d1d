import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # Files named test_zz_* run last.  The no-allocation entry point's test
    # lives there: a run that stops at the first failure (-x) has then run
    # every other test before it, and that test also checks that the shared
    # static scratch gives the same results after all the other work done in
    # this process.
    items.sort(key=lambda it: 1 if os.path.basename(str(it.fspath)).startswith("test_zz_") else 0)


def pytest_terminal_summary(terminalreporter):
    # counts that GPU tests report (e.g. rows accepted through the near-tie
    # hull), printed even when the tests pass
    from tests import notes
    if notes.LINES:
        terminalreporter.write_sep("-", "reported by the tests")
        for ln in notes.LINES:
            terminalreporter.write_line(ln)
