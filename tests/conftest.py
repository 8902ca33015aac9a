import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path")


def pytest_terminal_summary(terminalreporter):
    """Use of the cancellation allowance on the recorded (full-size) parity
    cases: one line per case, printed after the test results."""
    from tests import parity

    stats = parity.summarize_reports()
    if not stats:
        return
    terminalreporter.write_line("parity allowance record (n, over 1 ulp, admitted by the "
                                "cancellation allowance, max |err|/mag in 2^-24):")
    for name, s in sorted(stats.items()):
        terminalreporter.write_line(
            "  %s: n=%d over_1ulp=%d cancel_allowance_used=%d max_err_over_mag_u=%.2f max_ulp=%d"
            % (name, s["n"], s["over_1ulp"], s["cancel_allowance_used"],
               s["max_err_over_mag_u"], s["max_ulp"]))


def _build_module():
    """The library's build script, loaded by path (importing the package itself
    requires the built library)."""
    path = os.path.join(ROOT, "normalisation_rope_transformers_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_nr_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="session")
def lib_path():
    """Path of libnormrope.so, built (cross-compiled for sm_103a) if stale."""
    return _build_module().build()


@pytest.fixture(scope="session")
def nr(lib_path):
    """The CUDA binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import normalisation_rope_transformers_gb300 as nrt

    return nrt
