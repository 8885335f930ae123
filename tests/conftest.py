"""Shared pytest configuration.

Markers:
  gpu  -- needs a CUDA device (a GB300, sm_103a); runs the product kernels
          through the C ABI and compares them with the CPU oracle.
Tests without the marker run on any host: the oracle against its pins, the
host-side logic, and the C-ABI library's exported symbols.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_sessionstart(session):
    """Build the oracle and the C-ABI library if they are missing or stale
    (host compilers only; nothing here touches a GPU)."""
    import importlib.util

    from oracle import build as obuild
    obuild.build()
    # load the library's build script by path: importing the package itself
    # needs the library to exist already
    spec = importlib.util.spec_from_file_location(
        "_mx_lib_build", os.path.join(ROOT, "bit_gemm_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
