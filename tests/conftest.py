"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device with the compiled library; all other
tests run on the CPU alone (oracle pins, generator, host-side validation, ABI
symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
