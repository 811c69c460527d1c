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


def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_moe_expert_align_gb300 import build
    build.build()


_layers = {}


def _layer(name):
    _need_gpu()
    if name not in _layers:
        import synth
        from tests.gpu_util import DeviceLayer
        _layers[name] = DeviceLayer(synth.WORKLOADS[name].layer, seed=0)
    return _layers[name]


@pytest.fixture(scope="session")
def toy_layer():
    import synth
    return _layer(synth.TOY.name)


@pytest.fixture(scope="session")
def e384_layer():
    import synth
    return _layer(synth.DECODE.name)


@pytest.fixture(scope="session")
def e128_layer():
    import synth
    return _layer(synth.SECOND.name)


@pytest.fixture(scope="session")
def gpu():
    _need_gpu()
    return True
