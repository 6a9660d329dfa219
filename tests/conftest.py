import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _fresh_tuning():
    """Every test starts from the tuning overrides of its (restored)
    environment: the library reads CONV_* overrides once, so re-read them."""
    from transposed_conv_implicit_gb300 import _lib
    if _lib._lib is not None:
        _lib._lib.conv_testing_reload_tuning()
    yield


@pytest.fixture
def tuning(monkeypatch):
    """tuning(name, value) sets a CONV_* tuning override for this test
    (value None clears it) and makes the library re-read the overrides."""
    from transposed_conv_implicit_gb300 import _lib

    def set_override(name, value):
        if value is None:
            monkeypatch.delenv(name, raising=False)
        else:
            monkeypatch.setenv(name, str(value))
        _lib.lib().conv_testing_reload_tuning()
    return set_override
