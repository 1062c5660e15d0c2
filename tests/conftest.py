import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libpackedadam.so")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def built_package():
    """The binding, after building libpackedadam.so if needed (nvcc cross-compiles
    without a GPU); skips when no CUDA toolkit is installed."""
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_pa_build", os.path.join(ROOT, "adamw_update_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    try:
        mod.build()
    except RuntimeError as e:
        pytest.skip(str(e))
    import adamw_update_gb300

    return adamw_update_gb300
