import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def _load_oracle_from(pkg_dir):
    """Import the oracle package found in ``pkg_dir`` under the name "oracle"
    (the mutation tests point this at a copy with one planted mistake)."""
    spec = importlib.util.spec_from_file_location(
        "oracle", os.path.join(pkg_dir, "__init__.py"),
        submodule_search_locations=[pkg_dir])
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle"] = mod
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="session")
def orc():
    alt = os.environ.get("I8_ORACLE_DIR")
    if alt:
        oracle = _load_oracle_from(alt)
    else:
        import oracle
    oracle.build()
    return oracle
