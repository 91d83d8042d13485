import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


# A mutation test (tests/test_oracle_mutations.py) re-runs the oracle pins in a
# subprocess with FR_ORACLE_MUTANT pointing at a deliberately broken copy of
# the oracle source; it is swapped in here, before any test imports it.
_MUTANT = os.environ.get("FR_ORACLE_MUTANT")
if _MUTANT:
    import importlib.util

    import oracle as _oracle_pkg
    _spec = importlib.util.spec_from_file_location("oracle.fr_oracle", _MUTANT)
    _mod = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(_mod)
    sys.modules["oracle.fr_oracle"] = _mod
    for _name in _oracle_pkg.__all__:
        setattr(_oracle_pkg, _name, getattr(_mod, _name))
