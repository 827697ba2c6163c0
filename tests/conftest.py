import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The library and the oracle are built in-tree; build them (incrementally)
# before any test module imports them.
import __graft_entry__  # noqa: E402

__graft_entry__._load_libbuild().build()
from oracle import build as _oracle_build  # noqa: E402

_oracle_build.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
