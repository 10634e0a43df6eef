import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_sessionstart(session):
    # (Re)build the C-ABI library when its sources changed; a no-op otherwise.
    from collective_datapath_reduce_gb300 import _build
    _build.build()
