import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # Build (or reuse, by source-hash stamp) the in-tree library so the ABI tests can load it.
    from tensor_sharded_linear_gqa_gb300 import build
    build.build()
