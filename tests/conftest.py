"""pytest configuration: the ``gpu`` marker and the import path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Kernel waits are bounded; in tests a stuck pipeline should report within 1 s.
os.environ.setdefault("ATTN_WAIT_LIMIT_NS", "1000000000")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); run with -m gpu on a GB300")
