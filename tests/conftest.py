import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need the in-tree library; build it once if it is missing
    if any(item.get_closest_marker("gpu") for item in items):
        from normalization_gemm_tcgen05_gb300 import build as _b
        if not os.path.exists(_b.LIB_PATH):
            _b.build()
