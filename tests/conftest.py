import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--flce-debug-lib", action="store_true", default=False,
                     help="run against libflce_debug.so, the build that checks every kernel store "
                          "against its buffer")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of oracle time)")
    if config.getoption("--flce-debug-lib"):
        from linear_cross_entropy_tiled_gb300 import _lib
        _lib.use_debug_library()
