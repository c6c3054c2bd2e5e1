import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")
    # the library is built in-tree; (re)build it when sources changed so both the
    # CPU ABI tests and the GPU tests load the current code
    try:
        from bit_vector_lut_gb300 import build as b
        b.build()
    except Exception as e:  # nvcc missing: the ABI tests skip, GPU tests fail loudly
        sys.stderr.write(f"[conftest] library build skipped: {e}\n")
