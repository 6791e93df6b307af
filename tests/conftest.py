import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU test")
    # the oracle (gcc) and the CUDA library (nvcc, cross-compiled for sm_103a)
    # are built in-tree when missing or stale; the library needs no GPU to load
    from oracle import build as obuild
    from block_quantized_weight_dequant_gb300 import build as lbuild

    obuild.compile_oracle()
    lbuild.build()
