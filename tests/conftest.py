import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built libvp.so")
    # libvp.so is a build product, not checked in: (re)build it when missing or older
    # than its sources (nvcc cross-compiles for sm_103a; a no-op when up to date)
    from vocab_lm_head_vp_b300 import build
    build.build()
