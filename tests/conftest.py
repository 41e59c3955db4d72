import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The library picks CTA pairs for the row-grouped expert GEMMs only for large layers; the
# tests' shapes are small, so they ask for pairs wherever an expert can fill a pair tile
# (MOE_GEMM_PAIR=1) to exercise the pair kernels.  test_gpu_schedule.py checks that pairs,
# single CTAs and the automatic choice give bitwise the same results.
os.environ.setdefault("MOE_GEMM_PAIR", "1")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
