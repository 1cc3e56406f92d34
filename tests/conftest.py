import os
import sys

# The fp64 oracle runs its matrix products on a thread pool, one product per
# thread: BLAS itself stays single-threaded so that the pool's threads do not
# oversubscribe the cores (set before numpy is first imported).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import pytest  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cpattn():
    """The library binding, built in-tree (nvcc cross-compiles without a GPU)."""
    import context_attention_cpattn_gb300 as m
    m.build()
    m.lib()
    return m
