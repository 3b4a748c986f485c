import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle


@pytest.fixture(scope="session")
def zs():
    """The product binding with its CUDA library built (nvcc cross-compiles
    without a GPU; loading the library needs no device)."""
    from zero_partitioned_mixed_partition_gb300 import binding, build
    build.build(checked=os.environ.get("ZS_CHECKED") == "1")
    binding.lib()
    return binding


@pytest.fixture(autouse=True)
def _index_checks(request):
    """Under the debug build (ZS_CHECKED=1), every GPU test must leave the
    kernels' index checks without a recorded failure."""
    yield
    if os.environ.get("ZS_CHECKED") == "1" and request.node.get_closest_marker("gpu"):
        from zero_partitioned_mixed_partition_gb300 import binding
        built, fault = binding.zero_debug_checks()
        assert built, "ZS_CHECKED=1 but the loaded library has no index checks"
        assert fault == 0, f"index check failed: site {fault >> 48}, element {fault & ((1 << 48) - 1)}"


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda", 0)
