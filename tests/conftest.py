import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # The tests call the library through its C ABI; build it in-tree if this
    # checkout has not been built yet (nvcc cross-compiles without a GPU).
    lib = os.path.join(ROOT, "conv2d_implicit_gemm_gb300", "liboidnx.so")
    if not os.path.exists(lib):
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "_oidnx_build", os.path.join(ROOT, "conv2d_implicit_gemm_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
