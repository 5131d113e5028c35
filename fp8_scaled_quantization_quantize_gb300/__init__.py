"""fp8q: FP8 scaled quantization and scaled GEMM for GB300 (sm_103a).

The compute lives in libfp8q.so (C ABI in include/fp8q.h, CUDA kernels in
csrc/); ``api`` is its thin PyTorch binding and ``inputs`` draws the seeded
synthetic workloads.  Importing the package does not load the library; the
first call through ``api`` does, and raises if it has not been built.
"""
from . import inputs  # noqa: F401

__all__ = ["api", "inputs", "build"]


def __getattr__(name):
    if name == "api":
        import importlib
        return importlib.import_module(__name__ + ".api")
    raise AttributeError(name)
