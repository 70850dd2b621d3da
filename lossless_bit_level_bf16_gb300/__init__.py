"""Lossless bit-level codecs for ML tensors on GB300 (sm_103a).

Two codecs behind one C-ABI library (``include/zc.h``):

* ZipCCL-style exponent coding of bf16 buffers (``zc_plan``, ``zc_compress``,
  ``zc_decompress``);
* IBP invariant bit packing (``ibp_build_meta``, ``ibp_compress``,
  ``ibp_decompress``).

The Python layer only marshals arguments; every step runs in the CUDA kernels
of ``liblbb16.so``.  Importing this package does not load the library; the
first call does, and raises if the library has not been built.
"""
from . import workloads  # noqa: F401  (seeded inputs; no codec arithmetic)

__all__ = ["workloads"]


def __getattr__(name):
    if name in ("zipccl", "ibp", "abi"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
