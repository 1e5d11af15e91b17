"""Megatron-LM intra-layer tensor-parallel MLP block on one GB300 (sm_103a).

The compute path is libtpmlp.so (hand-written tcgen05/TMA CUDA kernels behind
a C ABI, see include/tp_mlp.h); ``binding`` is its ctypes binding with the
same names and ``mlp.TensorParallelMLP`` a thin object wrapper.  Submodules
load lazily, so importing the package (e.g. for ``workloads``) does not load
the shared library.
"""
import importlib

__all__ = ["binding", "build", "mlp", "workloads", "TensorParallelMLP"]


def __getattr__(name):
    if name in ("binding", "build", "mlp", "workloads"):
        return importlib.import_module(f".{name}", __name__)
    if name == "TensorParallelMLP":
        return importlib.import_module(".mlp", __name__).TensorParallelMLP
    raise AttributeError(name)
