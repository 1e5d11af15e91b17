"""Megatron-LM intra-layer tensor-parallel MLP block on one GB300 (sm_103a).

The compute path is libtpmlp.so (hand-written tcgen05/TMA CUDA kernels behind
a C ABI, see include/tp_mlp.h and include/tp_attn.h); ``binding`` is its
ctypes binding with the same names, ``mlp.TensorParallelMLP`` and
``attention.TensorParallelAttention`` thin object wrappers.  Submodules
load lazily, so importing the package (e.g. for ``workloads``) does not load
the shared library.
"""
import importlib

__all__ = ["attention", "binding", "build", "mlp", "workloads",
           "TensorParallelAttention", "TensorParallelMLP"]


def __getattr__(name):
    if name in ("attention", "binding", "build", "mlp", "workloads"):
        return importlib.import_module(f".{name}", __name__)
    if name == "TensorParallelMLP":
        return importlib.import_module(".mlp", __name__).TensorParallelMLP
    if name == "TensorParallelAttention":
        return importlib.import_module(".attention",
                                       __name__).TensorParallelAttention
    raise AttributeError(name)
