"""Tensor-parallel Transformer MLP block for GB300 (sm_103a).

    Z = GeLU(X A + a) B + b,  A split by columns and B by rows into t shards,

all t shards on one GPU, the shard all-reduce done as a fixed-order on-device
sum.  The compute lives in ``libtpmlp.so`` (hand-written CUDA, C ABI declared in
``include/tpmlp.h``); :mod:`.tpmlp` is the thin ctypes binding over it.  The
binding is imported lazily so that :mod:`.inputs` and :mod:`.workloads` can be
used without the compiled library.
"""
__all__ = ["inputs", "workloads", "tpmlp"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
