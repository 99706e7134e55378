"""GB300-native token-level hot path of speculative decoding.

The compute path is the C-ABI library ``libspecmarkov.so`` (hand-written sm_103a CUDA kernels);
``spec`` is its thin ctypes binding. ``workloads`` draws the seeded synthetic inputs.
Importing the package does not load the library; the first call into ``spec`` does, and it
raises if the library has not been built.
"""
__all__ = ["spec", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
