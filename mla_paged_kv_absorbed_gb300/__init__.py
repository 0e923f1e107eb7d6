"""GB300-native paged, absorbed MLA decode.

The compute path is the C-ABI library ``libmla.so`` (hand-written sm_103a CUDA,
declared in ``include/mla.h``); ``api`` is its thin ctypes binding over torch
tensors. ``inputs`` draws the seeded synthetic workloads.

Importing the package does not load the CUDA library; the first call into
``api`` does, and raises if it is missing.
"""
__version__ = "0.1.0"


def __getattr__(name):
    if name in ("api", "inputs", "build"):
        import importlib
        return importlib.import_module(f".{'_build' if name == 'build' else name}", __name__)
    from . import api as _api
    if hasattr(_api, name):
        return getattr(_api, name)
    raise AttributeError(name)
