"""EntropyCache decode-and-gate and selective-recompute attention on B300 (sm_103a).

The compute path is ``libec.so`` (hand-written CUDA kernels behind the C ABI in
``include/ec.h``); ``_native`` is its ctypes binding.  ``synth`` builds the
seeded synthetic inputs.  Importing the package does not load the library; the
first binding call does, and fails loudly if it has not been built.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "native"]


def native():
    """The binding module (imports torch and loads ``libec.so`` on first call)."""
    from . import _native
    _native.lib()
    return _native
