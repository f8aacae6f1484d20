"""GB300 (sm_103a) mHC sublayer boundary.

The boundary itself is the CUDA library ``lib/libmhc_boundary.so`` behind the
C ABI in ``include/mhc_boundary.h``; ``capi`` binds it with the same names and
``Boundary`` wraps it for PyTorch tensors.  ``synth`` draws seeded synthetic
inputs.  Build the library with ``build.build()``.
"""
import importlib

from . import synth  # noqa: F401

__all__ = ["Boundary", "build", "capi", "synth"]


def __getattr__(name):
    # the binding loads the CUDA library: import it only when asked for
    if name == "Boundary":
        return importlib.import_module(".boundary", __name__).Boundary
    if name in ("capi", "build", "boundary"):
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
