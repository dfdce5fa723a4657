"""GB300 (sm_103a) sparse-decode attention: Hamming SCORE -> TOPK -> GATHER-ATT.

The compute lives in the CUDA library ``libhashattn.so`` (C ABI in
``include/hashattn.h``); ``hashattn`` is its ctypes binding, ``workloads`` the
seeded synthetic inputs. Importing the package does not load the library; the
first call into ``hashattn`` does, and raises if it has not been built.
"""

from . import workloads  # noqa: F401

__all__ = ["hashattn", "workloads", "build"]


def build(force: bool = False, verbose: bool = False) -> str:
    from ._build import build as _b
    return _b(force=force, verbose=verbose)
