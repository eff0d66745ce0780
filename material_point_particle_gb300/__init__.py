"""GB300-native Material Point Method particle/grid transfer.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/mpm.h``): cell-key binning, fixed-point P2G scatter, grid update and
G2P gather.  ``_lib`` binds it with ctypes under the same function names;
``system.MPMSystem`` holds device tensors for one grid; ``workloads`` draws
seeded synthetic particle sets.
"""
from . import workloads  # noqa: F401  (numpy only)

__all__ = ["workloads", "library", "MPMSystem"]


def library():
    """The loaded CUDA library (built in-tree on first use)."""
    from . import _lib
    return _lib.library()


def __getattr__(name):
    if name == "MPMSystem":
        from .system import MPMSystem
        return MPMSystem
    raise AttributeError(name)
