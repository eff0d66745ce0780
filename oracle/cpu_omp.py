"""ctypes front end of the multi-core CPU baseline (``mpm_cpu_omp.c``).

TEST INFRASTRUCTURE, like the oracle whose source it is built from: imported
only by the test suite and ``bench.py``'s CPU-baseline leg.  One fixed-point
MPM step on all host cores with OpenMP (private per-thread int64 grids merged
by integer add); the new state comes back in bin order.  ``available()`` is
False where the host compiler has no OpenMP.
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

from . import oracle as O

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mpm_cpu_omp.c")
_DEPS = (_SRC, os.path.join(_HERE, "mpm_oracle.c"))
_OUT = os.path.join(_HERE, "_build", "libmpm_cpu_omp.so")
_lock = threading.Lock()
_lib = None
_error = None


def build(force: bool = False) -> str:
    """Compiles the baseline with gcc -fopenmp (contraction off, as the oracle)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    newest = max(os.path.getmtime(p) for p in _DEPS)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < newest:
        tmp = _OUT + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *O.CFLAGS, "-fopenmp", "-I", _HERE, "-o", tmp, _SRC, "-lm"], check=True,
                       capture_output=True)
        os.replace(tmp, _OUT)
    return _OUT


def available() -> bool:
    try:
        lib()
        return True
    except (OSError, subprocess.CalledProcessError) as e:
        global _error
        _error = str(e)
        return False


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ct.CDLL(build())
            L.orc_omp_max_threads.argtypes = []
            L.orc_omp_max_threads.restype = ct.c_int
            L.orc_omp_step_fixed.argtypes = [ct.POINTER(O.Desc), ct.c_float, O._P, ct.c_int64, O._PP, O._PP, O._PP,
                                             O._P, O._PP, O._PP, O._PP, O._P, O._P, O._P, O._P, ct.c_int, O._P]
            L.orc_omp_step_fixed.restype = ct.c_int64
            _lib = L
    return _lib


def max_threads() -> int:
    return int(lib().orc_omp_max_threads())


def phase_seconds() -> dict:
    """Seconds of the last step's phases."""
    arr = (ct.c_double * 6).in_dll(lib(), "orc_omp_phase_seconds")
    return dict(zip(("bin", "permute", "p2g", "merge", "grid_update", "g2p"), (round(float(t), 4) for t in arr)))


def buffers(grid: dict, n: int) -> dict:
    """Arrays for step_fixed's results (the new state, perm) and its grid scratch (acc, vel), to be reused
    from step to step (their pages are mapped once)."""
    dim = grid["dim"]
    nodes = O.grid_nodes(grid)
    return dict(x=np.empty((dim, n), np.float32), v=np.empty((dim, n), np.float32),
                C=np.empty((dim * dim, n), np.float32), m=np.empty(n, np.float32), perm=np.empty(n, np.uint32),
                acc=np.empty((dim + 1, nodes), np.int64), vel=np.empty((dim, nodes), np.float32))


def step_fixed(grid: dict, x, v, C, m, threads: int = 0, out: dict | None = None):
    """One step on `threads` cores (0: all).  Returns perm, acc, vel, counts, moved and the new
    x, v, C, m in bin order (column j is the new state of input particle perm[j]), in `out` (from
    buffers(); it must not hold the inputs) or in new arrays."""
    x, v, C, m = (O._f32(a) for a in (x, v, C, m))
    n = x.shape[1]
    if out is None:
        out = buffers(grid, n)
    counts = np.zeros(2, dtype=np.int64)
    dtg = O.dtg_of(grid)
    moved = lib().orc_omp_step_fixed(ct.byref(O.desc_from(grid)), ct.c_float(grid["dt"]), O._ptr(dtg), n,
                                     O._rows(x), O._rows(v), O._rows(C), O._ptr(m), O._rows(out["x"]),
                                     O._rows(out["v"]), O._rows(out["C"]), O._ptr(out["m"]), O._ptr(out["perm"]),
                                     O._ptr(out["acc"]), O._ptr(out["vel"]), int(threads), O._ptr(counts))
    return dict(out, counts=counts, moved=int(moved))
