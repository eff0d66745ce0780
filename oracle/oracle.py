"""ctypes front end of the CPU oracle (``mpm_oracle.c``).

TEST INFRASTRUCTURE: imported only by the test suite, ``__graft_entry__`` (its
smoke check and its build step) and ``bench.py``'s CPU-baseline leg.  It shares
no code with the CUDA library and never loads it.
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mpm_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libmpm_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
          "-std=gnu11", "-Wall", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (contraction off) into ``oracle/_build``."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        tmp = _OUT + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _OUT)
    return _OUT


class Desc(ct.Structure):
    _fields_ = [("dim", ct.c_int32), ("n", ct.c_int32 * 3), ("dx", ct.c_float),
                ("inv_dx", ct.c_float), ("order", ct.c_int32), ("acc_mode", ct.c_int32),
                ("scale_log2", ct.c_int32), ("tile", ct.c_int32), ("boundary_nodes", ct.c_int32)]


def desc_from(grid: dict) -> Desc:
    d = Desc()
    d.dim = grid["dim"]
    for i in range(3):
        d.n[i] = grid["n"][i] if i < len(grid["n"]) else 1
    d.dx = grid["dx"]
    d.inv_dx = grid["inv_dx"]
    d.order = grid["order"]
    d.acc_mode = grid["acc_mode"]
    d.scale_log2 = grid["scale_log2"]
    d.tile = grid["tile"]
    d.boundary_nodes = grid["boundary_nodes"]
    return d


_P = ct.c_void_p
_PP = ct.POINTER(ct.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ct.CDLL(build())
            L.orc_nodes.argtypes = [ct.POINTER(Desc)]
            L.orc_nodes.restype = ct.c_int64
            L.orc_num_tiles.argtypes = [ct.POINTER(Desc)]
            L.orc_num_tiles.restype = ct.c_int64
            L.orc_quadratic_weights.argtypes = [ct.c_float, _P]
            L.orc_quadratic_weights.restype = None
            L.orc_quadratic_weights_many.argtypes = [ct.c_int64, _P, _P]
            L.orc_quadratic_weights_many.restype = None
            L.orc_bin.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _P, _P, _P]
            L.orc_bin.restype = ct.c_int64
            L.orc_p2g_fixed.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _PP, _PP, _P, _P, _P]
            L.orc_p2g_fixed.restype = ct.c_uint32
            L.orc_scatter_range.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _PP, _PP, _P, _P, _P]
            L.orc_scatter_range.restype = ct.c_float
            L.orc_max_cover.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP]
            L.orc_max_cover.restype = ct.c_int64
            L.orc_bound_ok.argtypes = [ct.POINTER(Desc), ct.c_float, ct.c_int64]
            L.orc_bound_ok.restype = ct.c_int
            L.orc_p2g_float.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _PP, _PP, _P, _P, _P]
            L.orc_p2g_float.restype = ct.c_uint32
            L.orc_grid_update_fixed.argtypes = [ct.POINTER(Desc), _P, _P, _P]
            L.orc_grid_update_fixed.restype = None
            L.orc_grid_update_float.argtypes = [ct.POINTER(Desc), _P, _P, _P]
            L.orc_grid_update_float.restype = None
            L.orc_g2p.argtypes = [ct.POINTER(Desc), _P, ct.c_int64, _PP, _PP, _PP, ct.c_float]
            L.orc_g2p.restype = ct.c_int64
            L.orc_p2g_fixed_vol.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _PP, _PP, _P, _P, _P, _P]
            L.orc_p2g_fixed_vol.restype = ct.c_uint32
            L.orc_p2g_float_vol.argtypes = [ct.POINTER(Desc), ct.c_int64, _PP, _PP, _PP, _P, _P, _P, _P]
            L.orc_p2g_float_vol.restype = ct.c_uint32
            L.orc_grid_volume_fixed.argtypes = [ct.POINTER(Desc), _P, _P]
            L.orc_grid_volume_fixed.restype = None
            L.orc_grid_volume_float.argtypes = [ct.POINTER(Desc), _P, _P]
            L.orc_grid_volume_float.restype = None
            L.orc_g2p_volume.argtypes = [ct.POINTER(Desc), _P, ct.c_int64, _PP, _P]
            L.orc_g2p_volume.restype = ct.c_int64
            L.orc_g2p_elastic.argtypes = [ct.POINTER(Desc), _P, ct.c_int64, _PP, _PP, _PP, _PP, ct.c_float]
            L.orc_g2p_elastic.restype = ct.c_int64
            L.orc_log.argtypes = [ct.c_float]
            L.orc_log.restype = ct.c_float
            L.orc_kirchhoff.argtypes = [ct.c_int, ct.c_float, ct.c_float, _P, _P]
            L.orc_kirchhoff.restype = ct.c_int
            L.orc_stress_affine.argtypes = [ct.POINTER(Desc), ct.c_float, ct.c_float, ct.c_float, ct.c_int64,
                                            _PP, _PP, _PP, _P, _P, _PP]
            L.orc_stress_affine.restype = ct.c_int64
            L.orc_advective_speed.argtypes = [ct.c_int, ct.c_float, ct.c_int64, _PP, _PP]
            L.orc_advective_speed.restype = ct.c_float
            L.orc_rdiv.argtypes = [ct.c_int64, ct.c_int64]
            L.orc_rdiv.restype = ct.c_int64
            L.orc_cic_int_bound.argtypes = [ct.c_int, _P, ct.c_int64, _PP, _P, _PP]
            L.orc_cic_int_bound.restype = ct.c_int
            L.orc_cic_int_p2g.argtypes = [ct.c_int, _P, ct.c_int64, _PP, _P, _PP, _P, _P]
            L.orc_cic_int_p2g.restype = ct.c_int
            L.orc_cic_int_gather.argtypes = [ct.c_int, _P, ct.c_int64, _PP, _P, _PP]
            L.orc_cic_int_gather.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return ct.c_void_p(a.ctypes.data)


def _rows(a: np.ndarray):
    """Pointer array to the rows of a C-contiguous 2-D array (keeps ``a`` alive via caller)."""
    arr = (ct.c_void_p * a.shape[0])()
    for i in range(a.shape[0]):
        arr[i] = a[i].ctypes.data
    return arr


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def grid_nodes(grid: dict) -> int:
    return int(lib().orc_nodes(ct.byref(desc_from(grid))))


def num_tiles(grid: dict) -> int:
    return int(lib().orc_num_tiles(ct.byref(desc_from(grid))))


def quadratic_weights(f: float) -> np.ndarray:
    w = np.zeros(3, dtype=np.float32)
    lib().orc_quadratic_weights(ct.c_float(f), _ptr(w))
    return w


def quadratic_weights_many(f: np.ndarray) -> np.ndarray:
    f = _f32(f)
    w = np.zeros((f.shape[0], 3), dtype=np.float32)
    lib().orc_quadratic_weights_many(f.shape[0], _ptr(f), _ptr(w))
    return w


def bin_particles(grid: dict, x: np.ndarray):
    """Returns (key u32 [n], perm u32 [n], tile_count u32 [ntiles], n_valid)."""
    x = _f32(x)
    n = x.shape[1]
    d = desc_from(grid)
    key = np.zeros(n, dtype=np.uint32)
    perm = np.zeros(n, dtype=np.uint32)
    cnt = np.zeros(num_tiles(grid), dtype=np.uint32)
    valid = lib().orc_bin(ct.byref(d), n, _rows(x), _ptr(key), _ptr(perm), _ptr(cnt))
    return key, perm, cnt, int(valid)


def scatter_range(grid: dict, x, v, C, m, vol=None):
    """(R, in-domain count): R = max over the in-domain particles of the range R_p the
    bound is taken on (``mpm_oracle.c``, fixed-point P2G); NaN if any R_p is NaN."""
    x, v, C, m = _f32(x), _f32(v), _f32(C), _f32(m)
    d = desc_from(grid)
    valid = ct.c_int64(0)
    volp = None if vol is None else _ptr(_f32(vol))
    R = lib().orc_scatter_range(ct.byref(d), x.shape[1], _rows(x), _rows(v), _rows(C), _ptr(m), volp,
                                ct.byref(valid))
    return float(np.float32(R)), int(valid.value)


def max_cover(grid: dict, x) -> int:
    """The most in-domain particles whose stencil covers one node."""
    x = _f32(x)
    return int(lib().orc_max_cover(ct.byref(desc_from(grid)), x.shape[1], _rows(x)))


def bound_ok(grid: dict, R: float, count: int) -> bool:
    """The accumulator bound of the grid's mode for ``count`` particles of range R."""
    return bool(lib().orc_bound_ok(ct.byref(desc_from(grid)), float(R), int(count)))


def p2g_fixed(grid: dict, x, v, C, m, vol=None):
    """Fixed-point P2G: returns (acc int64 [(dim+1), nodes], status bits, counts[2]);
    with rest volumes ``vol`` the volume channel is a last plane (dim+2 planes).
    counts = (out-of-domain particles, in-domain particles left unscattered because
    the bound failed: all of them or none)."""
    x, v, C, m = _f32(x), _f32(v), _f32(C), _f32(m)
    d = desc_from(grid)
    nodes = grid_nodes(grid)
    acc = np.zeros((grid["dim"] + (1 if vol is None else 2), nodes), dtype=np.int64)
    counts = np.zeros(2, dtype=np.int64)
    if vol is None:
        st = lib().orc_p2g_fixed(ct.byref(d), x.shape[1], _rows(x), _rows(v), _rows(C), _ptr(m),
                                 _ptr(acc), _ptr(counts))
    else:
        vol = _f32(vol)
        st = lib().orc_p2g_fixed_vol(ct.byref(d), x.shape[1], _rows(x), _rows(v), _rows(C), _ptr(m), _ptr(vol),
                                     _ptr(acc), _ptr(counts))
    return acc, int(st), counts


def p2g_float(grid: dict, x, v, C, m, vol=None):
    """Float-atomic P2G with fp64 sums: returns (acc float64 [(dim+1), nodes], status, counts);
    with ``vol`` the volume channel is a last plane."""
    x, v, C, m = _f32(x), _f32(v), _f32(C), _f32(m)
    d = desc_from(grid)
    nodes = grid_nodes(grid)
    acc = np.zeros((grid["dim"] + (1 if vol is None else 2), nodes), dtype=np.float64)
    counts = np.zeros(2, dtype=np.int64)
    if vol is None:
        st = lib().orc_p2g_float(ct.byref(d), x.shape[1], _rows(x), _rows(v), _rows(C), _ptr(m),
                                 _ptr(acc), _ptr(counts))
    else:
        vol = _f32(vol)
        st = lib().orc_p2g_float_vol(ct.byref(d), x.shape[1], _rows(x), _rows(v), _rows(C), _ptr(m), _ptr(vol),
                                     _ptr(acc), _ptr(counts))
    return acc, int(st), counts


def grid_volume(grid: dict, plane) -> np.ndarray:
    """Node volume fractions from the volume channel (int64: fixed point, float64: float mode)."""
    phi = np.zeros(grid_nodes(grid), dtype=np.float32)
    if np.asarray(plane).dtype == np.int64:
        lib().orc_grid_volume_fixed(ct.byref(desc_from(grid)), _ptr(np.ascontiguousarray(plane)), _ptr(phi))
    else:
        plane = np.ascontiguousarray(plane, dtype=np.float64)
        lib().orc_grid_volume_float(ct.byref(desc_from(grid)), _ptr(plane), _ptr(phi))
    return phi


def g2p_volume(grid: dict, phi: np.ndarray, x, out=None):
    """Grid-recovered volume fraction of each in-domain particle (others keep ``out``'s values, 0 by default)."""
    phi, x = _f32(phi), _f32(x)
    res = np.zeros(x.shape[1], dtype=np.float32) if out is None else _f32(out).copy()
    lib().orc_g2p_volume(ct.byref(desc_from(grid)), _ptr(phi), x.shape[1], _rows(x), _ptr(res))
    return res


def dtg_of(grid: dict) -> np.ndarray:
    """dt * g, each product rounded to fp32 (the grid update adds this vector)."""
    dt = np.float32(grid["dt"])
    return np.array([dt * np.float32(c) for c in (list(grid["g"]) + [0.0] * 3)[:3]], dtype=np.float32)


def grid_update_fixed(grid: dict, acc: np.ndarray) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    vel = np.zeros((grid["dim"], grid_nodes(grid)), dtype=np.float32)
    dtg = dtg_of(grid)
    lib().orc_grid_update_fixed(ct.byref(desc_from(grid)), _ptr(acc), _ptr(dtg), _ptr(vel))
    return vel


def grid_update_float(grid: dict, acc: np.ndarray) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    vel = np.zeros((grid["dim"], grid_nodes(grid)), dtype=np.float32)
    dtg = dtg_of(grid)
    lib().orc_grid_update_float(ct.byref(desc_from(grid)), _ptr(acc), _ptr(dtg), _ptr(vel))
    return vel


def g2p(grid: dict, vel: np.ndarray, x, v=None, C=None):
    """G2P: returns (x', v', C', moved) as new fp32 arrays.  Particles outside
    the domain keep their inputs (zeros where ``v``/``C`` are not given)."""
    vel = _f32(vel)
    x = _f32(x).copy()
    dim = grid["dim"]
    n = x.shape[1]
    v = _f32(v).copy() if v is not None else np.zeros((dim, n), dtype=np.float32)
    C = _f32(C).copy() if C is not None else np.zeros((dim * dim, n), dtype=np.float32)
    moved = lib().orc_g2p(ct.byref(desc_from(grid)), _ptr(vel), n, _rows(x), _rows(v), _rows(C),
                          ct.c_float(grid["dt"]))
    return x, v, C, int(moved)


def g2p_elastic(grid: dict, vel: np.ndarray, x, v, C, F):
    """G2P that also advances the deformation gradient, F' = (I + dt C') F:
    returns (x', v', C', F', moved)."""
    vel = _f32(vel)
    x, v, C, F = (_f32(a).copy() for a in (x, v, C, F))
    moved = lib().orc_g2p_elastic(ct.byref(desc_from(grid)), _ptr(vel), x.shape[1], _rows(x), _rows(v), _rows(C),
                                  _rows(F), ct.c_float(grid["dt"]))
    return x, v, C, F, int(moved)


def log(J: float) -> float:
    """The fp32 natural logarithm both sides use for the Neo-Hookean ln J."""
    return float(lib().orc_log(ct.c_float(J)))


def kirchhoff(dim: int, mu: float, lam: float, F) -> tuple:
    """Neo-Hookean Kirchhoff stress tau = P F^T (dim x dim, fp32); (tau, ok)."""
    F = _f32(np.asarray(F).reshape(dim * dim))
    tau = np.zeros(dim * dim, dtype=np.float32)
    ok = lib().orc_kirchhoff(dim, ct.c_float(mu), ct.c_float(lam), _ptr(F), _ptr(tau))
    return tau.reshape(dim, dim), bool(ok)


def stress_affine(grid: dict, material: dict, x, C, F, vol, m):
    """The MLS fold C' = C - kappa tau: returns (C' fp32 [dim*dim, n], degenerate in-domain count)."""
    x, C, F, vol, m = _f32(x), _f32(C), _f32(F), _f32(vol), _f32(m)
    out = np.zeros_like(C)
    bad = lib().orc_stress_affine(ct.byref(desc_from(grid)), ct.c_float(grid["dt"]), ct.c_float(material["mu"]),
                                  ct.c_float(material["lambda"]), x.shape[1], _rows(x), _rows(C), _rows(F),
                                  _ptr(vol), _ptr(m), _rows(out))
    return out, int(bad)


def advective_speed(dim: int, dx: float, v, C) -> float:
    """max_p |v_p| + 1.5 dx |C_p|_F in fp32 (the advective step bound is dt <= dx / this)."""
    v, C = _f32(v), _f32(C)
    return float(lib().orc_advective_speed(dim, ct.c_float(dx), v.shape[1], _rows(v), _rows(C)))


def rdiv(a: int, b: int) -> int:
    return int(lib().orc_rdiv(a, b))


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def cic_int_bound(grid: dict, X, m, v) -> bool:
    X, m, v = _i32(X), _i64(m), _i64(v)
    n = np.array(grid["n"][:3], dtype=np.int32)
    return bool(lib().orc_cic_int_bound(grid["dim"], _ptr(n), X.shape[1], _rows(X), _ptr(m), _rows(v)))


def cic_int_p2g(grid: dict, X, m, v, order=None):
    """Integer CIC scatter in the given particle order; returns (acc, ok)."""
    X, m, v = _i32(X), _i64(m), _i64(v)
    dim = grid["dim"]
    n = np.array(grid["n"][:3], dtype=np.int32)
    nodes = int(np.prod(n[:dim]))
    acc = np.zeros((dim + 1, nodes), dtype=np.int64)
    o = _i64(order) if order is not None else None
    ok = lib().orc_cic_int_p2g(dim, _ptr(n), X.shape[1], _rows(X), _ptr(m), _rows(v),
                               _ptr(o) if o is not None else None, _ptr(acc))
    return acc, bool(ok)


def cic_int_gather(grid: dict, X, acc):
    X, acc = _i32(X), _i64(acc)
    dim = grid["dim"]
    n = np.array(grid["n"][:3], dtype=np.int32)
    out = np.zeros((dim, X.shape[1]), dtype=np.int64)
    lib().orc_cic_int_gather(dim, _ptr(n), X.shape[1], _rows(X), _ptr(acc), _rows(out))
    return out


def step_elastic(grid: dict, material: dict, x, v, C, m, F, vol):
    """One oracle step with the elastic stress: bin, fold, P2G, grid update, G2P with the F update."""
    key, perm, cnt, valid = bin_particles(grid, x)
    Cs, degenerate = stress_affine(grid, material, x, C, F, vol, m)
    if grid["acc_mode"] == 2:
        acc, st, counts = p2g_float(grid, x, v, Cs, m)
        vel = grid_update_float(grid, acc)
    else:
        acc, st, counts = p2g_fixed(grid, x, v, Cs, m)
        vel = grid_update_fixed(grid, acc)
    x2, v2, C2, F2, moved = g2p_elastic(grid, vel, x, v, C, F)
    return dict(key=key, perm=perm, tile_count=cnt, n_valid=valid, acc=acc, status=st, counts=counts,
                degenerate=degenerate, vel=vel, x=x2, v=v2, C=C2, F=F2)


def step_fixed(grid: dict, x, v, C, m):
    """One full oracle step in a fixed-point mode: bin, P2G, grid update, G2P."""
    key, perm, cnt, valid = bin_particles(grid, x)
    acc, st, counts = p2g_fixed(grid, x, v, C, m)
    vel = grid_update_fixed(grid, acc)
    x2, v2, C2, moved = g2p(grid, vel, x, v, C)
    return dict(key=key, perm=perm, tile_count=cnt, n_valid=valid, acc=acc, status=st,
                counts=counts, vel=vel, x=x2, v=v2, C=C2)
