"""ctypes binding of the C ABI in ``include/mpm.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: particles, grids and workspaces are torch tensors
whose device pointers are handed to the library.  The CUDA library must be
present (it is built in-tree by ``build.py``); there is no fallback.
"""
from __future__ import annotations

import ctypes as ct
import threading

import torch

from . import build as _build

MPM_OK, MPM_E_ARG, MPM_E_WORKSPACE, MPM_E_DOMAIN, MPM_E_BOUND, MPM_E_CUDA, MPM_E_TIMEOUT, MPM_E_NO_DEVICE = range(8)
MPM_ACC_I32, MPM_ACC_I64, MPM_ACC_F32, MPM_ACC_EXACT_INT = range(4)
(ST_FLAGS, ST_N_OUTSIDE, ST_N_OUT_OF_RANGE, ST_N_VALID, ST_N_SLICES, ST_N_ACTIVE, ST_MAX_NEIGHBOURS,
 ST_N_BIG_TILES, ST_N_RUNS, ST_N_LARGE_BUCKETS) = range(10)
ST_BIN_WORDS = 10   # status words 0..9 are written by mpm_bin
ST_N_DEGENERATE = 10  # elastic particles the last P2G scattered without stress (det F not positive normal)
ST_MAX_SPEED = 13   # fp32 bits of max |v'| + 1.5 dx |C'|_F over the particles the last G2P moved
ST_N_ESCAPED = 14   # mpm_step_fused: particles whose base cell left their tile (scattered into the global grid)
ST_RANGE = 15       # fp32 bits of R, the range the last fixed-point P2G checked its bound with
ST_SHARE_PATH = 16  # the last fixed-point P2G's shares: 0 below 2^22 (one fma each), 1 int64
MPM_BIN_KEYS_FROM_G2P = 1  # mpm_bin flag: the keys and histogram the last mpm_g2p_update wrote
ST_P2G_MASS = 20    # record: fp32 bits of max |m| over the particles the last P2G scattered
ST_P2G_VOLUME = 21  # record: fp32 bits of max rest volume in cells over the same
ST_G2P_RANGE = 22   # record: fp32 bits of max over the last G2P's particles of max(1, |v'_k| + 1.5 dx sum|C'_kl|)
MPM_STATUS_WORDS = 24
MPM_STATIC_WORKSPACE_BYTES = 16 << 20


class MPMError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} ({code})")
        self.code = code


class GridDesc(ct.Structure):
    _fields_ = [("dim", ct.c_int32), ("n", ct.c_int32 * 3), ("dx", ct.c_float), ("inv_dx", ct.c_float),
                ("order", ct.c_int32), ("acc_mode", ct.c_int32), ("scale_log2", ct.c_int32),
                ("tile", ct.c_int32), ("boundary_nodes", ct.c_int32), ("volume_channel", ct.c_int32)]


class Particles(ct.Structure):
    _fields_ = [("n", ct.c_int64), ("x", ct.c_void_p * 3), ("v", ct.c_void_p * 3), ("C", ct.c_void_p * 9),
                ("m", ct.c_void_p), ("id", ct.c_void_p), ("F", ct.c_void_p * 9), ("vol", ct.c_void_p),
                ("mu", ct.c_float), ("lambda_", ct.c_float), ("phi", ct.c_void_p)]


class Bins(ct.Structure):
    _fields_ = [("n", ct.c_int64), ("ntiles", ct.c_int64), ("max_slices", ct.c_int64),
                ("key", ct.c_void_p), ("perm", ct.c_void_p), ("tile_count", ct.c_void_p),
                ("tile_start", ct.c_void_p), ("slices", ct.c_void_p), ("active", ct.c_void_p),
                ("status", ct.c_void_p), ("scratch", ct.c_void_p), ("scratch_bytes", ct.c_size_t),
                ("range_from_g2p", ct.c_int32),
                ("next_keys", ct.c_int32)]


_lock = threading.Lock()
_L = None


def library() -> ct.CDLL:
    """Loads (building first if needed) the in-tree CUDA library."""
    global _L
    with _lock:
        if _L is None:
            path = _build.build()
            L = ct.CDLL(path)
            P, VP = ct.POINTER, ct.c_void_p
            L.mpm_version.restype = ct.c_int32
            L.mpm_strerror.argtypes = [ct.c_int]
            L.mpm_strerror.restype = ct.c_char_p
            L.mpm_workspace_bytes.argtypes = [P(GridDesc), ct.c_int64]
            L.mpm_workspace_bytes.restype = ct.c_size_t
            L.mpm_bins_init.argtypes = [P(GridDesc), ct.c_int64, VP, ct.c_size_t, P(Bins)]
            L.mpm_grid_acc_bytes.argtypes = [P(GridDesc)]
            L.mpm_grid_acc_bytes.restype = ct.c_size_t
            L.mpm_grid_vel_bytes.argtypes = [P(GridDesc)]
            L.mpm_grid_vel_bytes.restype = ct.c_size_t
            L.mpm_bin.argtypes = [P(GridDesc), P(Particles), P(Bins), ct.c_int, VP]
            L.mpm_p2g.argtypes = [P(GridDesc), P(Particles), P(Bins), VP, ct.c_float, VP]
            L.mpm_grid_update.argtypes = [P(GridDesc), VP, VP, P(ct.c_float), P(Bins), VP]
            L.mpm_g2p.argtypes = [P(GridDesc), VP, P(Particles), P(Bins), ct.c_float, VP]
            L.mpm_step.argtypes = [P(GridDesc), P(Particles), P(Bins), VP, VP, ct.c_float, P(ct.c_float), VP]
            L.mpm_g2p_sorted.argtypes = [P(GridDesc), VP, P(Particles), P(Particles), P(Bins), ct.c_float, VP]
            L.mpm_step_sorted.argtypes = [P(GridDesc), P(Particles), P(Particles), P(Bins), VP, VP, ct.c_float,
                                          P(ct.c_float), VP]
            L.mpm_step_host.argtypes = [P(GridDesc), P(Particles), P(Particles), P(Particles), P(Bins), VP, VP,
                                        ct.c_float, P(ct.c_float), VP]
            L.mpm_step_fused.argtypes = [P(GridDesc), P(Particles), P(Particles), P(Bins), VP, VP, ct.c_float,
                                         P(ct.c_float), VP]
            L.mpm_iterate.argtypes = [P(GridDesc), P(Particles), P(Bins), VP, VP, ct.c_int, VP]
            L.mpm_g2p_binned.argtypes = [P(GridDesc), VP, P(Particles), P(Particles), P(Bins), ct.c_float, VP]
            L.mpm_step_binned.argtypes = [P(GridDesc), P(Particles), P(Particles), P(Bins), VP, VP, ct.c_float,
                                          P(ct.c_float), VP]
            L.mpm_g2p_update.argtypes = [P(GridDesc), VP, P(ct.c_float), P(Particles), P(Bins), ct.c_float, VP]
            L.mpm_g2p_sorted_update.argtypes = [P(GridDesc), VP, P(ct.c_float), P(Particles), P(Particles), P(Bins),
                                                ct.c_float, VP]
            L.mpm_permute.argtypes = [P(GridDesc), P(Particles), P(Particles), P(Bins), VP]
            L.mpm_read_status.argtypes = [P(Bins), VP, VP]
            L.mpm_bin_static.argtypes = [P(GridDesc), P(Particles), ct.c_int, P(Bins), VP]
            for name in ("mpm_bins_init", "mpm_bin", "mpm_p2g", "mpm_grid_update", "mpm_g2p", "mpm_step",
                         "mpm_g2p_sorted", "mpm_step_sorted", "mpm_step_host", "mpm_permute", "mpm_read_status",
                         "mpm_bin_static", "mpm_step_fused", "mpm_iterate", "mpm_g2p_binned", "mpm_step_binned",
                         "mpm_g2p_update", "mpm_g2p_sorted_update"):
                getattr(L, name).restype = ct.c_int
            _L = L
    return _L


def strerror(code: int) -> str:
    return library().mpm_strerror(code).decode()


def _check(code: int, where: str):
    if code != MPM_OK:
        raise MPMError(code, where)


def _stream(stream) -> ct.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ct.c_void_p(stream.cuda_stream)


def grid_desc(grid: dict) -> GridDesc:
    d = GridDesc()
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
    d.volume_channel = int(grid.get("volume_channel", 0))
    return d


def particles(x: torch.Tensor, v: torch.Tensor, C: torch.Tensor | None, m: torch.Tensor,
              id: torch.Tensor | None = None, F: torch.Tensor | None = None, vol: torch.Tensor | None = None,
              mu: float = 0.0, lam: float = 0.0, phi: torch.Tensor | None = None) -> Particles:
    """SoA view of [dim, n] / [dim*dim, n] / [n] tensors (rows must be contiguous),
    with optional uint32-sized [n] particle ids, an optional elastic state
    (F [dim*dim, n], Lame constants mu and lam), rest volumes vol [n] and the
    volume-channel output phi [n]."""
    p = Particles()
    if F is not None:
        assert F.is_contiguous()
        for i in range(F.shape[0]):
            p.F[i] = F[i].data_ptr()
        p.mu = mu
        p.lambda_ = lam
    if vol is not None:
        assert vol.is_contiguous()
        p.vol = vol.data_ptr()
    if phi is not None:
        assert phi.is_contiguous()
        p.phi = phi.data_ptr()
    if id is not None:
        assert id.is_contiguous() and id.element_size() == 4
        p.id = id.data_ptr()
    p.n = int(x.shape[1])
    for rows, field in ((x, p.x), (v, p.v), (C, p.C)):
        if rows is None:
            continue
        assert rows.is_contiguous()
        for i in range(rows.shape[0]):
            field[i] = rows[i].data_ptr()
    assert m.is_contiguous()
    p.m = m.data_ptr()
    return p


def mpm_version() -> int:
    return int(library().mpm_version())


def mpm_strerror(code: int) -> str:
    return strerror(code)


def mpm_workspace_bytes(desc: GridDesc, n: int) -> int:
    return int(library().mpm_workspace_bytes(ct.byref(desc), n))


def mpm_grid_acc_bytes(desc: GridDesc) -> int:
    return int(library().mpm_grid_acc_bytes(ct.byref(desc)))


def mpm_grid_vel_bytes(desc: GridDesc) -> int:
    return int(library().mpm_grid_vel_bytes(ct.byref(desc)))


def mpm_bins_init(desc: GridDesc, n: int, ws: torch.Tensor) -> Bins:
    b = Bins()
    _check(library().mpm_bins_init(ct.byref(desc), n, ct.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                   ct.byref(b)), "mpm_bins_init")
    return b


def mpm_bin(desc: GridDesc, parts: Particles, bins: Bins, flags: int = 0, stream=None):
    _check(library().mpm_bin(ct.byref(desc), ct.byref(parts), ct.byref(bins), flags, _stream(stream)), "mpm_bin")


def mpm_p2g(desc: GridDesc, parts: Particles, bins: Bins, grid_acc: torch.Tensor, dt: float = 0.0, stream=None):
    _check(library().mpm_p2g(ct.byref(desc), ct.byref(parts), ct.byref(bins), ct.c_void_p(grid_acc.data_ptr()),
                             ct.c_float(dt), _stream(stream)), "mpm_p2g")


def _f3(vals) -> ct.Array:
    arr = (ct.c_float * 3)()
    for i, v in enumerate(list(vals)[:3]):
        arr[i] = float(v)
    return arr


def mpm_grid_update(desc: GridDesc, grid_acc: torch.Tensor, grid_vel: torch.Tensor, dtg, bins: Bins, stream=None):
    _check(library().mpm_grid_update(ct.byref(desc), ct.c_void_p(grid_acc.data_ptr()),
                                     ct.c_void_p(grid_vel.data_ptr()), _f3(dtg), ct.byref(bins), _stream(stream)),
           "mpm_grid_update")


def mpm_g2p(desc: GridDesc, grid: torch.Tensor, parts: Particles, bins: Bins | None, dt: float, stream=None):
    _check(library().mpm_g2p(ct.byref(desc), ct.c_void_p(grid.data_ptr()), ct.byref(parts),
                             ct.byref(bins) if bins is not None else None, ct.c_float(dt), _stream(stream)),
           "mpm_g2p")


def mpm_step(desc: GridDesc, parts: Particles, bins: Bins, grid_acc: torch.Tensor, grid_vel: torch.Tensor,
             dt: float, dtg, stream=None):
    _check(library().mpm_step(ct.byref(desc), ct.byref(parts), ct.byref(bins), ct.c_void_p(grid_acc.data_ptr()),
                              ct.c_void_p(grid_vel.data_ptr()), ct.c_float(dt), _f3(dtg), _stream(stream)),
           "mpm_step")


def mpm_g2p_sorted(desc: GridDesc, grid_vel: torch.Tensor, src: Particles, dst: Particles, bins: Bins, dt: float,
                   stream=None):
    _check(library().mpm_g2p_sorted(ct.byref(desc), ct.c_void_p(grid_vel.data_ptr()), ct.byref(src), ct.byref(dst),
                                    ct.byref(bins), ct.c_float(dt), _stream(stream)), "mpm_g2p_sorted")


def mpm_g2p_update(desc: GridDesc, grid_acc: torch.Tensor, dtg, parts: Particles, bins: Bins, dt: float,
                   stream=None):
    _check(library().mpm_g2p_update(ct.byref(desc), ct.c_void_p(grid_acc.data_ptr()), _f3(dtg), ct.byref(parts),
                                    ct.byref(bins), ct.c_float(dt), _stream(stream)), "mpm_g2p_update")


def mpm_g2p_sorted_update(desc: GridDesc, grid_acc: torch.Tensor, dtg, src: Particles, dst: Particles, bins: Bins,
                          dt: float, stream=None):
    _check(library().mpm_g2p_sorted_update(ct.byref(desc), ct.c_void_p(grid_acc.data_ptr()), _f3(dtg),
                                           ct.byref(src), ct.byref(dst), ct.byref(bins), ct.c_float(dt),
                                           _stream(stream)), "mpm_g2p_sorted_update")


def mpm_step_fused(desc: GridDesc, src: Particles, dst: Particles, bins: Bins, acc_read: torch.Tensor,
                   acc_write: torch.Tensor, dt: float, dtg, stream=None):
    _check(library().mpm_step_fused(ct.byref(desc), ct.byref(src), ct.byref(dst), ct.byref(bins),
                                    ct.c_void_p(acc_read.data_ptr()), ct.c_void_p(acc_write.data_ptr()),
                                    ct.c_float(dt), _f3(dtg), _stream(stream)), "mpm_step_fused")


def mpm_iterate(desc: GridDesc, parts: Particles, bins: Bins, acc_a: torch.Tensor, acc_b: torch.Tensor,
                iterations: int, stream=None):
    _check(library().mpm_iterate(ct.byref(desc), ct.byref(parts), ct.byref(bins), ct.c_void_p(acc_a.data_ptr()),
                                 ct.c_void_p(acc_b.data_ptr()), int(iterations), _stream(stream)), "mpm_iterate")


def mpm_g2p_binned(desc: GridDesc, grid_vel: torch.Tensor, src: Particles, dst: Particles, bins: Bins, dt: float,
                   stream=None):
    _check(library().mpm_g2p_binned(ct.byref(desc), ct.c_void_p(grid_vel.data_ptr()), ct.byref(src), ct.byref(dst),
                                    ct.byref(bins), ct.c_float(dt), _stream(stream)), "mpm_g2p_binned")


def mpm_step_binned(desc: GridDesc, src: Particles, dst: Particles, bins: Bins, grid_acc: torch.Tensor,
                    grid_vel: torch.Tensor, dt: float, dtg, stream=None):
    _check(library().mpm_step_binned(ct.byref(desc), ct.byref(src), ct.byref(dst), ct.byref(bins),
                                     ct.c_void_p(grid_acc.data_ptr()), ct.c_void_p(grid_vel.data_ptr()),
                                     ct.c_float(dt), _f3(dtg), _stream(stream)), "mpm_step_binned")


def mpm_step_sorted(desc: GridDesc, src: Particles, dst: Particles, bins: Bins, grid_acc: torch.Tensor,
                    grid_vel: torch.Tensor, dt: float, dtg, stream=None):
    _check(library().mpm_step_sorted(ct.byref(desc), ct.byref(src), ct.byref(dst), ct.byref(bins),
                                     ct.c_void_p(grid_acc.data_ptr()), ct.c_void_p(grid_vel.data_ptr()),
                                     ct.c_float(dt), _f3(dtg), _stream(stream)), "mpm_step_sorted")


def mpm_step_host(desc: GridDesc, host: Particles, dev_in: Particles, dev_out: Particles, bins: Bins,
                  grid_acc: torch.Tensor, grid_vel: torch.Tensor, dt: float, dtg, stream=None):
    _check(library().mpm_step_host(ct.byref(desc), ct.byref(host), ct.byref(dev_in), ct.byref(dev_out),
                                   ct.byref(bins), ct.c_void_p(grid_acc.data_ptr()), ct.c_void_p(grid_vel.data_ptr()),
                                   ct.c_float(dt), _f3(dtg), _stream(stream)), "mpm_step_host")


def mpm_permute(desc: GridDesc, src: Particles, dst: Particles, bins: Bins, stream=None):
    _check(library().mpm_permute(ct.byref(desc), ct.byref(src), ct.byref(dst), ct.byref(bins), _stream(stream)),
           "mpm_permute")


def mpm_read_status(bins: Bins, out: torch.Tensor, stream=None):
    """Asynchronous copy of the status words into ``out`` (uint32-sized int32 CPU tensor, 16 entries)."""
    assert out.numel() >= MPM_STATUS_WORDS and out.element_size() == 4 and out.device.type == "cpu"
    _check(library().mpm_read_status(ct.byref(bins), ct.c_void_p(out.data_ptr()), _stream(stream)),
           "mpm_read_status")


def mpm_bin_static(desc: GridDesc, parts: Particles, flags: int = 0, stream=None) -> Bins:
    """Bins into the library's own fixed-size device workspace (no allocation
    by anyone) and returns the bins, whose arrays point into that workspace.

    For callers that cannot allocate device memory where they bin.  One such
    workspace exists per device and process: the next call overwrites it, so
    calls (and the steps that read the returned bins) must not overlap; keep
    them on one stream.  The first call on a device sets the workspace up, so
    make it before any stream capture begins.
    """
    b = Bins()
    code = library().mpm_bin_static(ct.byref(desc), ct.byref(parts), flags, ct.byref(b), _stream(stream))
    if code == MPM_E_WORKSPACE:
        need = mpm_workspace_bytes(desc, int(parts.n))
        raise MPMError(code, f"mpm_bin_static: {int(parts.n)} particles need {need} bytes of workspace, the static "
                             f"workspace holds {MPM_STATIC_WORKSPACE_BYTES}; use mpm_bins_init with your own memory")
    _check(code, "mpm_bin_static")
    return b
