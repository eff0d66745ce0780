"""Device-resident particle set, grid and workspace for one grid descriptor.

A convenience holder over the C ABI (``_lib``): it allocates torch tensors for
the particle SoA, the accumulator and velocity grids and the binning
workspace, and calls the library's entry points on them.  It computes nothing
of the method itself.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L


def dt_times_g(grid: dict) -> list[float]:
    """dt*g per component, each product rounded to fp32 (the grid update adds it)."""
    dt = np.float32(grid["dt"])
    g = (list(grid["g"]) + [0.0, 0.0, 0.0])[:3]
    return [float(dt * np.float32(c)) for c in g]


class MPMSystem:
    def __init__(self, grid: dict, n: int, device: str | torch.device = "cuda"):
        self.grid = dict(grid)
        self.desc = L.grid_desc(grid)
        self.dim = grid["dim"]
        self.n = int(n)
        self.device = torch.device(device)
        dim = self.dim
        ws_bytes = L.mpm_workspace_bytes(self.desc, self.n)
        if ws_bytes == 0:
            raise L.MPMError(L.MPM_E_ARG, "mpm_workspace_bytes")
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        self.bins = L.mpm_bins_init(self.desc, self.n, self.ws)
        acc_bytes = L.mpm_grid_acc_bytes(self.desc)
        self.nodes = int(np.prod(grid["n"][:dim]))
        mode = grid["acc_mode"]
        acc_dtype = {L.MPM_ACC_I32: torch.int32, L.MPM_ACC_I64: torch.int64, L.MPM_ACC_F32: torch.float32,
                     L.MPM_ACC_EXACT_INT: torch.int64}[mode]
        self.vc = int(grid.get("volume_channel", 0))
        self.acc = torch.zeros((dim + 1 + self.vc, self.nodes), dtype=acc_dtype, device=self.device)
        assert self.acc.numel() * self.acc.element_size() == acc_bytes
        self.vel = torch.zeros((dim + self.vc, self.nodes), dtype=torch.float32, device=self.device)
        self.status_host = torch.zeros(L.MPM_STATUS_WORDS, dtype=torch.int32).pin_memory() \
            if torch.cuda.is_available() else torch.zeros(L.MPM_STATUS_WORDS, dtype=torch.int32)
        self.dt = float(grid.get("dt", 0.0))
        self.dtg = dt_times_g(grid) if "g" in grid else [0.0, 0.0, 0.0]
        self.x = self.v = self.C = self.m = None
        self.id = self.id2 = None
        self.F = self.vol = self.F2 = self.vol2 = None
        self.phi = self.phi2 = None
        self.material = {"mu": 0.0, "lambda": 0.0}
        self.parts = self.parts2 = None

    # -- particle state -------------------------------------------------------
    def load(self, x, v, C, m):
        """Copies host arrays ([dim, n], [dim, n], [dim*dim, n], [n]) to the device."""
        mode = self.grid["acc_mode"]
        if mode == L.MPM_ACC_EXACT_INT:
            self.x = torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)).to(self.device)
            self.v = torch.as_tensor(np.ascontiguousarray(v, dtype=np.int64)).to(self.device)
            self.C = None
            self.m = torch.as_tensor(np.ascontiguousarray(m, dtype=np.int64)).to(self.device)
        else:
            f32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(self.device)
            self.x, self.v, self.C, self.m = f32(x), f32(v), f32(C), f32(m)
        assert self.x.shape[1] <= self.n
        self.parts = self._parts(self.x, self.v, self.C, self.m, None, self.F, self.vol, self.phi)
        return self

    def load_volume(self, vol):
        """Rest volumes [n] for the volume channel; phi (the gathered volume fraction) starts at zero."""
        f32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(self.device)
        self.vol = f32(vol)
        self.phi = torch.zeros_like(self.vol)
        self.parts = self._parts(self.x, self.v, self.C, self.m, self.id, self.F, self.vol, self.phi)
        return self

    def load_elastic(self, F, vol, material: dict):
        """Adds the elastic state: deformation gradients F [dim*dim, n], rest
        volumes vol [n] and the Neo-Hookean constants {"mu", "lambda"}."""
        f32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(self.device)
        self.F, self.vol = f32(F), f32(vol)
        if self.vc and self.phi is None:
            self.phi = torch.zeros_like(self.vol)
        self.material = {"mu": float(material["mu"]), "lambda": float(material["lambda"])}
        self.parts = self._parts(self.x, self.v, self.C, self.m, self.id, self.F, self.vol, self.phi)
        return self

    def _parts(self, x, v, C, m, id, F, vol, phi=None):
        return L.particles(x, v, C, m, id, F, vol, self.material["mu"], self.material["lambda"], phi)

    def elastic_state(self):
        """(F, vol) as numpy arrays."""
        torch.cuda.synchronize(self.device)
        return self.F.cpu().numpy(), self.vol.cpu().numpy()

    def state(self):
        """(x, v, C) as numpy arrays."""
        torch.cuda.synchronize(self.device)
        C = self.C.cpu().numpy() if self.C is not None else None
        return self.x.cpu().numpy(), self.v.cpu().numpy(), C

    def use_range_records(self, on: bool = True):
        """With ``on``, mpm_p2g takes its bound's range from the records the last P2G and
        G2P on these bins wrote instead of a pass over v, C and m (see mpm_p2g)."""
        self.bins.range_from_g2p = 1 if on else 0
        return self

    def use_next_keys(self, on: bool = True):
        """With ``on``, mpm_g2p_update (in place, int64) also writes the keys of the particles' new
        positions and their tile histogram, which bin(keys_from_g2p=True) then takes (see mpm_g2p_update)."""
        self.bins.next_keys = 1 if on else 0
        return self

    # -- the library calls ----------------------------------------------------
    def bin(self, stream=None, keys_from_g2p: bool = False):
        L.mpm_bin(self.desc, self.parts, self.bins, L.MPM_BIN_KEYS_FROM_G2P if keys_from_g2p else 0, stream)

    def p2g(self, stream=None):
        L.mpm_p2g(self.desc, self.parts, self.bins, self.acc, self.dt, stream)

    def grid_update(self, stream=None):
        L.mpm_grid_update(self.desc, self.acc, self.vel, self.dtg, self.bins, stream)

    def g2p(self, stream=None):
        grid = self.acc if self.grid["acc_mode"] == L.MPM_ACC_EXACT_INT else self.vel
        L.mpm_g2p(self.desc, grid, self.parts, self.bins, self.dt, stream)

    def g2p_update(self, stream=None):
        """The grid update applied as G2P loads each tile's accumulators (mpm_g2p_update): in place, the
        accumulators consumed, no velocity grid."""
        L.mpm_g2p_update(self.desc, self.acc, self.dtg, self.parts, self.bins, self.dt, stream)

    def step_update(self, stream=None):
        """bin, p2g and mpm_g2p_update: a whole step without a velocity grid."""
        self.bin(stream)
        self.p2g(stream)
        self.g2p_update(stream)

    def step(self, stream=None):
        L.mpm_step(self.desc, self.parts, self.bins, self.acc, self.vel, self.dt, self.dtg, stream)

    # -- steps that keep the particles in bin order (ping-pong buffers) --------
    def enable_sorted(self, with_ids: bool = True):
        """Allocates the second particle buffer and (optionally) particle ids 0..n-1."""
        n = self.x.shape[1]
        if with_ids:
            self.id = torch.arange(n, dtype=torch.int32, device=self.device)
            self.id2 = torch.empty_like(self.id)
        else:
            self.id = self.id2 = None
        self.x2, self.v2, self.C2, self.m2 = (torch.empty_like(t) for t in (self.x, self.v, self.C, self.m))
        if self.F is not None:
            self.F2 = torch.empty_like(self.F)
        if self.vol is not None:
            self.vol2 = torch.empty_like(self.vol)
        if self.phi is not None:
            self.phi2 = torch.zeros_like(self.phi)
        self.parts = self._parts(self.x, self.v, self.C, self.m, self.id, self.F, self.vol, self.phi)
        self.parts2 = self._parts(self.x2, self.v2, self.C2, self.m2, self.id2, self.F2, self.vol2, self.phi2)
        return self

    def swap(self):
        self.x, self.x2 = self.x2, self.x
        self.v, self.v2 = self.v2, self.v
        self.C, self.C2 = self.C2, self.C
        self.m, self.m2 = self.m2, self.m
        self.id, self.id2 = self.id2, self.id
        self.F, self.F2 = self.F2, self.F
        self.vol, self.vol2 = self.vol2, self.vol
        self.phi, self.phi2 = self.phi2, self.phi
        self.parts, self.parts2 = self.parts2, self.parts

    def g2p_sorted(self, stream=None):
        L.mpm_g2p_sorted(self.desc, self.vel, self.parts, self.parts2, self.bins, self.dt, stream)
        self.swap()

    def g2p_sorted_update(self, stream=None):
        L.mpm_g2p_sorted_update(self.desc, self.acc, self.dtg, self.parts, self.parts2, self.bins, self.dt, stream)
        self.swap()

    def step_sorted_update(self, stream=None):
        self.bin(stream)
        self.p2g(stream)
        self.g2p_sorted_update(stream)

    def g2p_binned(self, stream=None):
        L.mpm_g2p_binned(self.desc, self.vel, self.parts, self.parts2, self.bins, self.dt, stream)
        self.swap()

    def step_binned(self, stream=None):
        L.mpm_step_binned(self.desc, self.parts, self.parts2, self.bins, self.acc, self.vel, self.dt, self.dtg,
                          stream)
        self.swap()

    def step_sorted(self, stream=None):
        L.mpm_step_sorted(self.desc, self.parts, self.parts2, self.bins, self.acc, self.vel, self.dt, self.dtg,
                          stream)
        self.swap()

    # -- the fused step: the accumulators of the current positions in, the next ones out --
    def enable_fused(self):
        """Second accumulator grid for mpm_step_fused; fills the first with the
        P2G of the current positions (bin + p2g).  Needs enable_sorted()."""
        self.acc2 = torch.zeros_like(self.acc)
        self.bin()
        self.p2g()
        return self

    def step_fused(self, stream=None):
        L.mpm_step_fused(self.desc, self.parts, self.parts2, self.bins, self.acc, self.acc2, self.dt, self.dtg,
                         stream)
        self.swap()
        self.acc, self.acc2 = self.acc2, self.acc

    def status(self) -> np.ndarray:
        L.mpm_read_status(self.bins, self.status_host)
        torch.cuda.synchronize(self.device)
        return self.status_host.numpy().astype(np.uint32).copy()

    def ws_view(self, ptr: int, count: int) -> torch.Tensor:
        """uint32 words of the workspace at device address ``ptr`` (as int32)."""
        off = int(ptr) - self.ws.data_ptr()
        assert 0 <= off and off + 4 * count <= self.ws.numel() and off % 4 == 0
        return self.ws[off:off + 4 * count].view(torch.int32)

    def bins_arrays(self):
        """(key, perm, tile_count) copied to the host as uint32."""
        torch.cuda.synchronize(self.device)
        n = self.x.shape[1]
        nt = int(self.bins.ntiles)
        grab = lambda ptr, cnt: self.ws_view(ptr, cnt).cpu().numpy().view(np.uint32)
        return grab(self.bins.key, n), grab(self.bins.perm, n), grab(self.bins.tile_count, nt)
