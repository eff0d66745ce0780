"""Seeded synthetic particle sets for the MPM transfer path.

This module draws random numbers and lays them out as arrays. It holds none of
the transfer arithmetic (no weights, no shares, no grid), so that the oracle
side and the CUDA side can both consume its arrays without sharing any of the
method's code.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", 2014), written out below from its published definition.
Uniforms take the top 24 bits (fp32-exact) or 53 bits (fp64) of each draw;
normals come from the Box-Muller transform in fp64 and are then rounded to fp32.

The five workloads follow the particle sets the pages describe:

* ``cic_int``     -- 2D integer cloud-in-cell transfer, 8x8 cells, 256 particles
  ("particle to grid transfer in checked integer arithmetic", section "the program").
* ``mls2d``       -- 2D quadratic B-spline, 128^2 nodes, 65,536 particles uniform
  in [0.25, 0.75]^2, int32 fixed point at scale 2^20.
* ``dambreak3d``  -- 3D quadratic, 128^3 nodes, 2,097,152 particles on a lattice
  at 8 per cell starting at 0.05, gravity -9.8 along y, dt 1e-4.
* ``blobs3d``     -- 3D quadratic, 256^3 nodes, 16,777,216 particles in 64
  Gaussian blobs (sigma 0.02, centres U[0.1, 0.9]^3), int64 fixed point.
* ``sphere3d``    -- 3D quadratic, 512^3 nodes, 67,108,864 particles uniform in a
  ball of radius 0.4, rigid rotation omega = (0, 0, 2) plus N(0, 0.05) noise.

Every builder takes ``n_particles`` to draw a smaller set with the same
distribution (the parity tests use these), and returns a dict of numpy arrays
plus the grid parameters.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SEED_BASE = 0x4D504D00
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+count-1`` of the splitmix64 sequence for ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        return _mix(state)


def _substream_seed(seed: int, tag: int) -> int:
    with np.errstate(over="ignore"):
        return int(_mix(np.array([seed ^ (tag * 0x632BE59BD9B4E019 & 0xFFFFFFFFFFFFFFFF)],
                                 dtype=np.uint64))[0])


class Stream:
    """A named, seeded source of uniforms and normals (counter based)."""

    def __init__(self, seed: int, tag: int):
        self.seed = _substream_seed(seed, tag)
        self.pos = 0

    def bits(self, count: int) -> np.ndarray:
        out = splitmix64(self.seed, count, self.pos)
        self.pos += count
        return out

    CHUNK = 1 << 20

    def _chunks(self, count: int, per: int, fill) -> None:
        """fill(lo, hi, bits) for each chunk [lo, hi) of `count` outputs, each taking `per` draws per
        output from its own place in the sequence; chunks run on a thread pool (numpy releases the GIL
        in these loops), and the counter-based sequence makes the result that of one sequential pass."""
        base = self.pos
        spans = [(lo, min(count, lo + self.CHUNK)) for lo in range(0, count, self.CHUNK)]

        def one(span):
            lo, hi = span
            fill(lo, hi, splitmix64(self.seed, per * (hi - lo), base + per * lo))

        if len(spans) > 1:
            with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as ex:
                list(ex.map(one, spans))
        elif spans:
            one(spans[0])
        self.pos = base + per * count

    def _uniform(self, count: int, shift: int, scale: float) -> np.ndarray:
        out = np.empty(count, dtype=np.float64)

        def fill(lo, hi, b):
            out[lo:hi] = (b >> np.uint64(shift)).astype(np.float64) * scale

        self._chunks(count, 1, fill)
        return out

    def uniform24(self, count: int) -> np.ndarray:
        """fp32-exact uniforms on [0, 1): multiples of 2^-24."""
        return self._uniform(count, 40, 2.0 ** -24)

    def uniform53(self, count: int) -> np.ndarray:
        return self._uniform(count, 11, 2.0 ** -53)

    def normal(self, count: int, sigma: float = 1.0, dtype=np.float64) -> np.ndarray:
        """Box-Muller on consecutive draw pairs (2i, 2i+1): pair i gives r cos(th)
        at output i and r sin(th) at output half + i.  With dtype float32 the fp64
        values are rounded to fp32 as they are stored."""
        half = (count + 1) // 2
        z = np.empty(2 * half, dtype=dtype)

        def fill(lo, hi, b):
            d = (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
            u1 = 1.0 - d[0::2]    # (0, 1]
            u2 = d[1::2]
            r = np.sqrt(-2.0 * np.log(u1))
            th = 2.0 * math.pi * u2
            z[lo:hi] = r * np.cos(th) * sigma
            z[half + lo:half + hi] = r * np.sin(th) * sigma

        self._chunks(half, 2, fill)
        return z[:count]


def scrambled_order(n: int, a: int, b: int) -> np.ndarray:
    """Index map k -> (k*a + b) mod n; a permutation when gcd(a, n) == 1."""
    k = np.arange(n, dtype=np.int64)
    return (k * a + b) % n


def _grid(dim, n, order, acc_mode, scale_log2, tile, dt=1e-4, g=(0.0, 0.0, 0.0), boundary_nodes=3):
    n = list(n) + [1] * (3 - len(n))
    dx = np.float32(1.0 / n[0])
    return dict(dim=dim, n=n, dx=float(dx), inv_dx=float(np.float32(n[0])), order=order,
                acc_mode=acc_mode, scale_log2=scale_log2, tile=tile,
                boundary_nodes=boundary_nodes, dt=float(np.float32(dt)),
                g=[float(np.float32(c)) for c in g])


ACC_I32, ACC_I64, ACC_F32, ACC_EXACT_INT = 0, 1, 2, 3


def cic_int(n_particles: int = 256, seed: int = SEED_BASE + 1):
    """Integer CIC cloud: positions in 1/65,536 of a cell on 8x8 cells, masses
    1..1000, velocities -1000..1000 per component."""
    s = Stream(seed, 1)
    X = np.floor(s.uniform24(2 * n_particles) * (8 * 65536)).astype(np.int32).reshape(2, n_particles)
    m = (1 + np.floor(s.uniform53(n_particles) * 1000)).astype(np.int64)
    v = (-1000 + np.floor(s.uniform53(2 * n_particles) * 2001)).astype(np.int64).reshape(2, n_particles)
    grid = _grid(2, (9, 9), 1, ACC_EXACT_INT, 0, 8)
    return dict(name="cic_int", X=X, m=m, v=v, grid=grid)


def _fp32_particles(x, v, C, m):
    return dict(x=np.ascontiguousarray(x, dtype=np.float32),
                v=np.ascontiguousarray(v, dtype=np.float32),
                C=np.ascontiguousarray(C, dtype=np.float32),
                m=np.ascontiguousarray(m, dtype=np.float32))


def mls2d(n_particles: int = 65536, seed: int = SEED_BASE + 2, n: int = 128):
    s = Stream(seed, 2)
    x = 0.25 + 0.5 * s.uniform24(2 * n_particles).reshape(2, n_particles)
    v = s.normal(2 * n_particles, 0.5).reshape(2, n_particles)
    C = s.normal(4 * n_particles, 0.1).reshape(4, n_particles)
    m = np.ones(n_particles)
    out = _fp32_particles(x, v, C, m)
    out.update(name="mls2d", grid=_grid(2, (n, n), 2, ACC_I32, 20, 8))
    return out


def dambreak3d(n_particles: int = 2097152, seed: int = SEED_BASE + 3, n: int = 128,
               acc_mode: int = ACC_I64, scale_log2: int = 21):
    """Lattice block: 128^3 particles spaced dx/2 from 0.05 (8 per cell); a
    smaller ``n_particles`` keeps the spacing and takes the leading sub-block."""
    side = max(1, int(round(n_particles ** (1.0 / 3.0))))
    while side ** 3 > n_particles:
        side -= 1
    count = side ** 3
    i = np.arange(side, dtype=np.float64)
    coord = 0.05 + (i + 0.5) / (2.0 * n)
    zz, yy, xx = np.meshgrid(coord, coord, coord, indexing="ij")
    x = np.stack([xx.ravel(), yy.ravel(), zz.ravel()])
    v = np.zeros((3, count))
    C = np.zeros((9, count))
    m = np.ones(count)
    out = _fp32_particles(x, v, C, m)
    out.update(name="dambreak3d",
               grid=_grid(3, (n, n, n), 2, acc_mode, scale_log2 if acc_mode != ACC_F32 else 0, 4,
                          dt=1e-4, g=(0.0, -9.8, 0.0)))
    return out


def blobs3d(n_particles: int = 16777216, seed: int = SEED_BASE + 4, n: int = 256,
            n_blobs: int = 64, sigma: float = 0.02, scale_log2: int = 19):
    """Gaussian blobs, stored blob-major; samples outside [2dx, 1-2dx] are redrawn."""
    s = Stream(seed, 4)
    centres = 0.1 + 0.8 * s.uniform53(3 * n_blobs).reshape(n_blobs, 3)
    per = np.full(n_blobs, n_particles // n_blobs)
    per[: n_particles - per.sum()] += 1
    lo, hi = 2.0 / n, 1.0 - 2.0 / n
    x = np.empty((3, n_particles))
    pos = 0
    for b in range(n_blobs):
        cnt = int(per[b])
        pts = centres[b][:, None] + s.normal(3 * cnt, sigma).reshape(cnt, 3).T
        bad = np.any((pts < lo) | (pts >= hi), axis=0)
        while bad.any():
            k = int(bad.sum())
            pts[:, bad] = centres[b][:, None] + s.normal(3 * k, sigma).reshape(k, 3).T
            bad = np.any((pts < lo) | (pts >= hi), axis=0)
        x[:, pos:pos + cnt] = pts
        pos += cnt
    v = s.normal(3 * n_particles, 1.0, dtype=np.float32).reshape(3, n_particles)
    C = s.normal(9 * n_particles, 0.1, dtype=np.float32).reshape(9, n_particles)
    m = np.ones(n_particles)
    out = _fp32_particles(x, v, C, m)
    out.update(name="blobs3d", grid=_grid(3, (n, n, n), 2, ACC_I64, scale_log2, 4))
    return out


def sphere3d(n_particles: int = 67108864, seed: int = SEED_BASE + 5, n: int = 512,
             radius: float = 0.4, scale_log2: int = 21):
    """Uniform in a ball (rejection from the cube), rigid rotation about z plus noise."""
    s = Stream(seed, 5)
    c = np.array([0.5, 0.5, 0.5])
    x64 = np.empty((3, n_particles))
    x = np.empty((3, n_particles), dtype=np.float32)
    v = np.empty((3, n_particles), dtype=np.float32)
    got = 0
    while got < n_particles:
        want = int((n_particles - got) * 2.0) + 1024
        u = s.uniform53(3 * want).reshape(want, 3)
        # candidates in chunks (threads), the accepted ones kept in candidate order
        spans = [(lo, min(want, lo + Stream.CHUNK)) for lo in range(0, want, Stream.CHUNK)]

        def accept(span):
            p = (u[span[0]:span[1]] * 2.0 - 1.0) * radius
            return p[np.sum(p * p, axis=1) < radius * radius]

        with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
            keeps = list(ex.map(accept, spans))
        for keep in keeps:
            take = min(len(keep), n_particles - got)
            if take <= 0:
                break
            x64[:, got:got + take] = (keep[:take] + c).T
            got += take
        del u, keeps
    noise = s.normal(3 * n_particles, 0.05).reshape(3, n_particles)
    omega = np.array([0.0, 0.0, 2.0])
    spans = [(lo, min(n_particles, lo + Stream.CHUNK)) for lo in range(0, n_particles, Stream.CHUNK)]

    def rotate(span):
        lo, hi = span
        r = x64[:, lo:hi] - c[:, None]
        v[:, lo:hi] = np.cross(omega[None, :], r.T).T + noise[:, lo:hi]
        x[:, lo:hi] = x64[:, lo:hi]

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(rotate, spans))
    del noise, x64
    C = s.normal(9 * n_particles, 0.1, dtype=np.float32).reshape(9, n_particles)
    m = np.ones(n_particles, dtype=np.float32)
    out = dict(x=x, v=v, C=C, m=m)
    out.update(name="sphere3d", grid=_grid(3, (n, n, n), 2, ACC_I64, scale_log2, 4))
    return out


def small_cloud(dim: int, n_particles: int, n: int, seed: int, acc_mode: int = ACC_I64,
                scale_log2: int = 20, lo: float = 0.3, hi: float = 0.7, vsig: float = 1.0,
                csig: float = 0.5, tile: int | None = None, mass_lo: float = 1.0,
                mass_hi: float = 1.0):
    """A small random cloud for parity and pin tests."""
    s = Stream(seed, 7)
    x = lo + (hi - lo) * s.uniform24(dim * n_particles).reshape(dim, n_particles)
    v = s.normal(dim * n_particles, vsig).reshape(dim, n_particles)
    C = s.normal(dim * dim * n_particles, csig).reshape(dim * dim, n_particles)
    m = mass_lo + (mass_hi - mass_lo) * s.uniform24(n_particles)
    out = _fp32_particles(x, v, C, m)
    nn = (n,) * dim
    out.update(name=f"cloud{dim}d", grid=_grid(dim, nn, 2, acc_mode, scale_log2,
                                                 tile if tile else (4 if dim == 3 else 8)))
    return out


def with_elastic(cloud: dict, seed: int, fsig: float = 0.05, ppc: float = 8.0, mu: float = 1.0e7,
                 lam: float = 1.0e7) -> dict:
    """Adds an elastic state to `cloud`: deformation gradients F = I + N(0, fsig) per
    entry (dim*dim planes, row-major like C), rest volumes V0 = dx^dim / ppc and a
    Neo-Hookean material {mu, lambda}.  The defaults make the stress term of the
    affine matrix comparable to C on the small test grids (dt = 1e-4, m ~ 1)."""
    dim = cloud["grid"]["dim"]
    n = cloud["x"].shape[1]
    s = Stream(seed, 11)
    F = s.normal(dim * dim * n, fsig).reshape(dim * dim, n)
    for k in range(dim):
        F[k * dim + k] += 1.0
    vol = np.full(n, cloud["grid"]["dx"] ** dim / ppc)
    out = dict(cloud)
    out.update(F=np.ascontiguousarray(F, dtype=np.float32), vol=np.ascontiguousarray(vol, dtype=np.float32),
               material={"mu": float(np.float32(mu)), "lambda": float(np.float32(lam))})
    return out


CONFIGS = {
    "cic_int": cic_int,
    "mls2d": mls2d,
    "dambreak3d": dambreak3d,
    "blobs3d": blobs3d,
    "sphere3d": sphere3d,
}
