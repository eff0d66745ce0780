"""The grid-recovered volume channel through the C ABI against the oracle.

P2G scatters each particle's rest volume in cells into a last accumulator
channel (bit for bit in the fixed-point modes), the grid update turns it into
a node volume fraction, and G2P gathers the particle's volume fraction back
(bit for bit).  Also with the elastic state, in float mode (within the float
tolerance), and through the sorted G2P, which carries vol and phi along.
"""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import oracle as O
from test_gpu_parity import sorted_output_order

pytestmark = pytest.mark.gpu


def volume_cloud(dim, count, n, seed, mode=W.ACC_I64, scale=19):
    cloud = W.with_elastic(W.small_cloud(dim, count, n, seed=seed, acc_mode=mode, scale_log2=scale, lo=0.05,
                                         hi=0.95, vsig=1.0, csig=1.0, mass_lo=0.5, mass_hi=1.5), seed=seed + 1)
    x = cloud["x"].copy()
    s = W.Stream(seed + 2, 3)
    idx = (s.bits(6) % np.uint64(count)).astype(np.int64)
    x[0, idx[:3]] = -0.1
    x[-1, idx[3:]] = 2.0
    vol = (cloud["vol"] * (0.5 + s.uniform24(count))).astype(np.float32)
    cloud.update(x=x, vol=vol)
    cloud["grid"] = dict(cloud["grid"], volume_channel=1)
    return cloud


def make(cloud, elastic):
    n = cloud["x"].shape[1]
    sys = MPMSystem(cloud["grid"], n).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    if elastic:
        return sys.load_elastic(cloud["F"], cloud["vol"], cloud["material"])
    return sys.load_volume(cloud["vol"])


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


CASES = [(3, W.ACC_I64, 19, 32, 6007, False), (3, W.ACC_I32, 19, 24, 2500, False),
         (2, W.ACC_I64, 20, 64, 6000, False), (2, W.ACC_I32, 20, 48, 3001, False),
         (3, W.ACC_I64, 19, 32, 5003, True), (2, W.ACC_I64, 20, 64, 4001, True)]


@pytest.mark.parametrize("dim,mode,scale,n,count,elastic", CASES)
def test_volume_step_fixed_bit_exact(dim, mode, scale, n, count, elastic):
    cloud = volume_cloud(dim, count, n, seed=2000 + 7 * dim + n + count, mode=mode, scale=scale)
    grid = cloud["grid"]
    sys = make(cloud, elastic)
    assert sys.acc.shape[0] == dim + 2 and sys.vel.shape[0] == dim + 1
    sys.bin()
    sys.p2g()
    torch.cuda.synchronize()
    acc = sys.acc.cpu().numpy().astype(np.int64)
    C = cloud["C"]
    if elastic:
        C, _ = O.stress_affine(grid, cloud["material"], cloud["x"], cloud["C"], cloud["F"], cloud["vol"],
                               cloud["m"])
    oacc, _, ocounts = O.p2g_fixed(grid, cloud["x"], cloud["v"], C, cloud["m"], vol=cloud["vol"])
    st = sys.status()
    assert ocounts[1] == 0 and st[L.ST_N_OUT_OF_RANGE] == 0 and not st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    assert np.array_equal(acc, oacc)
    sys.grid_update()
    vel = sys.vel.cpu().numpy()
    ovel = O.grid_update_fixed(grid, oacc[: dim + 1])
    ophi = O.grid_volume(grid, oacc[dim + 1])
    assert np.array_equal(bits(vel[:dim]), bits(ovel))
    assert np.array_equal(bits(vel[dim]), bits(ophi))
    assert not sys.acc.any().item(), "the grid update must clear every channel"
    sys.g2p()
    torch.cuda.synchronize()
    phi = sys.phi.cpu().numpy()
    ophi_p = O.g2p_volume(grid, ophi, cloud["x"])
    assert np.array_equal(bits(phi), bits(ophi_p))
    x, v, Cn = sys.state()
    if elastic:
        ox, ov, oC, oF, _ = O.g2p_elastic(grid, ovel, cloud["x"], cloud["v"], cloud["C"], cloud["F"])
    else:
        ox, ov, oC, _ = O.g2p(grid, ovel, cloud["x"], cloud["v"], cloud["C"])
    for a, b in ((x, ox), (v, ov), (Cn, oC)):
        assert np.array_equal(bits(a), bits(b))


@pytest.mark.parametrize("dim,n,count", [(3, 32, 6007), (2, 64, 6000)])
def test_volume_float_within_tolerance(dim, n, count):
    cloud = volume_cloud(dim, count, n, seed=2100 + dim, mode=W.ACC_F32, scale=0)
    grid = cloud["grid"]
    sys = make(cloud, False)
    sys.bin()
    sys.p2g()
    torch.cuda.synchronize()
    acc = sys.acc.cpu().numpy()
    oacc, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol=cloud["vol"])
    o = oacc.astype(np.float64)
    scale = np.abs(o).max(axis=-1, keepdims=True)
    assert np.all(np.abs(acc - o) <= np.maximum(1e-5 * np.abs(o), 1e-6 * scale))
    sys.grid_update()
    sys.g2p()
    torch.cuda.synchronize()
    phi = sys.phi.cpu().numpy().astype(np.float64)
    ophi = O.g2p_volume(grid, O.grid_volume(grid, oacc[dim + 1]), cloud["x"]).astype(np.float64)
    assert np.max(np.abs(phi - ophi)) <= 1e-5 * (1.0 + np.abs(ophi).max())


def test_volume_sorted_g2p_carries_vol_and_phi():
    dim, count, n = 3, 7001, 32
    cloud = volume_cloud(dim, count, n, seed=2200)
    grid = cloud["grid"]
    sys = make(cloud, False).enable_sorted()
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    valid = int(sys.status()[L.ST_N_VALID])
    sys.p2g()
    sys.grid_update()
    sys.g2p_sorted()
    torch.cuda.synchronize()
    phi, vol = sys.phi.cpu().numpy(), sys.vol.cpu().numpy()
    ids = sys.id.cpu().numpy().astype(np.int64)
    oacc, _, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol=cloud["vol"])
    ophi = O.g2p_volume(grid, O.grid_volume(grid, oacc[dim + 1]), cloud["x"])
    p = sorted_output_order(key, perm, cnt, valid, dim, grid["tile"])
    assert np.array_equal(ids, p)
    assert np.array_equal(vol, cloud["vol"][p])
    assert np.array_equal(bits(phi), bits(ophi[p]))


def test_volume_fraction_of_a_rest_packing_is_one():
    """8 particles per cell on a lattice, each carrying 1/8 of a cell: the
    interior reads one (the guide's 1/ppc emission)."""
    n, dim = 32, 3
    h = 0.5
    ax = (np.arange(8 * 2, 24 * 2) + 0.5) * h / n
    mesh = np.meshgrid(ax, ax, ax, indexing="ij")
    x = np.stack([m.ravel() for m in mesh]).astype(np.float32)
    count = x.shape[1]
    grid = dict(W.small_cloud(3, 1, n, seed=1, scale_log2=19)["grid"], volume_channel=1)
    z3, z9 = np.zeros((3, count), np.float32), np.zeros((9, count), np.float32)
    sys = MPMSystem(grid, count).load(x, z3, z9, np.ones(count, np.float32))
    sys.load_volume(np.full(count, grid["dx"] ** 3 / 8, np.float32))
    sys.step()
    torch.cuda.synchronize()
    phi = sys.phi.cpu().numpy()
    inside = np.all((x * n >= 10.5) & (x * n <= 21.5), axis=0)
    assert inside.sum() > 1000
    assert np.max(np.abs(phi[inside] - 1.0)) <= 1e-4
