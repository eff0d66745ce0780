"""The MLS-MPM elastic stress (Neo-Hookean stress folded into P2G's affine
matrix, F advanced by G2P) through the C ABI against the oracle.

Fixed-point modes match bit for bit: the accumulator grid (which carries the
stress through the shares), the velocity grid, and every particle's x, v, C
and F after G2P; the count of particles left unstressed (det F not a positive
normal number) matches the oracle's.  The float-atomic mode matches within
the float tolerance.  Sorted G2P and the host-buffer step carry F and the rest
volume along with the particle.
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


def elastic_cloud(dim, count, n, seed, mode=W.ACC_I64, scale=19, degenerate=True, **kw):
    cloud = W.with_elastic(W.small_cloud(dim, count, n, seed=seed, acc_mode=mode, scale_log2=scale, lo=0.05,
                                         hi=0.95, vsig=1.0, csig=1.0, mass_lo=0.5, mass_hi=1.5), seed=seed + 1,
                           **kw)
    x, F = cloud["x"].copy(), cloud["F"].copy()
    s = W.Stream(seed + 2, 3)
    idx = (s.bits(12) % np.uint64(count)).astype(np.int64)
    x[0, idx[:3]] = -0.1                          # outside the domain
    x[-1, idx[3:5]] = 2.0
    if degenerate:
        F[:, idx[5]] = 0.0                        # collapsed
        F[0, idx[6]] = -F[0, idx[6]]              # inverted (det < 0) ...
        F[1 if dim == 2 else 3, idx[6]] = 0.0
        F[:, idx[7]] = 0.0                        # ... and one collapsed particle outside the domain
        x[0, idx[7]] = -0.2
    cloud.update(x=x, F=F)
    return cloud


def make(cloud):
    n = cloud["x"].shape[1]
    return (MPMSystem(cloud["grid"], n).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
            .load_elastic(cloud["F"], cloud["vol"], cloud["material"]))


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


FIXED = [(3, W.ACC_I64, 19, 32, 6007), (3, W.ACC_I32, 19, 24, 2500), (2, W.ACC_I64, 20, 64, 6000),
         (2, W.ACC_I32, 20, 48, 3001)]


@pytest.mark.parametrize("dim,mode,scale,n,count", FIXED)
def test_elastic_step_fixed_bit_exact(dim, mode, scale, n, count):
    cloud = elastic_cloud(dim, count, n, seed=1000 + 7 * dim + n, mode=mode, scale=scale)
    grid, mat = cloud["grid"], cloud["material"]
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    torch.cuda.synchronize()
    acc = sys.acc.cpu().numpy().astype(np.int64)
    Cs, degenerate = O.stress_affine(grid, mat, cloud["x"], cloud["C"], cloud["F"], cloud["vol"], cloud["m"])
    oacc, ost, ocounts = O.p2g_fixed(grid, cloud["x"], cloud["v"], Cs, cloud["m"])
    assert degenerate == 2
    st = sys.status()
    assert st[L.ST_N_DEGENERATE] == degenerate
    assert ocounts[1] == 0 and st[L.ST_N_OUT_OF_RANGE] == 0 and not st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    assert np.array_equal(acc, oacc)
    sys.grid_update()
    vel = sys.vel.cpu().numpy()
    ovel = O.grid_update_fixed(grid, oacc)
    assert np.array_equal(bits(vel), bits(ovel))
    sys.g2p()
    x, v, C = sys.state()
    F, vol = sys.elastic_state()
    ox, ov, oC, oF, moved = O.g2p_elastic(grid, ovel, cloud["x"], cloud["v"], cloud["C"], cloud["F"])
    for a, b in ((x, ox), (v, ov), (C, oC), (F, oF)):
        assert np.array_equal(bits(a), bits(b))
    assert np.array_equal(vol, cloud["vol"])


def test_elastic_stress_changes_the_grid():
    """The stress is not a no-op: the same particles without F give another grid."""
    cloud = elastic_cloud(3, 3000, 32, seed=1100, degenerate=False)
    a = make(cloud)
    a.bin()
    a.p2g()
    b = MPMSystem(cloud["grid"], 3000).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    b.bin()
    b.p2g()
    torch.cuda.synchronize()
    ga, gb = a.acc.cpu().numpy(), b.acc.cpu().numpy()
    assert np.array_equal(ga[0], gb[0])                       # mass: unchanged
    assert np.array_equal(ga[1:].sum(axis=1), gb[1:].sum(axis=1))  # total momentum: unchanged
    assert np.count_nonzero(ga[1:] != gb[1:]) > 0.5 * np.count_nonzero(gb[1:])


@pytest.mark.parametrize("dim,n,count", [(3, 32, 6007), (2, 64, 6000)])
def test_elastic_step_float_within_tolerance(dim, n, count):
    cloud = elastic_cloud(dim, count, n, seed=1200 + dim, mode=W.ACC_F32, scale=0)
    grid, mat = cloud["grid"], cloud["material"]
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    torch.cuda.synchronize()
    acc = sys.acc.cpu().numpy()
    Cs, degenerate = O.stress_affine(grid, mat, cloud["x"], cloud["C"], cloud["F"], cloud["vol"], cloud["m"])
    oacc, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], Cs, cloud["m"])
    assert sys.status()[L.ST_N_DEGENERATE] == degenerate
    o = oacc.astype(np.float64)
    scale = np.abs(o).max(axis=-1, keepdims=True)
    assert np.all(np.abs(acc - o) <= np.maximum(1e-5 * np.abs(o), 1e-6 * scale))


@pytest.mark.parametrize("dim,n,count", [(3, 32, 7001), (2, 64, 5003)])
def test_elastic_sorted_g2p_carries_F_and_volume(dim, n, count):
    cloud = elastic_cloud(dim, count, n, seed=1300 + dim)
    cloud["vol"] = (cloud["vol"] * (1.0 + np.arange(count) / count)).astype(np.float32)  # distinct volumes
    grid, mat = cloud["grid"], cloud["material"]
    sys = make(cloud).enable_sorted()
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    valid = int(sys.status()[L.ST_N_VALID])
    sys.p2g()
    sys.grid_update()
    sys.g2p_sorted()
    x, v, C = sys.state()
    F, vol = sys.elastic_state()
    ids = sys.id.cpu().numpy().astype(np.int64)
    out = O.step_elastic(grid, mat, cloud["x"], cloud["v"], cloud["C"], cloud["m"], cloud["F"], cloud["vol"])
    p = sorted_output_order(key, perm, cnt, valid, dim, grid["tile"])
    assert np.array_equal(ids, p)
    for a, b in ((x, out["x"]), (v, out["v"]), (C, out["C"]), (F, out["F"])):
        assert np.array_equal(bits(a), bits(b[:, p]))
    assert np.array_equal(vol, cloud["vol"][p])
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    assert speed == O.advective_speed(dim, grid["dx"], out["v"][:, p[:valid]], out["C"][:, p[:valid]])


def test_elastic_steps_sorted_match_oracle_over_several_steps():
    """Three sorted steps in a row: the particles (found by id) keep matching
    the oracle's in-place steps bit for bit."""
    cloud = elastic_cloud(3, 5000, 32, seed=1400, degenerate=False, fsig=0.02)
    grid, mat = cloud["grid"], cloud["material"]
    sys = make(cloud).enable_sorted()
    x, v, C, m, F, vol = (cloud[k].copy() for k in ("x", "v", "C", "m", "F", "vol"))
    for _ in range(3):
        sys.step_sorted()
        out = O.step_elastic(grid, mat, x, v, C, m, F, vol)
        x, v, C, F = out["x"], out["v"], out["C"], out["F"]
    gx, gv, gC = sys.state()
    gF, gvol = sys.elastic_state()
    ids = sys.id.cpu().numpy().astype(np.int64)
    for a, b in ((gx, x), (gv, v), (gC, C), (gF, F)):
        assert np.array_equal(bits(a), bits(b[:, ids]))
    assert np.array_equal(gvol, vol[ids])
    assert sys.status()[L.ST_N_DEGENERATE] == 0


def test_elastic_step_host_equals_device_sorted_step():
    cloud = elastic_cloud(3, 20000, 32, seed=1500, degenerate=False)
    a = make(cloud).enable_sorted()
    a.step_sorted()
    xa, va, Ca = a.state()
    Fa, vola = a.elastic_state()
    ida = a.id.cpu().numpy()
    b = make(cloud).enable_sorted()
    pin = lambda arr: torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
    hx, hv, hC, hm = pin(cloud["x"]), pin(cloud["v"]), pin(cloud["C"]), pin(cloud["m"])
    hF, hvol = pin(cloud["F"]), pin(cloud["vol"])
    hid = pin(np.arange(20000, dtype=np.int32))
    b.x.zero_()
    b.F.zero_()
    host = L.particles(hx, hv, hC, hm, hid, hF, hvol, cloud["material"]["mu"], cloud["material"]["lambda"])
    L.mpm_step_host(b.desc, host, b.parts, b.parts2, b.bins, b.acc, b.vel, b.dt, b.dtg)
    torch.cuda.synchronize()
    assert np.array_equal(hid.numpy(), ida)
    assert np.array_equal(hx.numpy(), xa) and np.array_equal(hv.numpy(), va) and np.array_equal(hC.numpy(), Ca)
    assert np.array_equal(hF.numpy(), Fa) and np.array_equal(hvol.numpy(), vola)


def test_permute_carries_F_and_volume():
    cloud = elastic_cloud(3, 3001, 24, seed=1600)
    a = make(cloud).enable_sorted()
    a.bin()
    _, perm, _ = a.bins_arrays()
    L.mpm_permute(a.desc, a.parts, a.parts2, a.bins)
    torch.cuda.synchronize()
    p = perm.astype(np.int64)
    assert np.array_equal(a.F2.cpu().numpy(), cloud["F"][:, p])
    assert np.array_equal(a.vol2.cpu().numpy(), cloud["vol"][p])
    assert np.array_equal(a.C2.cpu().numpy(), cloud["C"][:, p])
