"""mpm_g2p_binned (the sorted G2P without the bank-class interleave, one warp
per work item) against the oracle: the new state of every particle bit for bit
(with the elastic state's F and the volume channel's phi), written in bin
order, out[j] = new state of in[perm[j]], the particles outside the domain
copied after them; and several binned steps in a row (found by id)."""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def cloud_with_outliers(dim, count, n, seed, **kw):
    cloud = W.small_cloud(dim, count, n, seed=seed, scale_log2=19, lo=0.05, hi=0.95, vsig=1.0, csig=2.0, **kw)
    x = cloud["x"].copy()
    x[0, :5] = -0.1
    x[-1, 5:9] = 2.0
    cloud["x"] = x
    return cloud


@pytest.mark.parametrize("dim,n,count,variant", [(3, 32, 7001, "plain"), (2, 64, 5003, "plain"),
                                                 (3, 32, 6007, "elastic"), (3, 32, 6007, "volume"),
                                                 (2, 48, 4001, "volume")])
def test_g2p_binned_matches_the_oracle(dim, n, count, variant):
    cloud = cloud_with_outliers(dim, count, n, seed=5000 + dim + n)
    grid = cloud["grid"]
    el = W.with_elastic(cloud, seed=5001)
    if variant == "volume":
        grid = dict(grid, volume_channel=1)
    sys = MPMSystem(grid, count).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    if variant == "elastic":
        sys.load_elastic(el["F"], el["vol"], el["material"])
    elif variant == "volume":
        sys.load_volume(el["vol"])
    sys.enable_sorted()
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    sys.p2g()
    sys.grid_update()
    vel = sys.vel.cpu().numpy()
    sys.g2p_binned()
    torch.cuda.synchronize()
    x, v, C = sys.state()
    ids = sys.id.cpu().numpy().astype(np.int64)
    p = perm.astype(np.int64)
    assert np.array_equal(ids, p)
    if variant == "elastic":
        ox, ov, oC, oF, _ = O.g2p_elastic(grid, vel[:dim], cloud["x"], cloud["v"], cloud["C"], el["F"])
        F, vol = sys.elastic_state()
        assert np.array_equal(bits(F), bits(oF[:, p]))
        assert np.array_equal(vol, el["vol"][p])
    else:
        ox, ov, oC, _ = O.g2p(grid, vel[:dim], cloud["x"], cloud["v"], cloud["C"])
    if variant == "volume":
        ophi = O.g2p_volume(grid, vel[dim], cloud["x"])
        inside = np.nonzero(key != 0xFFFFFFFF)[0]
        got = sys.phi.cpu().numpy()
        valid = int(sys.status()[L.ST_N_VALID])
        assert np.array_equal(bits(got[:valid]), bits(ophi[p[:valid]]))
        assert inside.size == valid
    for a, b in ((x, ox), (v, ov), (C, oC)):
        assert np.array_equal(bits(a), bits(b[:, p]))
    assert np.array_equal(sys.m.cpu().numpy(), cloud["m"][p])
    valid = int(sys.status()[L.ST_N_VALID])
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    assert speed == O.advective_speed(dim, grid["dx"], ov[:, p[:valid]], oC[:, p[:valid]])


def test_binned_steps_in_a_row_match_the_oracle():
    cloud = cloud_with_outliers(3, 6007, 32, seed=5100)
    grid = cloud["grid"]
    sys = MPMSystem(grid, 6007).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    x, v, C, m = (cloud[k].copy() for k in ("x", "v", "C", "m"))
    for _ in range(3):
        sys.step_binned()
        out = O.step_fixed(grid, x, v, C, m)
        x, v, C = out["x"], out["v"], out["C"]
    gx, gv, gC = sys.state()
    ids = sys.id.cpu().numpy().astype(np.int64)
    for a, b in ((gx, x), (gv, v), (gC, C)):
        assert np.array_equal(bits(a), bits(b[:, ids]))
