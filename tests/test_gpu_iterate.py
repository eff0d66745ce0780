"""The transfer loop at fixed positions (mpm_iterate) against the oracle.

After K iterations the particles' v and C (the displacement d and its
gradient D of the position-based solver) must equal, bit for bit, K rounds of
the oracle's P2G -> grid update without gravity -> G2P without advection,
starting from the P2G of the initial state; x, m and the particles outside
the domain are unchanged, and both accumulator grids are left zero.
"""
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


@pytest.mark.parametrize("dim,n,count,iterations", [(3, 32, 6007, 4), (2, 64, 6000, 3), (3, 24, 2500, 1),
                                                    (3, 16, 20000, 5)])
def test_iterations_match_the_oracle(dim, n, count, iterations):
    cloud = W.small_cloud(dim, count, n, seed=4000 + dim + n + iterations, scale_log2=19, lo=0.05, hi=0.95,
                          vsig=1.0, csig=2.0)
    x = cloud["x"].copy()
    x[0, :4] = -0.1
    cloud["x"] = x
    grid = dict(cloud["grid"], g=[0.0, 0.0, 0.0])     # the loop adds no gravity
    sys = MPMSystem(grid, count).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    sys.bin()
    sys.p2g()
    acc_b = torch.zeros_like(sys.acc)
    L.mpm_iterate(sys.desc, sys.parts, sys.bins, sys.acc, acc_b, iterations)
    torch.cuda.synchronize()
    gx, gv, gC = sys.state()
    x, v, C, m = (cloud[k].copy() for k in ("x", "v", "C", "m"))
    ogrid = dict(grid, dt=0.0)                         # G2P without advection
    for _ in range(iterations):
        acc, _, _ = O.p2g_fixed(ogrid, x, v, C, m)
        vel = O.grid_update_fixed(ogrid, acc)
        x2, v, C, _ = O.g2p(ogrid, vel, x, v, C)
        assert np.array_equal(bits(x2), bits(x))
    assert np.array_equal(bits(gx), bits(cloud["x"]))
    assert np.array_equal(bits(gv), bits(v))
    assert np.array_equal(bits(gC), bits(C))
    assert not sys.acc.any().item() and not acc_b.any().item()
    assert sys.status()[L.ST_FLAGS] == 0


def test_iterate_is_refused_outside_its_scope():
    cloud = W.small_cloud(3, 1000, 16, seed=4100, acc_mode=W.ACC_I32, scale_log2=19)
    sys = MPMSystem(cloud["grid"], 1000).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    with pytest.raises(L.MPMError) as e:
        L.mpm_iterate(sys.desc, sys.parts, sys.bins, sys.acc, torch.zeros_like(sys.acc), 2)
    assert e.value.code == L.MPM_E_ARG
