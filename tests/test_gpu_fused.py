"""The fused gather-scatter step (mpm_step_fused) against the oracle.

Each call must leave, bit for bit: the particles of the oracle's grid update
+ G2P of the accumulators it was given (in bin order, found by id), the next
accumulators equal to the oracle's P2G of the new state, and the accumulators
it read cleared.  Cases: 3D and 2D, several steps in a row,
particles that move more than a cell (scattered straight into the global
grid) and particles that leave the domain.
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


def fused_system(cloud):
    n = cloud["x"].shape[1]
    return MPMSystem(cloud["grid"], n).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted() \
        .enable_fused()


def run_and_check(cloud, steps):
    grid = cloud["grid"]
    sys = fused_system(cloud)
    x, v, C, m = (cloud[k].copy() for k in ("x", "v", "C", "m"))
    escaped = 0
    prev_ids = np.arange(cloud["x"].shape[1])
    for _ in range(steps):
        sys.step_fused()
        torch.cuda.synchronize()
        st = sys.status()
        # the oracle's step from the same state, particles in index order
        acc, _, _ = O.p2g_fixed(grid, x, v, C, m)
        vel = O.grid_update_fixed(grid, acc)
        inside = O.bin_particles(grid, x)[0] != 0xFFFFFFFF
        x, v, C, moved = O.g2p(grid, vel, x, v, C)
        ids = sys.id.cpu().numpy().astype(np.int64)
        gx, gv, gC = sys.state()
        for a, b in ((gx, x), (gv, v), (gC, C)):
            assert np.array_equal(bits(a), bits(b[:, ids]))
        # the next accumulators: the oracle's P2G of the new state
        nacc, _, counts = O.p2g_fixed(grid, x, v, C, m)
        assert np.array_equal(sys.acc.cpu().numpy(), nacc)
        assert st[L.ST_N_OUT_OF_RANGE] == 0 and counts[1] == 0
        assert not sys.acc2.any().item(), "the accumulators read must be cleared"
        # the order is bin order: out[j] = in[perm[j]] (indices into this step's input, whose ids are prev_ids)
        key, perm, cnt = sys.bins_arrays()
        assert np.array_equal(ids, prev_ids[perm.astype(np.int64)])
        prev_ids = ids
        speed = np.array([st[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
        assert speed == O.advective_speed(grid["dim"], grid["dx"], v[:, inside], C[:, inside])
        escaped += int(st[L.ST_N_ESCAPED])
    return escaped


@pytest.mark.parametrize("dim,n,count", [(3, 32, 6007), (2, 64, 6000), (3, 24, 257)])
def test_fused_steps_match_the_oracle(dim, n, count):
    cloud = W.small_cloud(dim, count, n, seed=3000 + dim + n, scale_log2=19, lo=0.05, hi=0.95, vsig=1.0, csig=2.0)
    x = cloud["x"].copy()
    x[0, :5] = -0.1                      # outside the domain from the start
    cloud["x"] = x
    cloud["grid"]["g"] = [0.0, -9.8, 0.0]
    run_and_check(cloud, steps=3)


def test_fused_particles_moving_more_than_a_cell():
    """dt large enough that many particles cross more than one cell in a step
    (and some leave the domain): those leaving their tile are scattered into
    the global grid with the same shares."""
    cloud = W.small_cloud(3, 4001, 32, seed=3100, scale_log2=19, lo=0.05, hi=0.95, vsig=2.0, csig=0.5)
    cloud["grid"]["dt"] = float(np.float32(0.03))    # |v| dt up to ~4 cells
    escaped = run_and_check(cloud, steps=2)
    assert escaped > 100


def test_fused_is_refused_outside_its_scope():
    cloud = W.small_cloud(3, 1000, 16, seed=3200, acc_mode=W.ACC_I32, scale_log2=19)
    sys = MPMSystem(cloud["grid"], 1000).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    acc2 = torch.zeros_like(sys.acc)
    with pytest.raises(L.MPMError) as e:
        L.mpm_step_fused(sys.desc, sys.parts, sys.parts2, sys.bins, sys.acc, acc2, sys.dt, sys.dtg)
    assert e.value.code == L.MPM_E_ARG


def test_fused_step_beyond_22_bit_shares_is_undone():
    """The fused step forms its new state and scatters it in one kernel, so it can
    only test each particle as it goes: a particle whose new shares would not fit
    22 bits (mass 10^5 at S = 2^19) undoes the step's scatter (the written grid is
    left zero) and sets the bound flag; the gathered state is still the oracle's."""
    cloud = W.small_cloud(3, 6007, 32, seed=3100, scale_log2=19, lo=0.2, hi=0.8)
    cloud["m"][123] = 1e5
    grid = cloud["grid"]
    sys = fused_system(cloud)
    st = sys.status()
    assert st[L.ST_SHARE_PATH] == 1 and not st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    sys.step_fused()
    st = sys.status()
    assert st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    assert st[L.ST_N_OUT_OF_RANGE] == 1
    assert not sys.acc.any().item() and not sys.acc2.any().item()
    acc, _, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    x, v, C, _ = O.g2p(grid, O.grid_update_fixed(grid, acc), cloud["x"], cloud["v"], cloud["C"])
    ids = sys.id.cpu().numpy().astype(np.int64)
    gx, gv, gC = sys.state()
    for a, b in ((gx, x), (gv, v), (gC, C)):
        assert np.array_equal(bits(a), bits(b[:, ids]))
