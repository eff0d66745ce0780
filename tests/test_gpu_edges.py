"""Edge cases of every stepping path: no particles, one, a ragged 33, and a
set that lies wholly outside the domain, through the sorted, bin-order and
fused steps, the transfer loop, and the elastic and volume-channel steps;
each result against the oracle's step (particles found by id)."""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import oracle as O

pytestmark = pytest.mark.gpu

CASES = ["empty", "one", "ragged", "outside"]


def edge_cloud(case, dim=3):
    count = {"empty": 0, "one": 1, "ragged": 33, "outside": 50}[case]
    cloud = W.small_cloud(dim, count, 16, seed=6000 + count, scale_log2=19, lo=0.2, hi=0.8)
    if case == "outside":
        x = cloud["x"].copy()
        x[0] = -0.5
        cloud["x"] = x
    return cloud


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def check_against_oracle(sys, cloud, out):
    x, v, C = sys.state()
    ids = sys.id.cpu().numpy().astype(np.int64)
    n = cloud["x"].shape[1]
    assert np.array_equal(np.sort(ids), np.arange(n))
    for a, b in ((x, out["x"]), (v, out["v"]), (C, out["C"])):
        assert np.array_equal(bits(a), bits(b[:, ids]))


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("path", ["sorted", "binned", "fused"])
def test_step_paths_on_edge_inputs(case, path):
    cloud = edge_cloud(case)
    n = cloud["x"].shape[1]
    sys = MPMSystem(cloud["grid"], max(n, 1)).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    if path == "sorted":
        sys.step_sorted()
    elif path == "binned":
        sys.step_binned()
    else:
        sys.enable_fused().step_fused()
    torch.cuda.synchronize()
    st = sys.status()
    valid = 0 if case in ("empty", "outside") else n
    assert st[L.ST_N_VALID] == valid and st[L.ST_N_OUTSIDE] == n - valid
    if n:
        check_against_oracle(sys, cloud, O.step_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"],
                                                      cloud["m"]))
    assert not sys.acc.any().item() if path != "fused" else not sys.acc2.any().item()


@pytest.mark.parametrize("case", CASES)
def test_transfer_loop_on_edge_inputs(case):
    cloud = edge_cloud(case)
    n = cloud["x"].shape[1]
    grid = dict(cloud["grid"], g=[0.0, 0.0, 0.0])
    sys = MPMSystem(grid, max(n, 1)).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    sys.bin()
    sys.p2g()
    acc_b = torch.zeros_like(sys.acc)
    L.mpm_iterate(sys.desc, sys.parts, sys.bins, sys.acc, acc_b, 3)
    torch.cuda.synchronize()
    gx, gv, gC = sys.state()
    x, v, C, m = (cloud[k].copy() for k in ("x", "v", "C", "m"))
    og = dict(grid, dt=0.0)
    for _ in range(3):
        acc, _, _ = O.p2g_fixed(og, x, v, C, m)
        x, v, C, _ = O.g2p(og, O.grid_update_fixed(og, acc), x, v, C)
    for a, b in ((gx, x), (gv, v), (gC, C)):
        assert np.array_equal(bits(a), bits(b))
    assert not sys.acc.any().item() and not acc_b.any().item()


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("variant", ["elastic", "volume"])
def test_variant_steps_on_edge_inputs(case, variant):
    cloud = edge_cloud(case)
    n = cloud["x"].shape[1]
    el = W.with_elastic(cloud, seed=6100)
    grid = dict(cloud["grid"], volume_channel=1) if variant == "volume" else cloud["grid"]
    sys = MPMSystem(grid, max(n, 1)).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    if variant == "elastic":
        sys.load_elastic(el["F"], el["vol"], el["material"])
    else:
        sys.load_volume(el["vol"])
    sys.enable_sorted()
    sys.step_binned()
    torch.cuda.synchronize()
    if not n:
        return
    if variant == "elastic":
        out = O.step_elastic(grid, el["material"], cloud["x"], cloud["v"], cloud["C"], cloud["m"], el["F"], el["vol"])
        check_against_oracle(sys, cloud, out)
        F, _ = sys.elastic_state()
        ids = sys.id.cpu().numpy().astype(np.int64)
        assert np.array_equal(bits(F), bits(out["F"][:, ids]))
    else:
        check_against_oracle(sys, cloud, O.step_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"],
                                                      cloud["m"]))
        oacc, _, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol=el["vol"])
        ophi = O.g2p_volume(grid, O.grid_volume(grid, oacc[3 + 1]), cloud["x"])
        ids = sys.id.cpu().numpy().astype(np.int64)
        assert np.array_equal(bits(sys.phi.cpu().numpy()), bits(ophi[ids]))
