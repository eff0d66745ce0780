"""The multi-core CPU baseline (OpenMP, private per-thread grids merged by
integer add) against the single-threaded oracle: the same permutation, the
same grid and node velocities, and the same new state of every particle, bit
for bit, for several thread counts (the merge order must not matter)."""
import numpy as np
import pytest

from material_point_particle_gb300 import workloads as W
from oracle import cpu_omp
from oracle import oracle as O

pytestmark = pytest.mark.skipif(not cpu_omp.available(), reason="no OpenMP in the host compiler")


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("dim,n,count", [(3, 32, 6007), (2, 64, 6000), (3, 16, 33), (3, 16, 0)])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_omp_step_matches_the_oracle(dim, n, count, threads):
    cloud = W.small_cloud(dim, count, n, seed=7000 + dim + n + count, scale_log2=19, lo=0.05, hi=0.95,
                          vsig=1.0, csig=2.0, mass_lo=0.5, mass_hi=1.5)
    x = cloud["x"].copy()
    x[0, :3] = -0.1                          # outside the domain
    cloud["x"] = x
    grid = dict(cloud["grid"], g=[0.0, -9.8, 0.0])
    out = cpu_omp.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], threads=threads)
    ref = O.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert np.array_equal(out["perm"], ref["perm"])
    assert np.array_equal(out["acc"], ref["acc"])
    assert np.array_equal(bits(out["vel"]), bits(ref["vel"]))
    assert np.array_equal(out["counts"], ref["counts"])
    p = out["perm"].astype(np.int64)
    for k in ("x", "v", "C"):
        assert np.array_equal(bits(out[k]), bits(ref[k][:, p]))
    assert np.array_equal(out["m"], cloud["m"][p])


def test_omp_step_on_the_blobs_sample():
    """The benchmark's sample shape (clustered blobs on the 256^3 grid), fewer particles."""
    cloud = W.blobs3d(n_particles=40000, n_blobs=4)
    grid = cloud["grid"]
    out = cpu_omp.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], threads=4)
    ref = O.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert np.array_equal(out["acc"], ref["acc"])
    p = out["perm"].astype(np.int64)
    for k in ("x", "v", "C"):
        assert np.array_equal(bits(out[k]), bits(ref[k][:, p]))
    assert out["moved"] == cloud["x"].shape[1]


def test_omp_step_matches_the_oracle_at_wide_scale():
    """At S = 2^32 (shares far past 2^22) and S = 2^19 with one heavy particle."""
    for scale, heavy in [(32, False), (19, True)]:
        cloud = W.small_cloud(3, 6007, 32, seed=7100 + scale, scale_log2=scale, lo=0.05, hi=0.95,
                              vsig=1.0, csig=2.0)
        if heavy:
            cloud["m"][17] = 1e5
        grid = cloud["grid"]
        out = cpu_omp.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], threads=5)
        ref = O.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert np.array_equal(out["acc"], ref["acc"]) and np.abs(ref["acc"]).max() > 2 ** 31
        assert np.array_equal(bits(out["vel"]), bits(ref["vel"]))
        p = out["perm"].astype(np.int64)
        for k in ("x", "v", "C"):
            assert np.array_equal(bits(out[k]), bits(ref[k][:, p]))


def test_omp_step_bound_failure_scatters_nothing():
    cloud = W.small_cloud(3, 2000, 24, seed=7200, scale_log2=32)
    cloud["m"][5] = 1e15
    grid = cloud["grid"]
    out = cpu_omp.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], threads=4)
    ref = O.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert not out["acc"].any() and not ref["acc"].any()
    assert np.array_equal(out["counts"], ref["counts"]) and out["counts"][1] == 2000
