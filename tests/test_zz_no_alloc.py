"""mpm_bin_static (binning into the library's own static workspace) against
mpm_bin with a caller workspace, through the C ABI.

Binning is integer work, so the two must agree exactly: the permutation (read
back through mpm_permute of particle ids), the status words after binning,
and the P2G grid built from each set of bins.  Two calls in a row on different
particle sets check that the second call reuses the workspace correctly.
"""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem

pytestmark = pytest.mark.gpu

BIN_WORDS = L.ST_BIN_WORDS   # the status words mpm_bin writes


def _status(bins):
    out = torch.zeros(L.MPM_STATUS_WORDS, dtype=torch.int32).pin_memory()
    L.mpm_read_status(bins, out)
    torch.cuda.synchronize()
    return out.numpy().astype(np.uint32)[:BIN_WORDS].copy()


def _perm_via_ids(sys, bins):
    """perm as seen through mpm_permute: the ids 0..n-1 reordered by it."""
    n = sys.x.shape[1]
    ids = torch.arange(n, dtype=torch.int32, device="cuda")
    out = [torch.empty_like(t) for t in (sys.x, sys.v, sys.C, sys.m)]
    ids_out = torch.empty_like(ids)
    src = L.particles(sys.x, sys.v, sys.C, sys.m, ids)
    dst = L.particles(*out, ids_out)
    L.mpm_permute(sys.desc, src, dst, bins)
    torch.cuda.synchronize()
    return ids_out.cpu().numpy().view(np.uint32)


def _p2g(sys, bins):
    acc = torch.zeros_like(sys.acc)
    L.mpm_p2g(sys.desc, sys.parts, bins, acc)
    torch.cuda.synchronize()
    return acc.cpu().numpy()


def _clouds():
    a = W.blobs3d(30000, n=64, n_blobs=4, seed=21)
    b = W.small_cloud(2, 5003, 64, seed=22, lo=0.02, hi=0.98)
    b["x"][0, 7] = -0.25      # one particle outside the domain
    return [a, b]


def _check_one(cloud):
    sys = MPMSystem(cloud["grid"], cloud["x"].shape[1]).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    sys.bin()
    ref_status = _status(sys.bins)
    ref_perm = _perm_via_ids(sys, sys.bins)
    ref_acc = _p2g(sys, sys.bins)

    bins = L.mpm_bin_static(sys.desc, sys.parts, 0)
    assert bins.n == sys.x.shape[1] and bins.ntiles == sys.bins.ntiles
    assert np.array_equal(_status(bins), ref_status)
    assert np.array_equal(_perm_via_ids(sys, bins), ref_perm)
    assert np.array_equal(_p2g(sys, bins), ref_acc)


def test_static_bins_equal_workspace_bins_twice():
    for cloud in _clouds():          # two calls in a row, different problems
        _check_one(cloud)


def test_static_bins_allocate_no_device_memory():
    """Repeated calls leave the device's free memory unchanged (measured by the
    driver, outside any caching allocator): the call uses only the library's
    file-scope array and the caller's particle arrays."""
    cloud = W.blobs3d(30000, n=64, n_blobs=4, seed=24)
    sys = MPMSystem(cloud["grid"], cloud["x"].shape[1]).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    L.mpm_bin_static(sys.desc, sys.parts, 0)        # the first call may load the library's device code
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        L.mpm_bin_static(sys.desc, sys.parts, 0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_bins_reject_oversize():
    cloud = W.small_cloud(3, 16, 64, seed=23)
    desc = L.grid_desc(cloud["grid"])
    n = 1 << 22                      # needs far more than the static workspace
    assert L.mpm_workspace_bytes(desc, n) > L.MPM_STATIC_WORKSPACE_BYTES
    buf = torch.zeros(n, dtype=torch.float32, device="cuda")
    p = L.Particles()
    p.n = n
    for i in range(3):
        p.x[i] = p.v[i] = buf.data_ptr()
    for i in range(9):
        p.C[i] = buf.data_ptr()
    p.m = buf.data_ptr()
    with pytest.raises(L.MPMError) as e:
        L.mpm_bin_static(desc, p, 0)
    assert e.value.code == L.MPM_E_WORKSPACE
    assert "static workspace" in str(e.value)
