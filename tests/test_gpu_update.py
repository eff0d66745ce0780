"""G2P with the grid update applied on load (mpm_g2p_update, mpm_g2p_sorted_update)
against the separate calls (mpm_grid_update, then mpm_g2p or mpm_g2p_sorted), and
so against the oracle, whose step the separate calls match bit for bit: every
particle's new state bit for bit, the status words the G2P writes, and the
accumulators left zero (consumed, as the grid update leaves them)."""
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


def cloud_for(dim, mode, n, count, seed, state="plain", lo=0.05, hi=0.95):
    cloud = W.small_cloud(dim, count, n, seed=seed, acc_mode=mode, scale_log2=19 if dim == 3 else 20, lo=lo,
                          hi=hi, vsig=1.0, csig=2.0, mass_lo=0.5, mass_hi=1.5)
    cloud["grid"]["g"] = [0.0, -9.8, 0.0]
    if state == "elastic":
        cloud = W.with_elastic(cloud, seed=seed + 1)
    if state == "volume":
        cloud["grid"]["volume_channel"] = 1
        cloud = W.with_elastic(cloud, seed=seed + 1)
    x = cloud["x"].copy()
    if count > 20:
        x[0, :3] = -0.1                      # outside the domain
    cloud["x"] = x
    return cloud


def make(cloud, sorted_=False):
    n = cloud["x"].shape[1]
    s = MPMSystem(cloud["grid"], max(n, 1)).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    if "F" in cloud and not cloud["grid"].get("volume_channel"):
        s.load_elastic(cloud["F"], cloud["vol"], cloud["material"])
    if cloud["grid"].get("volume_channel"):
        s.load_volume(cloud["vol"])
    if sorted_:
        s.enable_sorted()
    return s


def same_state(a, b):
    xa, va, Ca = a.state()
    xb, vb, Cb = b.state()
    for u, w in ((xa, xb), (va, vb), (Ca, Cb)):
        assert np.array_equal(bits(u), bits(w))
    if a.F is not None:
        assert np.array_equal(bits(a.elastic_state()[0]), bits(b.elastic_state()[0]))
    if a.phi is not None:
        assert np.array_equal(bits(a.phi.cpu().numpy()), bits(b.phi.cpu().numpy()))
    sa, sb = a.status(), b.status()
    for w in (L.ST_MAX_SPEED, L.ST_G2P_RANGE, L.ST_N_VALID, L.ST_FLAGS):
        assert sa[w] == sb[w], w


CASES = [(3, W.ACC_I64, 32, 6007, "plain"), (3, W.ACC_I32, 24, 2500, "plain"), (2, W.ACC_I64, 64, 6000, "plain"),
         (2, W.ACC_I32, 48, 3001, "plain"), (3, W.ACC_I64, 21, 3000, "plain"), (3, W.ACC_I64, 19, 2000, "plain"),
         (2, W.ACC_I64, 45, 2000, "plain"), (3, W.ACC_I64, 32, 6007, "elastic"), (3, W.ACC_I64, 32, 6007, "volume"),
         (2, W.ACC_I32, 48, 3001, "volume")]


@pytest.mark.parametrize("dim,mode,n,count,state", CASES)
def test_g2p_update_matches_the_separate_calls(dim, mode, n, count, state):
    cloud = cloud_for(dim, mode, n, count, seed=9000 + 13 * dim + n + count, state=state)
    a, b = make(cloud), make(cloud)
    for _ in range(3):                     # three steps in a row: the grids must come back zero every time
        a.step_update()
        b.bin()
        b.p2g()
        b.grid_update()
        b.g2p()
        torch.cuda.synchronize()
        same_state(a, b)
        assert not a.acc.any().item(), "the accumulators must be consumed"
        assert not b.acc.any().item()


def test_g2p_update_matches_the_oracle_step():
    cloud = cloud_for(3, W.ACC_I64, 32, 6007, seed=9100)
    a = make(cloud)
    a.step_update()
    ref = O.step_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    x, v, C = a.state()
    for u, k in ((x, "x"), (v, "v"), (C, "C")):
        assert np.array_equal(bits(u), bits(ref[k]))


@pytest.mark.parametrize("dim,mode,n,count,state", [c for c in CASES if c[4] != "volume"][:6] +
                         [(3, W.ACC_I64, 32, 6007, "elastic"), (2, W.ACC_I64, 64, 6000, "volume")])
def test_g2p_sorted_update_matches_the_separate_calls(dim, mode, n, count, state):
    cloud = cloud_for(dim, mode, n, count, seed=9200 + 13 * dim + n + count, state=state)
    a, b = make(cloud, True), make(cloud, True)
    for k in range(3):
        a.step_sorted_update()
        b.step_sorted()
        torch.cuda.synchronize()
        same_state(a, b)
        assert np.array_equal(a.id.cpu().numpy(), b.id.cpu().numpy())
        assert np.array_equal(a.m.cpu().numpy(), b.m.cpu().numpy())
        assert not a.acc.any().item()


def test_g2p_update_on_a_dense_cell_and_many_slices():
    """Tiles of several work items each (slices of 1024): a block's count of readers
    spans every slice of its tiles."""
    s = W.Stream(9300, 1)
    cnt = 30000
    x = (0.45 + 0.1 * s.uniform24(3 * cnt)).reshape(3, cnt)
    cloud = dict(x=x.astype(np.float32), v=s.normal(3 * cnt, 1.0).reshape(3, cnt).astype(np.float32),
                 C=s.normal(9 * cnt, 1.0).reshape(9, cnt).astype(np.float32), m=np.ones(cnt, np.float32),
                 grid=W.small_cloud(3, 1, 32, seed=1, scale_log2=19)["grid"])
    a, b = make(cloud), make(cloud)
    for _ in range(2):
        a.step_update()
        b.step()
        torch.cuda.synchronize()
        same_state(a, b)
        assert not a.acc.any().item()


@pytest.mark.parametrize("count", [0, 1, 33])
def test_g2p_update_edge_inputs(count):
    cloud = cloud_for(3, W.ACC_I64, 16, count, seed=9400 + count)
    a, b = make(cloud), make(cloud)
    a.step_update()
    b.step()
    torch.cuda.synchronize()
    if count:
        same_state(a, b)
    assert not a.acc.any().item()
    # every particle outside the domain: left unchanged
    k = max(count, 1)
    far = dict(grid=cloud["grid"], x=np.full((3, k), 2.0, np.float32), v=np.ones((3, k), np.float32),
               C=np.zeros((9, k), np.float32), m=np.ones(k, np.float32))
    c = make(far)
    c.step_update()
    torch.cuda.synchronize()
    x, v, _ = c.state()
    assert np.array_equal(x, far["x"]) and np.array_equal(v, far["v"])


def test_g2p_update_rejects_float_mode():
    cloud = W.small_cloud(3, 100, 16, seed=1, acc_mode=W.ACC_F32, scale_log2=0)
    a = make(cloud)
    a.bin()
    a.p2g()
    with pytest.raises(L.MPMError):
        a.g2p_update()


@pytest.mark.parametrize("state", ["plain", "elastic", "volume"])
def test_bin_with_keys_from_g2p_equals_computed_bin(state):
    """In-place steps whose G2P writes the next keys and their histogram (bins.next_keys) and whose binning
    takes them (MPM_BIN_KEYS_FROM_G2P) give, step after step, the keys, permutation, tile counts, status
    words and particle state of steps that compute them (particles outside the domain included)."""
    cloud = cloud_for(3, W.ACC_I64, 32, 6007, seed=9500, state=state)
    a, b = make(cloud), make(cloud)
    b.use_next_keys(True)
    for step in range(4):
        a.bin()
        b.bin(keys_from_g2p=step > 0)
        torch.cuda.synchronize()
        ka, pa, ca = a.bins_arrays()
        kb, pb, cb = b.bins_arrays()
        assert np.array_equal(ka, kb) and np.array_equal(pa, pb) and np.array_equal(ca, cb), step
        sa, sb = a.status(), b.status()
        for w in range(L.ST_BIN_WORDS):
            assert sa[w] == sb[w], (step, w)
        a.p2g()
        b.p2g()
        a.g2p_update()
        b.g2p_update()
        torch.cuda.synchronize()
        same_state(a, b)


def test_next_keys_refused_outside_int64():
    cloud = cloud_for(3, W.ACC_I32, 24, 2500, seed=9600)
    a = make(cloud).use_next_keys(True)
    a.bin()
    a.p2g()
    with pytest.raises(L.MPMError):
        a.g2p_update()
    with pytest.raises(L.MPMError):
        a.bin(keys_from_g2p=True)
