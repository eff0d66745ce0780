"""CUDA path against the oracle at the workloads' full sizes.

- The 3D dam break (2,097,152 particles, 128^3 nodes): one full step, every
  output compared with the oracle (bit for bit in int64 mode, within the float
  tolerance in float-atomic mode).
- The clustered blobs (16,777,216 particles, 256^3 nodes) in the launch
  configuration the benchmark times (three sorted warm-up steps, then
  in-place steps with a sorted one every eighth: one of each checked, and a
  bin-order step),
  and the sphere (67,108,864 particles, 512^3 nodes) from its generated order:
  one step checked piece by piece: the whole permutation against the oracle's
  binning; the P2G grid through the exact conservation identities and, on
  sampled tiles, against the oracle's P2G of the particles that reach them;
  the whole velocity grid where there is mass against the oracle's grid update
  of the GPU's accumulators; and the G2P on sampled particles (found through
  their ids) against the oracle's G2P.
- The blobs as the benchmark's elastic row times them (the Neo-Hookean state),
  checked the same way with the stress fold and the F update.
- The blobs stepped by the fused kernel: the new state on sampled particles,
  the next accumulators in total and on sampled tiles, the read grid cleared.
"""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _system(cloud):
    n = cloud["x"].shape[1]
    return MPMSystem(cloud["grid"], n).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])


def _float_close(g, o):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    scale = np.abs(o).max(axis=-1, keepdims=True)
    return np.all(np.abs(g - o) <= np.maximum(1e-5 * np.abs(o), 1e-6 * scale))


@pytest.mark.parametrize("mode", [W.ACC_I64, W.ACC_F32])
def test_dambreak_full_size_step(mode):
    cloud = W.dambreak3d(acc_mode=mode)
    grid = cloud["grid"]
    assert cloud["x"].shape[1] == 2097152 and grid["n"][0] == 128
    sys = _system(cloud)
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(grid, cloud["x"])
    assert np.array_equal(key, okey) and np.array_equal(perm, operm) and np.array_equal(cnt, ocnt)
    sys.p2g()
    torch.cuda.synchronize()
    acc = sys.acc.cpu().numpy()
    if mode == W.ACC_I64:
        oacc, _, counts = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert counts.sum() == 0
        assert np.array_equal(acc, oacc)
        ovel = O.grid_update_fixed(grid, oacc)
    else:
        oacc, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert _float_close(acc, oacc)
        ovel = O.grid_update_float(grid, oacc)
    sys.grid_update()
    sys.g2p()
    x, v, C = sys.state()
    ox, ov, oC, moved = O.g2p(grid, ovel, cloud["x"], cloud["v"], cloud["C"])
    assert moved == valid
    if mode == W.ACC_I64:
        assert np.array_equal(sys.vel.cpu().numpy().view(np.uint32), ovel.view(np.uint32))
        for a, b in ((x, ox), (v, ov), (C, oC)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    else:
        assert np.max(np.abs(v - ov)) <= 1e-4 * (1 + np.abs(ov).max())
        assert np.max(np.abs(x - ox)) <= 1e-6


def _quantities(grid, x, v, m):
    """Per particle: Q_m = rint(m*S), Q_k = rint(fp32(m*S) * v_k) (fp32 products, ties to even)."""
    Mt = (m.astype(np.float32) * np.float32(2.0 ** grid["scale_log2"])).astype(np.float32)
    Q = [np.rint(Mt).astype(np.int64)]
    for k in range(grid["dim"]):
        Q.append(np.rint((Mt * v[k].astype(np.float32)).astype(np.float32)).astype(np.int64))
    return Q


def _check_step(sys, grid, n, n_tiles_sampled=6, out="sorted"):
    """One step of `sys` whose G2P writes `out` ("sorted", "bin_order" or
    "in_place"), checked piece by piece against the oracle (with the stress fold
    and the F update when the particles are elastic)."""
    x0, v0, C0 = sys.state()
    m0 = sys.m.cpu().numpy()
    ids0 = sys.id.cpu().numpy().astype(np.int64)
    elastic = sys.F is not None
    if elastic:
        F0, vol0 = sys.elastic_state()

    # binning: the whole permutation
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(grid, x0)
    assert np.array_equal(key, okey) and np.array_equal(perm, operm) and np.array_equal(cnt, ocnt)

    # P2G: exact conservation, and sampled tiles against the oracle
    sys.p2g()
    torch.cuda.synchronize()
    st = sys.status()
    assert st[L.ST_FLAGS] == 0 and st[L.ST_N_OUT_OF_RANGE] == 0
    acc = sys.acc.cpu().numpy()
    inside = perm[:valid].astype(np.int64)
    Q = _quantities(grid, x0[:, inside], v0[:, inside], m0[inside])
    for c in range(grid["dim"] + 1):
        assert int(acc[c].sum()) == int(Q[c].sum()), f"channel {c} not conserved"
    T, nn = grid["tile"], grid["n"][0]
    nt = (nn - 2 + T - 1) // T          # tiles per axis: base cells 0 .. n-3
    base = np.floor(x0.astype(np.float32) * np.float32(grid["inv_dx"]) - np.float32(0.5)).astype(np.int64)
    tiles = np.nonzero(cnt)[0]
    s = W.Stream(31, 31)
    pick = list(tiles[(s.bits(n_tiles_sampled) % np.uint64(tiles.size)).astype(np.int64)]) + [int(np.argmax(cnt))]
    for t in pick:
        o = np.array([t % nt, (t // nt) % nt, t // (nt * nt)]) * T
        # nodes of tile t's own block get shares only from base cells in [o - 2, o + T)
        near = np.all((base >= (o - 2)[:, None]) & (base < (o + T)[:, None]), axis=0)
        sub = np.nonzero(near)[0]
        Cs = C0[:, sub]
        if elastic:
            Cs, _ = O.stress_affine(grid, sys.material, x0[:, sub], C0[:, sub], F0[:, sub], vol0[sub], m0[sub])
        oacc, _, counts = O.p2g_fixed(grid, x0[:, sub], v0[:, sub], Cs, m0[sub])
        assert counts.sum() == 0
        gx, gy, gz = np.meshgrid(*(np.arange(oi, oi + T) for oi in o), indexing="ij")
        nodes = ((gz * nn + gy) * nn + gx).ravel()
        assert np.array_equal(acc[:, nodes], oacc[:, nodes]), f"tile {t}"

    # grid update: the whole velocity grid where there is mass
    sys.grid_update()
    torch.cuda.synchronize()
    vel = sys.vel.cpu().numpy()
    ovel = O.grid_update_fixed(grid, acc)
    massive = acc[0] != 0
    assert np.array_equal(vel[:, massive].view(np.uint32), ovel[:, massive].view(np.uint32))
    del acc, ovel
    assert not sys.acc.any().item(), "grid update must leave the accumulators zero"

    # G2P: sampled in-domain particles, found through their ids
    {"sorted": sys.g2p_sorted, "bin_order": sys.g2p_binned, "in_place": sys.g2p}[out]()
    x1, v1, C1 = sys.state()
    ids1 = sys.id.cpu().numpy().astype(np.int64)
    # the advective step bound: the largest term over the moved particles (all in the domain)
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    mv = inside if out == "in_place" else np.arange(valid)   # where the moved particles now sit
    assert speed == O.advective_speed(grid["dim"], grid["dx"], v1[:, mv], C1[:, mv])
    if out == "bin_order":   # out[j] = in[perm[j]]
        assert np.array_equal(ids1, ids0[perm.astype(np.int64)])
    if out == "in_place":
        assert np.array_equal(ids1, ids0)
    where = np.empty(n, dtype=np.int64)
    where[ids1] = np.arange(n)
    samp = inside[(W.Stream(32, 32).bits(20000) % np.uint64(inside.size)).astype(np.int64)]
    at = where[ids0[samp]]
    if elastic:
        ox, ov, oC, oF, moved = O.g2p_elastic(grid, vel, x0[:, samp], v0[:, samp], C0[:, samp], F0[:, samp])
        F1, vol1 = sys.elastic_state()
        assert np.array_equal(F1[:, at].view(np.uint32), oF.view(np.uint32))
        assert np.array_equal(vol1[at], vol0[samp])
    else:
        ox, ov, oC, moved = O.g2p(grid, vel, x0[:, samp], v0[:, samp], C0[:, samp])
    assert moved == samp.size
    for a, b in ((x1[:, at], ox), (v1[:, at], ov), (C1[:, at], oC)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_blobs_full_size_bench_configuration():
    """The benchmark's schedule: three sorted warm-up steps, then in-place steps
    with a sorted one every eighth; an in-place step and a sorted step checked,
    and a bin-order step between them."""
    cloud = W.blobs3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    assert n == 16777216 and grid["n"][0] == 256
    sys = _system(cloud).enable_sorted()
    del cloud
    for _ in range(3):                       # the warm-up steps
        sys.step_sorted()
    for _ in range(5):
        sys.step()
    _check_step(sys, grid, n, n_tiles_sampled=3, out="in_place")
    _check_step(sys, grid, n, n_tiles_sampled=2, out="bin_order")
    _check_step(sys, grid, n, n_tiles_sampled=3)


def test_sphere_full_size_step():
    """The 512^3, 67,108,864-particle sphere: one full step from the generated order."""
    cloud = W.sphere3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    assert n == 67108864 and grid["n"][0] == 512
    sys = _system(cloud).enable_sorted()
    del cloud
    _check_step(sys, grid, n, n_tiles_sampled=3)


def test_blobs_full_size_elastic():
    """The bench's elastic row: the blobs with F = I + N(0, 0.05), V0 = dx^3 and
    mu = lambda = 1e9, one sorted step checked after three steady-state steps."""
    cloud = W.blobs3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    el = W.with_elastic(cloud, seed=77, fsig=0.05, ppc=1.0, mu=1.0e9, lam=1.0e9)
    sys = _system(cloud).load_elastic(el["F"], el["vol"], el["material"]).enable_sorted()
    del cloud, el
    for _ in range(3):
        sys.step_sorted()
    _check_step(sys, grid, n, n_tiles_sampled=4)
    assert sys.status()[L.ST_N_DEGENERATE] == 0


def test_blobs_full_size_fused_step():
    """mpm_step_fused on the blobs in their steady-state order: the new state on
    sampled particles, the next accumulators on sampled tiles and in total, and
    the grid it read cleared."""
    cloud = W.blobs3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    sys = _system(cloud).enable_sorted()
    del cloud
    for _ in range(3):
        sys.step_sorted()
    sys.enable_fused()
    torch.cuda.synchronize()
    x0, v0, C0 = sys.state()
    m0 = sys.m.cpu().numpy()
    ids0 = sys.id.cpu().numpy().astype(np.int64)
    R = sys.acc.cpu().numpy()
    vel = O.grid_update_fixed(grid, R)
    sys.step_fused()
    torch.cuda.synchronize()
    st = sys.status()
    assert st[L.ST_FLAGS] == 0 and 0 < st[L.ST_N_ESCAPED] < n // 20   # tile changes: a few per cent
    assert not sys.acc2.any().item(), "the grid read must be cleared"
    x1, v1, C1 = sys.state()
    ids1 = sys.id.cpu().numpy().astype(np.int64)
    where = np.empty(n, dtype=np.int64)
    where[ids1] = np.arange(n)
    inside = np.nonzero(O.bin_particles(grid, x0)[0] != 0xFFFFFFFF)[0]
    samp = inside[(W.Stream(33, 33).bits(20000) % np.uint64(inside.size)).astype(np.int64)]
    ox, ov, oC, moved = O.g2p(grid, vel, x0[:, samp], v0[:, samp], C0[:, samp])
    at = where[ids0[samp]]
    for a, b in ((x1[:, at], ox), (v1[:, at], ov), (C1[:, at], oC)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # the next accumulators: exact totals and sampled tiles of the new positions
    Wacc = sys.acc.cpu().numpy()
    m1 = sys.m.cpu().numpy()
    key1, _, cnt1, _ = O.bin_particles(grid, x1)
    inside1 = np.nonzero(key1 != 0xFFFFFFFF)[0]
    Q = _quantities(grid, x1[:, inside1], v1[:, inside1], m1[inside1])
    for c in range(4):
        assert int(Wacc[c].sum()) == int(Q[c].sum()), f"channel {c} not conserved"
    T, nn = grid["tile"], grid["n"][0]
    nt = (nn - 2 + T - 1) // T
    base = np.floor(x1.astype(np.float32) * np.float32(grid["inv_dx"]) - np.float32(0.5)).astype(np.int64)
    tiles = np.nonzero(cnt1)[0]
    for t in tiles[(W.Stream(34, 34).bits(4) % np.uint64(tiles.size)).astype(np.int64)]:
        o = np.array([t % nt, (t // nt) % nt, t // (nt * nt)]) * T
        near = np.all((base >= (o - 2)[:, None]) & (base < (o + T)[:, None]), axis=0)
        sub = np.nonzero(near)[0]
        oacc, _, counts = O.p2g_fixed(grid, x1[:, sub], v1[:, sub], C1[:, sub], m1[sub])
        gx, gy, gz = np.meshgrid(*(np.arange(oi, oi + T) for oi in o), indexing="ij")
        nodes = ((gz * nn + gy) * nn + gx).ravel()
        assert np.array_equal(Wacc[:, nodes], oacc[:, nodes]), f"tile {t}"
