"""CUDA path against the oracle at the workloads' full sizes, every array compared.

The oracle's step is taken from the same state the GPU steps: single-threaded
(``oracle.oracle``) where it finishes in seconds, else the OpenMP build of the
oracle's own per-particle and per-node code (``oracle.cpu_omp``), which the CPU
tests pin bit for bit against the single-threaded oracle for any thread count.

- The 3D dam break (2,097,152 particles, 128^3 nodes) at S = 2^21 and at
  S = 2^32 (int64 shares) and in float-atomic mode: one step.
- The clustered blobs (16,777,216 particles, 256^3 nodes) in the launch
  configuration the benchmark times (three sorted warm-up steps, then in-place
  steps with a sorted one every eighth, the bound's range taken from the
  previous P2G and G2P): an in-place, a bin-order and a sorted step; and one
  step at S = 2^32.
- The sphere (67,108,864 particles, 512^3 nodes) from its generated order.
- The blobs as the benchmark's elastic row times them (the Neo-Hookean state).
- The blobs stepped by the fused kernel: the new state and the next accumulators.

Each checked step compares the whole permutation, keys and tile counts, the
whole accumulator grid, the velocity grid on every node the grid update
writes (every node of a block next to an occupied tile, which includes every
node with mass) and every particle's x, v and C (and F) bit for bit.
"""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import cpu_omp
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


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("mode,scale", [(W.ACC_I64, 21), (W.ACC_I64, 32), (W.ACC_F32, 0)])
def test_dambreak_full_size_step(mode, scale):
    cloud = W.dambreak3d(acc_mode=mode, scale_log2=scale)
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
        assert sys.status()[L.ST_SHARE_PATH] == (1 if scale == 32 else 0)
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
        assert np.array_equal(bits(sys.vel.cpu().numpy()), bits(ovel))
        for a, b in ((x, ox), (v, ov), (C, oC)):
            assert np.array_equal(bits(a), bits(b))
    else:
        # particles gather from an order-dependent fp32 grid: per entry, the
        # node tolerance carried through the gather's weights (they sum to one)
        assert np.max(np.abs(v - ov)) <= 1e-4 * (1 + np.abs(ov).max())
        assert np.max(np.abs(x - ox)) <= 1e-6


def _updated_nodes(grid, cnt):
    """Nodes mpm_grid_update writes: those of the node blocks (tile^dim nodes) next to a tile holding
    particles, block b receiving from tiles b - delta, delta in {0,1}^dim (the rest of the velocity grid
    is not read by any G2P of these particles and keeps what it held)."""
    T, n = grid["tile"], grid["n"][0]
    nt = (n - 2 + T - 1) // T
    nb = (n + T - 1) // T
    occ = (cnt.reshape(nt, nt, nt) > 0)          # [tz, ty, tx]
    act = np.zeros((nb, nb, nb), dtype=bool)
    for d in range(8):
        dz, dy, dx = (d >> 2) & 1, (d >> 1) & 1, d & 1
        lz, ly, lx = min(nt, nb - dz), min(nt, nb - dy), min(nt, nb - dx)
        act[dz:dz + lz, dy:dy + ly, dx:dx + lx] |= occ[:lz, :ly, :lx]
    b = np.arange(n) // T
    return act[b[:, None, None], b[None, :, None], b[None, None, :]].reshape(-1)


def _oracle_step(grid, x0, v0, C0, m0, F0=None, vol0=None, material=None):
    """The oracle's step from the given state: perm, key, tile counts, the P2G grid,
    the velocity grid and the new state of every particle in input order."""
    key, perm, cnt, valid = O.bin_particles(grid, x0)
    if F0 is None:
        ref = cpu_omp.step_fixed(grid, x0, v0, C0, m0)
        assert np.array_equal(ref["perm"], perm)
        p = perm.astype(np.int64)
        new = {}
        for k in ("x", "v", "C"):
            a = np.empty_like(ref[k])
            a[:, p] = ref[k]                  # column j of the OpenMP result is input particle perm[j]
            new[k] = a
        return dict(key=key, perm=perm, cnt=cnt, valid=valid, acc=ref["acc"], vel=ref["vel"],
                    counts=ref["counts"], **new)
    Cs, _ = O.stress_affine(grid, material, x0, C0, F0, vol0, m0)
    acc, _, counts = O.p2g_fixed(grid, x0, v0, Cs, m0)
    vel = O.grid_update_fixed(grid, acc)
    x1, v1, C1, F1, moved = O.g2p_elastic(grid, vel, x0, v0, C0, F0)
    return dict(key=key, perm=perm, cnt=cnt, valid=valid, acc=acc, vel=vel, counts=counts, x=x1, v=v1, C=C1,
                F=F1)


def _check_step(sys, grid, n, out="sorted"):
    """One step of `sys` whose G2P writes `out` ("sorted", "bin_order" or
    "in_place"), every output compared with the oracle's step from the same state."""
    x0, v0, C0 = sys.state()
    m0 = sys.m.cpu().numpy()
    ids0 = sys.id.cpu().numpy().astype(np.int64)
    elastic = sys.F is not None
    F0 = vol0 = None
    if elastic:
        F0, vol0 = sys.elastic_state()
    ref = _oracle_step(grid, x0, v0, C0, m0, F0, vol0, sys.material)
    assert ref["counts"].sum() == n - ref["valid"]        # no bound failure

    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    assert np.array_equal(key, ref["key"]) and np.array_equal(perm, ref["perm"])
    assert np.array_equal(cnt, ref["cnt"])

    sys.p2g()
    torch.cuda.synchronize()
    st = sys.status()
    assert st[L.ST_FLAGS] == 0 and st[L.ST_N_OUT_OF_RANGE] == 0
    assert np.array_equal(sys.acc.cpu().numpy(), ref["acc"])

    sys.grid_update()
    torch.cuda.synchronize()
    upd = _updated_nodes(grid, ref["cnt"])
    assert upd[ref["acc"][0] != 0].all()
    assert np.array_equal(bits(sys.vel.cpu().numpy()[:, upd]), bits(ref["vel"][:, upd]))
    assert not sys.acc.any().item(), "grid update must leave the accumulators zero"

    {"sorted": sys.g2p_sorted, "bin_order": sys.g2p_binned, "in_place": sys.g2p}[out]()
    x1, v1, C1 = sys.state()
    ids1 = sys.id.cpu().numpy().astype(np.int64)
    if out == "bin_order":   # out[j] = in[perm[j]]
        assert np.array_equal(ids1, ids0[perm.astype(np.int64)])
    if out == "in_place":
        assert np.array_equal(ids1, ids0)
    # every particle: GPU entry j holds the particle with id ids1[j], i.e. input particle where0[ids1[j]]
    where0 = np.empty(n, dtype=np.int64)
    where0[ids0] = np.arange(n)
    src = where0[ids1]
    for a, k in ((x1, "x"), (v1, "v"), (C1, "C")):
        assert np.array_equal(bits(a), bits(ref[k][:, src])), k
    if elastic:
        F1, vol1 = sys.elastic_state()
        assert np.array_equal(bits(F1), bits(ref["F"][:, src]))
        assert np.array_equal(vol1, vol0[src])
    assert np.array_equal(sys.m.cpu().numpy(), m0[src])
    # the advective step bound: the largest term over the moved (in-domain) particles
    moved = ref["perm"][:ref["valid"]].astype(np.int64)
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    assert speed == O.advective_speed(grid["dim"], grid["dx"], ref["v"][:, moved], ref["C"][:, moved])


def test_blobs_full_size_bench_configuration():
    """The benchmark's schedule: three sorted warm-up steps, then in-place steps
    with a sorted one every eighth and the bound's range from the records; an
    in-place step, a bin-order step and a sorted step each checked in full."""
    cloud = W.blobs3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    assert n == 16777216 and grid["n"][0] == 256
    sys = _system(cloud).enable_sorted()
    del cloud
    for _ in range(3):                       # the warm-up steps
        sys.step_sorted()
    sys.use_range_records(True)
    for _ in range(5):
        sys.step()
    _check_step(sys, grid, n, out="in_place")
    assert sys.status()[L.ST_SHARE_PATH] == 0
    _check_step(sys, grid, n, out="bin_order")
    _check_step(sys, grid, n)


def test_blobs_full_size_int64_shares():
    """The blobs at S = 2^32: every share takes the int64 path."""
    cloud = W.blobs3d(scale_log2=32)
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    sys = _system(cloud).enable_sorted()
    del cloud
    sys.step_sorted()
    _check_step(sys, grid, n, out="in_place")
    assert sys.status()[L.ST_SHARE_PATH] == 1


def test_sphere_full_size_step():
    """The 512^3, 67,108,864-particle sphere: one full step from the generated order."""
    cloud = W.sphere3d()
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    assert n == 67108864 and grid["n"][0] == 512
    sys = _system(cloud).enable_sorted()
    del cloud
    _check_step(sys, grid, n)


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
    _check_step(sys, grid, n)
    assert sys.status()[L.ST_N_DEGENERATE] == 0


def test_blobs_full_size_fused_step():
    """mpm_step_fused on the blobs in their steady-state order: every particle's
    new state, the whole next accumulator grid, and the grid it read cleared."""
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
    ref = _oracle_step(grid, x0, v0, C0, m0)
    assert np.array_equal(sys.acc.cpu().numpy(), ref["acc"])
    sys.step_fused()
    torch.cuda.synchronize()
    st = sys.status()
    assert st[L.ST_FLAGS] == 0 and 0 < st[L.ST_N_ESCAPED] < n // 20   # tile changes: a few per cent
    assert not sys.acc2.any().item(), "the grid read must be cleared"
    x1, v1, C1 = sys.state()
    ids1 = sys.id.cpu().numpy().astype(np.int64)
    where0 = np.empty(n, dtype=np.int64)
    where0[ids0] = np.arange(n)
    src = where0[ids1]
    for a, k in ((x1, "x"), (v1, "v"), (C1, "C")):
        assert np.array_equal(bits(a), bits(ref[k][:, src])), k
    # the next accumulators: the oracle's P2G of the new state (every node)
    m1 = sys.m.cpu().numpy()
    nxt = cpu_omp.step_fixed(grid, x1, v1, C1, m1)
    assert np.array_equal(sys.acc.cpu().numpy(), nxt["acc"])
