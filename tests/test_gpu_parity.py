"""CUDA path (through the C ABI) against the CPU oracle, on the same seeded inputs.

Fixed-point modes must match bit for bit: keys, permutation, tile counts,
accumulator grids, velocity grids and the particle state after G2P.  The
float-atomic mode must match within |g - o| <= max(1e-5 |o|, 1e-6 max|o|) per
node and channel.
"""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def make(cloud, n=None):
    n = cloud["x"].shape[1] if n is None else n
    return MPMSystem(cloud["grid"], max(n, 1)).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])


def acc_np(sys):
    torch.cuda.synchronize()
    return sys.acc.cpu().numpy()


def float_close(g, o):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    scale = np.abs(o).max(axis=-1, keepdims=True) if o.size else 0.0
    return np.all(np.abs(g - o) <= np.maximum(1e-5 * np.abs(o), 1e-6 * scale))


def with_outliers(cloud, k=11):
    x = cloud["x"].copy()
    n = x.shape[1]
    s = W.Stream(5, 5)
    idx = (s.bits(k) % np.uint64(n)).astype(np.int64)
    x[0, idx[: k // 2]] = -0.1
    x[-1, idx[k // 2:]] = 2.0
    cloud = dict(cloud)
    cloud["x"] = x
    return cloud


# --------------------------------------------------------------------------
# binning

@pytest.mark.parametrize("dim,n,count", [(2, 64, 5003), (3, 40, 4099), (3, 24, 257), (2, 130, 31),
                                         # whole spans of 128 keys only, and one key either side of a span
                                         (3, 32, 4096), (3, 32, 128), (3, 32, 127), (2, 64, 129)])
def test_bin_matches_oracle(dim, n, count):
    cloud = with_outliers(W.small_cloud(dim, count, n, seed=10 * dim + n, lo=0.02, hi=0.98))
    sys = make(cloud)
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(cloud["grid"], cloud["x"])
    st = sys.status()
    assert np.array_equal(key, okey)
    assert np.array_equal(perm, operm)
    assert np.array_equal(cnt, ocnt)
    assert st[L.ST_N_VALID] == valid and st[L.ST_N_OUTSIDE] == count - valid
    assert st[L.ST_N_RUNS] == n_runs(cloud["grid"], okey)


def n_runs(grid, key):
    """Maximal ranges of consecutive indices whose particles share a bucket."""
    key = np.asarray(key, dtype=np.uint64)
    if key.size == 0:
        return 0
    cpt_log2 = grid["dim"] * int(np.log2(grid["tile"]))
    b = np.where(key == 0xFFFFFFFF, np.uint64(1 << 40), key >> np.uint64(cpt_log2))   # outside: one bucket
    return 1 + int(np.count_nonzero(b[1:] != b[:-1]))


@pytest.mark.parametrize("where", ["tile", "outside"])
@pytest.mark.parametrize("cnt", [2000, 20000])
def test_bin_bucket_with_many_runs(where, cnt):
    """One bucket whose particles alternate with another bucket's, so every
    particle is a run of its own: 1,000 runs take the block sort in shared
    memory, 10,000 the block sort in global memory.  The permutation is
    still the stable sort."""
    s = W.Stream(77, 1)
    # base cells 16..19 on every axis: one 4^3 tile of a 32^3 grid
    a = ((16.5 + 3.99 * s.uniform24(3 * cnt)) / 32.0).reshape(3, cnt)
    if where == "tile":
        other = ((8.5 + 3.99 * s.uniform24(3 * cnt)) / 32.0).reshape(3, cnt)   # tile at cells 8..11
    else:
        other = np.full((3, cnt), 5.0)
    x = np.empty((3, 2 * cnt))
    x[:, 0::2] = a
    x[:, 1::2] = other
    n = x.shape[1]
    cloud = dict(x=x.astype(np.float32), v=np.zeros((3, n), np.float32), C=np.zeros((9, n), np.float32),
                 m=np.ones(n, np.float32), grid=W.small_cloud(3, 1, 32, seed=1)["grid"])
    sys = make(cloud)
    sys.bin()
    key, perm, cnt_t = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(cloud["grid"], cloud["x"])
    st = sys.status()
    assert st[L.ST_N_RUNS] == n_runs(cloud["grid"], okey) == n
    assert st[L.ST_N_LARGE_BUCKETS] == 2
    assert st[L.ST_N_BIG_TILES] == (2 if cnt > 8192 else 0)
    assert np.array_equal(key, okey) and np.array_equal(perm, operm) and np.array_equal(cnt_t, ocnt)


def test_bin_sorted_input_has_one_run_per_bucket():
    """Particles already in bin order: each bucket is one run."""
    cloud = W.small_cloud(3, 30000, 64, seed=5, lo=0.05, hi=0.95)
    okey, operm, ocnt, valid = O.bin_particles(cloud["grid"], cloud["x"])
    srt = {k: (v[..., operm] if k in ("x", "v", "C", "m") else v) for k, v in cloud.items()}
    sys = make(srt)
    sys.bin()
    key, perm, cnt_t = sys.bins_arrays()
    st = sys.status()
    assert np.array_equal(perm, np.arange(perm.size, dtype=np.uint32))
    assert st[L.ST_N_RUNS] == st[L.ST_N_ACTIVE] + (1 if st[L.ST_N_OUTSIDE] else 0)


@pytest.mark.parametrize("frac", [0.002, 0.03, 0.3])
def test_bin_nearly_sorted_input(frac):
    """Bin order with a fraction of the particles moved elsewhere (as after a
    step): buckets of a few long runs, some of more than 32."""
    cloud = W.small_cloud(3, 60000, 16, seed=6, lo=0.05, hi=0.95)   # 64 tiles, ~900 particles each
    okey, operm, _, _ = O.bin_particles(cloud["grid"], cloud["x"])
    srt = {k: (v[..., operm] if k in ("x", "v", "C", "m") else v) for k, v in cloud.items()}
    s = W.Stream(8, 8)
    n = srt["x"].shape[1]
    moved = (s.bits(int(frac * n)) % np.uint64(n)).astype(np.int64)
    srt["x"][:, moved] = (0.05 + 0.9 * s.uniform24(3 * moved.size)).reshape(3, -1).astype(np.float32)
    sys = make(srt)
    sys.bin()
    key, perm, cnt_t = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(srt["grid"], srt["x"])
    st = sys.status()
    assert np.array_equal(key, okey) and np.array_equal(perm, operm) and np.array_equal(cnt_t, ocnt)
    assert st[L.ST_N_RUNS] == n_runs(srt["grid"], okey)


def test_bin_tiny_and_empty():
    for count in (0, 1, 2, 33):
        cloud = W.small_cloud(3, count, 16, seed=3 + count)
        sys = make(cloud)
        sys.step()
        st = sys.status()
        assert st[L.ST_N_VALID] == count
        if count:
            key, perm, cnt = sys.bins_arrays()
            okey, operm, ocnt, valid = O.bin_particles(cloud["grid"], cloud["x"])
            assert np.array_equal(perm, operm)


# --------------------------------------------------------------------------
# P2G, grid update, G2P

def expected_path(grid, R):
    """The share path the bound selects: 0 when wmax*S*R*(1 + 2^-10) <= 2^22 - 4096."""
    wmax = 0.421875 if grid["dim"] == 3 else 0.5625
    return 0 if wmax * 2.0 ** grid["scale_log2"] * R * (1 + 2.0 ** -10) <= 4190208.0 else 1


def check_bound(sys, cloud, ost, vol=None):
    """Status of the bound against the oracle's: the flag, and on success R and the path."""
    st = sys.status()
    failed = bool(ost & 2)
    assert bool(st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)) == failed
    assert st[L.ST_N_OUT_OF_RANGE] == 0
    if not failed:
        R, _ = O.scatter_range(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol)
        assert np.uint32(st[L.ST_RANGE]) == np.array([R], np.float32).view(np.uint32)[0]
        assert st[L.ST_SHARE_PATH] == expected_path(cloud["grid"], R)
    return st


FIXED_CASES = [
    (2, W.ACC_I32, 20, 64, 6000),
    (2, W.ACC_I64, 20, 48, 3001),
    (3, W.ACC_I64, 19, 32, 6007),
    (3, W.ACC_I32, 19, 24, 2500),
    # shares past 2^22: the int64 share path
    (2, W.ACC_I64, 32, 48, 3001),
    (3, W.ACC_I64, 32, 32, 6007),
    (3, W.ACC_I64, 40, 24, 2000),
    (2, W.ACC_I32, 24, 96, 3000),
]


@pytest.mark.parametrize("dim,mode,scale,n,count", FIXED_CASES)
def test_step_fixed_bit_exact(dim, mode, scale, n, count):
    cloud = with_outliers(W.small_cloud(dim, count, n, seed=100 + dim * 7 + n, acc_mode=mode, scale_log2=scale,
                                        lo=0.05, hi=0.95, vsig=1.0, csig=2.0, mass_lo=0.5, mass_hi=1.5))
    cloud["grid"]["g"] = [0.0, -9.8, 0.0]
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    acc = acc_np(sys)
    oacc, ost, ocounts = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert np.array_equal(acc.astype(np.int64), oacc)
    check_bound(sys, cloud, ost)
    assert not ost & 2
    sys.grid_update()
    vel = sys.vel.cpu().numpy()
    ovel = O.grid_update_fixed(cloud["grid"], oacc)
    assert np.array_equal(vel.view(np.uint32), ovel.view(np.uint32))
    assert not acc_np(sys).any(), "grid update must leave the accumulators zero"
    sys.g2p()
    x, v, C = sys.state()
    ox, ov, oC, moved = O.g2p(cloud["grid"], ovel, cloud["x"], cloud["v"], cloud["C"])
    assert np.array_equal(x.view(np.uint32), ox.view(np.uint32))
    assert np.array_equal(v.view(np.uint32), ov.view(np.uint32))
    assert np.array_equal(C.view(np.uint32), oC.view(np.uint32))
    # the advective step bound over the particles G2P moved
    inside = O.bin_particles(cloud["grid"], cloud["x"])[0] != 0xFFFFFFFF
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    assert speed == O.advective_speed(dim, cloud["grid"]["dx"], ov[:, inside], oC[:, inside])


@pytest.mark.parametrize("dim,n,count", [(2, 64, 6000), (3, 32, 6007)])
def test_step_float_within_tolerance(dim, n, count):
    cloud = W.small_cloud(dim, count, n, seed=200 + dim, acc_mode=W.ACC_F32, scale_log2=0, lo=0.05, hi=0.95,
                          csig=2.0)
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    acc = acc_np(sys)
    oacc, _, _ = O.p2g_float(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert float_close(acc, oacc)
    sys.grid_update()
    sys.g2p()
    x, v, C = sys.state()
    ovel = O.grid_update_float(cloud["grid"], oacc)
    ox, ov, oC, _ = O.g2p(cloud["grid"], ovel, cloud["x"], cloud["v"], cloud["C"])
    tol = float_step_tolerance(cloud)
    assert np.max(np.abs(v - ov)) <= tol["v"]
    assert np.max(np.abs(C - oC)) <= tol["C"]
    assert np.max(np.abs(x - ox)) <= tol["x"]


def float_step_tolerance(cloud):
    """First-order bounds on how far the fp32-atomic step's particle state can sit from
    the oracle's, which sums the same fp32 terms in fp64 and rounds each sum once.

    Both sides form every term w m (v + C d) with the same fp32 operations, so they
    differ only in the sums: any order of fp32 additions of k terms errs by at most
    (k - 1) u sum|term| (u = 2^-24), and sum|term| <= M_i V over a node of mass M_i,
    V bounding |v_a| + 1.5 dx sum_b |C_ab| (+ |dt g|) over the particles.  So P/M at
    a node differs by at most (2k + 6) u V (P's and M's errors, the oracle's roundings,
    the division and the gravity add).  The gather is the same fp32 code on both sides:
    it passes the node error through with weights summing to one and adds at most
    two roundings per each of its 27 steps, so |dv| <= (2k + 60) u V.  C scales the
    same sum by 4 inv_dx with |a - f| <= 1.5 cells: |dC| <= 6 inv_dx (2k + 64) u V.
    x' = x + dt v' adds a rounding of x' on each side.  k is the most particles any
    node receives, counted from the bases; 1 % covers second-order terms."""
    g = cloud["grid"]
    dim, n_ = g["dim"], g["n"]
    x = np.asarray(cloud["x"], np.float32)
    fx = x * np.float32(1.0 / g["dx"]) if "inv_dx" not in g else x * np.float32(g["inv_dx"])
    inside = np.all((fx >= 0.5) & (fx < np.array(n_[:dim], np.float32)[:, None] - 1.5), axis=0)
    b = np.floor(fx[:, inside] - np.float32(0.5)).astype(np.int64)
    hits = np.zeros([k + 2 for k in n_[:dim]], np.int64)
    for off in np.ndindex(*(3,) * dim):
        np.add.at(hits, tuple(b[l] + off[l] for l in range(dim)), 1)
    k = int(hits.max()) + 2
    v = np.abs(np.asarray(cloud["v"], np.float64))
    C = np.abs(np.asarray(cloud["C"], np.float64)).reshape(dim, dim, -1)
    V = float((v + 1.5 * g["dx"] * C.sum(axis=1)).max()) + float(np.abs(O.dtg_of(g)).max())
    u = 2.0 ** -24
    dv = 1.01 * (2 * k + 60) * u * V
    return dict(v=dv, C=1.01 * 6.0 / g["dx"] * (2 * k + 64) * u * V,
                x=1.01 * (g["dt"] * dv + 2 * u * float(np.abs(x).max() + g["dt"] * V)))


def test_scrambled_input_order_gives_identical_results():
    cloud = W.small_cloud(3, 8192, 32, seed=301, scale_log2=19, lo=0.2, hi=0.8)
    a = make(cloud)
    a.step()
    base_acc = None
    xa, va, Ca = a.state()
    for (mul, add) in [(97, 13), (1, 4095), (5, 1)]:
        pi = W.scrambled_order(8192, mul, add)
        c2 = dict(cloud, x=cloud["x"][:, pi], v=cloud["v"][:, pi], C=cloud["C"][:, pi], m=cloud["m"][pi])
        b = make(c2)
        b.bin()
        b.p2g()
        acc_b = acc_np(b)
        if base_acc is None:
            a2 = make(cloud)
            a2.bin()
            a2.p2g()
            base_acc = acc_np(a2)
        assert np.array_equal(acc_b, base_acc)
        b.grid_update()
        b.g2p()
        xb, vb, Cb = b.state()
        assert np.array_equal(xb, xa[:, pi]) and np.array_equal(vb, va[:, pi]) and np.array_equal(Cb, Ca[:, pi])


def test_dense_single_cell_matches():
    s = W.Stream(9, 9)
    cnt = 5000
    x = np.full((3, cnt), 0.5 + 0.3 / 16, dtype=np.float64) + 0.2 / 16 * s.uniform24(3 * cnt).reshape(3, cnt)
    cloud = dict(x=x.astype(np.float32), v=s.normal(3 * cnt, 1.0).reshape(3, cnt).astype(np.float32),
                 C=s.normal(9 * cnt, 1.0).reshape(9, cnt).astype(np.float32), m=np.ones(cnt, np.float32),
                 grid=W.small_cloud(3, 1, 16, seed=1, scale_log2=19)["grid"])
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    oacc, _, _ = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert np.array_equal(acc_np(sys), oacc)


def test_full_slice_of_largest_shares():
    """1,024 particles on one point, each with the largest mass the share
    range allows: their centre-node shares sum past 2^31, so a halo kept in
    int32 must be flushed part-way through the slice."""
    cnt = 1024
    grid = W.small_cloud(3, 1, 32, seed=1, scale_log2=20)["grid"]
    x = np.full((3, cnt), 10.0 / 32.0, dtype=np.float32)   # base cell 9, f = 1: centre weight 0.75^3
    m = np.full(cnt, 9.4, dtype=np.float32)                # 0.421875 * 9.4 * 2^20 just under 2^22 - 4096
    cloud = dict(x=x, v=np.zeros((3, cnt), np.float32), C=np.zeros((9, cnt), np.float32), m=m, grid=grid)
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    oacc, ost, ocounts = O.p2g_fixed(grid, x, cloud["v"], cloud["C"], m)
    assert ocounts[1] == 0 and oacc[0].max() > 2 ** 31
    assert np.array_equal(acc_np(sys), oacc)


@pytest.mark.parametrize("mode", [W.ACC_I64, W.ACC_I32])
@pytest.mark.parametrize("bad", ["huge", "nan", "inf"])
def test_bound_failure_scatters_nothing(mode, bad):
    """One particle whose range breaks the accumulator bound: nothing at all is
    scattered (the grid stays zero) and the status reports the bound, as the oracle."""
    cloud = W.small_cloud(3, 3000, 24, seed=401, scale_log2=19, acc_mode=mode)
    if bad == "huge":
        cloud["m"][77] = 1e15
    elif bad == "nan":
        cloud["v"][1, 100] = np.nan
    else:
        cloud["C"][4, 2999] = np.inf
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    oacc, ost, ocounts = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert ost & 2 and ocounts[1] == 3000 and not oacc.any()
    check_bound(sys, cloud, ost)
    assert not acc_np(sys).any()


def test_one_large_particle_takes_the_wide_path():
    """At S = 2^19 a particle of mass 10^5 has shares far past 2^22: the bound still
    holds, the whole launch takes the int64 share path, and the grid is the oracle's."""
    cloud = W.small_cloud(3, 3000, 24, seed=402, scale_log2=19)
    cloud["m"][[5, 77, 2999]] = 1e5
    sys = make(cloud)
    sys.bin()
    sys.p2g()
    oacc, ost, _ = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert ost == 0 and np.abs(oacc).max() > 2 ** 31
    st = check_bound(sys, cloud, ost)
    assert st[L.ST_SHARE_PATH] == 1
    assert np.array_equal(acc_np(sys), oacc)


def test_int32_accumulator_bound_stops_before_any_scatter():
    """600 stencils over one node: at S = 2^22 the int32 form fails (600 * B > 2^31),
    at S = 2^10 it holds; both as the oracle decides."""
    cnt = 600
    s = W.Stream(4, 4)
    x = (0.5 + 0.01 * s.uniform24(2 * cnt)).reshape(2, cnt)
    for scale, fails in [(22, True), (10, False)]:
        cloud = W.small_cloud(2, cnt, 64, seed=1, acc_mode=W.ACC_I32, scale_log2=scale)
        cloud["x"] = x.astype(np.float32)
        sys = make(cloud)
        sys.bin()
        sys.p2g()
        oacc, ost, _ = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert bool(ost & 2) == fails
        st = check_bound(sys, cloud, ost)
        assert st[L.ST_MAX_NEIGHBOURS] == cnt == O.max_cover(cloud["grid"], cloud["x"])
        assert np.array_equal(acc_np(sys), oacc)


def test_range_records_replace_the_pass():
    """Steps whose bound takes its range from the previous P2G and G2P (no pass over
    v, C, m) give the same bits as steps with the pass; breaking the promise (v
    changed after the G2P) undoes that P2G's scatter and reports the bound."""
    cloud = W.small_cloud(3, 20000, 32, seed=404, scale_log2=19, lo=0.2, hi=0.8)
    a = make(cloud)
    b = make(cloud).use_range_records(False)
    a.step()
    b.step()
    a.use_range_records(True)
    for _ in range(3):
        a.bin()
        a.p2g()
        b.bin()
        b.p2g()
        assert np.array_equal(acc_np(a), acc_np(b))
        sa, sb = a.status(), b.status()
        assert sa[L.ST_FLAGS] == sb[L.ST_FLAGS] == 0
        assert sa[L.ST_RANGE] >= sb[L.ST_RANGE]
        for s in (a, b):
            s.grid_update()
            s.g2p()
        xa, va, Ca = a.state()
        xb, vb, Cb = b.state()
        assert np.array_equal(xa, xb) and np.array_equal(va, vb) and np.array_equal(Ca, Cb)
    # the promise broken: one particle's velocity raised after the G2P
    with torch.no_grad():
        a.v[0, 123] = 1e4
    a.bin()
    a.p2g()
    st = a.status()
    assert st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    assert st[L.ST_N_OUT_OF_RANGE] == 1
    assert not acc_np(a).any()
@pytest.mark.parametrize("name,kw", [
    ("mls2d", {}),
    ("dambreak3d", dict(n_particles=32768)),
    ("dambreak3d_float", dict(n_particles=32768, acc_mode=W.ACC_F32)),
    ("blobs3d", dict(n_particles=262144)),
    ("sphere3d", dict(n_particles=100000, n=128)),
])
def test_workload_step_matches_oracle(name, kw):
    builder = {"mls2d": W.mls2d, "dambreak3d": W.dambreak3d, "dambreak3d_float": W.dambreak3d,
               "blobs3d": W.blobs3d, "sphere3d": W.sphere3d}[name]
    cloud = builder(**kw)
    grid = cloud["grid"]
    sys = make(cloud)
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    okey, operm, ocnt, valid = O.bin_particles(grid, cloud["x"])
    assert np.array_equal(perm, operm)
    sys.p2g()
    acc = acc_np(sys)
    fixed = grid["acc_mode"] != W.ACC_F32
    if fixed:
        oacc, _, ocounts = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert ocounts.sum() == 0
        assert np.array_equal(acc.astype(np.int64), oacc)
        ovel = O.grid_update_fixed(grid, oacc)
    else:
        oacc, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
        assert float_close(acc, oacc)
        ovel = O.grid_update_float(grid, oacc)
    sys.grid_update()
    sys.g2p()
    x, v, C = sys.state()
    ox, ov, oC, _ = O.g2p(grid, ovel, cloud["x"], cloud["v"], cloud["C"])
    if fixed:
        assert np.array_equal(sys.vel.cpu().numpy().view(np.uint32), ovel.view(np.uint32))
        assert np.array_equal(x.view(np.uint32), ox.view(np.uint32))
        assert np.array_equal(v.view(np.uint32), ov.view(np.uint32))
        assert np.array_equal(C.view(np.uint32), oC.view(np.uint32))
    else:
        assert np.max(np.abs(v - ov)) <= 1e-4 * (1 + np.abs(ov).max())
        assert np.max(np.abs(x - ox)) <= 1e-6


SLICE = 1024   # particles per work item (a slice of one tile)


def cell_class(key, dim, tile):
    """Bank class of a base cell: its offset in the compact (tile+2)^dim halo, mod 32."""
    key = key.astype(np.int64)
    h, lg = tile + 2, int(np.log2(tile))
    lx, ly = key & (tile - 1), (key >> lg) & (tile - 1)
    lz = (key >> (2 * lg)) & (tile - 1) if dim == 3 else 0
    return (lx + h * ly + h * h * lz) & 31


def sorted_output_order(key, perm, tile_count, n_valid, dim=3, tile=4):
    """Where mpm_g2p_sorted puts each particle: slice by slice in bin order,
    each slice of more than 32 particles stably sorted by bank class and dealt
    out column by column over rounds of 32."""
    out = perm.astype(np.int64).copy()
    start = np.concatenate([[0], np.cumsum(tile_count.astype(np.int64))])
    for t in np.nonzero(tile_count)[0]:
        for first in range(0, int(tile_count[t]), SLICE):
            beg = int(start[t]) + first
            cnt = min(SLICE, int(tile_count[t]) - first)
            idx = perm[beg:beg + cnt].astype(np.int64)
            if cnt <= 32:            # one round: bin order kept
                continue
            srt = np.empty(cnt, np.int64)
            srt[np.argsort(cell_class(key[idx], dim, tile), kind="stable")] = np.arange(cnt)
            R = -(-cnt // 32)
            Lf = cnt - 32 * (R - 1)
            lane = np.where(srt < Lf * R, srt // R, Lf + (srt - Lf * R) // max(R - 1, 1))
            rho = np.where(srt < Lf * R, srt % R, (srt - Lf * R) % max(R - 1, 1))
            pos = rho * 32 + lane
            assert np.array_equal(np.sort(pos), np.arange(cnt))
            out[beg + pos] = idx
    assert int(start[-1]) == n_valid
    return out


def test_g2p_sorted_moves_particles_into_bin_order():
    cloud = with_outliers(W.small_cloud(3, 7001, 32, seed=502, scale_log2=19, lo=0.05, hi=0.95))
    sys = make(cloud).enable_sorted()
    sys.bin()
    key, perm, cnt = sys.bins_arrays()
    valid = int(sys.status()[L.ST_N_VALID])
    sys.p2g()
    sys.grid_update()
    sys.g2p_sorted()
    x, v, C = sys.state()
    m, ids = sys.m.cpu().numpy(), sys.id.cpu().numpy()
    oacc, _, _ = O.p2g_fixed(cloud["grid"], cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    ovel = O.grid_update_fixed(cloud["grid"], oacc)
    ox, ov, oC, moved = O.g2p(cloud["grid"], ovel, cloud["x"], cloud["v"], cloud["C"])
    assert moved == valid
    p = sorted_output_order(key, perm, cnt, valid)
    assert np.array_equal(ids, p)
    assert np.array_equal(x.view(np.uint32), ox[:, p].view(np.uint32))
    assert np.array_equal(v.view(np.uint32), ov[:, p].view(np.uint32))
    assert np.array_equal(C.view(np.uint32), oC[:, p].view(np.uint32))
    assert np.array_equal(m, cloud["m"][p])
    speed = np.array([sys.status()[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0]
    assert speed == O.advective_speed(3, cloud["grid"]["dx"], ov[:, p], oC[:, p])


@pytest.mark.parametrize("pinned", [True, False])
def test_step_host_equals_device_sorted_step(pinned):
    """From and back to host arrays: page-locked ones (copied by a kernel through their device view) and
    ordinary ones (one copy per array)."""
    cloud = W.small_cloud(3, 20000, 32, seed=501, scale_log2=19)
    a = make(cloud).enable_sorted()
    a.step_sorted()
    xa, va, Ca = a.state()
    ida = a.id.cpu().numpy()
    b = make(cloud).enable_sorted()
    if pinned:
        pin = lambda arr: torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
    else:
        pin = lambda arr: torch.from_numpy(np.array(arr, copy=True, order="C"))
    hx, hv, hC, hm = pin(cloud["x"]), pin(cloud["v"]), pin(cloud["C"]), pin(cloud["m"])
    hid = pin(np.arange(20000, dtype=np.int32))
    b.x.zero_()
    host = L.particles(hx, hv, hC, hm, hid)
    L.mpm_step_host(b.desc, host, b.parts, b.parts2, b.bins, b.acc, b.vel, b.dt, b.dtg)
    torch.cuda.synchronize()
    assert np.array_equal(hid.numpy(), ida)
    assert np.array_equal(hx.numpy(), xa) and np.array_equal(hv.numpy(), va) and np.array_equal(hC.numpy(), Ca)


def test_sorted_steps_track_the_in_place_steps():
    """Three sorted steps give, particle by particle (through the ids), the
    same state as three in-place steps."""
    cloud = W.small_cloud(3, 30000, 48, seed=503, scale_log2=19, lo=0.2, hi=0.8)
    a = make(cloud)
    b = make(cloud).enable_sorted()
    for _ in range(3):
        a.step()
        b.step_sorted()
    xa, va, Ca = a.state()
    xb, vb, Cb = b.state()
    ids = b.id.cpu().numpy().astype(np.int64)
    assert np.array_equal(xb, xa[:, ids]) and np.array_equal(vb, va[:, ids]) and np.array_equal(Cb, Ca[:, ids])


def test_permute_reorders_by_perm():
    cloud = W.small_cloud(3, 5000, 32, seed=601)
    a = make(cloud)
    a.bin()
    _, perm, _ = a.bins_arrays()
    out = make(cloud)
    L.mpm_permute(a.desc, a.parts, out.parts, a.bins)
    x, v, C = out.state()
    assert np.array_equal(x, cloud["x"][:, perm]) and np.array_equal(C, cloud["C"][:, perm])
    assert np.array_equal(out.m.cpu().numpy(), cloud["m"][perm])


# --------------------------------------------------------------------------
# the integer CIC transfer page

def _cic_sys(cfg):
    return MPMSystem(cfg["grid"], cfg["X"].shape[1]).load(cfg["X"], cfg["v"], None, cfg["m"])


def test_cic_int_grid_and_gather_match_oracle():
    cfg = W.cic_int()
    sys = _cic_sys(cfg)
    sys.p2g()
    acc = acc_np(sys)
    oacc, ok = O.cic_int_p2g(cfg["grid"], cfg["X"], cfg["m"], cfg["v"])
    assert ok and np.array_equal(acc, oacc)
    st = sys.status()
    assert st[L.ST_FLAGS] == 0
    sys.g2p()
    torch.cuda.synchronize()
    assert np.array_equal(sys.v.cpu().numpy(), O.cic_int_gather(cfg["grid"], cfg["X"], oacc))


def test_cic_int_all_scrambled_orders_identical_on_gpu():
    cfg = W.cic_int()
    oacc, _ = O.cic_int_p2g(cfg["grid"], cfg["X"], cfg["m"], cfg["v"])
    for a in range(1, 256, 2):
        pi = W.scrambled_order(256, a, 13)
        sys = MPMSystem(cfg["grid"], 256).load(cfg["X"][:, pi], cfg["v"][:, pi], None, cfg["m"][pi])
        sys.p2g()
        assert np.array_equal(acc_np(sys), oacc), a


def test_cic_int_bounds_line_scatters_nothing():
    cfg = W.cic_int()
    m = cfg["m"].copy()
    m[3] = 2 ** 40
    sys = MPMSystem(cfg["grid"], 256).load(cfg["X"], cfg["v"], None, m)
    sys.p2g()
    st = sys.status()
    assert st[L.ST_FLAGS] & (1 << L.MPM_E_BOUND)
    assert not acc_np(sys).any()
    X = cfg["X"].copy()
    X[1, 7] = 8 * 65536
    sys = MPMSystem(cfg["grid"], 256).load(X, cfg["v"], None, cfg["m"])
    sys.p2g()
    st = sys.status()
    assert st[L.ST_FLAGS] & (1 << L.MPM_E_DOMAIN) and st[L.ST_N_OUTSIDE] == 1
    assert not acc_np(sys).any()
