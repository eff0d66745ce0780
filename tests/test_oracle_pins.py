"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own arithmetic: closed forms
(the quadratic B-spline, its moments), exact rational arithmetic (Python
``Fraction`` with round-half-even), brute-force all-nodes loops in fp64 with
the B-spline written as a function of distance, library routines (numpy's
stable argsort), invariants (conservation, order independence, APIC's
reproduction of affine fields) and the values the integer-transfer page prints.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from material_point_particle_gb300 import workloads as W
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# independent helpers

def phi2(r):
    """Cardinal quadratic B-spline of the distance r (in cells), fp64."""
    r = np.abs(np.asarray(r, dtype=np.float64))
    return np.where(r < 0.5, 0.75 - r * r, np.where(r < 1.5, 0.5 * (1.5 - r) ** 2, 0.0))


def node_coords(grid):
    dim = grid["dim"]
    axes = [np.arange(grid["n"][l]) for l in range(dim)]
    mesh = np.meshgrid(*axes[::-1], indexing="ij")[::-1]  # node index (k*n1 + j)*n0 + i
    return np.stack([m.ravel() for m in mesh]).astype(np.float64)  # [dim, nodes]


def brute_force_p2g(grid, x, v, C, m):
    """All nodes x all particles in fp64: mass and APIC momentum m w (v + C (x_i - x_p))."""
    dim = grid["dim"]
    X = node_coords(grid)
    dx = float(grid["dx"])
    xi = x.astype(np.float64) * float(grid["inv_dx"])
    nodes = X.shape[1]
    mass = np.zeros(nodes)
    mom = np.zeros((dim, nodes))
    absterm = np.zeros(nodes)
    for p in range(x.shape[1]):
        w = np.ones(nodes)
        for l in range(dim):
            w *= phi2(X[l] - xi[l, p])
        dvec = (X - xi[:, p:p + 1]) * dx
        Cp = C[:, p].astype(np.float64).reshape(dim, dim)
        vel = v[:, p:p + 1].astype(np.float64) + Cp @ dvec
        mass += m[p] * w
        mom += m[p] * w * vel
        absterm += np.abs(m[p] * w) * (1.0 + np.abs(vel).sum(axis=0))
    return mass, mom, absterm


def rne_fraction(fr: Fraction) -> int:
    return round(fr)  # Fraction.__round__ rounds half to even


# --------------------------------------------------------------------------
# B-spline weights (tensor-core PIC page, shape functions Eq. 12: non-negative,
# partition of unity; the quadratic moments are textbook identities)

def test_weights_closed_form_and_moments():
    s = W.Stream(12345, 1)
    f = (0.5 + s.uniform24(1_000_000)).astype(np.float32)
    f = np.concatenate([f, np.float32([0.5, 1.0, np.nextafter(np.float32(1.5), np.float32(0))])])
    w = O.quadratic_weights_many(f).astype(np.float64)
    fd = f.astype(np.float64)
    a = np.arange(3, dtype=np.float64)[None, :]
    e = a - fd[:, None]
    assert np.all(w >= 0.0)
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-6
    assert np.max(np.abs((w * e).sum(axis=1))) <= 1e-6
    assert np.max(np.abs((w * e * e).sum(axis=1) - 0.25)) <= 1e-6
    ref = phi2(e)
    assert np.max(np.abs(w - ref)) <= 2e-7


# --------------------------------------------------------------------------
# binning: keys name the stencil base cell; perm is the stable counting sort
# by tile ("Particle Worlds, part 3", Step 3: counting sort)

@pytest.mark.parametrize("dim,n,tile", [(2, 40, 8), (3, 24, 4), (3, 21, 4)])
def test_bin_is_stable_sort_of_base_cells(dim, n, tile):
    cloud = W.small_cloud(dim, 3000, n, seed=11 + dim + n, lo=-0.05, hi=1.05, tile=tile)
    grid, x = cloud["grid"], cloud["x"]
    key, perm, cnt, valid = O.bin_particles(grid, x)
    xi = x.astype(np.float64) * float(np.float32(grid["inv_dx"]))
    inside = np.all((xi >= 0.5) & (xi < np.array(grid["n"][:dim])[:, None] - 1.5), axis=0)
    assert valid == int(inside.sum())
    assert np.all(key[~inside] == 0xFFFFFFFF)
    # decode key -> base cell and check that the particle lies in [b+0.5, b+1.5)
    T = tile
    ntl = [(grid["n"][l] - 2 + T - 1) // T for l in range(dim)]
    k = key[inside].astype(np.int64)
    local, tid = k % (T ** dim), k // (T ** dim)
    b = np.zeros((dim, k.size), dtype=np.int64)
    for l in range(dim):
        b[l] = (tid % ntl[l]) * T + (local % T)
        tid //= ntl[l]
        local //= T
    fr = xi[:, inside] - b
    assert np.all((fr >= 0.5) & (fr < 1.5))
    assert np.all((b >= 0) & (b <= np.array(grid["n"][:dim])[:, None] - 3))
    # perm: numpy's stable argsort of the tile ids of the in-domain particles
    # (ties in index order), then the out-of-domain ones in index order
    idx = np.nonzero(inside)[0]
    tile_of = key[idx].astype(np.int64) // (T ** dim)
    expect = np.concatenate([idx[np.argsort(tile_of, kind="stable")], np.nonzero(~inside)[0]])
    assert np.array_equal(perm.astype(np.int64), expect)
    assert np.array_equal(cnt.astype(np.int64),
                          np.bincount(key[idx] // (T ** dim), minlength=cnt.size))


# --------------------------------------------------------------------------
# fixed-point P2G against brute force, conservation and order independence

@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("scale_log2", [18, 32])
def test_p2g_fixed_matches_brute_force(dim, scale_log2):
    n = 8
    cloud = W.small_cloud(dim, 48, n, seed=100 + dim, lo=0.2, hi=0.8, vsig=1.0, csig=3.0,
                          scale_log2=scale_log2, mass_lo=0.5, mass_hi=2.0)
    grid = cloud["grid"]
    acc, st, counts = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert st == 0 and counts.sum() == 0
    S = 2.0 ** grid["scale_log2"]
    mass, mom, absterm = brute_force_p2g(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    touched = np.zeros(mass.size)
    xi = cloud["x"].astype(np.float64) * grid["inv_dx"]
    X = node_coords(grid)
    for p in range(xi.shape[1]):
        inside = np.ones(mass.size, dtype=bool)
        for l in range(dim):
            inside &= np.abs(X[l] - xi[l, p]) < 1.5
        touched += inside
    tol = (13.5 * touched + 1.0) / S + 2e-6 * absterm
    assert np.all(np.abs(acc[0] / S - mass) <= tol)
    for k in range(dim):
        assert np.all(np.abs(acc[1 + k] / S - mom[k]) <= tol)
    # the affine term is large here: dropping it would fail the bound by far
    assert np.max(np.abs(mom)) > 0 and np.max(absterm) > 0


@pytest.mark.parametrize("dim", [2, 3])
def test_p2g_float_matches_brute_force(dim):
    n = 8
    cloud = W.small_cloud(dim, 48, n, seed=200 + dim, lo=0.2, hi=0.8, vsig=1.0, csig=3.0,
                          acc_mode=W.ACC_F32, scale_log2=0, mass_lo=0.5, mass_hi=2.0)
    grid = cloud["grid"]
    acc, st, counts = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    mass, mom, absterm = brute_force_p2g(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    tol = 2e-6 * absterm + 1e-12
    assert np.all(np.abs(acc[0] - mass) <= tol)
    for k in range(dim):
        assert np.all(np.abs(acc[1 + k] - mom[k]) <= tol)


@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("scale_log2", [17, 32])
def test_grid_totals_equal_particle_totals(dim, scale_log2):
    cloud = W.small_cloud(dim, 4000, 32, seed=300 + dim, vsig=2.0, csig=1.0, scale_log2=scale_log2,
                          mass_lo=0.25, mass_hi=3.0)
    grid = cloud["grid"]
    acc, st, counts = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert st == 0
    S = np.float32(2.0 ** grid["scale_log2"])
    Mt = cloud["m"].astype(np.float32) * S
    # particle totals Q: rint of the fp32 scaled mass and of its fp32 product with v
    Qm = sum(int(q) for q in np.rint(Mt.astype(np.float64)))
    assert int(acc[0].sum()) == Qm
    for k in range(dim):
        Qk = (Mt * cloud["v"][k].astype(np.float32)).astype(np.float32)
        assert int(acc[1 + k].sum()) == sum(int(q) for q in np.rint(Qk.astype(np.float64)))


@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("scale_log2", [19, 32])
def test_scrambled_orders_give_identical_grids(dim, scale_log2):
    cloud = W.small_cloud(dim, 2048, 24, seed=400 + dim, scale_log2=scale_log2)
    grid = cloud["grid"]
    base, _, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    for a, b in [(97, 13), (1, 13), (1023, 5), (3, 2047)]:
        pi = W.scrambled_order(2048, a, b)
        acc, _, _ = O.p2g_fixed(grid, cloud["x"][:, pi], cloud["v"][:, pi], cloud["C"][:, pi],
                                cloud["m"][pi])
        assert np.array_equal(acc, base)


def test_out_of_domain_particles_are_counted_not_scattered():
    cloud = W.small_cloud(3, 64, 16, seed=501, scale_log2=19)
    grid = cloud["grid"]
    x, v, C, m = cloud["x"].copy(), cloud["v"].copy(), cloud["C"].copy(), cloud["m"].copy()
    x[0, 3] = 0.0            # below the lowest stencil
    x[1, 7] = 1.0            # above the highest
    x[2, 9] = np.nan
    v[1, 7] = np.inf         # outside the domain: its range does not enter the bound
    acc, st, counts = O.p2g_fixed(grid, x, v, C, m)
    assert st == 1 and counts[0] == 3 and counts[1] == 0
    keep = np.ones(64, dtype=bool)
    keep[[3, 7, 9]] = False
    ref, st2, _ = O.p2g_fixed(grid, x[:, keep], v[:, keep], C[:, keep], m[keep])
    assert st2 == 0 and np.array_equal(acc, ref)


# --------------------------------------------------------------------------
# the bound before any scatter ("particle to grid transfer in checked integer
# arithmetic", the program: the bounds line runs first; if it fails nothing is
# scattered)

@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("scale_log2", [20, 32, 40])
def test_bound_covers_every_particles_shares(dim, scale_log2):
    """A particle's shares of each channel sum in absolute value to at most
    S*R_p*(1 + 2^-10) + 28: each particle scattered alone, its grid holds exactly its
    shares.  C is large, so the affine term dominates most particles' ranges; the
    first 20 have C = 0, where the bound is tight on their largest momentum channel."""
    cloud = W.small_cloud(dim, 200, 10, seed=600 + dim, lo=0.25, hi=0.75, vsig=3.0, csig=40.0,
                          scale_log2=scale_log2, mass_lo=0.1, mass_hi=4.0)
    cloud["C"][:, :20] = 0.0
    grid = cloud["grid"]
    S = 2.0 ** scale_log2
    worst = 0.0
    for p in range(200):
        sl = slice(p, p + 1)
        acc, st, _ = O.p2g_fixed(grid, cloud["x"][:, sl], cloud["v"][:, sl], cloud["C"][:, sl],
                                 cloud["m"][sl])
        assert st == 0
        R, valid = O.scatter_range(grid, cloud["x"][:, sl], cloud["v"][:, sl], cloud["C"][:, sl],
                                   cloud["m"][sl])
        assert valid == 1
        bound = S * R * (1 + 2.0 ** -10) + 28
        for c in range(dim + 1):
            total = sum(abs(int(t)) for t in acc[c])
            assert total <= bound
            worst = max(worst, total / bound)
    assert worst > 0.99     # the bound is tight for some particle and channel


def test_bound_failure_scatters_nothing():
    cloud = W.small_cloud(3, 64, 16, seed=502, scale_log2=32)
    grid = cloud["grid"]
    x, v, C, m = cloud["x"], cloud["v"].copy(), cloud["C"], cloud["m"].copy()
    acc, st, counts = O.p2g_fixed(grid, x, v, C, m)
    assert st == 0 and acc.any()
    for bad in ("inf", "nan", "huge"):
        v2, m2 = v.copy(), m.copy()
        if bad == "inf":
            v2[1, 12] = np.inf
        elif bad == "nan":
            m2[30] = np.nan
        else:
            m2[11] = 1e15       # 64 * 1e15 * |v| * 2^32 > 2^62
        acc, st, counts = O.p2g_fixed(grid, x, v2, C, m2)
        assert st == 2 and counts[0] == 0 and counts[1] == 64
        assert not acc.any()


def test_int64_bound_on_the_integer_pages_magnitudes():
    """The integer-transfer page's workload magnitudes (256 particles, m <= 1000,
    |v| <= 1000; its bounds line: 256 * 1000 * 1000 fits int64) carried over to the
    fp32 path with C = 0: R = max |m| * max(1, |v|) = 10^6 exactly, so the int64 form
    256 * (S * 10^6 * (1 + 2^-10) + 28) <= 2^62 holds up to S = 2^34 (4.40e18) and
    fails at 2^35 (8.80e18), by hand."""
    cfg = W.cic_int()
    X, mi, vi = cfg["X"], cfg["m"], cfg["v"]
    x = ((X.astype(np.float64) / 65536.0 + 0.5) / 10.0).astype(np.float32)     # inside a 10-node grid
    v = vi.astype(np.float32)
    m = mi.astype(np.float32)
    v[0, 0], m[0] = 1000.0, 1000.0                   # make the maxima exact
    C = np.zeros((4, 256), np.float32)
    for s_log2, ok in [(32, True), (34, True), (35, False)]:
        grid = W.small_cloud(2, 1, 10, seed=1, scale_log2=s_log2)["grid"]
        R, valid = O.scatter_range(grid, x, v, C, m)
        assert R == 1.0e6 and valid == 256
        total = 256 * (2.0 ** s_log2 * 1.0e6 * (1 + 2.0 ** -10) + 28)
        assert (total <= 2.0 ** 62) == ok
        assert O.bound_ok(grid, R, valid) == ok
        acc, st, counts = O.p2g_fixed(grid, x, v, C, m)
        assert (st == 0) == ok and acc.any() == ok


def test_int32_bound_counts_stencils_per_node():
    """int32 accumulators use the neighbourhood form: the most stencils covering one
    node (counted here by brute force over all nodes) times the per-particle bound.
    Just inside the int32 limit the grid holds the exact sums (checked against the
    int64 grid); just outside, nothing is scattered."""
    n = 12
    cloud = W.small_cloud(2, 300, n, seed=610, lo=0.3, hi=0.45, vsig=0.5, csig=0.2,
                          acc_mode=W.ACC_I32, scale_log2=20)
    grid = cloud["grid"]
    x, v, C, m = cloud["x"], cloud["v"], cloud["C"], cloud["m"]
    xi = x.astype(np.float64) * grid["inv_dx"]
    X = node_coords(grid)
    cover = np.zeros(X.shape[1], dtype=np.int64)
    for p in range(x.shape[1]):
        inside = np.ones(X.shape[1], dtype=bool)
        for l in range(2):
            b = np.floor(xi[l, p] - 0.5)
            inside &= (X[l] >= b) & (X[l] <= b + 2)
        cover += inside
    assert O.max_cover(grid, x) == cover.max()
    R, valid = O.scatter_range(grid, x, v, C, m)
    # the largest scale whose bound fits int32, then one more bit
    s_fit = max(s for s in range(0, 31)
                if cover.max() * (2.0 ** s * R * (1 + 2.0 ** -10) + 28) <= 2 ** 31 - 1024)
    for s_log2, ok in [(s_fit, True), (s_fit + 1, False)]:
        g32 = dict(grid, scale_log2=s_log2)
        acc, st, counts = O.p2g_fixed(g32, x, v, C, m)
        assert (st == 0) == ok
        if ok:
            g64 = dict(g32, acc_mode=W.ACC_I64)
            ref, _, _ = O.p2g_fixed(g64, x, v, C, m)
            assert np.array_equal(acc, ref) and np.abs(ref).max() < 2 ** 31
        else:
            assert not acc.any() and counts[1] == valid


# --------------------------------------------------------------------------
# grid update: hand-made nodes (implementation guide 2.1 / 3.3.2 sign test)

def test_grid_update_cases():
    grid = W.small_cloud(3, 1, 10, seed=1)["grid"]
    grid["dt"] = float(np.float32(0.5))
    grid["g"] = [0.0, -2.0, 0.0]
    nodes = 1000
    acc = np.zeros((4, nodes), dtype=np.int64)

    def idx(i, j, k):
        return (k * 10 + j) * 10 + i

    acc[:, idx(5, 5, 5)] = [4, 8, -4, 2]      # v = (2, -1, 0.5) + (0, -1, 0)
    acc[:, idx(1, 5, 5)] = [2, -2, 0, 0]      # x < 3 and v_x < 0: stopped
    acc[:, idx(1, 6, 5)] = [2, 2, 0, 0]       # moving away from the wall: kept
    acc[:, idx(8, 5, 5)] = [2, 2, 0, 0]       # x > n-1-3 and v_x > 0: stopped
    acc[:, idx(4, 2, 4)] = [2, 0, 0, 0]       # y near floor, gravity pulls down: stopped
    acc[:, idx(4, 4, 4)] = [0, 5, 5, 5]       # empty node: zero
    vel = O.grid_update_fixed(grid, acc)
    assert list(vel[:, idx(5, 5, 5)]) == [2.0, -2.0, 0.5]
    assert list(vel[:, idx(1, 5, 5)]) == [0.0, -1.0, 0.0]
    assert list(vel[:, idx(1, 6, 5)]) == [1.0, -1.0, 0.0]
    assert list(vel[:, idx(8, 5, 5)]) == [0.0, -1.0, 0.0]
    assert list(vel[:, idx(4, 2, 4)]) == [0.0, 0.0, 0.0]
    assert list(vel[:, idx(4, 4, 4)]) == [0.0, 0.0, 0.0]
    assert np.count_nonzero(vel) == 7


# --------------------------------------------------------------------------
# G2P: quadratic B-splines reproduce affine fields; APIC recovers the gradient

@pytest.mark.parametrize("dim", [2, 3])
def test_g2p_reproduces_affine_velocity_field(dim):
    n = 16
    cloud = W.small_cloud(dim, 500, n, seed=600 + dim, lo=0.15, hi=0.85)
    grid = cloud["grid"]
    s = W.Stream(77, dim)
    A = s.normal(dim * dim, 1.0).reshape(dim, dim)
    c = s.normal(dim, 1.0)
    X = node_coords(grid) * grid["dx"]
    vel = (A @ X + c[:, None]).astype(np.float32)
    grid["dt"] = float(np.float32(1e-3))
    x2, v2, C2, moved = O.g2p(grid, vel, cloud["x"])
    assert moved == 500
    xp = cloud["x"].astype(np.float64)
    vexp = A @ xp + c[:, None]
    assert np.max(np.abs(v2 - vexp)) <= 2e-5
    assert np.max(np.abs(C2 - A.reshape(dim * dim, 1))) <= 2e-3
    assert np.max(np.abs(x2 - (xp + grid["dt"] * v2.astype(np.float64)))) <= 1e-6


@pytest.mark.parametrize("mode", ["fixed", "float"])
def test_single_particle_apic_round_trip(mode):
    """P2G -> grid update -> G2P of one particle returns its v and C (APIC is
    exact for affine velocity fields; no gravity, no walls nearby)."""
    dim = 3
    grid = W.small_cloud(3, 1, 32, seed=1, scale_log2=20)["grid"]
    grid["g"] = [0.0, 0.0, 0.0]
    if mode == "float":
        grid["acc_mode"] = W.ACC_F32
    s = W.Stream(99, 3)
    for trial in range(20):
        x = (0.3 + 0.4 * s.uniform24(3)).astype(np.float32).reshape(3, 1)
        v = s.normal(3, 1.0).astype(np.float32).reshape(3, 1)
        C = s.normal(9, 2.0).astype(np.float32).reshape(9, 1)
        m = np.float32([1.0])
        if mode == "fixed":
            acc, st, _ = O.p2g_fixed(grid, x, v, C, m)
            vel = O.grid_update_fixed(grid, acc)
            tol_v, tol_c = 1e-4, 2e-2
        else:
            acc, st, _ = O.p2g_float(grid, x, v, C, m)
            vel = O.grid_update_float(grid, acc)
            tol_v, tol_c = 1e-5, 2e-3
        assert st == 0
        x2, v2, C2, moved = O.g2p(grid, vel, x)
        assert moved == 1
        assert np.max(np.abs(v2 - v)) <= tol_v * (1 + np.abs(v).max())
        assert np.max(np.abs(C2 - C)) <= tol_c * (1 + np.abs(C).max())


def test_step_conserves_momentum_without_gravity_or_walls():
    cloud = W.small_cloud(3, 3000, 32, seed=701, lo=0.3, hi=0.7, scale_log2=19)
    grid = cloud["grid"]
    out = O.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    p0 = (cloud["m"][None, :].astype(np.float64) * cloud["v"]).sum(axis=1)
    p1 = (cloud["m"][None, :].astype(np.float64) * out["v"]).sum(axis=1)
    assert np.max(np.abs(p1 - p0)) <= 1e-3 * np.abs(cloud["v"]).sum() / 3000 * 10


# --------------------------------------------------------------------------
# the integer CIC transfer page

def test_rdiv_is_round_half_even_division():
    s = W.Stream(2024, 9)
    raw = s.bits(4000)
    qs = (raw[:2000].astype(np.int64) >> np.int64(20)) - (1 << 42)
    Fs = (raw[2000:] % np.uint64(65536)).astype(np.int64)
    cases = list(zip(qs.tolist(), Fs.tolist()))
    cases += [(1, 32768), (3, 32768), (-1, 32768), (-3, 32768), (5, 0), (-7, 65535), (0, 12345),
              (2**46, 65535), (-(2**46), 65535)]
    for q, F in cases:
        far = O.rdiv(q * F, 65536)
        assert far == rne_fraction(Fraction(q * F, 65536))
        assert far + (q - far) == q
    for a, b in [(7, 2), (5, 2), (-5, 2), (-7, 2), (9, -4), (-9, -4), (10, 4), (100, 7)]:
        assert O.rdiv(a, b) == rne_fraction(Fraction(a, b))


def _cic_setup():
    cfg = W.cic_int()
    return cfg["grid"], cfg["X"], cfg["m"], cfg["v"]


def test_cic_int_totals_are_an_identity():
    grid, X, m, v = _cic_setup()
    acc, ok = O.cic_int_p2g(grid, X, m, v)
    assert ok
    mom = [int(sum(int(a) * int(b) for a, b in zip(m, v[k]))) for k in range(2)]
    assert int(acc[0].sum()) == int(m.sum())
    assert [int(acc[1].sum()), int(acc[2].sum())] == mom
    # each particle's four mass shares: Fraction check of the two-stage split
    Xq = X.astype(np.int64)
    for p in range(0, 256, 17):
        one, _ = O.cic_int_p2g(grid, X[:, p:p + 1], m[p:p + 1], v[:, p:p + 1])
        cx, fx = Xq[0, p] >> 16, Xq[0, p] & 0xFFFF
        cy, fy = Xq[1, p] >> 16, Xq[1, p] & 0xFFFF
        far_x = rne_fraction(Fraction(int(m[p]) * int(fx), 65536))
        parts = {cx: int(m[p]) - far_x, cx + 1: far_x}
        for col, q in parts.items():
            far_y = rne_fraction(Fraction(q * int(fy), 65536))
            assert one[0, cy * 9 + col] == q - far_y
            assert one[0, (cy + 1) * 9 + col] == far_y


def test_cic_int_every_scrambled_order_matches():
    grid, X, m, v = _cic_setup()
    base, ok = O.cic_int_p2g(grid, X, m, v)
    assert ok
    rows = [tuple(int(t) for t in ln.split()) for ln in open(os.path.join(GOLDEN, "p4_scrambled_orders.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert [r[0] for r in rows] == list(range(1, 256, 2))
    for a, float_diff, int_diff in rows:
        acc, ok = O.cic_int_p2g(grid, X, m, v, W.scrambled_order(256, a, 13))
        differing = int(np.any(acc != base, axis=0).sum())
        assert differing == int_diff == 0
        assert float_diff > 0   # the page's float scatter differs in every order


def test_cic_int_gather_is_rounded_cell_mean():
    grid, X, m, v = _cic_setup()
    acc, ok = O.cic_int_p2g(grid, X, m, v)
    out = O.cic_int_gather(grid, X, acc)
    Xq = X.astype(np.int64)
    for p in range(256):
        cx, cy = Xq[0, p] >> 16, Xq[1, p] >> 16
        nodes = [cy * 9 + cx, cy * 9 + cx + 1, (cy + 1) * 9 + cx, (cy + 1) * 9 + cx + 1]
        M = int(acc[0, nodes].sum())
        for k in range(2):
            assert out[k, p] == rne_fraction(Fraction(int(acc[1 + k, nodes].sum()), M))


def test_cic_int_bounds_line_stops_before_any_scatter():
    grid, X, m, v = _cic_setup()
    m2 = m.copy()
    m2[5] = 2**40                      # 256 * 2^40 * 1000 > 2^63
    acc, ok = O.cic_int_p2g(grid, X, m2, v)
    assert not ok and not acc.any()
    X2 = X.copy()
    X2[0, 9] = 8 * 65536               # a stencil past the last node
    acc, ok = O.cic_int_p2g(grid, X2, m, v)
    assert not ok and not acc.any()


def test_float_and_double_order_table_qualitatively():
    """The page's arithmetic table: exact arithmetic (integer, double with
    dyadic positions) matches in all 128 orders; float, and double with
    positions in 1/65,535, do not.  Plain numpy scatter, independent of the
    oracle."""
    grid, X, m, v = _cic_setup()
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "p4_arithmetic_table.txt"))
            if ln.strip() and not ln.startswith("#")]

    def scatter(dtype, denom, order):
        g = np.zeros((3, 81), dtype=dtype)
        for p in order:
            fx = dtype(X[0, p] % 65536) / dtype(denom) if denom == 65536 else dtype(X[0, p]) / dtype(denom)
            fy = dtype(X[1, p] % 65536) / dtype(denom) if denom == 65536 else dtype(X[1, p]) / dtype(denom)
            if denom != 65536:
                cx, cy = int(np.floor(fx)), int(np.floor(fy))
                fx, fy = fx - dtype(cx), fy - dtype(cy)
            else:
                cx, cy = int(X[0, p] >> 16), int(X[1, p] >> 16)
            q = [dtype(m[p]), dtype(m[p]) * dtype(v[0, p]), dtype(m[p]) * dtype(v[1, p])]
            for (i, j, w) in [(cx, cy, (dtype(1) - fx) * (dtype(1) - fy)), (cx + 1, cy, fx * (dtype(1) - fy)),
                              (cx, cy + 1, (dtype(1) - fx) * fy), (cx + 1, cy + 1, fx * fy)]:
                if 0 <= i < 9 and 0 <= j < 9:
                    for c in range(3):
                        g[c, j * 9 + i] = dtype(g[c, j * 9 + i] + dtype(q[c] * w))
        return g

    for name, denom, _, matching in rows:
        if name == "integer":
            continue
        dt = np.float32 if name == "float" else np.float64
        denom = int(denom)
        base = scatter(dt, denom, range(256))
        same = 0
        for a in range(1, 256, 2):
            g = scatter(dt, denom, W.scrambled_order(256, a, 13))
            same += int(np.array_equal(g, base))
        if int(matching) == 128:
            assert same == 128
        else:
            assert same < 128


# --------------------------------------------------------------------------
# the advective step bound (implementation guide 3.3.2, rule 6)

def test_advective_speed_special_cases():
    # 3-4-5: |v| = 5 exactly; C = 0
    v = np.array([[3.0], [4.0], [0.0]], np.float32)
    C = np.zeros((9, 1), np.float32)
    assert O.advective_speed(3, 0.25, v, C) == 5.0
    # v = 0, C with |C|_F = 5 exactly (entries 3 and 4): 1.5 * 0.25 * 5
    C[0, 0], C[4, 0] = 3.0, 4.0
    assert O.advective_speed(3, 0.25, np.zeros((3, 1), np.float32), C) == 1.875
    # both terms add
    assert O.advective_speed(3, 0.25, v, C) == 6.875
    # 2D reads two components and four entries
    assert O.advective_speed(2, 0.5, np.array([[6.0], [8.0]], np.float32), np.zeros((4, 1), np.float32)) == 10.0
    # no particle
    assert O.advective_speed(3, 0.25, np.zeros((3, 0), np.float32), np.zeros((9, 0), np.float32)) == 0.0


def test_advective_speed_is_the_largest_particle_term():
    s = W.Stream(41, 41)
    n = 5000
    v = s.normal(3 * n, 2.0).reshape(3, n).astype(np.float32)
    C = s.normal(9 * n, 5.0).reshape(9, n).astype(np.float32)
    dx = 1.0 / 64
    got = O.advective_speed(3, dx, v, C)
    terms = (np.sqrt((v.astype(np.float64) ** 2).sum(axis=0))
             + 1.5 * dx * np.sqrt((C.astype(np.float64) ** 2).sum(axis=0)))
    assert got == pytest.approx(terms.max(), rel=1e-6)
    # attained by one particle, and no particle is larger
    k = int(np.argmax(terms))
    assert O.advective_speed(3, dx, v[:, k:k + 1], C[:, k:k + 1]) == got
    assert O.advective_speed(3, dx, np.delete(v, k, axis=1), np.delete(C, k, axis=1)) <= got


# --------------------------------------------------------------------------
# MLS-MPM elastic stress (implementation guide, section 3.1, Part 2: the
# Neo-Hookean P and sigma; section 3.3.2: F <- (I + D) F)

def _pages_fold_fp64(grid, material, C, F, vol, m):
    """C - dt V sigma (4/dx^2) / m per particle, the stress written exactly as
    the guide prints it (F^-T, P, sigma = P F^T / J, V = V0 J), in fp64."""
    dim = grid["dim"]
    mu, lam = material["mu"], material["lambda"]
    out = np.zeros(C.shape, dtype=np.float64)
    for p in range(C.shape[1]):
        Fp = F[:, p].astype(np.float64).reshape(dim, dim)
        J = np.linalg.det(Fp)
        FinvT = np.linalg.inv(Fp).T
        P = mu * (Fp - FinvT) + lam * np.log(J) * FinvT
        sigma = P @ Fp.T / J
        V = vol[p] * J
        term = -grid["dt"] * V * sigma * 4.0 / grid["dx"] ** 2 / m[p]
        out[:, p] = C[:, p] + term.reshape(-1)
    return out


def test_log_series_matches_the_logarithm():
    s = W.Stream(4242, 1)
    J = np.exp(s.uniform53(200000) * 80.0 - 40.0).astype(np.float32)
    near1 = (1.0 + (s.uniform53(20000) - 0.5) * 1e-3).astype(np.float32)
    J = np.concatenate([J, near1, np.float32([1.0, 2.0, 0.5, 3.0, 2.0 ** -126, 3.4e38])])
    got = np.array([O.log(float(j)) for j in J], dtype=np.float64)
    ref = np.log(J.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 * ulp + 1e-45)
    assert O.log(1.0) == 0.0
    # outside the domain (not positive, subnormal, infinite, NaN): 0
    for bad in (0.0, -1.0, 1e-40, float("inf"), float("nan")):
        assert O.log(bad) == 0.0


@pytest.mark.parametrize("dim", [2, 3])
def test_kirchhoff_vanishes_at_rest_and_under_rotation(dim):
    tau, ok = O.kirchhoff(dim, 3.0e6, 5.0e6, np.eye(dim))
    assert ok and np.all(tau == 0.0)
    s = W.Stream(31, dim)
    for _ in range(20):
        q, _ = np.linalg.qr(s.normal(dim * dim, 1.0).reshape(dim, dim))
        if np.linalg.det(q) < 0:
            q[:, 0] = -q[:, 0]
        tau, ok = O.kirchhoff(dim, 3.0e6, 5.0e6, q)
        assert ok and np.max(np.abs(tau)) <= 3.0e6 * 1e-6


@pytest.mark.parametrize("dim", [2, 3])
def test_kirchhoff_uniform_stretch_closed_form(dim):
    for sc in (0.5, 0.8, 1.25, 1.5, 2.0):
        mu, lam = 2.0e3, 7.0e3
        tau, ok = O.kirchhoff(dim, mu, lam, sc * np.eye(dim))
        expect = mu * (sc * sc - 1.0) + lam * dim * np.log(sc)
        assert ok
        assert np.max(np.abs(tau - expect * np.eye(dim))) <= 1e-6 * (abs(expect) + mu)


@pytest.mark.parametrize("dim", [2, 3])
def test_stress_fold_matches_the_guides_formulas_in_fp64(dim):
    cloud = W.with_elastic(W.small_cloud(dim, 400, 32, seed=900 + dim, lo=0.1, hi=0.9, csig=1.0,
                                         mass_lo=0.5, mass_hi=2.0), seed=901 + dim, fsig=0.15)
    g, mat = cloud["grid"], cloud["material"]
    Cs, bad = O.stress_affine(g, mat, cloud["x"], cloud["C"], cloud["F"], cloud["vol"], cloud["m"])
    ref = _pages_fold_fp64(g, mat, cloud["C"], cloud["F"], cloud["vol"], cloud["m"])
    assert bad == 0
    # fp32 error model: a few roundings of C, of mu * (F F^T)_kk (mu (F F^T - I) cancels) and of lambda ln J
    n = cloud["x"].shape[1]
    kappa = g["dt"] * cloud["vol"].astype(np.float64) * 4.0 / g["dx"] ** 2 / cloud["m"]
    Fm = cloud["F"].astype(np.float64).T.reshape(n, dim, dim)
    bnorm = np.einsum("pkj,pkj->p", Fm, Fm)
    logJ = np.abs(np.log(np.linalg.det(Fm)))
    scale = np.abs(cloud["C"]).max(axis=0) + kappa * (mat["mu"] * bnorm + mat["lambda"] * logJ)
    assert np.all(np.abs(Cs - ref) <= 1e-6 * scale[None, :])
    # the stress term is not small next to C here: dropping it fails by far
    assert np.median(np.abs(ref - cloud["C"])) > 0.3 * np.median(np.abs(cloud["C"]))


@pytest.mark.parametrize("dim", [2, 3])
def test_stress_scatter_is_the_mls_nodal_force(dim):
    """With v = 0 and C = 0 the momentum the fold scatters is the MLS force
    impulse -dt V sigma (4/dx^2) w_i (x_i - x_p), summed in fp64 over all nodes."""
    cloud = W.with_elastic(W.small_cloud(dim, 24, 8, seed=910 + dim, lo=0.25, hi=0.75, scale_log2=18,
                                         mass_lo=0.5, mass_hi=2.0), seed=911 + dim, fsig=0.2, mu=2.0e5,
                           lam=3.0e5)
    g, mat = cloud["grid"], cloud["material"]
    n = cloud["x"].shape[1]
    v0 = np.zeros((dim, n), dtype=np.float32)
    C0 = np.zeros((dim * dim, n), dtype=np.float32)
    Cs, bad = O.stress_affine(g, mat, cloud["x"], C0, cloud["F"], cloud["vol"], cloud["m"])
    acc, st, counts = O.p2g_fixed(g, cloud["x"], v0, Cs, cloud["m"])
    assert bad == 0 and st == 0
    ref_C = _pages_fold_fp64(g, mat, C0, cloud["F"], cloud["vol"], cloud["m"])
    mass, mom, absterm = brute_force_p2g(g, cloud["x"], v0, ref_C, cloud["m"])
    S = 2.0 ** g["scale_log2"]
    assert np.max(np.abs(mom)) > 1e3 / S
    tol = (13.5 * n + 1.0) / S + 2e-6 * absterm
    for k in range(dim):
        assert np.all(np.abs(acc[1 + k] / S - mom[k]) <= tol)
    # momentum is unchanged by the stress: the shares of each particle sum to rint(m S v) = 0
    assert np.all(acc[1:].sum(axis=1) == 0)


def test_degenerate_deformation_is_counted_and_unstressed():
    cloud = W.with_elastic(W.small_cloud(3, 6, 16, seed=920, lo=0.3, hi=0.7), seed=921)
    F = cloud["F"].copy()
    F[:, 0] = [1, 0, 0, 0, 1, 0, 0, 0, -1]          # inverted
    F[:, 1] = [1, 2, 3, 2, 4, 6, 0, 0, 1]           # singular
    F[:, 2] = [1e-20, 0, 0, 0, 1e-20, 0, 0, 0, 1]   # J subnormal
    x = cloud["x"].copy()
    x[:, 2] = -1.0                                  # ... but outside the domain: not counted
    Cs, bad = O.stress_affine(cloud["grid"], cloud["material"], x, cloud["C"], F, cloud["vol"], cloud["m"])
    assert bad == 2
    assert np.array_equal(Cs[:, :3].view(np.uint32), cloud["C"][:, :3].view(np.uint32))
    assert not np.array_equal(Cs[:, 3:], cloud["C"][:, 3:])


@pytest.mark.parametrize("dim", [2, 3])
def test_g2p_advances_F_by_the_new_affine_matrix(dim):
    """In an affine velocity field v = A x + c the gathered C is A, and F becomes
    (I + dt A) F: A on the left (a transposed or right-multiplied update fails)."""
    n = 16
    cloud = W.with_elastic(W.small_cloud(dim, 300, n, seed=930 + dim, lo=0.15, hi=0.85), seed=931 + dim,
                           fsig=0.3)
    grid = cloud["grid"]
    grid["dt"] = float(np.float32(1e-2))
    s = W.Stream(78, dim)
    A = s.normal(dim * dim, 1.0).reshape(dim, dim)
    c = s.normal(dim, 1.0)
    X = node_coords(grid) * grid["dx"]
    vel = (A @ X + c[:, None]).astype(np.float32)
    x2, v2, C2, F2, moved = O.g2p_elastic(grid, vel, cloud["x"], cloud["v"], cloud["C"], cloud["F"])
    assert moved == 300
    x3, v3, C3, moved3 = O.g2p(grid, vel, cloud["x"], cloud["v"], cloud["C"])
    assert np.array_equal(C2, C3) and np.array_equal(v2, v3) and np.array_equal(x2, x3)
    for p in range(300):
        Fp = cloud["F"][:, p].astype(np.float64).reshape(dim, dim)
        Cp = C2[:, p].astype(np.float64).reshape(dim, dim)
        expect = (np.eye(dim) + grid["dt"] * Cp) @ Fp
        assert np.max(np.abs(F2[:, p].reshape(dim, dim) - expect)) <= 1e-6 * (1 + np.abs(expect).max())
        assert np.max(np.abs(Cp - A)) <= 2e-3
    wrong = np.stack([(cloud["F"][:, p].reshape(dim, dim) @ (np.eye(dim) + grid["dt"] * A)).ravel()
                      for p in range(300)], axis=1)
    assert np.max(np.abs(F2 - wrong)) > 1e-3


def test_elastic_step_keeps_grid_totals_an_identity():
    cloud = W.with_elastic(W.small_cloud(3, 2000, 32, seed=940, lo=0.2, hi=0.8, scale_log2=19), seed=941)
    grid = cloud["grid"]
    out = O.step_elastic(grid, cloud["material"], cloud["x"], cloud["v"], cloud["C"], cloud["m"], cloud["F"],
                         cloud["vol"])
    assert out["status"] == 0 and out["degenerate"] == 0
    S = np.float32(2.0 ** grid["scale_log2"])
    Mt = (cloud["m"] * S).astype(np.float32)
    assert int(out["acc"][0].sum()) == int(np.rint(Mt).astype(np.int64).sum())
    for k in range(3):
        Qk = np.rint((Mt * cloud["v"][k]).astype(np.float32)).astype(np.int64)
        assert int(out["acc"][1 + k].sum()) == int(Qk.sum())


# --------------------------------------------------------------------------
# grid-recovered volume (implementation guide, section 3.3.2: each particle
# scatters its rest volume as a fraction of a cell, so a rest-packed node sums
# to about one; G2P gathers it back)

def _lattice(n, per_cell_axis, lo_cell, hi_cell, dim=3):
    """Particles on a regular lattice, per_cell_axis per cell edge, cells lo..hi-1."""
    h = 1.0 / per_cell_axis
    ax = (np.arange(lo_cell * per_cell_axis, hi_cell * per_cell_axis) + 0.5) * h / n
    mesh = np.meshgrid(*([ax] * dim), indexing="ij")
    return np.stack([m.ravel() for m in mesh]).astype(np.float32)


@pytest.mark.parametrize("dim", [2, 3])
def test_volume_channel_sums_to_one_on_a_rest_packing(dim):
    n = 16
    x = _lattice(n, 2, 3, 13, dim)
    npart = x.shape[1]
    grid = W.small_cloud(dim, 1, n, seed=1, scale_log2=20)["grid"]
    dx = grid["dx"]
    vol = np.full(npart, dx ** dim / 2 ** dim, dtype=np.float32)   # 1/ppc of a cell each
    z = np.zeros((dim, npart), np.float32)
    acc, st, counts = O.p2g_fixed(grid, x, z, np.zeros((dim * dim, npart), np.float32),
                                  np.ones(npart, np.float32), vol=vol)
    assert st == 0 and acc.shape[0] == dim + 2
    S = 2.0 ** grid["scale_log2"]
    assert int(acc[dim + 1].sum()) == npart * int(np.rint(S / 2 ** dim))      # totals: an identity
    phi = O.grid_volume(grid, acc[dim + 1])
    X = node_coords(grid)
    interior = np.all((X >= 5) & (X <= 10), axis=0)
    assert np.max(np.abs(phi[interior] - 1.0)) <= 27 * 2 ** dim / S
    assert np.all(phi[~np.all((X >= 2) & (X <= 14), axis=0)] == 0.0)
    # gathered back: particles well inside read a rest packing
    pp = O.g2p_volume(grid, phi, x)
    inside = np.all((x * n >= 5.5) & (x * n <= 10.5), axis=0)
    assert np.max(np.abs(pp[inside] - 1.0)) <= 1e-5
    # compressed: the same particles at twice the density read two
    acc2, _, _ = O.p2g_fixed(grid, x, z, np.zeros((dim * dim, npart), np.float32),
                             np.ones(npart, np.float32), vol=vol * 2)
    pp2 = O.g2p_volume(grid, O.grid_volume(grid, acc2[dim + 1]), x)
    assert np.max(np.abs(pp2[inside] - 2.0)) <= 2e-5


@pytest.mark.parametrize("dim", [2, 3])
def test_volume_channel_matches_brute_force(dim):
    n = 8
    cloud = W.with_elastic(W.small_cloud(dim, 40, n, seed=950 + dim, lo=0.2, hi=0.8, scale_log2=20), seed=951)
    grid = cloud["grid"]
    vol = (cloud["vol"] * (0.5 + W.Stream(952, 1).uniform24(40))).astype(np.float32)
    acc, st, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol=vol)
    accf, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], vol=vol)
    base, _, _ = O.p2g_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    assert st == 0 and np.array_equal(acc[: dim + 1], base)      # the other channels are unchanged
    q = vol.astype(np.float64) / grid["dx"] ** dim
    ones = np.ones((dim, 40))
    mass, _, absterm = brute_force_p2g(grid, cloud["x"], 0 * ones, np.zeros((dim * dim, 40)), q)
    S = 2.0 ** grid["scale_log2"]
    assert np.all(np.abs(acc[dim + 1] / S - mass) <= 27.0 * 40 / S + 1e-6 * absterm)
    assert np.all(np.abs(accf[dim + 1] - mass) <= 2e-6 * absterm + 1e-12)


@pytest.mark.parametrize("dim", [2, 3])
def test_volume_gather_reproduces_affine_fields(dim):
    """The quadratic B-spline reproduces affine functions: gathering phi = a.x + b
    returns a.x_p + b (a transposed node index or a wrong weight fails)."""
    n = 16
    cloud = W.small_cloud(dim, 500, n, seed=960 + dim, lo=0.15, hi=0.85)
    grid = cloud["grid"]
    a = np.array([0.7, -1.3, 2.1][:dim])
    X = node_coords(grid) * grid["dx"]
    phi = (a @ X + 0.25).astype(np.float32)
    pp = O.g2p_volume(grid, phi, cloud["x"])
    expect = a @ cloud["x"].astype(np.float64) + 0.25
    assert np.max(np.abs(pp - expect)) <= 2e-6
