"""The seeded input generator: published splitmix64 outputs, determinism, and
independence from the internal chunk size (both sides of every parity test
consume these arrays)."""
import numpy as np

from material_point_particle_gb300 import workloads as W


def test_splitmix64_published_outputs():
    # Vigna's reference splitmix64: seed 0 and seed 1234567, first three outputs
    assert [int(v) for v in W.splitmix64(0, 3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(v) for v in W.splitmix64(1234567, 3)] == [6457827717110365317, 3203168211198807973,
                                                           9817491932198370423]


def test_streams_do_not_depend_on_chunking(monkeypatch):
    ref = W.Stream(99, 3).normal(300001)
    refu = W.Stream(99, 4).uniform24(300001)
    monkeypatch.setattr(W.Stream, "CHUNK", 1 << 10)
    assert np.array_equal(W.Stream(99, 3).normal(300001), ref)
    assert np.array_equal(W.Stream(99, 4).uniform24(300001), refu)


def test_workloads_are_deterministic_and_in_domain():
    for build, kw in [(W.mls2d, {}), (W.dambreak3d, dict(n_particles=4096)), (W.blobs3d, dict(n_particles=8192)),
                      (W.sphere3d, dict(n_particles=8192, n=64))]:
        a, b = build(**kw), build(**kw)
        for k in ("x", "v", "C", "m"):
            assert np.array_equal(a[k], b[k])
        g = a["grid"]
        xi = a["x"].astype(np.float64) * g["inv_dx"]
        assert np.all(xi >= 0.5) and np.all(xi < np.array(g["n"][:g["dim"]])[:, None] - 1.5)
    cfg = W.cic_int()
    assert cfg["X"].shape == (2, 256) and cfg["X"].min() >= 0 and cfg["X"].max() < 8 * 65536
    assert cfg["m"].min() >= 1 and cfg["m"].max() <= 1000 and np.abs(cfg["v"]).max() <= 1000
