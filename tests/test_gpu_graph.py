"""The stepping calls captured in a CUDA graph (the bench's headline timing replays one): a period of 16
steps (bin, P2G with the range records, G2P with the update on load, sorted every 8th step) captured once
and replayed must leave the same particle state, bit for bit, as the same steps run eagerly; and the
capture itself must run nothing."""
import numpy as np
import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W
from material_point_particle_gb300.system import MPMSystem

pytestmark = pytest.mark.gpu

PERIOD, SORT = 16, 8


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def make(cloud):
    n = cloud["x"].shape[1]
    s = MPMSystem(cloud["grid"], n).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    s.bin()
    s.p2g()
    s.grid_update()
    s.step_sorted()
    s.use_range_records(True)
    torch.cuda.synchronize()
    return s


def period(s, stream=None):
    for k in range(PERIOD):
        s.bin(stream)
        s.p2g(stream)
        if (k + 1) % SORT == 0:
            s.g2p_sorted_update(stream)
        else:
            s.g2p_update(stream)


@pytest.mark.parametrize("dim,n,count", [(3, 32, 20000), (2, 64, 12000)])
def test_graph_replay_matches_eager_steps(dim, n, count):
    cloud = W.small_cloud(dim, count, n, seed=7100 + dim, scale_log2=19 if dim == 3 else 20, lo=0.1, hi=0.9,
                          vsig=1.0, csig=2.0)
    cloud["grid"]["g"] = [0.0, -9.8, 0.0]
    a, b = make(cloud), make(cloud)
    period(a)
    period(a)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    before = [t.clone() for t in (b.x, b.v, b.C)]
    with torch.cuda.graph(g, stream=side):
        period(b)
    torch.cuda.synchronize()
    for t, u in zip((b.x, b.v, b.C), before):
        assert torch.equal(t, u), "the capture ran work"
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    xa, va, Ca = a.state()
    xb, vb, Cb = b.state()
    for u, w in ((xa, xb), (va, vb), (Ca, Cb)):
        assert np.array_equal(bits(u), bits(w))
    assert np.array_equal(a.id.cpu().numpy(), b.id.cpu().numpy())
    sa, sb = a.status(), b.status()
    assert sa[L.ST_FLAGS] == sb[L.ST_FLAGS] == 0
    for w in (L.ST_N_VALID, L.ST_MAX_SPEED, L.ST_G2P_RANGE, L.ST_RANGE, L.ST_SHARE_PATH):
        assert sa[w] == sb[w], w


def test_graph_replay_of_fused_steps_matches_eager():
    """mpm_step_fused (bin, the fused gather-scatter kernel, the clear) captured for 16 steps (both buffer
    pairs back in place) and replayed twice, against 32 eager fused steps."""
    cloud = W.small_cloud(3, 20000, 32, seed=7200, scale_log2=19, lo=0.1, hi=0.9, vsig=1.0, csig=2.0)
    cloud["grid"]["g"] = [0.0, -9.8, 0.0]
    a, b = make(cloud), make(cloud)
    a.enable_fused()
    b.enable_fused()
    for _ in range(2 * PERIOD):
        a.step_fused()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(PERIOD):
            b.step_fused()
    torch.cuda.synchronize()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    xa, va, Ca = a.state()
    xb, vb, Cb = b.state()
    for u, w in ((xa, xb), (va, vb), (Ca, Cb)):
        assert np.array_equal(bits(u), bits(w))
    assert a.status()[L.ST_FLAGS] == b.status()[L.ST_FLAGS] == 0
