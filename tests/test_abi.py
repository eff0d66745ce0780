"""The C-ABI library: builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes as ct
import os
import re
import subprocess

import pytest
import torch

from material_point_particle_gb300 import _lib as L
from material_point_particle_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mpm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mpm_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = L.library()
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(lib, name), name
        assert hasattr(L, name), f"binding lacks {name}"
    assert L.mpm_version() >= 1


def _aligned_ws(nbytes):
    raw = torch.empty(nbytes + 256, dtype=torch.uint8)
    off = (-raw.data_ptr()) % 256
    return raw, raw[off:off + nbytes]


def _parts(dim, n):
    x = torch.zeros(dim, n)
    return L.particles(x, torch.zeros(dim, n), torch.zeros(dim * dim, n), torch.zeros(n)), x


@pytest.mark.parametrize("bad", ["dim", "tile", "order", "n", "scale", "mode", "dx"])
def test_bad_descriptor_is_rejected(bad):
    grid = W.small_cloud(3, 8, 16, seed=1)["grid"]
    d = L.grid_desc(grid)
    if bad == "dim":
        d.dim = 4
    elif bad == "tile":
        d.tile = 8
    elif bad == "order":
        d.order = 3
    elif bad == "n":
        d.n[1] = 2
    elif bad == "scale":
        d.scale_log2 = 41
    elif bad == "mode":
        d.acc_mode = 9
    elif bad == "dx":
        d.dx = float("nan")
    assert L.mpm_workspace_bytes(d, 8) == 0
    assert L.mpm_grid_acc_bytes(d) == 0
    p, _ = _parts(3, 8)
    b = L.Bins()
    assert L.library().mpm_bin(ct.byref(d), ct.byref(p), ct.byref(b), 0, None) == L.MPM_E_ARG


def test_workspace_carving_and_size_checks():
    grid = W.small_cloud(3, 8, 16, seed=1)["grid"]
    d = L.grid_desc(grid)
    need = L.mpm_workspace_bytes(d, 1000)
    assert need > 3 * 4 * 1000
    raw, ws = _aligned_ws(need)
    b = L.mpm_bins_init(d, 1000, ws)
    base = ws.data_ptr()
    assert b.scratch == base and b.n == 1000 and b.ntiles == 64
    for name in ("key", "perm", "tile_count", "tile_start", "slices", "active", "status"):
        ptr = getattr(b, name)
        assert base <= ptr < base + need and (ptr - base) % 256 == 0, name
    with pytest.raises(L.MPMError) as e:
        L.mpm_bins_init(d, 1000, ws[: need - 256])
    assert e.value.code == L.MPM_E_WORKSPACE
    with pytest.raises(L.MPMError) as e:
        L.mpm_bins_init(d, 1000, raw[((-raw.data_ptr()) % 256) + 4:][:need])
    assert e.value.code == L.MPM_E_ARG  # misaligned workspace
    # particles beyond the carved count are refused
    p, _ = _parts(3, 1001)
    assert L.library().mpm_bin(ct.byref(d), ct.byref(p), ct.byref(b), 0, None) == L.MPM_E_ARG
    # null particle arrays are refused
    p, _ = _parts(3, 10)
    p.v[1] = None
    assert L.library().mpm_p2g(ct.byref(d), ct.byref(p), ct.byref(b), ct.c_void_p(base), 0.0, None) == L.MPM_E_ARG
    # an elastic state needs every F plane and the rest volumes
    p, keep = _parts(3, 10)
    F = torch.zeros((9, 10))
    for j in range(9):
        p.F[j] = F[j].data_ptr()
    assert L.library().mpm_p2g(ct.byref(d), ct.byref(p), ct.byref(b), ct.c_void_p(base), 0.0, None) == L.MPM_E_ARG
    p.vol = F[0].data_ptr()
    p.F[8] = None
    assert L.library().mpm_p2g(ct.byref(d), ct.byref(p), ct.byref(b), ct.c_void_p(base), 0.0, None) == L.MPM_E_ARG


def test_grid_byte_counts():
    for dim, mode, w in [(3, W.ACC_I64, 8), (3, W.ACC_I32, 4), (2, W.ACC_F32, 4)]:
        grid = W.small_cloud(dim, 8, 20, seed=1, acc_mode=mode)["grid"]
        d = L.grid_desc(grid)
        nodes = 20 ** dim
        assert L.mpm_grid_acc_bytes(d) == (dim + 1) * nodes * w
        assert L.mpm_grid_vel_bytes(d) == dim * nodes * 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_fails_loudly():
    grid = W.small_cloud(3, 8, 16, seed=1)["grid"]
    d = L.grid_desc(grid)
    raw, ws = _aligned_ws(L.mpm_workspace_bytes(d, 10))
    b = L.mpm_bins_init(d, 10, ws)
    p, _ = _parts(3, 10)
    code = L.library().mpm_bin(ct.byref(d), ct.byref(p), ct.byref(b), 0, None)
    assert code == L.MPM_E_NO_DEVICE
    assert "device" in L.strerror(code)


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of the C structs have the header's sizes and offsets."""
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stddef.h>
#include <stdio.h>
#include "mpm.h"
int main(void) {
    printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(mpm_grid_desc), sizeof(mpm_particles), sizeof(mpm_bins),
           offsetof(mpm_particles, id), offsetof(mpm_particles, F), offsetof(mpm_particles, vol),
           offsetof(mpm_particles, mu), offsetof(mpm_particles, lambda));
    return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(t) for t in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    P = L.Particles
    assert got == [ct.sizeof(L.GridDesc), ct.sizeof(P), ct.sizeof(L.Bins), P.id.offset, P.F.offset,
                   P.vol.offset, P.mu.offset, P.lambda_.offset]
