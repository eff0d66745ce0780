// api.cu -- the C ABI (include/mpm.h): argument checks, workspace carving,
// device facts, and the calls that sequence the kernels.  Host code only.
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mpm {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int ilog2(int v) {
    int r = 0;
    while ((1 << r) < v) ++r;
    return r;
}

// Validates the descriptor and derives the kernel parameters.
mpm_status make_grid(const mpm_grid_desc *d, GridP &g) {
    if (!d) return MPM_E_ARG;
    if (d->dim != 2 && d->dim != 3) return MPM_E_ARG;
    if (d->acc_mode < MPM_ACC_I32 || d->acc_mode > MPM_ACC_EXACT_INT) return MPM_E_ARG;
    if (d->volume_channel != 0 && d->volume_channel != 1) return MPM_E_ARG;
    if (d->volume_channel && d->acc_mode == MPM_ACC_EXACT_INT) return MPM_E_ARG;
    std::memset(&g, 0, sizeof(g));
    g.dim = d->dim;
    g.acc_mode = d->acc_mode;
    int64_t nodes = 1;
    for (int l = 0; l < 3; ++l) {
        g.n[l] = l < d->dim ? d->n[l] : 1;
        if (l < d->dim && (g.n[l] < 3 || g.n[l] > (1 << 20))) return MPM_E_ARG;
        nodes *= g.n[l];
    }
    g.nodes = nodes;
    if (d->acc_mode == MPM_ACC_EXACT_INT) {
        if (d->order != 1) return MPM_E_ARG;
        g.T = 1;
        return MPM_OK;
    }
    if (d->order != 2) return MPM_E_ARG;
    if (!(d->dx > 0.0f) || !(d->inv_dx > 0.0f) || !std::isfinite(d->dx) || !std::isfinite(d->inv_dx))
        return MPM_E_ARG;
    if (d->boundary_nodes < 0) return MPM_E_ARG;
    if (d->acc_mode != MPM_ACC_F32 && (d->scale_log2 < 0 || d->scale_log2 > 40)) return MPM_E_ARG;
    const int want_tile = d->dim == 3 ? 4 : 8;
    if (d->tile != want_tile || !is_pow2(d->tile)) return MPM_E_ARG;
    g.dx = d->dx;
    g.inv_dx = d->inv_dx;
    g.S = d->acc_mode == MPM_ACC_F32 ? 1.0f : std::ldexp(1.0f, d->scale_log2);
    g.T = d->tile;
    g.T_log2 = ilog2(d->tile);
    g.cpt_log2 = g.T_log2 * d->dim;
    g.ntiles = 1;
    g.nblocks = 1;
    for (int l = 0; l < 3; ++l) {
        g.nt[l] = l < d->dim ? (g.n[l] - 2 + g.T - 1) / g.T : 1;
        g.nb[l] = l < d->dim ? (g.n[l] + g.T - 1) / g.T : 1;
        g.ntiles *= g.nt[l];
        g.nblocks *= g.nb[l];
    }
    if ((g.ntiles << g.cpt_log2) >= (int64_t)0xFFFFFFFFll) return MPM_E_ARG;
    g.H = g.T + 2;
    g.halo_nodes = d->dim == 3 ? g.H * g.H * g.H : g.H * g.H;
    g.boundary = d->boundary_nodes;
    g.wmax = d->dim == 3 ? 0.421875f : 0.5625f;
    g.vc = d->volume_channel;
    g.vcell = d->inv_dx * d->inv_dx;
    if (d->dim == 3) g.vcell = g.vcell * d->inv_dx;
    g.inv_S = d->acc_mode == MPM_ACC_F32 ? 1.0f : std::ldexp(1.0f, -d->scale_log2);
    return MPM_OK;
}

struct Layout {
    size_t key, perm, heads, tails, count, start, hcnt, tcnt, active, slices, large_list, partial, status, cellcount,
        readers, count_next,
        scratch, total;
    int64_t max_slices;
};

Layout layout_of(const GridP &g, int64_t n) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off += align_up(bytes);
        return at;
    };
    if (g.acc_mode == MPM_ACC_EXACT_INT) {
        L.status = take(MPM_STATUS_WORDS * sizeof(uint32_t));
        L.scratch = take(2 * sizeof(uint64_t));
        L.total = off;
        return L;
    }
    const int64_t nb = g.ntiles + 1;
    L.max_slices = (n + kSliceParticles - 1) / kSliceParticles + std::min<int64_t>(g.ntiles, n) + 1;
    L.key = take(n * sizeof(uint32_t));
    L.perm = take(n * sizeof(uint32_t));
    L.heads = take(n * sizeof(uint32_t));
    L.tails = take(n * sizeof(uint32_t));
    L.count = take(nb * sizeof(uint32_t));
    L.start = take((nb + 1) * sizeof(uint32_t));
    L.hcnt = take(nb * sizeof(uint32_t));
    L.tcnt = take(nb * sizeof(uint32_t));
    L.active = take(g.ntiles * sizeof(uint32_t));
    L.slices = take(2 * L.max_slices * sizeof(uint32_t));
    L.large_list = take(nb * sizeof(uint32_t));
    L.partial = take(3 * ((nb + 1023) / 1024 + 1) * sizeof(uint32_t));
    L.status = take(MPM_STATUS_WORDS * sizeof(uint32_t));
    L.cellcount = g.acc_mode == MPM_ACC_I32 ? take((size_t)(g.ntiles << g.cpt_log2) * sizeof(uint32_t)) : 0;
    L.readers = take((size_t)g.nblocks * sizeof(uint32_t));
    L.count_next = take(nb * sizeof(uint32_t));
    L.scratch = take(2 * sizeof(uint64_t));
    L.total = off;
    return L;
}

WsView view_of(const GridP &g, const mpm_bins &b) {
    Layout L = layout_of(g, b.n);
    char *base = static_cast<char *>(b.scratch);
    WsView w{};
    w.status = reinterpret_cast<uint32_t *>(base + L.status);
    if (g.acc_mode == MPM_ACC_EXACT_INT) return w;
    w.key = reinterpret_cast<uint32_t *>(base + L.key);
    w.perm = reinterpret_cast<uint32_t *>(base + L.perm);
    w.heads = reinterpret_cast<uint32_t *>(base + L.heads);
    w.tails = reinterpret_cast<uint32_t *>(base + L.tails);
    w.count = reinterpret_cast<uint32_t *>(base + L.count);
    w.start = reinterpret_cast<uint32_t *>(base + L.start);
    w.hcnt = reinterpret_cast<uint32_t *>(base + L.hcnt);
    w.tcnt = reinterpret_cast<uint32_t *>(base + L.tcnt);
    w.active = reinterpret_cast<uint32_t *>(base + L.active);
    w.slices = reinterpret_cast<uint32_t *>(base + L.slices);
    w.large_list = reinterpret_cast<uint32_t *>(base + L.large_list);
    w.partial = reinterpret_cast<uint32_t *>(base + L.partial);
    w.cellcount = g.acc_mode == MPM_ACC_I32 ? reinterpret_cast<uint32_t *>(base + L.cellcount) : nullptr;
    w.readers = reinterpret_cast<uint32_t *>(base + L.readers);
    w.count_next = reinterpret_cast<uint32_t *>(base + L.count_next);
    return w;
}

// The bins must have been carved for this grid and at least n particles.
mpm_status check_bins(const GridP &g, const mpm_bins *b, int64_t n) {
    if (!b || !b->scratch || !b->status) return MPM_E_ARG;
    if (n < 0 || n > b->n) return MPM_E_ARG;
    if (g.acc_mode != MPM_ACC_EXACT_INT && b->ntiles != g.ntiles) return MPM_E_ARG;
    if (b->scratch_bytes < layout_of(g, b->n).total) return MPM_E_WORKSPACE;
    return MPM_OK;
}

mpm_status parts_f(const GridP &g, const mpm_particles *p, bool need_state, PartsF &out) {
    if (!p || p->n < 0 || p->n > 0xFFFFFFFEll) return MPM_E_ARG;
    std::memset(&out, 0, sizeof(out));
    out.n = p->n;
    for (int l = 0; l < g.dim; ++l) {
        out.x[l] = static_cast<float *>(p->x[l]);
        if (!out.x[l] && p->n) return MPM_E_ARG;
    }
    if (!need_state) return MPM_OK;
    for (int k = 0; k < g.dim; ++k) {
        out.v[k] = static_cast<float *>(p->v[k]);
        if (!out.v[k] && p->n) return MPM_E_ARG;
    }
    for (int j = 0; j < g.dim * g.dim; ++j) {
        out.C[j] = static_cast<float *>(p->C[j]);
        if (!out.C[j] && p->n) return MPM_E_ARG;
    }
    out.m = static_cast<const float *>(p->m);
    if (!out.m && p->n) return MPM_E_ARG;
    out.id = static_cast<uint32_t *>(p->id);
    if (p->F[0]) {  // elastic state: every F plane and vol
        for (int j = 0; j < g.dim * g.dim; ++j) {
            out.F[j] = static_cast<float *>(p->F[j]);
            if (!out.F[j]) return MPM_E_ARG;
        }
        out.vol = static_cast<float *>(p->vol);
        if (!out.vol) return MPM_E_ARG;
        out.mu = p->mu;
        out.lam = p->lambda;
    }
    if (g.vc) {  // volume channel: rest volumes in, volume fractions out
        out.vol = static_cast<float *>(p->vol);
        out.phi = static_cast<float *>(p->phi);
        if ((!out.vol || !out.phi) && p->n) return MPM_E_ARG;
    }
    return MPM_OK;
}

mpm_status parts_i(const GridP &g, const mpm_particles *p, PartsI &out) {
    if (!p || p->n < 0 || p->n > 0xFFFFFFFEll) return MPM_E_ARG;
    std::memset(&out, 0, sizeof(out));
    out.n = p->n;
    for (int l = 0; l < g.dim; ++l) {
        out.X[l] = static_cast<const int32_t *>(p->x[l]);
        out.v[l] = static_cast<int64_t *>(p->v[l]);
        if ((!out.X[l] || !out.v[l]) && p->n) return MPM_E_ARG;
    }
    out.m = static_cast<const int64_t *>(p->m);
    if (!out.m && p->n) return MPM_E_ARG;
    return MPM_OK;
}

std::mutex g_dev_mutex;
int g_sms[64] = {0};

}  // namespace

mpm_status device_info(DeviceInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MPM_E_NO_DEVICE;
    if (dev < 0 || dev >= 64) return MPM_E_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_sms[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return MPM_E_NO_DEVICE;
        g_sms[dev] = sms;
    }
    out.device = dev;
    out.sms = g_sms[dev];
    return MPM_OK;
}

}  // namespace mpm

using namespace mpm;

#define MPM_TRY(expr)                       \
    do {                                    \
        mpm_status _s = (expr);             \
        if (_s != MPM_OK) return _s;        \
    } while (0)

extern "C" {

int32_t mpm_version(void) { return (0 << 16) | 1; }

const char *mpm_strerror(mpm_status s) {
    switch (s) {
        case MPM_OK: return "ok";
        case MPM_E_ARG: return "invalid argument";
        case MPM_E_WORKSPACE: return "workspace too small";
        case MPM_E_DOMAIN: return "particles outside the domain";
        case MPM_E_BOUND: return "shares or accumulators would not fit";
        case MPM_E_CUDA: return "CUDA error";
        case MPM_E_TIMEOUT: return "bounded device wait gave up";
        case MPM_E_NO_DEVICE: return "no usable CUDA device";
    }
    return "unknown status";
}

size_t mpm_workspace_bytes(const mpm_grid_desc *desc, int64_t n) {
    GridP g;
    if (make_grid(desc, g) != MPM_OK || n < 0) return 0;
    return layout_of(g, n).total;
}

mpm_status mpm_bins_init(const mpm_grid_desc *desc, int64_t n, void *ws, size_t ws_bytes, mpm_bins *out) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (!out || !ws || n < 0 || n > 0xFFFFFFFEll) return MPM_E_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MPM_E_ARG;
    Layout L = layout_of(g, n);
    if (ws_bytes < L.total) return MPM_E_WORKSPACE;
    std::memset(out, 0, sizeof(*out));
    out->n = n;
    out->ntiles = g.acc_mode == MPM_ACC_EXACT_INT ? 0 : g.ntiles;
    out->max_slices = L.max_slices;
    out->scratch = ws;
    out->scratch_bytes = ws_bytes;
    WsView w = view_of(g, *out);
    out->status = w.status;
    out->key = w.key;
    out->perm = w.perm;
    out->tile_count = w.count;
    out->tile_start = w.start;
    out->slices = w.slices;
    out->active = w.active;
    return MPM_OK;
}

size_t mpm_grid_acc_bytes(const mpm_grid_desc *desc) {
    GridP g;
    if (make_grid(desc, g) != MPM_OK) return 0;
    const size_t w = (g.acc_mode == MPM_ACC_I64 || g.acc_mode == MPM_ACC_EXACT_INT) ? 8 : 4;
    return (size_t)(g.dim + 1 + g.vc) * (size_t)g.nodes * w;
}

size_t mpm_grid_vel_bytes(const mpm_grid_desc *desc) {
    GridP g;
    if (make_grid(desc, g) != MPM_OK) return 0;
    return (size_t)(g.dim + g.vc) * (size_t)g.nodes * sizeof(float);
}

mpm_status mpm_bin(const mpm_grid_desc *desc, const mpm_particles *parts, mpm_bins *bins, int flags, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT || (flags & ~MPM_BIN_KEYS_FROM_G2P) != 0) return MPM_E_ARG;
    const bool from_g2p = (flags & MPM_BIN_KEYS_FROM_G2P) != 0;
    if (from_g2p && g.acc_mode != MPM_ACC_I64) return MPM_E_ARG;
    PartsF p;
    MPM_TRY(parts_f(g, parts, false, p));
    MPM_TRY(check_bins(g, bins, p.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_bin(g, p, view_of(g, *bins), from_g2p, dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_p2g(const mpm_grid_desc *desc, const mpm_particles *parts, mpm_bins *bins, void *grid_acc,
                   float dt, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (!grid_acc) return MPM_E_ARG;
    DeviceInfo dev;
    if (g.acc_mode == MPM_ACC_EXACT_INT) {
        PartsI p;
        MPM_TRY(parts_i(g, parts, p));
        MPM_TRY(check_bins(g, bins, 0));
        MPM_TRY(device_info(dev));
        WsView w = view_of(g, *bins);
        Layout L = layout_of(g, bins->n);
        uint64_t *scratch = reinterpret_cast<uint64_t *>(static_cast<char *>(bins->scratch) + L.scratch);
        return launch_cic_int_p2g(g, p, static_cast<int64_t *>(grid_acc), w.status, scratch, dev,
                                  static_cast<cudaStream_t>(stream));
    }
    PartsF p;
    MPM_TRY(parts_f(g, parts, true, p));
    MPM_TRY(check_bins(g, bins, p.n));
    MPM_TRY(device_info(dev));
    return launch_p2g(g, p, view_of(g, *bins), grid_acc, dt, bins->range_from_g2p != 0, dev,
                      static_cast<cudaStream_t>(stream));
}

mpm_status mpm_grid_update(const mpm_grid_desc *desc, void *grid_acc, float *grid_vel, const float dtg[3],
                           mpm_bins *bins, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT || !grid_acc || !grid_vel || !dtg) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, 0));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_grid_update(g, grid_acc, grid_vel, dtg, view_of(g, *bins), dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_g2p(const mpm_grid_desc *desc, const void *grid, mpm_particles *parts, mpm_bins *bins, float dt,
                   void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (!grid) return MPM_E_ARG;
    DeviceInfo dev;
    if (g.acc_mode == MPM_ACC_EXACT_INT) {
        PartsI p;
        MPM_TRY(parts_i(g, parts, p));
        MPM_TRY(device_info(dev));
        return launch_cic_int_gather(g, p, static_cast<const int64_t *>(grid), dev, static_cast<cudaStream_t>(stream));
    }
    PartsF p;
    MPM_TRY(parts_f(g, parts, true, p));
    MPM_TRY(check_bins(g, bins, p.n));
    MPM_TRY(device_info(dev));
    return launch_g2p(g, static_cast<const float *>(grid), p, view_of(g, *bins), dt, dev,
                      static_cast<cudaStream_t>(stream));
}

mpm_status mpm_step(const mpm_grid_desc *desc, mpm_particles *parts, mpm_bins *bins, void *grid_acc, float *grid_vel,
                    float dt, const float dtg[3], void *stream) {
    MPM_TRY(mpm_bin(desc, parts, bins, 0, stream));
    MPM_TRY(mpm_p2g(desc, parts, bins, grid_acc, dt, stream));
    MPM_TRY(mpm_grid_update(desc, grid_acc, grid_vel, dtg, bins, stream));
    return mpm_g2p(desc, grid_vel, parts, bins, dt, stream);
}

mpm_status mpm_g2p_sorted(const mpm_grid_desc *desc, const float *grid_vel, const mpm_particles *in,
                          mpm_particles *out, mpm_bins *bins, float dt, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT || !grid_vel) return MPM_E_ARG;
    PartsF pi, po;
    MPM_TRY(parts_f(g, in, true, pi));
    MPM_TRY(parts_f(g, out, true, po));
    if (pi.n != po.n || (!pi.id) != (!po.id) || (!pi.F[0]) != (!po.F[0])) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, pi.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_g2p_sorted(g, grid_vel, pi, po, view_of(g, *bins), dt, dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_g2p_binned(const mpm_grid_desc *desc, const float *grid_vel, const mpm_particles *in,
                          mpm_particles *out, mpm_bins *bins, float dt, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT || !grid_vel) return MPM_E_ARG;
    PartsF pi, po;
    MPM_TRY(parts_f(g, in, true, pi));
    MPM_TRY(parts_f(g, out, true, po));
    if (pi.n != po.n || (!pi.id) != (!po.id) || (!pi.F[0]) != (!po.F[0])) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, pi.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_g2p_binned(g, grid_vel, pi, po, view_of(g, *bins), dt, dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_g2p_update(const mpm_grid_desc *desc, void *grid_acc, const float dtg[3], mpm_particles *parts,
                          mpm_bins *bins, float dt, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if ((g.acc_mode != MPM_ACC_I64 && g.acc_mode != MPM_ACC_I32) || !grid_acc || !dtg) return MPM_E_ARG;
    PartsF p;
    MPM_TRY(parts_f(g, parts, true, p));
    MPM_TRY(check_bins(g, bins, p.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    if (bins->next_keys && g.acc_mode != MPM_ACC_I64) return MPM_E_ARG;
    return launch_g2p_update(g, grid_acc, dtg, p, p, view_of(g, *bins), dt, false, bins->next_keys != 0, dev,
                             static_cast<cudaStream_t>(stream));
}

mpm_status mpm_g2p_sorted_update(const mpm_grid_desc *desc, void *grid_acc, const float dtg[3],
                                 const mpm_particles *in, mpm_particles *out, mpm_bins *bins, float dt, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if ((g.acc_mode != MPM_ACC_I64 && g.acc_mode != MPM_ACC_I32) || !grid_acc || !dtg) return MPM_E_ARG;
    PartsF pi, po;
    MPM_TRY(parts_f(g, in, true, pi));
    MPM_TRY(parts_f(g, out, true, po));
    if (pi.n != po.n || (!pi.id) != (!po.id) || (!pi.F[0]) != (!po.F[0])) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, pi.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_g2p_update(g, grid_acc, dtg, pi, po, view_of(g, *bins), dt, true, false, dev,
                             static_cast<cudaStream_t>(stream));
}

mpm_status mpm_step_binned(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                           void *grid_acc, float *grid_vel, float dt, const float dtg[3], void *stream) {
    MPM_TRY(mpm_bin(desc, in, bins, 0, stream));
    MPM_TRY(mpm_p2g(desc, in, bins, grid_acc, dt, stream));
    MPM_TRY(mpm_grid_update(desc, grid_acc, grid_vel, dtg, bins, stream));
    return mpm_g2p_binned(desc, grid_vel, in, out, bins, dt, stream);
}

mpm_status mpm_step_sorted(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                           void *grid_acc, float *grid_vel, float dt, const float dtg[3], void *stream) {
    MPM_TRY(mpm_bin(desc, in, bins, 0, stream));
    MPM_TRY(mpm_p2g(desc, in, bins, grid_acc, dt, stream));
    MPM_TRY(mpm_grid_update(desc, grid_acc, grid_vel, dtg, bins, stream));
    return mpm_g2p_sorted(desc, grid_vel, in, out, bins, dt, stream);
}

mpm_status mpm_step_fused(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                          void *acc_read, void *acc_write, float dt, const float dtg[3], void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode != MPM_ACC_I64 || g.vc || !acc_read || !acc_write || acc_read == acc_write || !dtg)
        return MPM_E_ARG;
    PartsF pi, po;
    MPM_TRY(parts_f(g, in, true, pi));
    MPM_TRY(parts_f(g, out, true, po));
    if (pi.F[0] || po.F[0]) return MPM_E_ARG;
    if (pi.n != po.n || (!pi.id) != (!po.id)) return MPM_E_ARG;
    MPM_TRY(mpm_bin(desc, in, bins, 0, stream));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_g2p2g(g, pi, po, view_of(g, *bins), acc_read, acc_write, dt, dtg, dev,
                        static_cast<cudaStream_t>(stream));
}

mpm_status mpm_iterate(const mpm_grid_desc *desc, mpm_particles *parts, mpm_bins *bins, void *acc_a, void *acc_b,
                       int iterations, void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode != MPM_ACC_I64 || g.vc || !acc_a || !acc_b || acc_a == acc_b || iterations < 1)
        return MPM_E_ARG;
    PartsF p;
    MPM_TRY(parts_f(g, parts, true, p));
    if (p.F[0]) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, p.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_iterate(g, p, view_of(g, *bins), acc_a, acc_b, iterations, dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_step_host(const mpm_grid_desc *desc, mpm_particles *host, mpm_particles *dev_in,
                         mpm_particles *dev_out, mpm_bins *bins, void *grid_acc, float *grid_vel, float dt,
                         const float dtg[3], void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT || !host || !dev_in || !dev_out) return MPM_E_ARG;
    PartsF ph, pa, pb;
    MPM_TRY(parts_f(g, host, true, ph));
    MPM_TRY(parts_f(g, dev_in, true, pa));
    MPM_TRY(parts_f(g, dev_out, true, pb));
    if (ph.n != pa.n || ph.n != pb.n) return MPM_E_ARG;
    if ((!ph.id) != (!pa.id) || (!ph.id) != (!pb.id)) return MPM_E_ARG;
    if ((!ph.F[0]) != (!pa.F[0]) || (!ph.F[0]) != (!pb.F[0])) return MPM_E_ARG;
    if ((!ph.vol) != (!pa.vol) || (!ph.vol) != (!pb.vol) || (!ph.phi) != (!pa.phi) || (!ph.phi) != (!pb.phi))
        return MPM_E_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)ph.n * sizeof(float);
    // the (host, device in, device out) arrays of the state, in one list
    const void *hs[kMaxCopies];
    void *di[kMaxCopies], *dout[kMaxCopies];
    int cnt = 0;
    auto add = [&](const void *h, void *i, void *o) {
        hs[cnt] = h;
        di[cnt] = i;
        dout[cnt] = o;
        ++cnt;
    };
    for (int l = 0; l < g.dim; ++l) add(ph.x[l], pa.x[l], pb.x[l]);
    for (int l = 0; l < g.dim; ++l) add(ph.v[l], pa.v[l], pb.v[l]);
    for (int j = 0; j < g.dim * g.dim; ++j) add(ph.C[j], pa.C[j], pb.C[j]);
    add(ph.m, const_cast<float *>(pa.m), const_cast<float *>(pb.m));
    if (ph.id) add(ph.id, pa.id, pb.id);
    if (ph.F[0])
        for (int j = 0; j < g.dim * g.dim; ++j) add(ph.F[j], pa.F[j], pb.F[j]);
    if (ph.vol) add(ph.vol, pa.vol, pb.vol);
    if (ph.phi) add(ph.phi, pa.phi, pb.phi);
    // pinned host arrays are copied by a kernel through their device view; otherwise one copy per array
    void *hview[kMaxCopies];
    bool pinned = bytes > 0;
    for (int a = 0; a < cnt && pinned; ++a) pinned = (hview[a] = device_view_of_host(hs[a])) != nullptr;
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    if (bytes) {
        if (pinned) {
            MPM_TRY(launch_copy_table(hview, di, cnt, (int64_t)bytes, dev, st));
        } else {
            for (int a = 0; a < cnt; ++a)
                if (cudaMemcpyAsync(di[a], hs[a], bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return MPM_E_CUDA;
        }
    }
    MPM_TRY(mpm_step_sorted(desc, dev_in, dev_out, bins, grid_acc, grid_vel, dt, dtg, stream));
    if (bytes) {
        if (pinned) {
            const void *from[kMaxCopies];
            for (int a = 0; a < cnt; ++a) from[a] = dout[a];
            MPM_TRY(launch_copy_table(from, hview, cnt, (int64_t)bytes, dev, st));
        } else {
            for (int a = 0; a < cnt; ++a)
                if (cudaMemcpyAsync(const_cast<void *>(hs[a]), dout[a], bytes, cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess)
                    return MPM_E_CUDA;
        }
    }
    return MPM_OK;
}

mpm_status mpm_permute(const mpm_grid_desc *desc, const mpm_particles *in, mpm_particles *out, const mpm_bins *bins,
                       void *stream) {
    GridP g;
    MPM_TRY(make_grid(desc, g));
    if (g.acc_mode == MPM_ACC_EXACT_INT) return MPM_E_ARG;
    PartsF pi, po;
    MPM_TRY(parts_f(g, in, true, pi));
    MPM_TRY(parts_f(g, out, true, po));
    if (pi.n != po.n) return MPM_E_ARG;
    MPM_TRY(check_bins(g, bins, pi.n));
    DeviceInfo dev;
    MPM_TRY(device_info(dev));
    return launch_permute(g, pi, po, bins->perm, dev, static_cast<cudaStream_t>(stream));
}

mpm_status mpm_read_status(const mpm_bins *bins, uint32_t *host_out, void *stream) {
    if (!bins || !bins->status || !host_out) return MPM_E_ARG;
    if (cudaMemcpyAsync(host_out, bins->status, MPM_STATUS_WORDS * sizeof(uint32_t), cudaMemcpyDeviceToHost,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MPM_E_CUDA;
    return MPM_OK;
}

}  // extern "C"
