// internal.h -- host-side declarations shared by the library's translation
// units (workspace view, device facts, kernel launchers).  Not part of the ABI.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mpm.h"

namespace mpm {

struct GridP;
struct PartsF;

// Device arrays carved from the caller's workspace (see mpm_bins_init).
struct WsView {
    uint32_t *key, *perm;
    uint32_t *heads;      // [n] run heads, each bucket's in its range [start, start + count); then sorted
    uint32_t *tails;      // [n] run tails, likewise; then the runs' offsets inside the bucket
    uint32_t *count;      // [ntiles + 1] particles per bucket (last: outside the domain)
    uint32_t *start;      // [ntiles + 2] exclusive prefix of count
    uint32_t *hcnt;       // [ntiles + 1] runs per bucket (heads appended)
    uint32_t *tcnt;       // [ntiles + 1] tails appended
    uint32_t *active;     // [ntiles]
    uint32_t *slices;     // [2 * max_slices]
    uint32_t *large_list; // [ntiles + 1] buckets of more than 512 runs
    uint32_t *partial;    // scan block totals, 3 words per 1024 buckets
    uint32_t *status;     // [MPM_STATUS_WORDS]
    uint32_t *cellcount;  // int32 mode only: [ntiles * T^dim], else null
    uint32_t *readers;    // [nblocks] work items that have read each node block (G2P with the update on load)
    uint32_t *count_next; // [ntiles + 1] the histogram of the next keys a G2P wrote (MPM_BIN_KEYS_FROM_G2P)
};

struct DeviceInfo {
    int device;
    int sms;
};

mpm_status device_info(DeviceInfo &out);

mpm_status launch_bin(const GridP &g, const PartsF &p, const WsView &w, bool keys_from_g2p, const DeviceInfo &dev,
                      cudaStream_t st);
mpm_status launch_p2g(const GridP &g, const PartsF &p, const WsView &w, void *grid_acc, float dt, bool records,
                      const DeviceInfo &dev, cudaStream_t st);
void launch_rollback(const GridP &g, void *grid_acc, const uint32_t *status, const DeviceInfo &dev,
                     cudaStream_t st);
mpm_status launch_grid_update(const GridP &g, void *grid_acc, float *vel, const float dtg[3], const WsView &w,
                              const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_g2p(const GridP &g, const float *vel, const PartsF &p, const WsView &w, float dt,
                      const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_g2p_sorted(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w,
                             float dt, const DeviceInfo &dev, cudaStream_t st);
void launch_copy_rest(const GridP &g, const PartsF &in, const PartsF &out, const WsView &w, const DeviceInfo &dev,
                      cudaStream_t st);
mpm_status launch_g2p2g(const GridP &g, const PartsF &in, const PartsF &out, const WsView &w, void *acc_read,
                        void *acc_write, float dt, const float dtg[3], const DeviceInfo &dev, cudaStream_t st);
void launch_clear_blocks(const GridP &g, long long *acc, const WsView &w, const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_iterate(const GridP &g, const PartsF &p, const WsView &w, void *acc_a, void *acc_b,
                          int iterations, const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_g2p_update(const GridP &g, const void *acc, const float dtg[3], const PartsF &in, const PartsF &out,
                             const WsView &w, float dt, bool sorted, bool next_keys, const DeviceInfo &dev,
                             cudaStream_t st);
mpm_status launch_g2p_binned(const GridP &g, const float *vel, const PartsF &in, const PartsF &out, const WsView &w,
                             float dt, const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_permute(const GridP &g, const PartsF &in, const PartsF &out, const uint32_t *perm,
                          const DeviceInfo &dev, cudaStream_t st);

// Whole-array copies by a kernel (host_copy.cu): `count` arrays of `bytes`
// each, src/dst device-addressable (device memory, or pinned host memory
// through its device view).
constexpr int kMaxCopies = 32;
void *device_view_of_host(const void *p);
mpm_status launch_copy_table(const void *const *src, void *const *dst, int count, int64_t bytes,
                             const DeviceInfo &dev, cudaStream_t st);

// Integer cloud-in-cell transfer (integer particles, int64 grid).
struct PartsI {
    const int32_t *X[3];
    int64_t *v[3];
    const int64_t *m;
    int64_t n;
};
mpm_status launch_cic_int_p2g(const GridP &g, const PartsI &p, int64_t *acc, uint32_t *status,
                              uint64_t *scratch, const DeviceInfo &dev, cudaStream_t st);
mpm_status launch_cic_int_gather(const GridP &g, const PartsI &p, const int64_t *acc, const DeviceInfo &dev,
                                 cudaStream_t st);

}  // namespace mpm
