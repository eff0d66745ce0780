// bin.cu -- cell keys and the stable counting sort of particles into tiles.
//
// "Particle Worlds, part 3", Step 3 and Step 4: a counting sort in three
// phases, histogram -> exclusive prefix sum -> scatter, the scan as per-block
// scans, a scan of the block totals and an add-back.  The page's scatter
// claims slots with an atomic cursor and so leaves the order inside a bucket
// unspecified; the implementation guide (section 2.1, caveat (b), and rule 3)
// asks for every such race to be neutralised by a sort on a stable key.
// Here the buckets are tiles of T^dim base cells (section 2.1: bin into
// tiles, sort an index buffer, particles never move), the atomic scatter
// fills each tile's range, and one CTA per tile then sorts the range by
// (cell, particle index) in shared memory, which makes the permutation the
// stable sort of the keys -- a deterministic function of the keys.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_keys          key per particle, warp-aggregated tile histogram,
//                   out-of-domain count (int32 mode: per-cell counts)
//   k_scan_reduce / k_scan_top / k_scan_final
//                   exclusive scans of (count, P2G slices, active flag) over
//                   the buckets; active-tile list, P2G work list, cursors
//   k_scatter       warp-aggregated atomic scatter of indices into buckets
//   k_tile_sort     per-bucket sort by (cell, index) in shared memory
//   k_big_sort      buckets too large for shared memory: a stable counting
//                   sort over the key array in index order
//   k_nbr_bound     int32 mode: most stencils covering one node (the
//                   accumulator bound, checked before any scatter)
#include "common.cuh"
#include "internal.h"

namespace mpm {

// --------------------------------------------------------------------------
__global__ void k_keys(GridP g, PartsF p, uint32_t *__restrict__ key, uint32_t *__restrict__ count,
                       uint32_t *__restrict__ cellcount, uint32_t *__restrict__ status) {
    const int64_t n = p.n;
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint32_t bucket_invalid = (uint32_t)g.ntiles;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < n;
         base += warps * 32) {
        const int64_t i = base + lane;
        uint32_t k = kKeyInvalid, bucket = 0xFFFFFFFFu;
        if (i < n) {
            int b[3] = {0, 0, 0};
            float f;
            bool ok = true;
            for (int l = 0; l < g.dim; ++l) ok = ok && base_frac(p.x[l][i], g.inv_dx, g.n[l], b[l], f);
            if (ok) {
                k = cell_key(g, b);
                bucket = k >> g.cpt_log2;
                if (cellcount) atomicAdd(&cellcount[k], 1u);
            } else {
                bucket = bucket_invalid;
            }
            key[i] = k;
        }
        // warp-aggregated histogram: one atomic per distinct bucket in the warp
        const uint32_t live = __ballot_sync(0xFFFFFFFFu, i < n);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bucket) & live;
        if (i < n && (peers & lanemask_lt()) == 0) {
            atomicAdd(&count[bucket], (uint32_t)__popc(peers));
            if (bucket == bucket_invalid) atomicAdd(&status[MPM_ST_N_OUTSIDE], (uint32_t)__popc(peers));
        }
    }
}

// --------------------------------------------------------------------------
// Scans over the nb = ntiles + 1 buckets (the last bucket holds the particles
// outside the domain).  Each thread of a 256-thread block owns 4 buckets.
constexpr int kScanThreads = 256;
constexpr int kScanItems = 4;
constexpr int kScanBlock = kScanThreads * kScanItems;

struct Tri {
    uint32_t a, b, c;
};

__device__ __forceinline__ Tri tri_add(Tri x, Tri y) { return {x.a + y.a, x.b + y.b, x.c + y.c}; }

__device__ __forceinline__ Tri bucket_values(const GridP &g, const uint32_t *count, int64_t nb, int64_t b) {
    if (b >= nb) return {0, 0, 0};
    uint32_t c = count[b];
    if (b == nb - 1) return {c, 0, 0};  // outside-the-domain bucket: no P2G work
    return {c, (c + kSliceParticles - 1) / kSliceParticles, c > 0 ? 1u : 0u};
}

// Block-wide exclusive scan of one Tri per thread; returns the block total.
__device__ Tri block_exclusive_scan(Tri v, Tri &excl) {
    __shared__ Tri warp_tot[kScanThreads / 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    Tri inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t a = __shfl_up_sync(0xFFFFFFFFu, inc.a, d);
        uint32_t b = __shfl_up_sync(0xFFFFFFFFu, inc.b, d);
        uint32_t c = __shfl_up_sync(0xFFFFFFFFu, inc.c, d);
        if ((int)lane >= d) inc = tri_add(inc, {a, b, c});
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    Tri before = {0, 0, 0}, total = {0, 0, 0};
    for (int w = 0; w < kScanThreads / 32; ++w) {
        if (w < (int)warp) before = tri_add(before, warp_tot[w]);
        total = tri_add(total, warp_tot[w]);
    }
    excl = {before.a + inc.a - v.a, before.b + inc.b - v.b, before.c + inc.c - v.c};
    __syncthreads();
    return total;
}

__global__ void k_scan_reduce(GridP g, const uint32_t *__restrict__ count, int64_t nb, Tri *__restrict__ partial) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tri s = {0, 0, 0};
    for (int j = 0; j < kScanItems; ++j) s = tri_add(s, bucket_values(g, count, nb, b0 + j));
    Tri excl;
    Tri tot = block_exclusive_scan(s, excl);
    if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// One block: exclusive scan of the block totals (in place) and the grand totals.
__global__ void k_scan_top(Tri *__restrict__ partial, int64_t nblocks, const uint32_t *__restrict__ count,
                           int64_t nb, uint32_t *__restrict__ status) {
    Tri carry = {0, 0, 0};
    for (int64_t base = 0; base < nblocks; base += kScanThreads) {
        int64_t i = base + threadIdx.x;
        Tri v = i < nblocks ? partial[i] : Tri{0, 0, 0};
        Tri excl;
        Tri tot = block_exclusive_scan(v, excl);
        if (i < nblocks) partial[i] = tri_add(carry, excl);
        carry = tri_add(carry, tot);
    }
    if (threadIdx.x == 0) {
        status[MPM_ST_N_VALID] = carry.a - count[nb - 1];
        status[MPM_ST_N_SLICES] = carry.b;
        status[MPM_ST_N_ACTIVE] = carry.c;
    }
}

__global__ void k_scan_final(GridP g, const uint32_t *__restrict__ count, int64_t nb, const Tri *__restrict__ partial,
                             uint32_t *__restrict__ start, uint32_t *__restrict__ cursor,
                             uint32_t *__restrict__ active, uint32_t *__restrict__ slices,
                             uint32_t *__restrict__ big, uint32_t *__restrict__ status, int sort_cap) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tri v[kScanItems];
    Tri s = {0, 0, 0};
    for (int j = 0; j < kScanItems; ++j) {
        v[j] = bucket_values(g, count, nb, b0 + j);
        s = tri_add(s, v[j]);
    }
    Tri excl;
    block_exclusive_scan(s, excl);
    Tri run = tri_add(partial[blockIdx.x], excl);
    for (int j = 0; j < kScanItems; ++j) {
        const int64_t b = b0 + j;
        if (b >= nb) break;
        start[b] = run.a;
        cursor[b] = run.a;
        if (v[j].c) active[run.c] = (uint32_t)b;
        for (uint32_t s2 = 0; s2 < v[j].b; ++s2) {
            slices[2 * (int64_t)(run.b + s2)] = (uint32_t)b;
            slices[2 * (int64_t)(run.b + s2) + 1] = s2 * kSliceParticles;
        }
        if (v[j].a > (uint32_t)sort_cap) big[atomicAdd(&status[MPM_ST_N_BIG_TILES], 1u)] = (uint32_t)b;
        run = tri_add(run, v[j]);
        if (b == nb - 1) start[nb] = run.a;
    }
}

// --------------------------------------------------------------------------
__global__ void k_scatter(GridP g, const uint32_t *__restrict__ key, int64_t n, uint32_t *__restrict__ cursor,
                          uint32_t *__restrict__ tmp) {
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint32_t bucket_invalid = (uint32_t)g.ntiles;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < n;
         base += warps * 32) {
        const int64_t i = base + lane;
        uint32_t bucket = 0xFFFFFFFFu;
        if (i < n) {
            uint32_t k = key[i];
            bucket = k == kKeyInvalid ? bucket_invalid : (k >> g.cpt_log2);
        }
        const uint32_t live = __ballot_sync(0xFFFFFFFFu, i < n);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bucket) & live;
        const uint32_t leader = __ffs(peers) - 1;
        uint32_t slot = 0;
        if (i < n && lane == leader) slot = atomicAdd(&cursor[bucket], (uint32_t)__popc(peers));
        slot = __shfl_sync(0xFFFFFFFFu, slot, leader);
        if (i < n) tmp[slot + __popc(peers & lanemask_lt())] = (uint32_t)i;
    }
}

// --------------------------------------------------------------------------
// Per-bucket sort by (cell within tile, particle index).  Composite keys are
// distinct, so any correct sort gives the stable order; a bitonic network in
// shared memory, padded to a power of two with all-ones sentinels.
template <typename K>
__device__ void bitonic_sort_smem(K *s, int n_pow2) {
    for (int k = 2; k <= n_pow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = threadIdx.x; t < (n_pow2 >> 1); t += blockDim.x) {
                const int i = (t / j) * 2 * j + (t % j);
                const int pr = i + j;
                const bool up = (i & k) == 0;
                K a = s[i], b = s[pr];
                if ((a > b) == up) {
                    s[i] = b;
                    s[pr] = a;
                }
            }
            __syncthreads();
        }
    }
}

template <typename K>
__global__ void k_tile_sort(GridP g, const uint32_t *__restrict__ key, const uint32_t *__restrict__ tmp,
                            const uint32_t *__restrict__ start, const uint32_t *__restrict__ count,
                            const uint32_t *__restrict__ active, int64_t nb, uint32_t *__restrict__ perm,
                            const uint32_t *__restrict__ status, int idx_bits, int cap) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    K *s = reinterpret_cast<K *>(smem_raw);
    const uint32_t n_active = status[MPM_ST_N_ACTIVE];
    const uint32_t local_mask = (1u << g.cpt_log2) - 1;
    // items: the active tiles, then the outside-the-domain bucket
    for (uint32_t item = blockIdx.x; item <= n_active; item += gridDim.x) {
        const uint32_t b = item < n_active ? active[item] : (uint32_t)(nb - 1);
        const uint32_t beg = start[b];
        const uint32_t cnt = count[b];
        if (cnt == 0 || cnt > (uint32_t)cap) continue;  // empty, or sorted by k_big_sort
        if (cnt == 1) {
            if (threadIdx.x == 0) perm[beg] = tmp[beg];
            continue;
        }
        int n_pow2 = 1;
        while (n_pow2 < (int)cnt) n_pow2 <<= 1;
        for (int r = threadIdx.x; r < n_pow2; r += blockDim.x) {
            K c = ~(K)0;
            if (r < (int)cnt) {
                const uint32_t idx = tmp[beg + r];
                const uint32_t k = key[idx];
                const K local = k == kKeyInvalid ? (K)0 : (K)(k & local_mask);
                c = (local << idx_bits) | (K)idx;
            }
            s[r] = c;
        }
        __syncthreads();
        bitonic_sort_smem(s, n_pow2);
        const K idx_mask = (idx_bits >= (int)(8 * sizeof(K))) ? ~(K)0 : (((K)1 << idx_bits) - 1);
        for (int r = threadIdx.x; r < (int)cnt; r += blockDim.x) perm[beg + r] = (uint32_t)(s[r] & idx_mask);
        __syncthreads();
    }
}

// Buckets above the shared-memory capacity: one CTA per bucket reads the key
// array in index order twice (cell histogram, then stable placement).  Slow
// (O(n) per bucket) and only reached by very dense inputs.
constexpr int kBigThreads = 256;
constexpr int kMaxCells = 4096;

__global__ void k_big_sort(GridP g, const uint32_t *__restrict__ key, int64_t n, const uint32_t *__restrict__ start,
                           const uint32_t *__restrict__ big, int64_t nb, uint32_t *__restrict__ perm,
                           const uint32_t *__restrict__ status) {
    __shared__ uint32_t cell_off[kMaxCells];
    __shared__ uint32_t warp_cnt[kBigThreads / 32][64];
    __shared__ uint32_t warp_off[kBigThreads / 32][64];
    const uint32_t nbig = status[MPM_ST_N_BIG_TILES];
    const uint32_t ncell = 1u << g.cpt_log2;
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    for (uint32_t item = blockIdx.x; item < nbig; item += gridDim.x) {
        const uint32_t b = big[item];
        const bool outside = b == (uint32_t)(nb - 1);
        const uint32_t cells = outside ? 1u : ncell;
        for (uint32_t c = threadIdx.x; c < cells; c += blockDim.x) cell_off[c] = 0;
        __syncthreads();
        // pass 1: cell histogram of this bucket
        for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t k = key[i];
            const uint32_t kb = k == kKeyInvalid ? (uint32_t)(nb - 1) : (k >> g.cpt_log2);
            if (kb == b) atomicAdd(&cell_off[outside ? 0u : (k & (ncell - 1))], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t run = start[b];
            for (uint32_t c = 0; c < cells; ++c) {
                uint32_t t = cell_off[c];
                cell_off[c] = run;
                run += t;
            }
        }
        __syncthreads();
        // pass 2: stable placement, 256 indices per round, cells in groups of 64
        for (int64_t base = 0; base < n; base += blockDim.x) {
            const int64_t i = base + threadIdx.x;
            uint32_t c = 0xFFFFFFFFu;
            if (i < n) {
                const uint32_t k = key[i];
                const uint32_t kb = k == kKeyInvalid ? (uint32_t)(nb - 1) : (k >> g.cpt_log2);
                if (kb == b) c = outside ? 0u : (k & (ncell - 1));
            }
            for (uint32_t group = 0; group < cells; group += 64) {
                const bool mine = c != 0xFFFFFFFFu && c >= group && c < group + 64;
                const uint32_t cg = mine ? c - group : 64u;
                const uint32_t peers = __match_any_sync(0xFFFFFFFFu, cg);
                if (lane < 64 / 2) {
                    warp_cnt[warp][lane] = 0;
                    warp_cnt[warp][lane + 32] = 0;
                }
                __syncwarp();
                if (mine && (peers & lanemask_lt()) == 0) warp_cnt[warp][cg] = __popc(peers);
                __syncthreads();
                if (threadIdx.x < 64 && group + threadIdx.x < cells) {
                    uint32_t run = cell_off[group + threadIdx.x];
                    for (int w = 0; w < kBigThreads / 32; ++w) {
                        warp_off[w][threadIdx.x] = run;
                        run += warp_cnt[w][threadIdx.x];
                    }
                    cell_off[group + threadIdx.x] = run;
                }
                __syncthreads();
                if (mine) perm[warp_off[warp][cg] + __popc(peers & lanemask_lt())] = (uint32_t)i;
                __syncthreads();
            }
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// int32 accumulators: for every node, the number of particles whose stencil
// covers it is the sum of the counts of the 3^dim base cells below it.
__global__ void k_nbr_bound(GridP g, const uint32_t *__restrict__ cellcount, uint32_t *__restrict__ status) {
    uint32_t best = 0;
    for (int64_t node = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; node < g.nodes;
         node += (int64_t)gridDim.x * blockDim.x) {
        int idx[3];
        idx[0] = (int)(node % g.n[0]);
        idx[1] = (int)((node / g.n[0]) % g.n[1]);
        idx[2] = (int)(node / ((int64_t)g.n[0] * g.n[1]));
        uint32_t sum = 0;
        for (int a2 = 0; a2 < (g.dim == 3 ? 3 : 1); ++a2)
            for (int a1 = 0; a1 < 3; ++a1)
                for (int a0 = 0; a0 < 3; ++a0) {
                    int b[3] = {idx[0] - a0, idx[1] - a1, g.dim == 3 ? idx[2] - a2 : 0};
                    bool ok = true;
                    for (int l = 0; l < g.dim; ++l) ok = ok && b[l] >= 0 && b[l] <= g.n[l] - 3;
                    if (ok) sum += cellcount[cell_key(g, b)];
                }
        best = max(best, sum);
    }
    for (int d = 16; d > 0; d >>= 1) best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, d));
    if (lane_id() == 0 && best > 0) {
        atomicMax(&status[MPM_ST_MAX_NEIGHBOURS], best);
        if (best > kI32MaxContributions) atomicOr(&status[MPM_ST_FLAGS], (1u << MPM_E_BOUND) | kFlagNoScatter);
    }
}

// --------------------------------------------------------------------------
mpm_status launch_bin(const GridP &g, const PartsF &p, const WsView &w, const DeviceInfo &dev,
                      cudaStream_t st) {
    const int64_t n = p.n;
    const int64_t nb = g.ntiles + 1;
    cudaMemsetAsync(w.status, 0, MPM_STATUS_WORDS * sizeof(uint32_t), st);
    cudaMemsetAsync(w.count, 0, nb * sizeof(uint32_t), st);
    if (w.cellcount) cudaMemsetAsync(w.cellcount, 0, (size_t)(g.ntiles << g.cpt_log2) * sizeof(uint32_t), st);
    const int threads = 256;
    const int grid_p = (int)std::max<int64_t>(1, std::min<int64_t>((n + threads - 1) / threads, dev.sms * 8));
    if (n > 0) k_keys<<<grid_p, threads, 0, st>>>(g, p, w.key, w.count, w.cellcount, w.status);
    const int64_t nblk = (nb + kScanBlock - 1) / kScanBlock;
    k_scan_reduce<<<(unsigned)nblk, kScanThreads, 0, st>>>(g, w.count, nb, (Tri *)w.partial);
    k_scan_top<<<1, kScanThreads, 0, st>>>((Tri *)w.partial, nblk, w.count, nb, w.status);
    const bool narrow = n <= (int64_t(1) << (32 - g.cpt_log2));
    const int cap = narrow ? kSortCap32 : kSortCap64;
    k_scan_final<<<(unsigned)nblk, kScanThreads, 0, st>>>(g, w.count, nb, (const Tri *)w.partial, w.start,
                                                          w.cursor, w.active, w.slices, w.big, w.status, cap);
    if (n > 0) {
        k_scatter<<<grid_p, threads, 0, st>>>(g, w.key, n, w.cursor, w.tmp);
        const int sort_blocks = dev.sms * 2;
        // the sort buffers are 64 KB of dynamic shared memory (above the 48 KB default)
        cudaFuncSetAttribute(k_tile_sort<uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSortCap32 * (int)sizeof(uint32_t));
        cudaFuncSetAttribute(k_tile_sort<uint64_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSortCap64 * (int)sizeof(uint64_t));
        if (narrow) {
            int idx_bits = 32 - g.cpt_log2;
            k_tile_sort<uint32_t><<<sort_blocks, 512, kSortCap32 * sizeof(uint32_t), st>>>(
                g, w.key, w.tmp, w.start, w.count, w.active, nb, w.perm, w.status, idx_bits, cap);
        } else {
            k_tile_sort<uint64_t><<<sort_blocks, 512, kSortCap64 * sizeof(uint64_t), st>>>(
                g, w.key, w.tmp, w.start, w.count, w.active, nb, w.perm, w.status, 32, cap);
        }
        k_big_sort<<<dev.sms, kBigThreads, 0, st>>>(g, w.key, n, w.start, w.big, nb, w.perm, w.status);
    }
    if (w.cellcount) k_nbr_bound<<<dev.sms * 4, 256, 0, st>>>(g, w.cellcount, w.status);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
