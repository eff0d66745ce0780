// bin.cu -- cell keys and the stable counting sort of particles into tiles.
//
// "Particle Worlds, part 3", Step 3 and Step 4: a counting sort in three
// phases, histogram -> exclusive prefix sum -> scatter, the scan as per-block
// scans, a scan of the block totals and an add-back.  The page's scatter
// claims slots with an atomic cursor and so leaves the order inside a bucket
// unspecified; the implementation guide (section 2.1, caveat (b), and rule 3)
// asks for every such race to be neutralised by a sort on a stable key.
// Here the buckets are tiles of T^dim base cells (section 2.1: bin into
// tiles, sort an index buffer) and the permutation is the STABLE counting
// sort by tile: each tile's particles in particle-index order, a
// deterministic function of the keys.
//
// The scatter works on runs, not on single particles.  A run is a maximal
// range of consecutive particle indices whose particles share one bucket; a
// bucket's particles in index order are its runs in order of their first
// index, each run in order.  So it is enough to collect each bucket's runs
// (their heads and tails, in any order), sort the heads and the tails of the
// bucket (runs of one bucket are disjoint, so the k-th smallest head and the
// k-th smallest tail belong to the same run), prefix-sum the run lengths and
// write perm position by position.  When the particles are already stored in
// bin order (as the sorted G2P leaves them) a tile holds a handful of runs
// and the sort is nearly free; in a random order every particle is a run and
// the same code sorts indices.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_keys          key per particle, tile histogram aggregated over runs
//                   (int32 mode: per-cell counts); skipped when the last G2P
//                   wrote both (MPM_BIN_KEYS_FROM_G2P)
//   k_scan_reduce / k_scan_top / k_scan_final
//                   exclusive scans of (count, P2G slices, active flag) over
//                   the buckets; active-tile list, P2G work list; clears the
//                   run counters
//   k_runs          run heads and tails, appended to their bucket's range
//   k_sort_runs     per bucket with 33..512 runs (one warp): heads and
//                   tails sorted in registers, run offsets
//   k_sort_runs_large  the same for more runs (one block; shared memory, or
//                   global memory above kSmemRuns)
//   k_emit          perm, position by position; sorts buckets of at most 32
//                   runs itself
//   k_nbr_bound     int32 mode: most stencils covering one node (for the
//                   accumulator bound mpm_p2g checks before any scatter)
#include "common.cuh"
#include "internal.h"

namespace mpm {

constexpr int kKeysUnroll = 4;   // particles per lane per iteration (loads in flight)

// Keys of the 32 * kKeysUnroll particles from `base` (FULL: all below n, so
// no bounds tests); tile histogram aggregated over runs of equal buckets
// among each 32 consecutive particles (one atomic per run: particles kept in
// bin order come in long runs).
template <int DIM, int T, bool FULL>
__device__ __forceinline__ void keys_span(const GridP &g, const PartsF &p, int64_t n, int64_t base, uint32_t lane,
                                          uint32_t *__restrict__ key, uint32_t *__restrict__ count,
                                          uint32_t *__restrict__ cellcount, uint32_t *__restrict__ status) {
    constexpr int LOG = T == 4 ? 2 : 3;
    const uint32_t bucket_invalid = (uint32_t)g.ntiles;
    const float *xs[DIM];
#pragma unroll
    for (int l = 0; l < DIM; ++l) xs[l] = p.x[l] + base + lane;
    uint32_t *ks = key + base + lane;
    float xv[kKeysUnroll][DIM];
#pragma unroll
    for (int u = 0; u < kKeysUnroll; ++u) {
        const bool in = FULL || base + u * 32 + lane < n;
#pragma unroll
        for (int l = 0; l < DIM; ++l) xv[u][l] = in ? xs[l][u * 32] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kKeysUnroll; ++u) {
        const bool in = FULL || base + u * 32 + lane < n;
        uint32_t k = kKeyInvalid, bucket = bucket_invalid;
        if (in) {
            int b[3] = {0, 0, 0};
            float f;
            bool ok = true;
#pragma unroll
            for (int l = 0; l < DIM; ++l) ok = base_frac(xv[u][l], g.inv_dx, g.n[l], b[l], f) && ok;
            if (ok) {
                k = cell_key_t<DIM, T>(g, b);
                bucket = k >> (DIM * LOG);
                if (cellcount) atomicAdd(&cellcount[k], 1u);
            }
            ks[u * 32] = k;
        }
        // runs of equal buckets: the head lane adds the run's length
        const uint32_t live = FULL ? 0xFFFFFFFFu : __ballot_sync(0xFFFFFFFFu, in);
        const uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, bucket, 1);
        const uint32_t heads = __ballot_sync(0xFFFFFFFFu, in && (lane == 0 || prev != bucket));
        if ((heads >> lane) & 1u) {
            const uint32_t later = heads & ~((2u << lane) - 1u);   // heads after this lane (lane 31: none)
            const uint32_t stop = later ? (uint32_t)(__ffs(later) - 1) : (uint32_t)(32 - __clz(live));
            atomicAdd(&count[bucket], stop - lane);
        }
    }
}

// Key per particle and tile histogram (keys_span).
template <int DIM, int T>
__global__ void __launch_bounds__(256) k_keys(GridP g, PartsF p, uint32_t *__restrict__ key,
                                              uint32_t *__restrict__ count, uint32_t *__restrict__ cellcount,
                                              uint32_t *__restrict__ status) {
    const int64_t n = p.n;
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    constexpr int64_t kSpan = 32 * kKeysUnroll;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kSpan; base < n;
         base += warps * kSpan) {
        if (base + kSpan <= n) keys_span<DIM, T, true>(g, p, n, base, lane, key, count, cellcount, status);
        else keys_span<DIM, T, false>(g, p, n, base, lane, key, count, cellcount, status);
    }
}

// --------------------------------------------------------------------------
// Scans over the nb = ntiles + 1 buckets (the last bucket holds the particles
// outside the domain).  Each thread of a 256-thread block owns 4 buckets.
// Three running totals: particles, P2G slices and active tiles.
constexpr int kScanThreads = 256;
constexpr int kScanItems = 4;
constexpr int kScanBlock = kScanThreads * kScanItems;

struct Tot3 {
    uint32_t v[3];
};

__device__ __forceinline__ Tot3 tot_add(const Tot3 &x, const Tot3 &y) {
    return Tot3{{x.v[0] + y.v[0], x.v[1] + y.v[1], x.v[2] + y.v[2]}};
}

__device__ __forceinline__ Tot3 tot_zero() { return Tot3{{0, 0, 0}}; }

__device__ __forceinline__ Tot3 bucket_values(const uint32_t *count, int64_t nb, int64_t b) {
    if (b >= nb) return tot_zero();
    const uint32_t c = count[b];
    const bool outside = b == nb - 1;
    Tot3 r;
    r.v[0] = c;
    r.v[1] = outside ? 0u : (c + kSliceParticles - 1) / kSliceParticles;  // no P2G work outside
    r.v[2] = (!outside && c > 0) ? 1u : 0u;
    return r;
}

// Block-wide exclusive scan of one Tot3 per thread; returns the block total.
__device__ Tot3 block_exclusive_scan(const Tot3 &v, Tot3 &excl) {
    __shared__ Tot3 warp_tot[kScanThreads / 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    Tot3 inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        Tot3 t;
#pragma unroll
        for (int i = 0; i < 3; ++i) t.v[i] = __shfl_up_sync(0xFFFFFFFFu, inc.v[i], d);
        if ((int)lane >= d) inc = tot_add(inc, t);
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    Tot3 before = tot_zero(), total = tot_zero();
    for (int w = 0; w < kScanThreads / 32; ++w) {
        if (w < (int)warp) before = tot_add(before, warp_tot[w]);
        total = tot_add(total, warp_tot[w]);
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) excl.v[i] = before.v[i] + inc.v[i] - v.v[i];
    __syncthreads();
    return total;
}

__global__ void k_scan_reduce(const uint32_t *__restrict__ count, int64_t nb, Tot3 *__restrict__ partial) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tot3 s = tot_zero();
    for (int j = 0; j < kScanItems; ++j) s = tot_add(s, bucket_values(count, nb, b0 + j));
    Tot3 excl;
    Tot3 tot = block_exclusive_scan(s, excl);
    if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// One block: exclusive scan of the block totals (in place) and the grand totals (with the
// in-domain and outside counts).
__global__ void k_scan_top(Tot3 *__restrict__ partial, int64_t nblocks, const uint32_t *__restrict__ count,
                           int64_t nb, uint32_t *__restrict__ status) {
    Tot3 carry = tot_zero();
    for (int64_t base = 0; base < nblocks; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        const Tot3 v = i < nblocks ? partial[i] : tot_zero();
        Tot3 excl;
        const Tot3 tot = block_exclusive_scan(v, excl);
        if (i < nblocks) partial[i] = tot_add(carry, excl);
        carry = tot_add(carry, tot);
    }
    if (threadIdx.x == 0) {
        status[MPM_ST_N_OUTSIDE] = count[nb - 1];
        status[MPM_ST_N_VALID] = carry.v[0] - count[nb - 1];
        status[MPM_ST_N_SLICES] = carry.v[1];
        status[MPM_ST_N_ACTIVE] = carry.v[2];
    }
}

__global__ void k_scan_final(const uint32_t *__restrict__ count, int64_t nb, const Tot3 *__restrict__ partial,
                             uint32_t *__restrict__ start, uint32_t *__restrict__ hcnt,
                             uint32_t *__restrict__ tcnt, uint32_t *__restrict__ active,
                             uint32_t *__restrict__ slices) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tot3 v[kScanItems];
    Tot3 s = tot_zero();
    for (int j = 0; j < kScanItems; ++j) {
        v[j] = bucket_values(count, nb, b0 + j);
        s = tot_add(s, v[j]);
    }
    Tot3 excl;
    block_exclusive_scan(s, excl);
    Tot3 run = tot_add(partial[blockIdx.x], excl);
    for (int j = 0; j < kScanItems; ++j) {
        const int64_t b = b0 + j;
        if (b >= nb) break;
        start[b] = run.v[0];
        hcnt[b] = 0;
        tcnt[b] = 0;
        if (v[j].v[2]) active[run.v[2]] = (uint32_t)b;
        for (uint32_t s2 = 0; s2 < v[j].v[1]; ++s2) {
            slices[2 * (int64_t)(run.v[1] + s2)] = (uint32_t)b;
            slices[2 * (int64_t)(run.v[1] + s2) + 1] = s2 * kSliceParticles;
        }
        run = tot_add(run, v[j]);
        if (b == nb - 1) start[nb] = run.v[0];
    }
}

// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bucket_of(uint32_t k, int cpt_log2, uint32_t bucket_invalid) {
    return k == kKeyInvalid ? bucket_invalid : (k >> cpt_log2);
}

// Run heads (first index of a run) and tails (last index), each appended to
// its bucket's range of `heads` / `tails` (a bucket has at most as many runs
// as particles, so its range [start, start + count) has room).
template <int DIM, int T, bool FULL>
__device__ __forceinline__ void runs_span(int64_t n, int64_t base, uint32_t lane, uint32_t binv,
                                          const uint32_t *__restrict__ key, const uint32_t *__restrict__ start,
                                          uint32_t *__restrict__ hcnt, uint32_t *__restrict__ tcnt,
                                          uint32_t *__restrict__ heads, uint32_t *__restrict__ tails) {
    constexpr int CPT = DIM * (T == 4 ? 2 : 3);
    constexpr int64_t kSpan = 32 * kKeysUnroll;
    const uint32_t *ks = key + base + lane;
    uint32_t bk[kKeysUnroll];
#pragma unroll
    for (int u = 0; u < kKeysUnroll; ++u)
        bk[u] = bucket_of((FULL || base + u * 32 + lane < n) ? ks[u * 32] : kKeyInvalid, CPT, binv);
    // the buckets just before and just after the span (lane 0 / lane 31 use them)
    const uint32_t bprev = (lane == 0 && base > 0) ? bucket_of(key[base - 1], CPT, binv) : binv;
    const uint32_t bnext = (lane == 31 && base + kSpan < n) ? bucket_of(key[base + kSpan], CPT, binv) : binv;
#pragma unroll
    for (int u = 0; u < kKeysUnroll; ++u) {
        const int64_t i = base + u * 32 + lane;
        const uint32_t up = __shfl_up_sync(0xFFFFFFFFu, bk[u], 1);
        const uint32_t dn = __shfl_down_sync(0xFFFFFFFFu, bk[u], 1);
        const uint32_t last_before = u > 0 ? __shfl_sync(0xFFFFFFFFu, bk[u > 0 ? u - 1 : 0], 31) : bprev;
        const uint32_t first_after =
            u + 1 < kKeysUnroll ? __shfl_sync(0xFFFFFFFFu, bk[u + 1 < kKeysUnroll ? u + 1 : u], 0) : bnext;
        const uint32_t bp = lane == 0 ? last_before : up;
        const uint32_t bn = lane == 31 ? first_after : dn;
        if (FULL || i < n) {
            const uint32_t b = bk[u];
            const bool head = i == 0 || bp != b;
            const bool tail = i == n - 1 || bn != b;
            if (head) heads[start[b] + atomicAdd(&hcnt[b], 1u)] = (uint32_t)i;
            if (tail) tails[start[b] + atomicAdd(&tcnt[b], 1u)] = (uint32_t)i;
        }
    }
}

template <int DIM, int T>
__global__ void __launch_bounds__(256) k_runs(GridP g, const uint32_t *__restrict__ key, int64_t n,
                                              const uint32_t *__restrict__ start, uint32_t *__restrict__ hcnt,
                                              uint32_t *__restrict__ tcnt, uint32_t *__restrict__ heads,
                                              uint32_t *__restrict__ tails) {
    const uint32_t lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const uint32_t binv = (uint32_t)g.ntiles;
    constexpr int64_t kSpan = 32 * kKeysUnroll;
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kSpan; base < n;
         base += warps * kSpan) {
        if (base + kSpan <= n) runs_span<DIM, T, true>(n, base, lane, binv, key, start, hcnt, tcnt, heads, tails);
        else runs_span<DIM, T, false>(n, base, lane, binv, key, start, hcnt, tcnt, heads, tails);
    }
}

// --------------------------------------------------------------------------
// Ascending bitonic sort of 32*E keys held E per lane (element e*32 + lane).
template <int E>
__device__ __forceinline__ void warp_bitonic(uint32_t (&v)[E]) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 32) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int e2 = e ^ (j >> 5);
                    if (e < e2) {
                        const bool asc = (((uint32_t)e * 32u + lane) & (uint32_t)k) == 0;
                        const uint32_t a = v[e], b = v[e2];
                        if ((a > b) == asc) {
                            v[e] = b;
                            v[e2] = a;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const bool asc = (((uint32_t)e * 32u + lane) & (uint32_t)k) == 0;
                    const uint32_t p = __shfl_xor_sync(0xFFFFFFFFu, v[e], j);
                    const bool lower = (lane & (uint32_t)j) == 0;
                    v[e] = (lower == asc) ? min(v[e], p) : max(v[e], p);
                }
            }
        }
    }
}

// One bucket's nr <= 32*E runs: sorted heads back into `heads`, and each
// run's offset inside the bucket (exclusive prefix of the lengths) into
// `tails`.
template <int E>
__device__ __forceinline__ void sort_runs_warp(uint32_t *heads, uint32_t *tails, uint32_t beg, uint32_t nr) {
    const uint32_t lane = lane_id();
    uint32_t h[E], t[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint32_t k = (uint32_t)e * 32u + lane;
        h[e] = k < nr ? heads[beg + k] : 0xFFFFFFFFu;
        t[e] = k < nr ? tails[beg + k] : 0xFFFFFFFFu;
    }
    if (nr > 1) {
        warp_bitonic<E>(h);
        warp_bitonic<E>(t);
    }
    uint32_t run = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint32_t k = (uint32_t)e * 32u + lane;
        const uint32_t len = k < nr ? t[e] - h[e] + 1u : 0u;
        uint32_t inc = len;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if ((int)lane >= d) inc += x;
        }
        if (k < nr) {
            heads[beg + k] = h[e];
            tails[beg + k] = run + inc - len;
        }
        run += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
}

constexpr int kWarpRuns = 512;           // most runs one warp sorts in registers
constexpr int kEmitRuns = 32;            // buckets of at most this many runs are sorted by k_emit itself
constexpr int kSortWarps = 8;

// Buckets with more than kEmitRuns runs (the active tiles, then the outside
// bucket), looked at 32 per warp: each such bucket is sorted by the warp, or
// listed for the block kernel above kWarpRuns.  Also counts all runs.
__global__ void __launch_bounds__(kSortWarps * 32) k_sort_runs(GridP g, const uint32_t *__restrict__ start,
                                                               const uint32_t *__restrict__ count,
                                                               const uint32_t *__restrict__ active,
                                                               const uint32_t *__restrict__ hcnt,
                                                               uint32_t *__restrict__ heads,
                                                               uint32_t *__restrict__ tails,
                                                               uint32_t *__restrict__ large_list,
                                                               uint32_t *__restrict__ status) {
    __shared__ uint32_t runs_sh;
    if (threadIdx.x == 0) runs_sh = 0;
    __syncthreads();
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const uint32_t nactive = status[MPM_ST_N_ACTIVE];
    const uint32_t nitems = nactive + (count[g.ntiles] > 0 ? 1u : 0u);
    const uint32_t nw = gridDim.x * kSortWarps;
    uint32_t my_runs = 0;
    for (uint32_t base = (blockIdx.x * kSortWarps + warp) * 32; base < nitems; base += nw * 32) {
        const uint32_t it = base + lane;
        uint32_t b = 0, nr = 0;
        if (it < nitems) {
            b = it < nactive ? active[it] : (uint32_t)g.ntiles;
            nr = hcnt[b];
        }
        my_runs += nr;
        uint32_t big = __ballot_sync(0xFFFFFFFFu, nr > (uint32_t)kEmitRuns);
        while (big) {
            const int j = __ffs(big) - 1;
            big &= big - 1;
            const uint32_t bj = __shfl_sync(0xFFFFFFFFu, b, j), nj = __shfl_sync(0xFFFFFFFFu, nr, j);
            const uint32_t beg = start[bj];
            if (nj <= 64) {
                sort_runs_warp<2>(heads, tails, beg, nj);
            } else if (nj <= 128) {
                sort_runs_warp<4>(heads, tails, beg, nj);
            } else if (nj <= 256) {
                sort_runs_warp<8>(heads, tails, beg, nj);
            } else if (nj <= (uint32_t)kWarpRuns) {
                sort_runs_warp<16>(heads, tails, beg, nj);
            } else if (lane == 0) {
                large_list[atomicAdd(&status[MPM_ST_N_LARGE_BUCKETS], 1u)] = bj;
            }
        }
    }
    my_runs = __reduce_add_sync(0xFFFFFFFFu, my_runs);
    if (lane == 0 && my_runs) atomicAdd(&runs_sh, my_runs);
    __syncthreads();
    if (threadIdx.x == 0 && runs_sh) atomicAdd(&status[MPM_ST_N_RUNS], runs_sh);
}

// Ascending sort of a[0..n) by a bitonic network whose comparators all put
// the smaller key at the lower index (the first merge step of each stage
// compares mirrored positions), so indices at or past n act as +infinity and
// are never touched.  Block-wide; `a` in shared or global memory.
__device__ void block_sort_u32(uint32_t *a, uint32_t n) {
    uint32_t np2 = 1;
    while (np2 < n) np2 <<= 1;
    for (uint32_t k = 2; k <= np2; k <<= 1) {
        const uint32_t half = k >> 1;
        for (uint32_t t = threadIdx.x; t < (np2 >> 1); t += blockDim.x) {
            const uint32_t blk = t / half, off = t % half;
            const uint32_t i = blk * k + off, l = blk * k + k - 1 - off;
            if (l < n) {
                const uint32_t x = a[i], y = a[l];
                if (x > y) {
                    a[i] = y;
                    a[l] = x;
                }
            }
        }
        __syncthreads();
        for (uint32_t j = half >> 1; j > 0; j >>= 1) {
            for (uint32_t t = threadIdx.x; t < (np2 >> 1); t += blockDim.x) {
                const uint32_t i = (t / j) * 2 * j + (t % j), l = i + j;
                if (l < n) {
                    const uint32_t x = a[i], y = a[l];
                    if (x > y) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

constexpr int kLargeThreads = 256;
constexpr uint32_t kSmemRuns = 8192;     // runs per list kept in shared memory (2 lists: 64 KB)

__device__ __forceinline__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t &total) {
    __shared__ uint32_t sh[kLargeThreads / 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if ((int)lane >= d) inc += t;
    }
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kLargeThreads / 32; ++w) {
        const uint32_t t = sh[w];
        before += (w < (int)warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + inc - v;
}

// One block per bucket with more than kWarpRuns runs.
__global__ void __launch_bounds__(kLargeThreads) k_sort_runs_large(const uint32_t *__restrict__ start,
                                                                  const uint32_t *__restrict__ hcnt,
                                                                  const uint32_t *__restrict__ large_list,
                                                                  uint32_t *__restrict__ heads,
                                                                  uint32_t *__restrict__ tails,
                                                                  uint32_t *__restrict__ status) {
    extern __shared__ uint32_t smem[];
    uint32_t *sh = smem, *st = smem + kSmemRuns;
    const uint32_t nitems = status[MPM_ST_N_LARGE_BUCKETS];
    for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
        const uint32_t b = large_list[it];
        const uint32_t beg = start[b], nr = hcnt[b];
        const bool in_smem = nr <= kSmemRuns;
        uint32_t *H = in_smem ? sh : heads + beg;
        uint32_t *Tl = in_smem ? st : tails + beg;
        if (in_smem) {
            for (uint32_t k = threadIdx.x; k < nr; k += blockDim.x) {
                sh[k] = heads[beg + k];
                st[k] = tails[beg + k];
            }
        } else if (threadIdx.x == 0) {
            atomicAdd(&status[MPM_ST_N_BIG_TILES], 1u);
        }
        __syncthreads();
        block_sort_u32(H, nr);
        block_sort_u32(Tl, nr);
        // offsets: exclusive prefix of the lengths, in chunks of the block size
        uint32_t run = 0;
        for (uint32_t base = 0; base < nr; base += blockDim.x) {
            const uint32_t k = base + threadIdx.x;
            uint32_t hk = 0, len = 0;
            if (k < nr) {
                hk = H[k];
                len = Tl[k] - hk + 1u;
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan_u32(len, tot);
            if (k < nr) {
                heads[beg + k] = hk;
                tails[beg + k] = run + ex;
            }
            run += tot;
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// perm, position by position.  Work items: the P2G slices (up to 1024
// positions of one tile), then the outside bucket in chunks of 1024; one
// warp per item.  A bucket of at most kEmitRuns runs is sorted here, in
// registers (lane k holds run k), and its runs that meet the item's
// positions are written one after another, 32 consecutive positions at a
// time.  Larger buckets come sorted, with their offsets, and each position
// binary-searches its run.
__global__ void __launch_bounds__(256) k_emit(GridP g, const uint32_t *__restrict__ start,
                                              const uint32_t *__restrict__ count,
                                              const uint32_t *__restrict__ hcnt,
                                              const uint32_t *__restrict__ heads,
                                              const uint32_t *__restrict__ tails,
                                              const uint32_t *__restrict__ slices,
                                              const uint32_t *__restrict__ status, uint32_t *__restrict__ perm) {
    const uint32_t lane = lane_id();
    const uint32_t nslices = status[MPM_ST_N_SLICES];
    const uint32_t nout = count[g.ntiles];
    const uint32_t nitems = nslices + (nout + kSliceParticles - 1) / kSliceParticles;
    const uint32_t nw = gridDim.x * (blockDim.x >> 5);
    for (uint32_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < nitems; it += nw) {
        uint32_t b, first;
        if (it < nslices) {
            b = slices[2 * (size_t)it];
            first = slices[2 * (size_t)it + 1];
        } else {
            b = (uint32_t)g.ntiles;
            first = (it - nslices) * kSliceParticles;
        }
        const uint32_t beg = start[b], cnt_b = start[b + 1] - beg, nr = hcnt[b];
        const uint32_t end = first + min((uint32_t)kSliceParticles, cnt_b - first);
        if (nr == 1) {
            const uint32_t h0 = heads[beg];
            for (uint32_t q = first + lane; q < end; q += 32) perm[beg + q] = h0 + q;
        } else if (nr <= (uint32_t)kEmitRuns) {
            uint32_t h[1], t[1];
            h[0] = lane < nr ? heads[beg + lane] : 0xFFFFFFFFu;
            t[0] = lane < nr ? tails[beg + lane] : 0xFFFFFFFFu;
            warp_bitonic<1>(h);
            warp_bitonic<1>(t);
            const uint32_t len = lane < nr ? t[0] - h[0] + 1u : 0u;
            uint32_t inc = len;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, inc, d);
                if ((int)lane >= d) inc += x;
            }
            const uint32_t off = inc - len;
            // run by run: run k fills positions [off_k, off_k + len_k) with h_k, h_k + 1, ...
            for (uint32_t k = 0; k < nr; ++k) {
                const uint32_t hk = __shfl_sync(0xFFFFFFFFu, h[0], k);
                const uint32_t ok = __shfl_sync(0xFFFFFFFFu, off, k);
                const uint32_t lk = __shfl_sync(0xFFFFFFFFu, len, k);
                const uint32_t lo = max(ok, first), hi = min(ok + lk, end);
                for (uint32_t q = lo + lane; q < hi; q += 32) perm[beg + q] = hk + (q - ok);
            }
        } else {
            for (uint32_t q = first + lane; q < end; q += 32) {
                uint32_t lo = 0, hi = nr - 1;
                while (lo < hi) {
                    const uint32_t mid = (lo + hi + 1) >> 1;
                    if (tails[beg + mid] <= q) lo = mid;
                    else hi = mid - 1;
                }
                perm[beg + q] = heads[beg + lo] + (q - tails[beg + lo]);
            }
        }
    }
}

// --------------------------------------------------------------------------
// int32 accumulators: for every node, the number of particles whose stencil
// covers it is the sum of the counts of the 3^dim base cells below it; the
// most of them enters mpm_p2g's bound.
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
    if (lane_id() == 0 && best > 0) atomicMax(&status[MPM_ST_MAX_NEIGHBOURS], best);
}

// --------------------------------------------------------------------------
mpm_status launch_bin(const GridP &g, const PartsF &p, const WsView &w, bool keys_from_g2p, const DeviceInfo &dev,
                      cudaStream_t st) {
    const int64_t n = p.n;
    const int64_t nb = g.ntiles + 1;
    // every status word but the records of the last P2G and G2P, which the next bound may use
    static_assert(MPM_ST_G2P_RANGE == MPM_ST_P2G_MASS + 2, "adjacent records");
    cudaMemsetAsync(w.status, 0, MPM_ST_P2G_MASS * sizeof(uint32_t), st);
    cudaMemsetAsync(&w.status[MPM_ST_G2P_RANGE + 1], 0, (MPM_STATUS_WORDS - MPM_ST_G2P_RANGE - 1) * sizeof(uint32_t),
                    st);
    const int threads = 256;
    const int64_t span = (int64_t)threads * kKeysUnroll;
    const int grid_p = (int)std::max<int64_t>(1, std::min<int64_t>((n + span - 1) / span, dev.sms * 8));
    if (keys_from_g2p) {
        // the keys (in place) and their histogram, written by the last G2P at the positions it wrote
        cudaMemcpyAsync(w.count, w.count_next, nb * sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
    } else {
        cudaMemsetAsync(w.count, 0, nb * sizeof(uint32_t), st);
        if (w.cellcount) cudaMemsetAsync(w.cellcount, 0, (size_t)(g.ntiles << g.cpt_log2) * sizeof(uint32_t), st);
    }
    if (n > 0 && !keys_from_g2p) {
        if (g.dim == 3)
            k_keys<3, 4><<<grid_p, threads, 0, st>>>(g, p, w.key, w.count, w.cellcount, w.status);
        else
            k_keys<2, 8><<<grid_p, threads, 0, st>>>(g, p, w.key, w.count, w.cellcount, w.status);
    }
    const int64_t nblk = (nb + kScanBlock - 1) / kScanBlock;
    k_scan_reduce<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.count, nb, (Tot3 *)w.partial);
    k_scan_top<<<1, kScanThreads, 0, st>>>((Tot3 *)w.partial, nblk, w.count, nb, w.status);
    k_scan_final<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.count, nb, (const Tot3 *)w.partial, w.start, w.hcnt,
                                                          w.tcnt, w.active, w.slices);
    if (n > 0) {
        if (g.dim == 3)
            k_runs<3, 4><<<grid_p, threads, 0, st>>>(g, w.key, n, w.start, w.hcnt, w.tcnt, w.heads, w.tails);
        else
            k_runs<2, 8><<<grid_p, threads, 0, st>>>(g, w.key, n, w.start, w.hcnt, w.tcnt, w.heads, w.tails);
        k_sort_runs<<<dev.sms * 4, kSortWarps * 32, 0, st>>>(g, w.start, w.count, w.active, w.hcnt, w.heads,
                                                             w.tails, w.large_list, w.status);
        const int smem = 2 * (int)kSmemRuns * (int)sizeof(uint32_t);
        cudaFuncSetAttribute(k_sort_runs_large, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        k_sort_runs_large<<<dev.sms, kLargeThreads, smem, st>>>(w.start, w.hcnt, w.large_list, w.heads, w.tails,
                                                                w.status);
        k_emit<<<dev.sms * 16, 256, 0, st>>>(g, w.start, w.count, w.hcnt, w.heads, w.tails, w.slices, w.status,
                                             w.perm);
    }
    if (w.cellcount) k_nbr_bound<<<dev.sms * 4, 256, 0, st>>>(g, w.cellcount, w.status);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
