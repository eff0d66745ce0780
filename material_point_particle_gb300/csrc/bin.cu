// bin.cu -- cell keys and the stable counting sort of particles into tiles.
//
// "Particle Worlds, part 3", Step 3 and Step 4: a counting sort in three
// phases, histogram -> exclusive prefix sum -> scatter, the scan as per-block
// scans, a scan of the block totals and an add-back.  The page's scatter
// claims slots with an atomic cursor and so leaves the order inside a bucket
// unspecified; the implementation guide (section 2.1, caveat (b), and rule 3)
// asks for every such race to be neutralised by a sort on a stable key.
// Here the buckets are tiles of T^dim base cells (section 2.1: bin into
// tiles, sort an index buffer), the atomic scatter fills each tile's range,
// and a warp or block per tile puts the range back in particle-index order,
// which makes the permutation the stable counting sort by tile -- a
// deterministic function of the keys.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_keys          key per particle, warp-aggregated tile histogram,
//                   out-of-domain count (int32 mode: per-cell counts)
//   k_scan_reduce / k_scan_top / k_scan_final
//                   exclusive scans of (count, P2G slices, active flag) over
//                   the buckets; active-tile list, P2G work list, cursors
//   k_scatter       warp-aggregated atomic scatter of indices into buckets
//   k_order_small   index order inside buckets of up to 256 entries (one warp)
//   k_order_claims  index order inside larger buckets (one warp): the
//                   atomic scatter's claims sorted and copied back in order
//   k_order_large   the same for buckets with too many claims (one block)
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
// Five running totals: particles, P2G slices, active tiles, and the buckets
// ordered by the warp kernel (small) and by the block kernel (large).
constexpr int kScanThreads = 256;
constexpr int kScanItems = 4;
constexpr int kScanBlock = kScanThreads * kScanItems;
constexpr uint32_t kSmallBucket = 256;   // buckets up to this size are ordered by one warp

struct Tot5 {
    uint32_t v[5];
};

__device__ __forceinline__ Tot5 tot_add(const Tot5 &x, const Tot5 &y) {
    Tot5 r;
#pragma unroll
    for (int i = 0; i < 5; ++i) r.v[i] = x.v[i] + y.v[i];
    return r;
}

__device__ __forceinline__ Tot5 tot_zero() { return Tot5{{0, 0, 0, 0, 0}}; }

__device__ __forceinline__ Tot5 bucket_values(const uint32_t *count, int64_t nb, int64_t b) {
    if (b >= nb) return tot_zero();
    const uint32_t c = count[b];
    const bool outside = b == nb - 1;
    Tot5 r;
    r.v[0] = c;
    r.v[1] = outside ? 0u : (c + kSliceParticles - 1) / kSliceParticles;  // no P2G work outside
    r.v[2] = (!outside && c > 0) ? 1u : 0u;
    r.v[3] = (c > 0 && c <= kSmallBucket) ? 1u : 0u;
    r.v[4] = c > kSmallBucket ? 1u : 0u;
    return r;
}

// Block-wide exclusive scan of one Tot5 per thread; returns the block total.
__device__ Tot5 block_exclusive_scan(const Tot5 &v, Tot5 &excl) {
    __shared__ Tot5 warp_tot[kScanThreads / 32];
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    Tot5 inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        Tot5 t;
#pragma unroll
        for (int i = 0; i < 5; ++i) t.v[i] = __shfl_up_sync(0xFFFFFFFFu, inc.v[i], d);
        if ((int)lane >= d) inc = tot_add(inc, t);
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    Tot5 before = tot_zero(), total = tot_zero();
    for (int w = 0; w < kScanThreads / 32; ++w) {
        if (w < (int)warp) before = tot_add(before, warp_tot[w]);
        total = tot_add(total, warp_tot[w]);
    }
#pragma unroll
    for (int i = 0; i < 5; ++i) excl.v[i] = before.v[i] + inc.v[i] - v.v[i];
    __syncthreads();
    return total;
}

__global__ void k_scan_reduce(const uint32_t *__restrict__ count, int64_t nb, Tot5 *__restrict__ partial) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tot5 s = tot_zero();
    for (int j = 0; j < kScanItems; ++j) s = tot_add(s, bucket_values(count, nb, b0 + j));
    Tot5 excl;
    Tot5 tot = block_exclusive_scan(s, excl);
    if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// One block: exclusive scan of the block totals (in place) and the grand totals.
__global__ void k_scan_top(Tot5 *__restrict__ partial, int64_t nblocks, const uint32_t *__restrict__ count,
                           int64_t nb, uint32_t *__restrict__ status) {
    Tot5 carry = tot_zero();
    for (int64_t base = 0; base < nblocks; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        const Tot5 v = i < nblocks ? partial[i] : tot_zero();
        Tot5 excl;
        const Tot5 tot = block_exclusive_scan(v, excl);
        if (i < nblocks) partial[i] = tot_add(carry, excl);
        carry = tot_add(carry, tot);
    }
    if (threadIdx.x == 0) {
        status[MPM_ST_N_VALID] = carry.v[0] - count[nb - 1];
        status[MPM_ST_N_SLICES] = carry.v[1];
        status[MPM_ST_N_ACTIVE] = carry.v[2];
        status[MPM_ST_N_SMALL_BUCKETS] = carry.v[3];
        status[MPM_ST_N_LARGE_BUCKETS] = carry.v[4];
    }
}

__global__ void k_scan_final(const uint32_t *__restrict__ count, int64_t nb, const Tot5 *__restrict__ partial,
                             uint32_t *__restrict__ start, uint32_t *__restrict__ cursor,
                             uint32_t *__restrict__ active, uint32_t *__restrict__ slices,
                             uint32_t *__restrict__ small_list, uint32_t *__restrict__ large_list) {
    const int64_t b0 = (int64_t)blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    Tot5 v[kScanItems];
    Tot5 s = tot_zero();
    for (int j = 0; j < kScanItems; ++j) {
        v[j] = bucket_values(count, nb, b0 + j);
        s = tot_add(s, v[j]);
    }
    Tot5 excl;
    block_exclusive_scan(s, excl);
    Tot5 run = tot_add(partial[blockIdx.x], excl);
    for (int j = 0; j < kScanItems; ++j) {
        const int64_t b = b0 + j;
        if (b >= nb) break;
        start[b] = run.v[0];
        cursor[b] = run.v[0];
        if (v[j].v[2]) active[run.v[2]] = (uint32_t)b;
        for (uint32_t s2 = 0; s2 < v[j].v[1]; ++s2) {
            slices[2 * (int64_t)(run.v[1] + s2)] = (uint32_t)b;
            slices[2 * (int64_t)(run.v[1] + s2) + 1] = s2 * kSliceParticles;
        }
        if (v[j].v[3]) small_list[run.v[3]] = (uint32_t)b;
        if (v[j].v[4]) large_list[run.v[4]] = (uint32_t)b;
        run = tot_add(run, v[j]);
        if (b == nb - 1) start[nb] = run.v[0];
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
// The order inside each tile: particle-index order (the stable counting sort
// with the tile as bucket).  The atomic scatter leaves each bucket as a set of
// "claims": one per warp-round and bucket, holding that warp's lanes of the
// bucket in lane (= index) order, all sharing w = idx >> 5 (a warp covers 32
// consecutive indices per round).  So ordering the claims by w puts the
// bucket in index order.
//
// Small buckets (at most 256 entries): one warp sorts the indices in
// registers with a bitonic network.
// Large buckets: one block.  Claims are placed by a table over a window of
// 2048 values of w around the bucket's median entry (in steady state almost
// every claim falls in it); the few claims outside are sorted and go before or
// after it.  Buckets above kOrderCap entries keep their working arrays in
// global scratch instead of shared memory.
constexpr int kOrderThreads = 256;
constexpr int kOrderWarps = kOrderThreads / 32;
constexpr int kOrderCap = 8192;
constexpr int kWindow = 2048;
constexpr int kFarCap = 256;             // far claims kept in shared memory (and sorted by one warp)
constexpr int kHeadCap = kOrderCap / 4;  // claim heads kept in shared memory

template <int E>
__device__ __forceinline__ void warp_bitonic(unsigned long long (&v)[E]) {
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
                        const unsigned long long a = v[e], b = v[e2];
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
                    const unsigned long long p = __shfl_xor_sync(0xFFFFFFFFu, v[e], j);
                    const bool lower = (lane & (uint32_t)j) == 0;
                    v[e] = (lower == asc) ? (v[e] < p ? v[e] : p) : (v[e] < p ? p : v[e]);
                }
            }
        }
    }
}

template <int E>
__device__ __forceinline__ void order_small(const uint32_t *tmp, uint32_t beg, uint32_t cnt, uint32_t *perm) {
    const uint32_t lane = lane_id();
    unsigned long long v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint32_t i = (uint32_t)e * 32u + lane;
        v[e] = i < cnt ? (unsigned long long)tmp[beg + i] : ~0ull;
    }
    warp_bitonic<E>(v);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint32_t i = (uint32_t)e * 32u + lane;
        if (i < cnt) perm[beg + i] = (uint32_t)v[e];
    }
}

__global__ void __launch_bounds__(256) k_order_small(const uint32_t *__restrict__ tmp,
                                                     const uint32_t *__restrict__ start,
                                                     const uint32_t *__restrict__ count,
                                                     const uint32_t *__restrict__ list, uint32_t *__restrict__ perm,
                                                     const uint32_t *__restrict__ status) {
    const uint32_t nitems = status[MPM_ST_N_SMALL_BUCKETS];
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const uint32_t nw = gridDim.x * (blockDim.x >> 5);
    for (uint32_t it = blockIdx.x * (blockDim.x >> 5) + warp; it < nitems; it += nw) {
        const uint32_t b = list[it];
        const uint32_t beg = start[b], cnt = count[b];
        if (cnt == 1) {
            if (lane == 0) perm[beg] = tmp[beg];
        } else if (cnt <= 32) {
            order_small<1>(tmp, beg, cnt, perm);
        } else if (cnt <= 64) {
            order_small<2>(tmp, beg, cnt, perm);
        } else if (cnt <= 128) {
            order_small<4>(tmp, beg, cnt, perm);
        } else {
            order_small<8>(tmp, beg, cnt, perm);
        }
    }
}

// Larger buckets whose claims number at most kClaimCap: one warp per bucket.
// Pass 1 records each claim head as a key (w << 37 | position << 6 | length-1)
// in the warp's shared slot, the warp sorts the keys in registers, scans the
// lengths in sorted order and copies each claim from tmp to its place in perm
// (one lane per entry).  Buckets with more claims (a cold particle order) or
// above 2^26 entries go to `fallback` for the block kernel.
constexpr int kClaimCap = 512;
constexpr int kClaimWarps = 8;

__global__ void __launch_bounds__(kClaimWarps * 32) k_order_claims(const uint32_t *__restrict__ tmp,
                                                                   const uint32_t *__restrict__ start,
                                                                   const uint32_t *__restrict__ count,
                                                                   const uint32_t *__restrict__ list,
                                                                   uint32_t *__restrict__ perm,
                                                                   uint32_t *__restrict__ fallback,
                                                                   uint32_t *__restrict__ status) {
    __shared__ unsigned long long keys[kClaimWarps][kClaimCap];
    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    unsigned long long *kw = keys[warp];
    const uint32_t nitems = status[MPM_ST_N_LARGE_BUCKETS];
    const uint32_t nw = gridDim.x * kClaimWarps;
    for (uint32_t it = blockIdx.x * kClaimWarps + warp; it < nitems; it += nw) {
        const uint32_t b = list[it];
        const uint32_t beg = start[b], cnt = count[b];
        // pass 1: claim heads (where idx >> 5 changes)
        uint32_t nclaims = 0, wlast = 0xFFFFFFFFu;
        for (uint32_t base = 0; base < cnt; base += 32) {
            const uint32_t i = base + lane;
            const uint32_t w = i < cnt ? (tmp[beg + i] >> 5) : 0xFFFFFFFFu;
            uint32_t wprev = __shfl_up_sync(0xFFFFFFFFu, w, 1);
            if (lane == 0) wprev = wlast;
            const bool head = i < cnt && w != wprev;
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, head);
            const uint32_t k = nclaims + __popc(m & lanemask_lt());
            if (head && k < (uint32_t)kClaimCap) kw[k] = ((unsigned long long)w << 37) | ((unsigned long long)i << 6);
            nclaims += __popc(m);
            wlast = __shfl_sync(0xFFFFFFFFu, w, 31);
        }
        if (nclaims > (uint32_t)kClaimCap || cnt >= (1u << 26)) {
            if (lane == 0) fallback[atomicAdd(&status[MPM_ST_N_FALLBACK], 1u)] = b;
            continue;
        }
        __syncwarp();
        // lengths (from the next head in bucket order), then sort by w
        unsigned long long v[kClaimCap / 32];
#pragma unroll
        for (int e = 0; e < kClaimCap / 32; ++e) {
            const uint32_t k = (uint32_t)e * 32u + lane;
            if (k < nclaims) {
                const unsigned long long key = kw[k];
                const uint32_t pos = (uint32_t)(key >> 6) & ((1u << 26) - 1);
                const uint32_t next = k + 1 < nclaims ? (uint32_t)(kw[k + 1] >> 6) & ((1u << 26) - 1) : cnt;
                v[e] = key | (unsigned long long)(next - pos - 1);
            } else {
                v[e] = ~0ull;
            }
        }
        __syncwarp();
        warp_bitonic<kClaimCap / 32>(v);
        // destinations: running sum of lengths in sorted order; claims back to shared memory
        uint32_t run = 0;
#pragma unroll
        for (int e = 0; e < kClaimCap / 32; ++e) {
            const uint32_t k = (uint32_t)e * 32u + lane;
            const uint32_t len = k < nclaims ? (uint32_t)(v[e] & 63u) + 1u : 0u;
            uint32_t inc = len;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
                if ((int)lane >= d) inc += t;
            }
            if (k < nclaims) {
                const uint32_t pos = (uint32_t)(v[e] >> 6) & ((1u << 26) - 1);
                kw[k] = ((unsigned long long)(run + inc - len) << 32) | ((unsigned long long)pos << 6) | (len - 1);
            }
            run += __shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        __syncwarp();
        // copy claim by claim (independent iterations, unrolled for memory parallelism)
        uint32_t j = 0;
        for (; j + 4 <= nclaims; j += 4) {
            uint32_t val[4], dst[4];
            bool on[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const unsigned long long c = kw[j + u];
                const uint32_t pos = (uint32_t)(c >> 6) & ((1u << 26) - 1), len = (uint32_t)(c & 63u) + 1u;
                dst[u] = (uint32_t)(c >> 32);
                on[u] = lane < len;
                val[u] = on[u] ? tmp[beg + pos + lane] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (on[u]) perm[beg + dst[u] + lane] = val[u];
        }
        for (; j < nclaims; ++j) {
            const unsigned long long c = kw[j];
            const uint32_t pos = (uint32_t)(c >> 6) & ((1u << 26) - 1), len = (uint32_t)(c & 63u) + 1u;
            if (lane < len) perm[beg + (uint32_t)(c >> 32) + lane] = tmp[beg + pos + lane];
        }
        __syncwarp();
    }
}

__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t &total, uint32_t *sh) {
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
    for (int w = 0; w < kOrderWarps; ++w) {
        const uint32_t t = sh[w];
        before += (w < (int)warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + inc - v;
}

// Ascending bitonic sort of n_pow2 keys, block-wide (shared or global memory).
__device__ void block_bitonic(unsigned long long *s, uint32_t n_pow2) {
    for (uint32_t k = 2; k <= n_pow2; k <<= 1) {
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t t = threadIdx.x; t < (n_pow2 >> 1); t += blockDim.x) {
                const uint32_t i = (t / j) * 2 * j + (t % j);
                const uint32_t pr = i + j;
                const bool up = (i & k) == 0;
                const unsigned long long a = s[i], b = s[pr];
                if ((a > b) == up) {
                    s[i] = b;
                    s[pr] = a;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kOrderThreads)
k_order_large(const uint32_t *__restrict__ tmp, const uint32_t *__restrict__ start,
              const uint32_t *__restrict__ count, const uint32_t *__restrict__ list, uint32_t *perm, uint32_t *gH,
              unsigned long long *gF, uint32_t *__restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint32_t *sA = reinterpret_cast<uint32_t *>(smem_raw);
    uint32_t *sH = sA + kOrderCap;  // kHeadCap + 1 entries
    __shared__ uint32_t table[kWindow];
    __shared__ unsigned long long sF[kFarCap];
    __shared__ uint32_t scan_sh[kOrderWarps];
    __shared__ uint32_t nfar_sh, nlow_sh;
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    const uint32_t nitems = status[MPM_ST_N_FALLBACK];
    for (uint32_t it = blockIdx.x; it < nitems; it += gridDim.x) {
        const uint32_t b = list[it];
        const uint32_t beg = start[b], cnt = count[b];
        const bool small = cnt <= (uint32_t)kOrderCap;
        if (!small && threadIdx.x == 0) atomicAdd(&status[MPM_ST_N_BIG_TILES], 1u);
        const uint32_t *A = small ? sA : tmp + beg;
        uint32_t *S = perm + beg;
        if (small)
            for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) sA[i] = tmp[beg + i];
        if (threadIdx.x == 0) nfar_sh = 0;
        for (uint32_t d = threadIdx.x; d < (uint32_t)kWindow; d += blockDim.x) table[d] = 0;
        __syncthreads();
        // claim heads: warp w scans the contiguous segment [w*hseg, (w+1)*hseg)
        // 32 entries at a time, counts its heads, then writes their positions
        const uint32_t hseg = (cnt + kOrderWarps - 1) / kOrderWarps;
        const uint32_t h0 = min(cnt, warp * hseg), h1 = min(cnt, h0 + hseg);
        uint32_t myheads = 0;
        for (uint32_t base = h0; base < h1; base += 32) {
            const uint32_t i = base + lane;
            const bool head = i < h1 && (i == 0 || (A[i] >> 5) != (A[i - 1] >> 5));
            myheads += __popc(__ballot_sync(0xFFFFFFFFu, head));
        }
        uint32_t nclaims;
        uint32_t k = block_excl_scan(lane == 0 ? myheads : 0u, nclaims, scan_sh);
        k = __shfl_sync(0xFFFFFFFFu, k, 0);
        uint32_t *H = (small && nclaims <= (uint32_t)kHeadCap) ? sH : gH + (size_t)beg + b;
        for (uint32_t base = h0; base < h1; base += 32) {
            const uint32_t i = base + lane;
            const bool head = i < h1 && (i == 0 || (A[i] >> 5) != (A[i - 1] >> 5));
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, head);
            if (head) H[k + __popc(m & lanemask_lt())] = i;
            k += __popc(m);
        }
        if (threadIdx.x == 0) H[nclaims] = cnt;
        __syncthreads();
        // window around the median entry; claims inside go to the table by w,
        // the others ("far") to a list sorted below
        const long long w_lo = (long long)(A[cnt / 2] >> 5) - kWindow / 2;
        for (uint32_t c = threadIdx.x; c < nclaims; c += blockDim.x) {
            const long long d = (long long)(A[H[c]] >> 5) - w_lo;
            if (d >= 0 && d < kWindow) table[d] = H[c + 1] - H[c];
            else atomicAdd(&nfar_sh, 1u);
        }
        __syncthreads();
        const uint32_t nfar = nfar_sh;
        unsigned long long *F = nfar <= (uint32_t)kFarCap ? sF : gF + 2 * (size_t)beg;
        __syncthreads();
        if (threadIdx.x == 0) nfar_sh = 0;
        __syncthreads();
        if (nfar > 0) {
            for (uint32_t c = threadIdx.x; c < nclaims; c += blockDim.x) {
                const uint32_t w = A[H[c]] >> 5;
                const long long d = (long long)w - w_lo;
                if (!(d >= 0 && d < kWindow)) F[atomicAdd(&nfar_sh, 1u)] = ((unsigned long long)w << 32) | c;
            }
            __syncthreads();
        }
        if (nfar > 1 && nfar <= (uint32_t)kFarCap) {
            if (warp == 0) {  // one warp sorts in registers
                unsigned long long v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t f = (uint32_t)e * 32u + lane;
                    v[e] = f < nfar ? F[f] : ~0ull;
                }
                warp_bitonic<8>(v);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t f = (uint32_t)e * 32u + lane;
                    if (f < nfar) F[f] = v[e];
                }
            }
            __syncthreads();
        } else if (nfar > (uint32_t)kFarCap) {
            uint32_t np2 = 1;
            while (np2 < nfar) np2 <<= 1;
            for (uint32_t f = nfar + threadIdx.x; f < np2; f += blockDim.x) F[f] = ~0ull;
            __syncthreads();
            block_bitonic(F, np2);
        }
        // far claims below the window come first: count them (binary search in
        // the sorted keys) and add up their lengths
        uint32_t nlow = 0, lowlen = 0;
        if (nfar > 0) {
            if (threadIdx.x == 0) {
                uint32_t lo2 = 0, hi2 = nfar;
                while (lo2 < hi2) {
                    const uint32_t mid = (lo2 + hi2) / 2;
                    if ((long long)(F[mid] >> 32) < w_lo) lo2 = mid + 1;
                    else hi2 = mid;
                }
                nlow_sh = lo2;
            }
            __syncthreads();
            nlow = nlow_sh;
            uint32_t mylow = 0;
            for (uint32_t f = threadIdx.x; f < nlow; f += blockDim.x) {
                const uint32_t c = (uint32_t)(F[f] & 0xFFFFFFFFu);
                mylow += H[c + 1] - H[c];
            }
            block_excl_scan(mylow, lowlen, scan_sh);
        }
        // table prefix (blocked, 8 slots per thread) -> destinations of the window claims
        constexpr int kPer = kWindow / kOrderThreads;
        uint32_t tv[kPer], tsum = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            tv[q] = table[threadIdx.x * kPer + q];
            tsum += tv[q];
        }
        uint32_t wintotal;
        uint32_t toff = block_excl_scan(tsum, wintotal, scan_sh);
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const uint32_t t = tv[q];
            table[threadIdx.x * kPer + q] = lowlen + toff;
            toff += t;
        }
        __syncthreads();
        // copy window claims: one warp per claim, lanes copy its entries
        for (uint32_t c = warp; c < nclaims; c += kOrderWarps) {
            const uint32_t src = H[c], len = H[c + 1] - H[c];
            const long long d = (long long)(A[src] >> 5) - w_lo;
            if (d >= 0 && d < kWindow && lane < len) S[table[d] + lane] = A[src + lane];
        }
        // copy far claims in sorted order (block-wide prefix of their lengths)
        uint32_t run = 0;
        for (uint32_t base = 0; base < nfar; base += blockDim.x) {
            const uint32_t f = base + threadIdx.x;
            uint32_t len = 0, c = 0;
            if (f < nfar) {
                c = (uint32_t)(F[f] & 0xFFFFFFFFu);
                len = H[c + 1] - H[c];
            }
            uint32_t tot;
            const uint32_t ex = run + block_excl_scan(len, tot, scan_sh);
            if (f < nfar) {
                const uint32_t dst = f < nlow ? ex : ex + wintotal;
                const uint32_t src = H[c];
                for (uint32_t e = 0; e < len; ++e) S[dst + e] = A[src + e];
            }
            run += tot;
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
    k_scan_reduce<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.count, nb, (Tot5 *)w.partial);
    k_scan_top<<<1, kScanThreads, 0, st>>>((Tot5 *)w.partial, nblk, w.count, nb, w.status);
    k_scan_final<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.count, nb, (const Tot5 *)w.partial, w.start, w.cursor,
                                                          w.active, w.slices, w.small_list, w.large_list);
    if (n > 0) {
        k_scatter<<<grid_p, threads, 0, st>>>(g, w.key, n, w.cursor, w.tmp);
        k_order_small<<<dev.sms * 4, 256, 0, st>>>(w.tmp, w.start, w.count, w.small_list, w.perm, w.status);
        k_order_claims<<<dev.sms * 4, kClaimWarps * 32, 0, st>>>(w.tmp, w.start, w.count, w.large_list, w.perm,
                                                                  w.fallback, w.status);
        const int smem = (kOrderCap + kHeadCap + 4) * (int)sizeof(uint32_t);
        cudaFuncSetAttribute(k_order_large, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        k_order_large<<<dev.sms * 2, kOrderThreads, smem, st>>>(w.tmp, w.start, w.count, w.fallback, w.perm, w.gH,
                                                               (unsigned long long *)w.gCW, w.status);
    }
    if (w.cellcount) k_nbr_bound<<<dev.sms * 4, 256, 0, st>>>(g, w.cellcount, w.status);
    return cudaGetLastError() == cudaSuccess ? MPM_OK : MPM_E_CUDA;
}

}  // namespace mpm
