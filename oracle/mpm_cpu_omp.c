/*
 * mpm_cpu_omp.c -- the multi-core CPU baseline of one fixed-point MPM step
 * (bin, P2G, grid update, G2P) on all host cores with OpenMP.
 *
 * TEST INFRASTRUCTURE, like the oracle it is built from: only the test suite
 * and the benchmark's CPU-baseline leg load it.  It includes the oracle's
 * source, so every per-particle and per-node operation is the oracle's own
 * code; what is added is the parallel structure around it:
 *
 *   bin      keys in parallel; per-thread tile histograms over contiguous
 *            index ranges, scanned tile-major then thread-major, so the
 *            scatter is the stable counting sort by tile (the oracle's
 *            (tile, index) order, then the particles outside the domain in
 *            index order)
 *   permute  the particle arrays copied into that order (the sorted SoA copy
 *            of the stable-scatter step)
 *   P2G      each thread scatters a contiguous range of the sorted particles
 *            into its own private int64 grid, zeroed and read back only over
 *            the node planes its particles reach (their tiles are contiguous,
 *            so that is a slab); the private grids are merged by integer
 *            add, plane by plane in parallel.  Integer addition is exact and
 *            order-free, so the grid is the oracle's bit for bit
 *   update   the oracle's node update, planes in parallel
 *   G2P      the oracle's gather on contiguous ranges of the sorted particles
 *
 * The new state is written in bin order: out[j] = new state of in[perm[j]].
 * int64 fixed point (the accumulator mode of the headline workload).
 */
#include "mpm_oracle.c"

#include <omp.h>

typedef struct {
    int64_t lo, hi; /* node-plane range [lo, hi) a thread's particles reach (planes of n0*n1 nodes in 3D, rows of n0 in 2D) */
} plane_range;

static int64_t plane_nodes(const orc_desc *d)
{
    return d->dim == 3 ? (int64_t)d->n[0] * d->n[1] : (int64_t)d->n[0];
}

static int64_t num_planes(const orc_desc *d)
{
    return d->dim == 3 ? d->n[2] : d->n[1];
}

/* The node planes reached by base cells in tiles t0 .. t1 (tile-major order,
 * so the slowest tile axis is the plane axis): tile rows tz0 .. tz1 cover base
 * planes tz0*T .. tz1*T + T - 1, whose stencils reach two planes further.    */
static plane_range planes_of_tiles(const orc_desc *d, uint32_t t0, uint32_t t1)
{
    int64_t per_row = 1;
    for (int l = 0; l < d->dim - 1; ++l)
        per_row *= tiles_per_axis(d, l);
    plane_range r;
    r.lo = (int64_t)(t0 / per_row) * d->tile;
    r.hi = (int64_t)(t1 / per_row) * d->tile + d->tile + 2;
    if (r.hi > num_planes(d))
        r.hi = num_planes(d);
    return r;
}

int orc_omp_max_threads(void) { return omp_get_max_threads(); }

/* Seconds of the last step's phases: bin, permute, P2G, merge, grid update,
 * G2P. */
double orc_omp_phase_seconds[6];

/* The private grids live from call to call (their pages are mapped once):
 * one (dim+1)*nodes int64 grid per thread, regrown when the grid or the
 * thread count grows.  Calls must not overlap.                            */
static int64_t **g_priv;
static int g_priv_threads;
static size_t g_priv_words;

static int64_t **private_grids(int T, size_t words)
{
    if (T > g_priv_threads || words > g_priv_words) {
        for (int t = 0; t < g_priv_threads; ++t)
            free(g_priv[t]);
        free(g_priv);
        g_priv = (int64_t **)calloc((size_t)T, sizeof(int64_t *));
        for (int t = 0; t < T; ++t)
            g_priv[t] = (int64_t *)malloc(sizeof(int64_t) * words);
        g_priv_threads = T;
        g_priv_words = words;
    }
    return g_priv;
}

/* One step.  x, v, C, m: the input state (np particles, fp32 planes).
 * xo, vo, Co, mo: the new state in bin order; perm: the order; acc:
 * (dim+1)*nodes int64 and vel: dim*nodes fp32 scratch (the grid of the step,
 * left holding it).  threads <= 0: all cores.  Returns the number of
 * particles moved (those in the domain); counts[0], counts[1] as the
 * oracle's P2G.                                                            */
int64_t orc_omp_step_fixed(const orc_desc *d, float dt, const float *dtg, int64_t np, const float *const *x,
                           const float *const *v, const float *const *C, const float *m, float *const *xo,
                           float *const *vo, float *const *Co, float *mo, uint32_t *perm, int64_t *acc,
                           float *vel, int threads, int64_t counts[2])
{
    int dim = d->dim;
    int64_t nodes = nodes_of(d);
    int64_t ntiles = orc_num_tiles(d);
    int64_t nb = ntiles + 1; /* bucket ntiles: outside the domain */
    uint32_t cells_per_tile = 1;
    for (int l = 0; l < dim; ++l)
        cells_per_tile *= (uint32_t)d->tile;
    int T = threads > 0 ? threads : omp_get_max_threads();
    counts[0] = counts[1] = 0;
    double t_start = omp_get_wtime();

    /* bin: bucket per particle, per-thread histograms */
    uint32_t *bucket = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(np > 0 ? np : 1));
    uint32_t *hist = (uint32_t *)calloc((size_t)T * (size_t)nb, sizeof(uint32_t));
#pragma omp parallel num_threads(T)
    {
        int t = omp_get_thread_num();
        int64_t p0 = np * t / T, p1 = np * (t + 1) / T;
        uint32_t *h = hist + (size_t)t * (size_t)nb;
        for (int64_t p = p0; p < p1; ++p) {
            int b[3];
            float f[3];
            uint32_t bk = (uint32_t)ntiles;
            if (base_frac(d, x, p, b, f))
                bk = key_of(d, b) / cells_per_tile;
            bucket[p] = bk;
            h[bk] += 1;
        }
    }
    /* exclusive scan, bucket-major then thread-major: hist becomes each
     * thread's first position in each bucket */
    {
        uint32_t run = 0;
        for (int64_t bk = 0; bk < nb; ++bk)
            for (int t = 0; t < T; ++t) {
                uint32_t c = hist[(size_t)t * (size_t)nb + (size_t)bk];
                hist[(size_t)t * (size_t)nb + (size_t)bk] = run;
                run += c;
            }
    }
#pragma omp parallel num_threads(T)
    {
        int t = omp_get_thread_num();
        int64_t p0 = np * t / T, p1 = np * (t + 1) / T;
        uint32_t *h = hist + (size_t)t * (size_t)nb;
        for (int64_t p = p0; p < p1; ++p)
            perm[h[bucket[p]]++] = (uint32_t)p;
    }
    free(hist);
    int64_t valid = 0;
    for (int64_t j = np - 1; j >= 0 && valid == 0; --j)
        if (bucket[perm[j]] != (uint32_t)ntiles)
            valid = j + 1;
    double t_bin = omp_get_wtime();

    /* permute the particle arrays into bin order */
#pragma omp parallel for num_threads(T) schedule(static)
    for (int64_t j = 0; j < np; ++j) {
        uint32_t p = perm[j];
        for (int l = 0; l < dim; ++l) {
            xo[l][j] = x[l][p];
            vo[l][j] = v[l][p];
        }
        for (int k = 0; k < dim * dim; ++k)
            Co[k][j] = C[k][p];
        mo[j] = m[p];
    }

    double t_perm = omp_get_wtime();

    /* the oracle's bound before any scatter: R over every in-domain
     * particle (the max is order-free), one test for the whole step        */
    float *Rt = (float *)calloc((size_t)T, sizeof(float));
#pragma omp parallel num_threads(T)
    {
        int t = omp_get_thread_num();
        int64_t j0 = valid * t / T, j1 = valid * (t + 1) / T;
        const float *xs[3], *vs[3], *Cs[9];
        for (int l = 0; l < dim; ++l) {
            xs[l] = xo[l] + j0;
            vs[l] = vo[l] + j0;
        }
        for (int k = 0; k < dim * dim; ++k)
            Cs[k] = Co[k] + j0;
        Rt[t] = orc_scatter_range(d, j1 - j0, xs, vs, Cs, mo + j0, NULL, NULL);
    }
    float R = 0.0f;
    for (int t = 0; t < T; ++t)
        R = max_nan(R, Rt[t]);
    free(Rt);
    int64_t count = d->acc_mode == 0 ? orc_max_cover(d, valid, (const float *const *)xo) : valid;
    int scatter = orc_bound_ok(d, R, count);
    counts[1] = scatter ? 0 : valid;

    /* P2G: private grids over each thread's slab, merged by integer add */
    int64_t pn = plane_nodes(d), nplanes = num_planes(d);
    int64_t **priv = private_grids(T, (size_t)(dim + 1) * (size_t)nodes);
    int *used = (int *)calloc((size_t)T, sizeof(int));
    plane_range *range = (plane_range *)calloc((size_t)T, sizeof(plane_range));
#pragma omp parallel num_threads(T)
    {
        int t = omp_get_thread_num();
        int64_t j0 = valid * t / T, j1 = valid * (t + 1) / T;
        range[t].lo = range[t].hi = 0;
        if (scatter && j1 > j0) {
            range[t] = planes_of_tiles(d, bucket[perm[j0]], bucket[perm[j1 - 1]]);
            used[t] = 1;
            /* only the slab is cleared and read back */
            for (int c = 0; c <= dim; ++c)
                memset(priv[t] + (size_t)c * (size_t)nodes + (size_t)(range[t].lo * pn), 0,
                       sizeof(int64_t) * (size_t)((range[t].hi - range[t].lo) * pn));
            const float *xs[3], *vs[3], *Cs[9];
            for (int l = 0; l < dim; ++l) {
                xs[l] = xo[l] + j0;
                vs[l] = vo[l] + j0;
            }
            for (int k = 0; k < dim * dim; ++k)
                Cs[k] = Co[k] + j0;
            int64_t outside = 0;
            scatter_fixed_all(d, j1 - j0, xs, vs, Cs, mo + j0, NULL, priv[t], &outside);
        }
    }
    counts[0] += np - valid;
    double t_p2g = omp_get_wtime();
#pragma omp parallel for num_threads(T) schedule(static)
    for (int64_t z = 0; z < nplanes; ++z)
        for (int c = 0; c <= dim; ++c) {
            int64_t *dst = acc + (size_t)c * (size_t)nodes + (size_t)(z * pn);
            memset(dst, 0, sizeof(int64_t) * (size_t)pn);
            for (int t = 0; t < T; ++t)
                if (used[t] && z >= range[t].lo && z < range[t].hi) {
                    const int64_t *src = priv[t] + (size_t)c * (size_t)nodes + (size_t)(z * pn);
                    for (int64_t i = 0; i < pn; ++i)
                        dst[i] += src[i];
                }
        }
    free(used);
    free(range);
    double t_merge = omp_get_wtime();

    /* grid update: the oracle's node update, planes in parallel */
#pragma omp parallel for num_threads(T) schedule(static)
    for (int64_t z = 0; z < nplanes; ++z) {
        int nj = dim == 3 ? d->n[1] : 1;
        for (int j = 0; j < nj; ++j)
            for (int i = 0; i < d->n[0]; ++i) {
                int jj = dim == 3 ? j : (int)z, kk = dim == 3 ? (int)z : 0;
                int64_t node = node_at(d, i, jj, kk);
                float P[3] = {0.0f, 0.0f, 0.0f}, out[3];
                for (int l = 0; l < dim; ++l)
                    P[l] = (float)acc[(int64_t)(1 + l) * nodes + node];
                update_node(d, i, jj, kk, (float)acc[node], P, dtg, out);
                for (int l = 0; l < dim; ++l)
                    vel[(int64_t)l * nodes + node] = out[l];
            }
    }

    double t_update = omp_get_wtime();

    /* G2P: the oracle's gather on contiguous ranges of the sorted particles */
    int64_t moved = 0;
#pragma omp parallel num_threads(T) reduction(+ : moved)
    {
        int t = omp_get_thread_num();
        int64_t j0 = valid * t / T, j1 = valid * (t + 1) / T;
        if (j1 > j0) {
            float *xs[3], *vs[3], *Cs[9];
            for (int l = 0; l < dim; ++l) {
                xs[l] = xo[l] + j0;
                vs[l] = vo[l] + j0;
            }
            for (int k = 0; k < dim * dim; ++k)
                Cs[k] = Co[k] + j0;
            moved += g2p_core(d, vel, j1 - j0, xs, vs, Cs, NULL, dt);
        }
    }
    free(bucket);
    double t_end = omp_get_wtime();
    orc_omp_phase_seconds[0] = t_bin - t_start;
    orc_omp_phase_seconds[1] = t_perm - t_bin;
    orc_omp_phase_seconds[2] = t_p2g - t_perm;
    orc_omp_phase_seconds[3] = t_merge - t_p2g;
    orc_omp_phase_seconds[4] = t_update - t_merge;
    orc_omp_phase_seconds[5] = t_end - t_update;
    return moved;
}
