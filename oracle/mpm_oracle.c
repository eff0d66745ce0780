/*
 * mpm_oracle.c -- plain, slow, single-threaded CPU oracle for the Material
 * Point Method particle/grid transfer: cell keys and a stable counting sort,
 * the particle-to-grid (P2G) scatter of mass and APIC/MLS affine momentum in
 * fixed-point integers (and in floating point), the grid update and the
 * grid-to-particle (G2P) gather, and the MLS-MPM elastic stress folded into
 * the affine matrix with the deformation-gradient update.  Also the integer
 * cloud-in-cell transfer of
 * "particle to grid transfer in checked integer arithmetic" exactly as that
 * page states it.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product (the CUDA
 * library) never links, loads or calls it, and it includes none of the
 * product's headers: every type below is declared here.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC.  Contraction
 * must be off: every fp32 operation below is one IEEE round-to-nearest-even
 * operation, and fused multiply-adds appear only where fmaf() is written.
 *
 * Arithmetic contract (the GPU must reproduce these bits in fixed-point mode):
 *   cell coordinates  xi = x * inv_dx;  b = floor(xi - 0.5);  f = xi - b
 *   1-D weights       w0 = 0.5*(1.5-f)^2, w1 = 0.75-(f-1)^2, w2 = 0.5*(f-0.5)^2
 *   scaled mass       Mt = m * S                         (S = 2^scale_log2)
 *   node weight       Wt(a) = ((wx[a0]*Mt) * wy[a1]) * wz[a2]
 *   node offset       d_l = (a_l - f_l) * dx
 *   node velocity     vel_k(a) = fma(C_k2,d_2, fma(C_k1,d_1, fma(C_k0,d_0, v_k)))
 *   shares            s_m(a) = rint(Wt(a));  s_k(a) = rint(Wt(a) x vel_k(a))
 *                     (exact product, rounded once, ties to even)
 *   particle totals   Q_m = rint(Mt);  Q_k = rint(Mt * v_k)
 *   centre node       s_c(1,1,1) = Q_c - sum of the other 26 shares
 * The centre-remainder rule is the quadratic-stencil reading of the integer
 * split ("the near node's share is q minus that"): the shares of one particle
 * sum to its quantity exactly, so grid totals equal particle totals.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t dim;            /* 2 or 3 */
    int32_t n[3];           /* nodes per axis (n[2] = 1 in 2D) */
    float dx, inv_dx;       /* node spacing and its reciprocal, both fp32 */
    int32_t order;          /* 2 = quadratic B-spline (1 = linear, integer path only) */
    int32_t acc_mode;       /* 0 int32, 1 int64, 2 fp32 atomics, 3 exact integer CIC */
    int32_t scale_log2;     /* fixed-point scale S = 2^scale_log2 */
    int32_t tile;           /* cells per tile edge */
    int32_t boundary_nodes; /* width of the velocity boundary band */
} orc_desc;

#define ORC_KEY_INVALID 0xFFFFFFFFu
#define ORC_ST_DOMAIN 1u
#define ORC_ST_BOUND 2u

/* ------------------------------------------------------------------------ */
/* Grid indexing: planar channels, node (i, j, k) at (k*n1 + j)*n0 + i.       */

static int64_t nodes_of(const orc_desc *d)
{
    return (int64_t)d->n[0] * d->n[1] * (d->dim == 3 ? d->n[2] : 1);
}

static int64_t node_at(const orc_desc *d, int i, int j, int k)
{
    return ((int64_t)k * d->n[1] + j) * d->n[0] + i;
}

int64_t orc_nodes(const orc_desc *d) { return nodes_of(d); }

/* ------------------------------------------------------------------------ */
/* Quadratic B-spline weights.  "Mass Matrix Assembly on Tensor Cores for
 * Implicit Particle-In-Cell Methods", shape functions (Eq. 12): the weight is
 * a product of 1-D B-splines of order n, non-negative, summing to one; for
 * second order the stencil is the nearest node and its two neighbours.  The
 * three values are the cardinal quadratic B-spline at distances f, f-1, f-2
 * from the stencil's first node, f in [0.5, 1.5).                           */

void orc_quadratic_weights(float f, float w[3])
{
    float t0 = 1.5f - f;
    float t1 = f - 1.0f;
    float t2 = f - 0.5f;
    w[0] = 0.5f * (t0 * t0);
    w[1] = 0.75f - (t1 * t1);
    w[2] = 0.5f * (t2 * t2);
}

/* The same weights for many fractions at once (w: 3 values per fraction). */
void orc_quadratic_weights_many(int64_t count, const float *f, float *w)
{
    for (int64_t i = 0; i < count; ++i)
        orc_quadratic_weights(f[i], w + 3 * i);
}

/* Stencil placement, same page: a fractional coordinate below one half uses
 * nodes {j-1, j, j+1}, otherwise {j, j+1, j+2}; that is base = floor(xi-1/2).
 * A particle is in the domain when its whole stencil lies on the grid:
 * 0 <= b and b + 2 <= n - 1, i.e. 0.5 <= xi < n - 1.5.  Returns 0 outside.  */
static int base_frac(const orc_desc *d, const float *const *x, int64_t p, int b[3], float f[3])
{
    for (int l = 0; l < 3; ++l) {
        b[l] = 0;
        f[l] = 0.0f;
    }
    for (int l = 0; l < d->dim; ++l) {
        float xi = x[l][p] * d->inv_dx;
        if (!(xi >= 0.5f && xi < (float)d->n[l] - 1.5f))
            return 0;
        b[l] = (int)floorf(xi - 0.5f);
        f[l] = xi - (float)b[l];
    }
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Cell keys and the stable counting sort.
 * "Particle Worlds, part 3", Step 3 (counting sort and the prefix sum): count
 * the particles of each bucket, an exclusive running total gives each
 * bucket's start, then each particle goes to its slot.  Here the bucket is
 * the particle's stencil base cell, numbered tile-major (tiles of T^d cells,
 * as the implementation guide's section 2.1 bins particles into tiles), and
 * the order inside a bucket is particle-index order (a stable sort).        */

static int tiles_per_axis(const orc_desc *d, int l)
{
    int cells = d->n[l] - 2;                 /* valid base cells 0 .. n-3 */
    return (cells + d->tile - 1) / d->tile;
}

int64_t orc_num_tiles(const orc_desc *d)
{
    int64_t t = 1;
    for (int l = 0; l < d->dim; ++l)
        t *= tiles_per_axis(d, l);
    return t;
}

static uint32_t key_of(const orc_desc *d, const int b[3])
{
    int T = d->tile;
    uint32_t tile_id = 0, local = 0;
    for (int l = d->dim - 1; l >= 0; --l) {
        tile_id = tile_id * (uint32_t)tiles_per_axis(d, l) + (uint32_t)(b[l] / T);
        local = local * (uint32_t)T + (uint32_t)(b[l] % T);
    }
    uint32_t cells_per_tile = 1;
    for (int l = 0; l < d->dim; ++l)
        cells_per_tile *= (uint32_t)T;
    return tile_id * cells_per_tile + local;
}

static int cmp_u64(const void *a, const void *b)
{
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return (x > y) - (x < y);
}

/* key[i] for every particle (ORC_KEY_INVALID outside the domain); perm = the
 * in-domain particles ordered by (tile, index) -- the stable counting sort
 * with the tile as bucket -- followed by the out-of-domain ones in index
 * order; tile_count[t] = particles whose base cell lies in tile t.  Returns
 * the number of in-domain particles.  (The pages leave the order inside a
 * bucket open: page 2's atomic scatter "doesn't put the particles in any
 * particular order within a cell"; the implementation guide, section 2.1,
 * asks that such a race be neutralised by sorting on a stable key.  Here the
 * key is the tile and ties keep particle-index order.)                      */
int64_t orc_bin(const orc_desc *d, int64_t np, const float *const *x,
                uint32_t *key, uint32_t *perm, uint32_t *tile_count)
{
    int64_t ntiles = orc_num_tiles(d);
    uint32_t cells_per_tile = 1;
    for (int l = 0; l < d->dim; ++l)
        cells_per_tile *= (uint32_t)d->tile;
    memset(tile_count, 0, sizeof(uint32_t) * (size_t)ntiles);
    uint64_t *pairs = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(np > 0 ? np : 1));
    int64_t valid = 0, invalid = 0;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (base_frac(d, x, p, b, f)) {
            key[p] = key_of(d, b);
            tile_count[key[p] / cells_per_tile] += 1;
            pairs[valid++] = ((uint64_t)(key[p] / cells_per_tile) << 32) | (uint64_t)p;
        } else {
            key[p] = ORC_KEY_INVALID;
        }
    }
    /* stable counting sort by tile: (tile, index) order */
    qsort(pairs, (size_t)valid, sizeof(uint64_t), cmp_u64);
    for (int64_t j = 0; j < valid; ++j)
        perm[j] = (uint32_t)(pairs[j] & 0xFFFFFFFFu);
    for (int64_t p = 0; p < np; ++p)
        if (key[p] == ORC_KEY_INVALID)
            perm[valid + invalid++] = (uint32_t)p;
    free(pairs);
    return valid;
}

/* ------------------------------------------------------------------------ */
/* Fixed-point P2G.
 * Implementation guide section 2.1 ("fixed-point atomics"): accumulate scaled
 * integers so the scatter is order-independent; section 3.3.1 and rule 1:
 * the encode rounds, it does not truncate, and the multiplier is a runtime
 * precision dial (any S = 2^scale_log2 here).  "particle to grid transfer in
 * checked integer arithmetic", "integers do not care about order": shares
 * are made integers by splitting, so a particle's shares sum to its quantity
 * exactly.  The momentum carried to a node is the APIC/MLS affine momentum
 * m w (v + C (x_i - x_p)) (implementation guide section 3.1, Part 1; the
 * PB-MPM reading in 3.3.2 scatters "momentum(d + D*offset)" with no stress).
 *
 * Bound (the same page, "the program": the bounds line runs before the loop,
 * and when it fails the program stops there, before any particle is
 * scattered).  The page bounds count * max m * max |v| by the int64 range.
 * Here a particle's quantity is spread over a stencil with an affine term,
 * so its range is taken per particle, in fp32, in this order:
 *     r_k = |v_k| + h*((|C_k0| + |C_k1|) + |C_k2|),   h = 1.5*dx
 *     r   = max(1, r_0, .., r_dim-1)
 *     R_p = max(|m|*r, |q|)          (q = rest volume in cells, volume channel)
 * with NaN making R_p NaN.  Since |x_i - x_p| <= 1.5 dx over the stencil and
 * the weights sum to one up to a few fp32 roundings, the absolute values of a
 * particle's shares of any channel sum to at most
 *     S*R_p*(1 + 2^-10) + 28
 * (26 shares each rounded by at most 1/2; the centre's remainder differs from
 * its own product by Q's rounding and the weights' and fma's roundings, which
 * are below 2^-16 relative).  A node's accumulator, and every partial sum on
 * the way to it, is at most the sum of these over the particles whose stencil
 * covers the node.  With R = max over the in-domain particles of R_p and
 * B = S*R*(1 + 2^-10) + 28 in fp64 (no contraction, this order):
 *     int64 accumulators:  n_in_domain * B <= 2^62
 *     int32 accumulators:  (most stencils covering one node) * B <= 2^31 - 1024
 * (the int32 form is the neighbourhood refinement of the global one).  If the
 * test fails (or R is NaN) nothing is scattered and the status reports the
 * bound.  The limits keep a margin below the types' maxima that covers the
 * fp64 rounding of the test itself.                                         */

#define ORC_I64_LIMIT 0x1p62
#define ORC_I32_LIMIT 2147482624.0 /* 2^31 - 1024 */

/* max that keeps NaN: NaN in either operand gives NaN */
static float max_nan(float a, float b)
{
    if (a != a || b != b)
        return NAN;
    return a > b ? a : b;
}

static float cells_of_volume(const orc_desc *d, float V0);

/* R_p of particle p (see above).  vol: rest volumes (volume channel) or NULL. */
static float particle_range(const orc_desc *d, const float *const *v, const float *const *C, const float *m,
                            const float *vol, int64_t p)
{
    int dim = d->dim;
    float h = 1.5f * d->dx;
    float r = 1.0f;
    for (int k = 0; k < dim; ++k) {
        float sc = fabsf(C[k * dim + 0][p]) + fabsf(C[k * dim + 1][p]);
        if (dim == 3)
            sc = sc + fabsf(C[k * dim + 2][p]);
        r = max_nan(r, fabsf(v[k][p]) + h * sc);
    }
    float R = fabsf(m[p]) * r;
    if (m[p] != m[p])
        R = NAN;
    if (vol)
        R = max_nan(R, fabsf(cells_of_volume(d, vol[p])));
    return R;
}

/* R = max of R_p over the in-domain particles (0 when there are none; NaN if
 * any R_p is NaN); *valid = their number.                                   */
float orc_scatter_range(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                        const float *const *C, const float *m, const float *vol, int64_t *valid)
{
    float R = 0.0f;
    int64_t nv = 0;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (!base_frac(d, x, p, b, f))
            continue;
        nv += 1;
        R = max_nan(R, particle_range(d, v, C, m, vol, p));
    }
    if (valid)
        *valid = nv;
    return R;
}

/* The most in-domain particles whose stencil covers one node: per base cell
 * the particle count, then per node the sum over the 3^dim base cells whose
 * stencil reaches it.                                                       */
int64_t orc_max_cover(const orc_desc *d, int64_t np, const float *const *x)
{
    int dim = d->dim;
    int64_t nodes = nodes_of(d);
    int64_t *cnt = (int64_t *)calloc((size_t)nodes, sizeof(int64_t)); /* indexed by the base node */
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (base_frac(d, x, p, b, f))
            cnt[node_at(d, b[0], b[1], dim == 3 ? b[2] : 0)] += 1;
    }
    int64_t best = 0;
    int nk = dim == 3 ? d->n[2] : 1;
    for (int k = 0; k < nk; ++k)
        for (int j = 0; j < d->n[1]; ++j)
            for (int i = 0; i < d->n[0]; ++i) {
                int64_t s = 0;
                for (int a2 = 0; a2 < (dim == 3 ? 3 : 1); ++a2)
                    for (int a1 = 0; a1 < 3; ++a1)
                        for (int a0 = 0; a0 < 3; ++a0) {
                            int bi = i - a0, bj = j - a1, bk = k - a2;
                            if (bi < 0 || bj < 0 || bk < 0)
                                continue;
                            s += cnt[node_at(d, bi, bj, bk)];
                        }
                if (s > best)
                    best = s;
            }
    free(cnt);
    return best;
}

/* 1 when the accumulators of this mode hold `count` particles of range R
 * (count = in-domain particles for int64, orc_max_cover for int32).        */
int orc_bound_ok(const orc_desc *d, float R, int64_t count)
{
    double S = ldexp(1.0, d->scale_log2);
    double B = S * (double)R;
    B = B * (1.0 + 0x1p-10);
    B = B + 28.0;
    double total = (double)count * B;
    double limit = d->acc_mode == 0 ? ORC_I32_LIMIT : ORC_I64_LIMIT;
    return total <= limit;
}

/* rint of the exact product a*b: the product of two fp32 values is exact in
 * fp64 (48 significant bits); nearbyint rounds it once, ties to even (the
 * default rounding mode).  Callers keep |a*b| below 2^62 by the bound.     */
static int64_t rint_product(float a, float b)
{
    return (int64_t)nearbyint((double)a * (double)b);
}

/* The grid-recovered volume channel (implementation guide, section 3.3.2,
 * "grid-recovered volume": each particle scatters its rest volume as a
 * fraction of a cell, 1/ppc for a rest packing, so that a node of a
 * rest-packed region sums to about one; G2P gathers the node values back).
 * The quantity is q = V0 * inv_dx^dim (inv_dx^3 = (inv_dx*inv_dx)*inv_dx),
 * scattered as the mass is: Vt = q*S, share rint(((wx*Vt)*wy)*wz), and the
 * centre node takes rint(Vt) minus the other shares.  It is the last plane
 * of acc and enters the bound through R_p.                                  */
static float cells_of_volume(const orc_desc *d, float V0)
{
    float c = d->inv_dx * d->inv_dx;
    if (d->dim == 3)
        c = c * d->inv_dx;
    return V0 * c;
}

/* Scatters every in-domain particle, no bound check (the callers check it
 * first).  counts[0] += out-of-domain particles.                           */
static void scatter_fixed_all(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                              const float *const *C, const float *m, const float *vol, int64_t *acc,
                              int64_t *outside);

static uint32_t p2g_fixed_core(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                               const float *const *C, const float *m, const float *vol, int64_t *acc,
                               int64_t counts[2]);

/* acc: (dim+1) planes of nodes_of(d) int64 values (mass, then momentum per
 * axis), zeroed by the caller.  counts[0] = out-of-domain particles,
 * counts[1] = in-domain particles left unscattered because the bound failed
 * (all of them, or none).  Returns the status bits.                         */
uint32_t orc_p2g_fixed(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                       const float *const *C, const float *m, int64_t *acc, int64_t counts[2])
{
    return p2g_fixed_core(d, np, x, v, C, m, NULL, acc, counts);
}

/* The same with the volume channel: acc has dim+2 planes, the last one the
 * rest volume in cells.                                                     */
uint32_t orc_p2g_fixed_vol(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                           const float *const *C, const float *m, const float *vol, int64_t *acc,
                           int64_t counts[2])
{
    return p2g_fixed_core(d, np, x, v, C, m, vol, acc, counts);
}

static uint32_t p2g_fixed_core(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                               const float *const *C, const float *m, const float *vol, int64_t *acc,
                               int64_t counts[2])
{
    int64_t valid = 0;
    float R = orc_scatter_range(d, np, x, v, C, m, vol, &valid);
    int64_t count = d->acc_mode == 0 ? orc_max_cover(d, np, x) : valid;
    counts[0] = np - valid;
    counts[1] = 0;
    if (!orc_bound_ok(d, R, count)) {
        counts[1] = valid;
        return (counts[0] ? ORC_ST_DOMAIN : 0u) | ORC_ST_BOUND;
    }
    int64_t outside = 0;
    scatter_fixed_all(d, np, x, v, C, m, vol, acc, &outside);
    return counts[0] ? ORC_ST_DOMAIN : 0u;
}

static void scatter_fixed_all(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                              const float *const *C, const float *m, const float *vol, int64_t *acc,
                              int64_t *outside)
{
    int dim = d->dim;
    int64_t nodes = nodes_of(d);
    float S = ldexpf(1.0f, d->scale_log2);
    int64_t vplane = (int64_t)(dim + 1) * nodes;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (!base_frac(d, x, p, b, f)) {
            *outside += 1;
            continue;
        }
        float Mt = m[p] * S;
        float Vt = vol ? cells_of_volume(d, vol[p]) * S : 0.0f;
        float w[3][3], dd[3][3];
        for (int l = 0; l < 3; ++l)
            for (int a = 0; a < 3; ++a) {
                w[l][a] = 1.0f;
                dd[l][a] = 0.0f;
            }
        for (int l = 0; l < dim; ++l) {
            orc_quadratic_weights(f[l], w[l]);
            for (int a = 0; a < 3; ++a)
                dd[l][a] = ((float)a - f[l]) * d->dx;
        }
        int64_t Q[4] = {0, 0, 0, 0};
        Q[0] = (int64_t)rintf(Mt);
        for (int k = 0; k < dim; ++k)
            Q[1 + k] = (int64_t)rintf(Mt * v[k][p]);
        int64_t rest[4] = {Q[0], Q[1], Q[2], Q[3]};
        int64_t vrest = (int64_t)rintf(Vt);
        int a2n = dim == 3 ? 3 : 1;
        for (int a0 = 0; a0 < 3; ++a0)
            for (int a1 = 0; a1 < 3; ++a1)
                for (int a2 = 0; a2 < a2n; ++a2) {
                    int centre = a0 == 1 && a1 == 1 && (dim == 2 || a2 == 1);
                    if (centre)
                        continue;
                    float Wt = (w[0][a0] * Mt) * w[1][a1];
                    if (dim == 3)
                        Wt = Wt * w[2][a2];
                    int64_t node = node_at(d, b[0] + a0, b[1] + a1, dim == 3 ? b[2] + a2 : 0);
                    int64_t sm = (int64_t)rintf(Wt);
                    acc[node] += sm;
                    rest[0] -= sm;
                    if (vol) {
                        float Wv = (w[0][a0] * Vt) * w[1][a1];
                        if (dim == 3)
                            Wv = Wv * w[2][a2];
                        int64_t sv = (int64_t)rintf(Wv);
                        acc[vplane + node] += sv;
                        vrest -= sv;
                    }
                    for (int k = 0; k < dim; ++k) {
                        float vel = fmaf(C[k * dim + 0][p], dd[0][a0], v[k][p]);
                        vel = fmaf(C[k * dim + 1][p], dd[1][a1], vel);
                        if (dim == 3)
                            vel = fmaf(C[k * dim + 2][p], dd[2][a2], vel);
                        int64_t sk = rint_product(Wt, vel);
                        acc[(int64_t)(1 + k) * nodes + node] += sk;
                        rest[1 + k] -= sk;
                    }
                }
        int64_t cnode = node_at(d, b[0] + 1, b[1] + 1, dim == 3 ? b[2] + 1 : 0);
        for (int c = 0; c <= dim; ++c)
            acc[(int64_t)c * nodes + cnode] += rest[c];
        if (vol)
            acc[vplane + cnode] += vrest;
    }
}

/* Float-atomic P2G for comparison (implementation guide section 2.1 caveat:
 * float atomics are order-dependent).  The node value is the sum over
 * particles of the fp32 terms u_m(a) = W(a), u_k(a) = W(a) * vel_k(a) with
 * W(a) = ((wx*m)*wy)*wz; the oracle adds them in fp64.                      */
static uint32_t p2g_float_core(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                               const float *const *C, const float *m, const float *vol, double *acc,
                               int64_t counts[2]);

uint32_t orc_p2g_float(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                       const float *const *C, const float *m, double *acc, int64_t counts[2])
{
    return p2g_float_core(d, np, x, v, C, m, NULL, acc, counts);
}

/* With the volume channel (last plane): the fp32 terms ((wx*q)*wy)*wz of
 * q = V0 * inv_dx^dim, summed in fp64.                                      */
uint32_t orc_p2g_float_vol(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                           const float *const *C, const float *m, const float *vol, double *acc,
                           int64_t counts[2])
{
    return p2g_float_core(d, np, x, v, C, m, vol, acc, counts);
}

static uint32_t p2g_float_core(const orc_desc *d, int64_t np, const float *const *x, const float *const *v,
                               const float *const *C, const float *m, const float *vol, double *acc,
                               int64_t counts[2])
{
    int dim = d->dim;
    int64_t nodes = nodes_of(d);
    int64_t vplane = (int64_t)(dim + 1) * nodes;
    counts[0] = counts[1] = 0;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (!base_frac(d, x, p, b, f)) {
            counts[0] += 1;
            continue;
        }
        float w[3][3], dd[3][3];
        for (int l = 0; l < 3; ++l)
            for (int a = 0; a < 3; ++a) {
                w[l][a] = 1.0f;
                dd[l][a] = 0.0f;
            }
        for (int l = 0; l < dim; ++l) {
            orc_quadratic_weights(f[l], w[l]);
            for (int a = 0; a < 3; ++a)
                dd[l][a] = ((float)a - f[l]) * d->dx;
        }
        int a2n = dim == 3 ? 3 : 1;
        for (int a0 = 0; a0 < 3; ++a0)
            for (int a1 = 0; a1 < 3; ++a1)
                for (int a2 = 0; a2 < a2n; ++a2) {
                    float W = (w[0][a0] * m[p]) * w[1][a1];
                    if (dim == 3)
                        W = W * w[2][a2];
                    int64_t node = node_at(d, b[0] + a0, b[1] + a1, dim == 3 ? b[2] + a2 : 0);
                    acc[node] += (double)W;
                    if (vol) {
                        float Wv = (w[0][a0] * cells_of_volume(d, vol[p])) * w[1][a1];
                        if (dim == 3)
                            Wv = Wv * w[2][a2];
                        acc[vplane + node] += (double)Wv;
                    }
                    for (int k = 0; k < dim; ++k) {
                        float vel = fmaf(C[k * dim + 0][p], dd[0][a0], v[k][p]);
                        vel = fmaf(C[k * dim + 1][p], dd[1][a1], vel);
                        if (dim == 3)
                            vel = fmaf(C[k * dim + 2][p], dd[2][a2], vel);
                        acc[(int64_t)(1 + k) * nodes + node] += (double)(W * vel);
                    }
                }
    }
    return counts[0] ? ORC_ST_DOMAIN : 0u;
}

/* ------------------------------------------------------------------------ */
/* MLS-MPM elastic stress (implementation guide, section 3.1, Part 2: the
 * Neo-Hookean model with Lame constants mu and lambda,
 *     J = det F,  P = mu (F - F^-T) + lambda ln(J) F^-T,  sigma = P F^T / J).
 * In MLS-MPM the stress enters the same affine scatter as the APIC matrix:
 * node momentum gains -dt V sigma D^-1 w (x_i - x_p), with V = V0 J the
 * particle's current volume and D^-1 = 4/dx^2 the quadratic B-spline's
 * inverse inertia (the guide's "D (= B*4)", section 3.3.2).  Dividing by the
 * particle mass folds it into C:
 *     C' = C - kappa tau,  kappa = dt V0 (4/dx^2) / m,  tau = J sigma = P F^T
 * and P F^T = mu (F F^T - I) + lambda ln(J) I, because F^-T F^T = I.  So the
 * scatter itself is unchanged; only the matrix it reads differs.
 *
 * Evaluation order (fp32, round to nearest even, no contraction), the
 * contract the GPU reproduces bit for bit:
 *   J (3D)  = (F00*(F11*F22 - F12*F21) - F01*(F10*F22 - F12*F20))
 *             + F02*(F10*F21 - F11*F20);      J (2D) = F00*F11 - F01*F10
 *   b_kl    = (F_k0*F_l0 + F_k1*F_l1) + F_k2*F_l2       (F F^T, index order)
 *   tau_kl  = mu*b_kl (k != l);  tau_kk = mu*(b_kk - 1) + lambda*ln(J)
 *   kappa   = ((dt*V0) * c4s) / m,  c4s = (4*inv_dx)*inv_dx
 *   C'_kl   = C_kl - kappa*tau_kl
 * A particle whose J is not a positive normal finite number (an inverted or
 * collapsed element; ln J undefined) keeps C' = C and is counted.
 *
 * ln is computed here, not taken from the C library, so that both sides
 * round identically: J = 2^e * r with r in [1/sqrt2, sqrt2), and
 * ln r = 2 atanh(s), s = (r - 1)/(r + 1), from the series
 * atanh(s) = s + s^3/3 + s^5/5 + s^7/7 + s^9/9 + ..., |s| <= 0.1716, so the
 * dropped terms are below 2e-9 relative.  ln 2 is split as
 * LN2_HI = 45426/65536 (e * LN2_HI exact for |e| < 256) plus LN2_LO.
 *   z = s*s;  p = ((1/9*z + 1/7)*z + 1/5)*z + 1/3   (each op rounded)
 *   ln r = 2*(s + s*(z*p));   ln J = e*LN2_HI + (e*LN2_LO + ln r)         */

#define ORC_LN2_HI 0x1.62e4p-1f       /* 45426 / 65536 */
#define ORC_LN2_LO 0x1.7f7d1cp-20f    /* ln 2 - LN2_HI, rounded to fp32 */
#define ORC_SQRT2 0x1.6a09e6p+0f      /* sqrt(2) rounded down to fp32 */

/* 1 if J > 0 is a normal finite fp32 number. */
static int orc_log_domain(float J)
{
    return J >= 0x1p-126f && J <= 0x1.fffffep+127f;
}

/* ln J for J in the log domain (above); 0 outside it. */
float orc_log(float J)
{
    if (!orc_log_domain(J))
        return 0.0f;
    uint32_t u;
    memcpy(&u, &J, sizeof u);
    int e = (int)(u >> 23) - 127;
    u = (u & 0x007FFFFFu) | 0x3F800000u;
    float r;
    memcpy(&r, &u, sizeof r);
    if (r > ORC_SQRT2) {
        r = r * 0.5f;
        e += 1;
    }
    float s = (r - 1.0f) / (r + 1.0f);
    float z = s * s;
    float p = (1.0f / 9.0f) * z + (1.0f / 7.0f);
    p = p * z + (1.0f / 5.0f);
    p = p * z + (1.0f / 3.0f);
    float lr = 2.0f * (s + s * (z * p));
    float fe = (float)e;
    return fe * ORC_LN2_HI + (fe * ORC_LN2_LO + lr);
}

/* Kirchhoff stress tau = P F^T of the Neo-Hookean model; F and tau are
 * dim x dim row-major (F[k*dim + l]).  Returns 0 (tau = 0) when J is
 * outside the log domain, else 1.                                           */
int orc_kirchhoff(int dim, float mu, float lambda, const float *F, float *tau)
{
    float J;
    if (dim == 3) {
        float c0 = F[4] * F[8] - F[5] * F[7];
        float c1 = F[3] * F[8] - F[5] * F[6];
        float c2 = F[3] * F[7] - F[4] * F[6];
        J = (F[0] * c0 - F[1] * c1) + F[2] * c2;
    } else {
        J = F[0] * F[3] - F[1] * F[2];
    }
    for (int j = 0; j < dim * dim; ++j)
        tau[j] = 0.0f;
    if (!orc_log_domain(J))
        return 0;
    float lj = lambda * orc_log(J);
    for (int k = 0; k < dim; ++k)
        for (int l = 0; l < dim; ++l) {
            float b = F[k * dim + 0] * F[l * dim + 0] + F[k * dim + 1] * F[l * dim + 1];
            if (dim == 3)
                b = b + F[k * dim + 2] * F[l * dim + 2];
            tau[k * dim + l] = k == l ? mu * (b - 1.0f) + lj : mu * b;
        }
    return 1;
}

/* C' = C - kappa tau for every particle (Cout may alias C).  Returns the
 * number of in-domain particles whose J is outside the log domain (those
 * keep C' = C); out-of-domain particles are folded too but not counted,
 * since P2G never scatters them.                                            */
int64_t orc_stress_affine(const orc_desc *d, float dt, float mu, float lambda, int64_t np,
                          const float *const *x, const float *const *C, const float *const *F,
                          const float *vol, const float *m, float *const *Cout)
{
    int dim = d->dim;
    float c4s = (4.0f * d->inv_dx) * d->inv_dx;
    int64_t degenerate = 0;
    for (int64_t p = 0; p < np; ++p) {
        float Fp[9] = {0}, tau[9];
        for (int j = 0; j < dim * dim; ++j)
            Fp[j] = F[j][p];
        int ok = orc_kirchhoff(dim, mu, lambda, Fp, tau);
        int b[3];
        float f[3];
        if (!ok) {
            if (base_frac(d, x, p, b, f))
                degenerate += 1;
            for (int j = 0; j < dim * dim; ++j)
                Cout[j][p] = C[j][p];
            continue;
        }
        float kappa = ((dt * vol[p]) * c4s) / m[p];
        for (int j = 0; j < dim * dim; ++j)
            Cout[j][p] = C[j][p] - kappa * tau[j];
    }
    return degenerate;
}

/* ------------------------------------------------------------------------ */
/* Grid update.  Implementation guide section 2.1 (the grid pass:
 * mass-normalise, collide, boundary) and section 3.3.2's note that the
 * velocity-form boundary is a sign test; rule 7: gravity is a solver
 * parameter.  v = P / M in fp32 (the scale cancels), then v += dt*g, then,
 * per axis, a node within `boundary_nodes` of a wall keeps no velocity
 * component pointing into that wall.  An empty node (M == 0) has v = 0.    */

static void update_node(const orc_desc *d, int i, int j, int k, float M, const float *P,
                        const float *dtg, float *out)
{
    int idx[3] = {i, j, k};
    int B = d->boundary_nodes;
    for (int l = 0; l < 3; ++l)
        out[l] = 0.0f;
    if (M == 0.0f)
        return;
    for (int l = 0; l < d->dim; ++l) {
        float vl = P[l] / M;
        vl = vl + dtg[l];
        if ((idx[l] < B && vl < 0.0f) || (idx[l] > d->n[l] - 1 - B && vl > 0.0f))
            vl = 0.0f;
        out[l] = vl;
    }
}

/* acc int64 planes (fixed-point sums); vel: dim planes of fp32.            */
void orc_grid_update_fixed(const orc_desc *d, const int64_t *acc, const float *dtg, float *vel)
{
    int64_t nodes = nodes_of(d);
    int nk = d->dim == 3 ? d->n[2] : 1;
    for (int k = 0; k < nk; ++k)
        for (int j = 0; j < d->n[1]; ++j)
            for (int i = 0; i < d->n[0]; ++i) {
                int64_t node = node_at(d, i, j, k);
                int64_t Mi = acc[node];
                float P[3] = {0.0f, 0.0f, 0.0f}, out[3];
                for (int l = 0; l < d->dim; ++l)
                    P[l] = (float)acc[(int64_t)(1 + l) * nodes + node];
                update_node(d, i, j, k, (float)Mi, P, dtg, out);
                for (int l = 0; l < d->dim; ++l)
                    vel[(int64_t)l * nodes + node] = out[l];
            }
}

/* Float mode: the fp64 sums are first rounded to fp32 (the precision the
 * float-atomic grid holds), then updated as above.                         */
void orc_grid_update_float(const orc_desc *d, const double *acc, const float *dtg, float *vel)
{
    int64_t nodes = nodes_of(d);
    int nk = d->dim == 3 ? d->n[2] : 1;
    for (int k = 0; k < nk; ++k)
        for (int j = 0; j < d->n[1]; ++j)
            for (int i = 0; i < d->n[0]; ++i) {
                int64_t node = node_at(d, i, j, k);
                float P[3] = {0.0f, 0.0f, 0.0f}, out[3];
                for (int l = 0; l < d->dim; ++l)
                    P[l] = (float)acc[(int64_t)(1 + l) * nodes + node];
                update_node(d, i, j, k, (float)acc[node], P, dtg, out);
                for (int l = 0; l < d->dim; ++l)
                    vel[(int64_t)l * nodes + node] = out[l];
            }
}

/* ------------------------------------------------------------------------ */
/* G2P.  Implementation guide section 1: each particle reads its stencil and
 * writes only itself; section 3.1 Part 1 (APIC) and 3.3.2 ("gather d and D
 * (= B*4)"): the new velocity is sum_a w v_a and the affine matrix is
 * C = B * 4/dx^2 with B = sum_a w v_a (x_a - x_p)^T, here in cell units so
 * C_kl = (sum_a w v_k(a) e_l(a)) * (4 * inv_dx).  Then x += dt v.
 *
 * Evaluation order (the contract): the stencil sum is taken axis by axis,
 * innermost axis first; a three-term sum is fma(w2,t2, fma(w1,t1, w0*t0)).
 * With we_l[a] = w_l[a] * e_l[a]:
 *   Z (a0,a1) = sum_a2 wz  vel      Zq(a0,a1) = sum_a2 wez vel
 *   Y (a0)    = sum_a1 wy  Z        Ye(a0)    = sum_a1 wey Z
 *   Yq(a0)    = sum_a1 wy  Zq
 *   v'        = sum_a0 wx  Y        B_0 = sum_a0 wex Y
 *   B_1       = sum_a0 wx  Ye       B_2 = sum_a0 wx  Yq
 * (2D: drop the z level; Y is the innermost sum over a1.)                   */

static float sum3(const float w[3], const float t[3])
{
    return fmaf(w[2], t[2], fmaf(w[1], t[1], w[0] * t[0]));
}

/* Out-of-domain particles are left unchanged.  Returns how many moved.
 * With F (not NULL) the deformation gradient of every moved particle is
 * advanced with its new C (implementation guide, section 3.3.2: F <- (I + D) F,
 * where the velocity form's D is dt C):
 *   F'_kl = fma(D_k2, F_2l, fma(D_k1, F_1l, fma(D_k0, F_0l, F_kl))),
 *   D_kj = dt * C'_kj        (2D: drop the third term).                   */
static int64_t g2p_core(const orc_desc *d, const float *vel, int64_t np, float *const *x, float *const *v,
                        float *const *C, float *const *F, float dt);

int64_t orc_g2p(const orc_desc *d, const float *vel, int64_t np, float *const *x, float *const *v,
                float *const *C, float dt)
{
    return g2p_core(d, vel, np, x, v, C, NULL, dt);
}

int64_t orc_g2p_elastic(const orc_desc *d, const float *vel, int64_t np, float *const *x, float *const *v,
                        float *const *C, float *const *F, float dt)
{
    return g2p_core(d, vel, np, x, v, C, F, dt);
}

static int64_t g2p_core(const orc_desc *d, const float *vel, int64_t np, float *const *x, float *const *v,
                        float *const *C, float *const *F, float dt)
{
    int dim = d->dim;
    int64_t nodes = nodes_of(d);
    float c4 = 4.0f * d->inv_dx;
    int64_t moved = 0;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (!base_frac(d, (const float *const *)x, p, b, f))
            continue;
        float w[3][3], we[3][3];
        for (int l = 0; l < dim; ++l) {
            orc_quadratic_weights(f[l], w[l]);
            for (int a = 0; a < 3; ++a)
                we[l][a] = w[l][a] * ((float)a - f[l]);
        }
        float vnew[3] = {0, 0, 0}, Bm[3][3] = {{0}};
        for (int k = 0; k < dim; ++k) {
            const float *vk = vel + (int64_t)k * nodes;
            if (dim == 3) {
                float Y[3], Ye[3], Yq[3];
                for (int a0 = 0; a0 < 3; ++a0) {
                    float Z[3], Zq[3];
                    for (int a1 = 0; a1 < 3; ++a1) {
                        float t[3];
                        for (int a2 = 0; a2 < 3; ++a2)
                            t[a2] = vk[node_at(d, b[0] + a0, b[1] + a1, b[2] + a2)];
                        Z[a1] = sum3(w[2], t);
                        Zq[a1] = sum3(we[2], t);
                    }
                    Y[a0] = sum3(w[1], Z);
                    Ye[a0] = sum3(we[1], Z);
                    Yq[a0] = sum3(w[1], Zq);
                }
                vnew[k] = sum3(w[0], Y);
                Bm[k][0] = sum3(we[0], Y);
                Bm[k][1] = sum3(w[0], Ye);
                Bm[k][2] = sum3(w[0], Yq);
            } else {
                float Y[3], Ye[3];
                for (int a0 = 0; a0 < 3; ++a0) {
                    float t[3];
                    for (int a1 = 0; a1 < 3; ++a1)
                        t[a1] = vk[node_at(d, b[0] + a0, b[1] + a1, 0)];
                    Y[a0] = sum3(w[1], t);
                    Ye[a0] = sum3(we[1], t);
                }
                vnew[k] = sum3(w[0], Y);
                Bm[k][0] = sum3(we[0], Y);
                Bm[k][1] = sum3(w[0], Ye);
            }
        }
        for (int k = 0; k < dim; ++k) {
            v[k][p] = vnew[k];
            for (int l = 0; l < dim; ++l)
                C[k * dim + l][p] = Bm[k][l] * c4;
        }
        for (int l = 0; l < dim; ++l)
            x[l][p] = fmaf(dt, vnew[l], x[l][p]);
        if (F) {
            float D[9], Fo[9];
            for (int j = 0; j < dim * dim; ++j) {
                D[j] = dt * C[j][p];
                Fo[j] = F[j][p];
            }
            for (int k = 0; k < dim; ++k)
                for (int l = 0; l < dim; ++l) {
                    float t = fmaf(D[k * dim + 0], Fo[0 * dim + l], Fo[k * dim + l]);
                    t = fmaf(D[k * dim + 1], Fo[1 * dim + l], t);
                    if (dim == 3)
                        t = fmaf(D[k * dim + 2], Fo[2 * dim + l], t);
                    F[k * dim + l][p] = t;
                }
        }
        moved += 1;
    }
    return moved;
}

/* Grid volume fraction from the volume channel: phi = (float)V * 2^-scale
 * (fixed point; the int64 sum rounded once, the scale exact), or the fp64 sum
 * rounded to fp32 (float mode).  vplane: the channel's nodes_of(d) values.  */
void orc_grid_volume_fixed(const orc_desc *d, const int64_t *vplane, float *phi)
{
    int64_t nodes = nodes_of(d);
    float inv_S = ldexpf(1.0f, -d->scale_log2);
    for (int64_t i = 0; i < nodes; ++i)
        phi[i] = (float)vplane[i] * inv_S;
}

void orc_grid_volume_float(const orc_desc *d, const double *vplane, float *phi)
{
    int64_t nodes = nodes_of(d);
    for (int64_t i = 0; i < nodes; ++i)
        phi[i] = (float)vplane[i];
}

/* The particle's grid-recovered volume fraction: sum_a w(a) phi(a), taken in
 * the G2P's order (innermost axis first, three-term sums as in sum3), from
 * the positions before advection.  Out-of-domain particles are left as they
 * are.  Returns how many were written.                                      */
int64_t orc_g2p_volume(const orc_desc *d, const float *phi, int64_t np, const float *const *x, float *out)
{
    int dim = d->dim;
    int64_t written = 0;
    for (int64_t p = 0; p < np; ++p) {
        int b[3];
        float f[3];
        if (!base_frac(d, x, p, b, f))
            continue;
        float w[3][3];
        for (int l = 0; l < dim; ++l)
            orc_quadratic_weights(f[l], w[l]);
        float Y[3];
        for (int a0 = 0; a0 < 3; ++a0) {
            if (dim == 3) {
                float Z[3];
                for (int a1 = 0; a1 < 3; ++a1) {
                    float t[3];
                    for (int a2 = 0; a2 < 3; ++a2)
                        t[a2] = phi[node_at(d, b[0] + a0, b[1] + a1, b[2] + a2)];
                    Z[a1] = sum3(w[2], t);
                }
                Y[a0] = sum3(w[1], Z);
            } else {
                float t[3];
                for (int a1 = 0; a1 < 3; ++a1)
                    t[a1] = phi[node_at(d, b[0] + a0, b[1] + a1, 0)];
                Y[a0] = sum3(w[1], t);
            }
        }
        out[p] = sum3(w[0], Y);
        written += 1;
    }
    return written;
}

/* The advective time-step bound of the implementation guide (section 3.3.2,
 * rule 6: the step must satisfy dt <= dx / max_p(|v_p| + 1.5 dx |C_p|_F)):
 * the largest |v_p| + 1.5 dx |C_p|_F over np particles, each term in fp32 as
 * sqrt((vx*vx + vy*vy) + vz*vz) + (1.5*dx) * sqrt(C0*C0 + C1*C1 + ... ), the
 * sums taken in index order.  0 for no particle.                            */
float orc_advective_speed(int dim, float dx, int64_t np, const float *const *v, const float *const *C)
{
    float best = 0.0f;
    float h = 1.5f * dx;
    for (int64_t p = 0; p < np; ++p) {
        float sv = 0.0f, sc = 0.0f;
        for (int k = 0; k < dim; ++k)
            sv = sv + v[k][p] * v[k][p];
        for (int j = 0; j < dim * dim; ++j)
            sc = sc + C[j][p] * C[j][p];
        float t = sqrtf(sv) + h * sqrtf(sc);
        if (t > best)
            best = t;
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* The integer cloud-in-cell transfer of "particle to grid transfer in
 * checked integer arithmetic".  Positions are integers in 1/65,536 of a cell;
 * for a quantity q and node fraction F/65,536 the far (upper) node's share is
 * q*F/65,536 rounded once to the nearest integer, the near node's share is q
 * minus that; the split is taken along x, then each part along y (and z).
 * Rounding ties go to even.                                                 */

int64_t orc_rdiv(int64_t a, int64_t b)
{
    int64_t q = a / b, r = a % b;
    uint64_t ar = r < 0 ? (uint64_t)0 - (uint64_t)r : (uint64_t)r;
    uint64_t br = b < 0 ? (uint64_t)0 - (uint64_t)b : (uint64_t)b;
    uint64_t other = br - ar;
    if (ar > other || (ar == other && (q & 1)))
        q += ((a < 0) != (b < 0)) ? -1 : 1;
    return q;
}

/* The page's bounds line, as an executable statement before any scatter:
 * the largest value a node can hold is the particle count times the largest
 * mass times the largest speed; it must fit int64.  The products q*F of the
 * split must fit too, and every position must be on the grid.  Returns 1 if
 * the scatter may run.                                                      */
int orc_cic_int_bound(int dim, const int32_t *n, int64_t np, const int32_t *const *X, const int64_t *m,
                      const int64_t *const *v)
{
    __int128 mmax = 0, vmax = 0;
    for (int64_t p = 0; p < np; ++p) {
        __int128 am = m[p] < 0 ? -(__int128)m[p] : (__int128)m[p];
        if (am > mmax)
            mmax = am;
        for (int k = 0; k < dim; ++k) {
            __int128 av = v[k][p] < 0 ? -(__int128)v[k][p] : (__int128)v[k][p];
            if (av > vmax)
                vmax = av;
        }
        for (int l = 0; l < dim; ++l)
            if (X[l][p] < 0 || (X[l][p] >> 16) > n[l] - 2)
                return 0;
    }
    /* q = largest |m|*|v| (or |m|); each factor is below 2^64, so q fits 128 bits */
    __int128 q = mmax * (vmax > 1 ? vmax : 1);
    if (q > (__int128)INT64_MAX / 65536)
        return 0;
    if (q * (__int128)np > (__int128)INT64_MAX)
        return 0;
    return 1;
}

static void cic_split_add(int dim, const int32_t *n, int64_t *plane, const int c[3], const int32_t F[3],
                          int axis, int idx[3], int64_t q)
{
    if (axis == dim) {
        int64_t node = ((int64_t)(dim == 3 ? idx[2] : 0) * n[1] + idx[1]) * n[0] + idx[0];
        plane[node] += q;
        return;
    }
    int64_t far = orc_rdiv(q * (int64_t)F[axis], 65536);
    int64_t near = q - far;
    idx[axis] = c[axis];
    cic_split_add(dim, n, plane, c, F, axis + 1, idx, near);
    idx[axis] = c[axis] + 1;
    cic_split_add(dim, n, plane, c, F, axis + 1, idx, far);
}

/* acc: (dim+1) planes of int64 (mass, momentum per axis), zeroed by the
 * caller.  order: the particle visiting order (NULL = 0..np-1).  Returns 0
 * (and scatters nothing) when the bounds line fails, 1 otherwise.          */
int orc_cic_int_p2g(int dim, const int32_t *n, int64_t np, const int32_t *const *X, const int64_t *m,
                    const int64_t *const *v, const int64_t *order, int64_t *acc)
{
    if (!orc_cic_int_bound(dim, n, np, X, m, v))
        return 0;
    int64_t nodes = (int64_t)n[0] * n[1] * (dim == 3 ? n[2] : 1);
    for (int64_t s = 0; s < np; ++s) {
        int64_t p = order ? order[s] : s;
        int c[3] = {0, 0, 0};
        int32_t F[3] = {0, 0, 0};
        for (int l = 0; l < dim; ++l) {
            c[l] = X[l][p] >> 16;
            F[l] = X[l][p] & 0xFFFF;
        }
        int idx[3] = {0, 0, 0};
        cic_split_add(dim, n, acc, c, F, 0, idx, m[p]);
        for (int k = 0; k < dim; ++k)
            cic_split_add(dim, n, acc + (int64_t)(1 + k) * nodes, c, F, 0, idx, m[p] * v[k][p]);
    }
    return 1;
}

/* Gather (same page, "the last lines gather velocity back for one particle
 * from its four nodes, with the division rounded by name"): the particle's
 * cell momentum over its cell mass, rounded to nearest, ties to even.      */
void orc_cic_int_gather(int dim, const int32_t *n, int64_t np, const int32_t *const *X, const int64_t *acc,
                        int64_t *const *vout)
{
    int64_t nodes = (int64_t)n[0] * n[1] * (dim == 3 ? n[2] : 1);
    int corners = 1 << dim;
    for (int64_t p = 0; p < np; ++p) {
        int c[3] = {0, 0, 0};
        for (int l = 0; l < dim; ++l)
            c[l] = X[l][p] >> 16;
        int64_t M = 0, P[3] = {0, 0, 0};
        for (int s = 0; s < corners; ++s) {
            int i = c[0] + (s & 1), j = c[1] + ((s >> 1) & 1), k = dim == 3 ? c[2] + ((s >> 2) & 1) : 0;
            int64_t node = ((int64_t)k * n[1] + j) * n[0] + i;
            M += acc[node];
            for (int l = 0; l < dim; ++l)
                P[l] += acc[(int64_t)(1 + l) * nodes + node];
        }
        for (int l = 0; l < dim; ++l)
            vout[l][p] = M != 0 ? orc_rdiv(P[l], M) : 0;
    }
}
