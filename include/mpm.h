/*
 * mpm.h -- C ABI of the GB300 (sm_103a) Material Point Method transfer library.
 *
 * One explicit MPM transfer step, in the four phases "reset -> particle-to-grid
 * (P2G) -> grid update -> grid-to-particle (G2P)" of "Implementation -- GPU
 * Optimization & Reference Codebases", section 1, plus the cell-key binning
 * that feeds P2G (section 2.1, "spatial sorting + tiling"; "Particle Worlds,
 * part 3", Step 3, the counting sort):
 *
 *   mpm_bin          cell keys, tile histogram, exclusive scan, stable scatter
 *   mpm_p2g          scatter of mass and APIC/MLS affine momentum, fixed point
 *                    (int32/int64) or float atomics
 *   mpm_grid_update  momentum -> velocity, gravity, boundary; clears the
 *                    accumulators it reads
 *   mpm_g2p          gather of velocity and affine matrix, advection
 *   mpm_step_fused   grid update, G2P and the next P2G in one kernel
 *   mpm_iterate      the position-based transfer loop, one kernel per iteration
 *
 * Conventions shared by every call:
 *  - All pointers inside the structs are DEVICE pointers unless a call says
 *    otherwise.  The caller owns all memory; the library allocates nothing.
 *  - Calls are asynchronous and stream ordered on the stream passed in (a
 *    cudaStream_t given as void*; NULL is the legacy default stream).
 *  - Argument errors are found on the host, returned at once, and launch
 *    nothing.  Data errors (particles outside the domain, shares out of range,
 *    a failed accumulator bound) are recorded in the device status words of
 *    mpm_bins; read them with mpm_read_status (asynchronous copy).
 *  - Particle arrays are structure-of-arrays, one array per component.  The
 *    affine matrix is C[k*dim + l] = d v_k / d x_l.
 *  - Grid arrays are planar: channel c of node (i, j, k) is at
 *    c*nodes + (k*n[1] + j)*n[0] + i.  Accumulator channels: mass, then
 *    momentum along each axis, then (volume_channel) the rest volume.
 *    Velocity channels: one per axis, then (volume_channel) the node's
 *    volume fraction.
 *  - Node i sits at position i*dx; the domain holds particles whose whole
 *    quadratic stencil lies on the grid, 0.5 <= x*inv_dx < n - 1.5 per axis.
 */
#ifndef MPM_GB300_H
#define MPM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mpm_status {
    MPM_OK = 0,
    MPM_E_ARG = 1,        /* bad descriptor, null pointer, unsupported combination */
    MPM_E_WORKSPACE = 2,  /* workspace too small */
    MPM_E_DOMAIN = 3,     /* (status bit) particles outside the domain were skipped */
    MPM_E_BOUND = 4,      /* (status bit) shares or accumulators would not fit */
    MPM_E_CUDA = 5,       /* a CUDA call failed (launch or copy) */
    MPM_E_TIMEOUT = 6,    /* reserved: a bounded device wait gave up */
    MPM_E_NO_DEVICE = 7   /* no usable CUDA device */
} mpm_status;

typedef enum mpm_acc_mode {
    MPM_ACC_I32 = 0,       /* fixed point, int32 node accumulators */
    MPM_ACC_I64 = 1,       /* fixed point, int64 node accumulators */
    MPM_ACC_F32 = 2,       /* fp32 atomics (order dependent; for comparison) */
    MPM_ACC_EXACT_INT = 3  /* integer particles, integer CIC split (see mpm_p2g) */
} mpm_acc_mode;

/* Dense grid descriptor. */
typedef struct mpm_grid_desc {
    int32_t dim;            /* 2 or 3 */
    int32_t n[3];           /* nodes per axis; n[2] ignored (1) in 2D */
    float dx;               /* node spacing (fp32; the same bits the oracle uses) */
    float inv_dx;           /* 1/dx, supplied by the caller (fp32) */
    int32_t order;          /* 2 = quadratic B-spline; 1 = linear (MPM_ACC_EXACT_INT only) */
    int32_t acc_mode;       /* mpm_acc_mode */
    int32_t scale_log2;     /* fixed-point scale S = 2^scale_log2, 0..40 */
    int32_t tile;           /* cells per tile edge: 4 (3D) or 8 (2D) */
    int32_t boundary_nodes; /* velocity boundary band width in nodes (e.g. 3) */
    int32_t volume_channel; /* 1: the grid-recovered volume channel (see mpm_p2g), else 0 */
} mpm_grid_desc;

/* Particle state (device SoA).  fp32 everywhere, except MPM_ACC_EXACT_INT:
 * x = int32 positions in 1/65,536 of a cell, v = int64, m = int64, C unused.
 * id: optional uint32 particle identities (NULL if unused); only the calls
 * that move particles (mpm_permute, mpm_g2p_sorted, mpm_step_sorted,
 * mpm_step_host) touch it, carrying it along with the particle.
 *
 * Elastic state (optional; F[0] == NULL for none, the APIC transfer alone):
 * F = deformation gradient, dim*dim fp32 planes in the layout of C
 * (F[k*dim + l]); vol = rest volume V0 per particle (fp32); mu, lambda = the
 * Lame constants of the particles' Neo-Hookean material.  With it, mpm_p2g
 * adds the MLS-MPM stress to the affine matrix it scatters and mpm_g2p
 * advances F (implementation guide, section 3.1, Part 2; section 3.3.2,
 * F <- (I + D) F); the calls that move particles carry F and vol along.
 * Not used by MPM_ACC_EXACT_INT.
 *
 * Grid-recovered volume (descriptors with volume_channel = 1): vol as above
 * (the rest volume V0, needed then even without F) and phi = fp32 output of
 * G2P, the particle's grid-recovered volume fraction (see mpm_g2p). */
typedef struct mpm_particles {
    int64_t n;
    void *x[3];
    void *v[3];
    void *C[9];
    const void *m;
    void *id;
    void *F[9];
    void *vol;
    float mu;
    float lambda;
    void *phi;
} mpm_particles;

/* Status words (device, uint32), in mpm_bins.status. */
enum {
    MPM_ST_FLAGS = 0,        /* bit (1 << MPM_E_DOMAIN) | (1 << MPM_E_BOUND) | ... */
    MPM_ST_N_OUTSIDE = 1,    /* particles outside the domain */
    MPM_ST_N_OUT_OF_RANGE = 2, /* particles found above the range the last P2G's bound was checked with
                                  (records given by the caller, or a fused step's new state beyond
                                  22-bit shares): that call's scatter was undone */
    MPM_ST_N_VALID = 3,      /* in-domain particles (length of the sorted part of perm) */
    MPM_ST_N_SLICES = 4,     /* P2G work items */
    MPM_ST_N_ACTIVE = 5,     /* tiles holding at least one particle */
    MPM_ST_MAX_NEIGHBOURS = 6, /* int32 mode: most particles whose stencil covers one node */
    MPM_ST_N_BIG_TILES = 7,  /* buckets whose runs were sorted in global memory (cold, huge buckets) */
    MPM_ST_N_RUNS = 8,       /* runs: maximal index ranges of one bucket (= buckets when already sorted) */
    MPM_ST_N_LARGE_BUCKETS = 9, /* buckets of more than 512 runs (sorted by one block each) */
    MPM_ST_N_DEGENERATE = 10, /* elastic particles the last P2G scattered without stress: det F
                                 not a positive normal fp32 number (inverted or collapsed) */
    MPM_ST_WORK_P2G = 11,    /* internal: work counter of the P2G launch */
    MPM_ST_WORK_G2P = 12,    /* internal: work counter of the G2P launch */
    MPM_ST_MAX_SPEED = 13,   /* fp32 bits of max over the particles the last G2P moved of
                                |v'| + 1.5 dx |C'|_F; the advective step bound is dt <= dx / it */
    MPM_ST_N_ESCAPED = 14,   /* mpm_step_fused: particles whose base cell left their tile in the step,
                                scattered straight into the global grid */
    MPM_ST_RANGE = 15,       /* fp32 bits of R, the range the last fixed-point P2G checked its bound
                                with (see mpm_p2g) */
    MPM_ST_SHARE_PATH = 16,  /* the last fixed-point P2G's shares: 0 below 2^22 (one fp32 fma each),
                                1 int64 (exact integer product); the bits are the same either way */
    MPM_ST_P2G_MASS = 20,    /* record: fp32 bits of max |m| over the particles the last P2G scattered */
    MPM_ST_P2G_VOLUME = 21,  /* record: fp32 bits of max |V0 inv_dx^dim| over the same (volume channel) */
    MPM_ST_G2P_RANGE = 22,   /* record: fp32 bits of max over the particles the last G2P moved of
                                max(1, |v'_k| + 1.5 dx sum_l |C'_kl|) */
    MPM_STATUS_WORDS = 24
};

/* Binning state: device arrays carved out of one caller workspace by
 * mpm_bins_init.  All read-only for the caller. */
typedef struct mpm_bins {
    int64_t n;               /* particle count the workspace was sized for */
    int64_t ntiles;          /* tiles of tile^dim base cells */
    int64_t max_slices;
    uint32_t *key;           /* [n] tile-major base-cell key; 0xFFFFFFFF outside the domain */
    uint32_t *perm;          /* [n] particle indices in (tile, index) order; the
                                in-domain ones first, then the others in index order */
    uint32_t *tile_count;    /* [ntiles] particles per tile */
    uint32_t *tile_start;    /* [ntiles + 1] exclusive prefix of tile_count */
    uint32_t *slices;        /* [2 * max_slices] P2G work items (tile, first) */
    uint32_t *active;        /* [ntiles] tiles with particles, ascending */
    uint32_t *status;        /* [MPM_STATUS_WORDS] */
    void *scratch;           /* internal */
    size_t scratch_bytes;
    int32_t range_from_g2p;  /* set by the caller (mpm_bins_init clears it): see mpm_p2g */
    int32_t next_keys;       /* set by the caller (mpm_bins_init clears it): see mpm_g2p_update */
} mpm_bins;

/* Bytes of workspace mpm_bins_init needs for n particles on this grid. */
size_t mpm_workspace_bytes(const mpm_grid_desc *desc, int64_t n);

/* Carves `ws` (device, 256-byte aligned, at least mpm_workspace_bytes) into
 * `out`.  Host only; launches nothing.  MPM_E_WORKSPACE if too small. */
mpm_status mpm_bins_init(const mpm_grid_desc *desc, int64_t n, void *ws, size_t ws_bytes, mpm_bins *out);

/* Bytes of the accumulator grid ((dim+1) channels of int32/int64/fp32) and of
 * the velocity grid (dim channels of fp32). */
size_t mpm_grid_acc_bytes(const mpm_grid_desc *desc);
size_t mpm_grid_vel_bytes(const mpm_grid_desc *desc);

/* Flags of mpm_bin.  MPM_BIN_KEYS_FROM_G2P: take the keys and the tile
 * histogram the last mpm_g2p_update on these bins wrote with bins->next_keys
 * set, instead of computing them (MPM_ACC_I64 only; see mpm_g2p_update). */
enum { MPM_BIN_DEFAULT = 0, MPM_BIN_KEYS_FROM_G2P = 1 };

/*
 * mpm_bin -- cell keys and a stable counting sort of the particles into tiles.
 * ("Particle Worlds, part 3", Step 3: histogram, exclusive prefix sum, scatter;
 *  implementation guide section 2.1: bin into tiles, sort an index buffer.)
 * key = tile-major id of the particle's stencil base cell b = floor(x*inv_dx - 1/2);
 * the tile is key >> log2(tile^dim).  perm = the in-domain particles in
 * ascending tile order, each tile in particle-index order (the stable counting
 * sort with the tile as bucket), then the out-of-domain particles in index
 * order, so the order is a deterministic function of the keys.  Also builds the active-tile list and
 * the P2G work list, resets the status words (all but the records
 * MPM_ST_P2G_MASS .. MPM_ST_G2P_RANGE), counts out-of-domain particles, and in
 * MPM_ACC_I32 mode counts the most stencils covering one node
 * (MPM_ST_MAX_NEIGHBOURS), which mpm_p2g's bound uses.
 */
mpm_status mpm_bin(const mpm_grid_desc *desc, const mpm_particles *parts, mpm_bins *bins, int flags,
                   void *stream);

/*
 * mpm_p2g -- particle-to-grid scatter into `grid_acc` (must be zero on entry;
 * mpm_grid_update leaves it zero).  Fixed-point modes compute, per particle,
 *   Mt = m*S, Wt(a) = ((wx[a0]*Mt)*wy[a1])*wz[a2],
 *   vel_k(a) = fma(C_k2, d_2, fma(C_k1, d_1, fma(C_k0, d_0, v_k))),  d_l = (a_l - f_l)*dx,
 *   share s_m(a) = rint(Wt(a)), s_k(a) = rint(Wt(a) * vel_k(a)) (exact product,
 *   one rounding, ties to even, at any S), and gives the centre node (1,1,1) the
 *   remainder Q - sum of the others, with Q_m = rint(Mt), Q_k = rint(Mt*v_k),
 * so grid totals equal particle totals exactly ("particle to grid transfer in
 * checked integer arithmetic": split rather than weight; implementation guide
 * 2.1 and 3.3.1: fixed-point atomics, round rather than truncate, the
 * multiplier a runtime precision dial).  The result is bit-identical for
 * every particle order.
 * Bound, before any particle is scattered (the same page's bounds line): with
 * r_k = |v_k| + h*((|C_k0| + |C_k1|) + |C_k2|), h = 1.5*dx, each particle's
 * range is R_p = max(|m| * max(1, r_0, .., r_dim-1), |V0 inv_dx^dim|) (the
 * last term with the volume channel; elastic particles use the stress-folded
 * matrix below; fp32, in this order, NaN propagating), R = max over the
 * binned particles, and B = S*R*(1 + 2^-10) + 28 (fp64) bounds the absolute
 * sum of one particle's shares of any channel.  The scatter proceeds when
 * N_valid * B <= 2^62 (int64 grids) or MPM_ST_MAX_NEIGHBOURS * B <= 2^31 - 1024
 * (int32 grids); otherwise MPM_E_BOUND is set and nothing is scattered.  R is
 * found by a pass over v, C and m before the scatter, or -- when the caller
 * sets bins->range_from_g2p, promising that the particles are those the last
 * mpm_p2g and mpm_g2p on these bins left (v, C, m unchanged since) -- from the
 * records those calls wrote (R = max(P2G_MASS * G2P_RANGE, P2G_VOLUME)), which
 * saves the pass.  With records each particle is verified against R as it is
 * scattered; a particle above it (the promise broken) makes the call undo its
 * scatter (the grid is left zero), set MPM_E_BOUND and count the particle in
 * MPM_ST_N_OUT_OF_RANGE.  Elastic particles always take the pass.
 * Shares below 2^22 in magnitude (wmax*S*R*(1 + 2^-10) <= 2^22 - 4096,
 * wmax = 0.75^dim) are formed with one fp32 fma each and summed in 32-bit
 * shared-memory tile accumulators; larger ones with an exact 24x24-bit integer
 * product and 64-bit sums (MPM_ST_SHARE_PATH says which ran).  R and the path
 * are written to MPM_ST_RANGE and MPM_ST_SHARE_PATH; the call also writes the
 * records MPM_ST_P2G_MASS and MPM_ST_P2G_VOLUME.
 * MPM_ACC_F32 adds the fp32 values Wt*vel with float atomics instead (no bound).
 * Elastic particles (parts->F[0] != NULL) scatter with C replaced by the
 * MLS-MPM affine matrix C' = C - kappa*tau (implementation guide, section
 * 3.1, Part 2: J = det F, P = mu (F - F^-T) + lambda ln(J) F^-T,
 * sigma = P F^T / J; the force -dt V sigma (4/dx^2) w (x_i - x_p) with
 * V = V0 J, divided by m): tau = J sigma = mu (F F^T - I) + lambda ln(J) I,
 * kappa = ((dt*V0)*c4s)/m, c4s = (4*inv_dx)*inv_dx, each step one fp32
 * rounding in the order the oracle states, ln computed by the library's own
 * series (not the CUDA math library) so that it is reproducible.  C' also
 * enters the range.  A particle whose det F is not a positive normal
 * fp32 number keeps C and is counted in MPM_ST_N_DEGENERATE.  `dt` is only
 * read for elastic particles.
 * With volume_channel = 1 a last accumulator channel receives each
 * particle's rest volume in cells, q = V0 * inv_dx^dim (inv_dx^3 taken as
 * (inv_dx*inv_dx)*inv_dx), as the mass is scattered: Vt = q*S, shares
 * rint(((wx*Vt)*wy)*wz), remainder at the centre (implementation guide,
 * section 3.3.2, "grid-recovered volume": 1/ppc per particle, so a rest-packed
 * node sums to about one).  MPM_ACC_F32 adds the fp32 terms ((wx*q)*wy)*wz.
 * MPM_ACC_EXACT_INT (2D or 3D, order 1): integer positions X (1/65,536 cell),
 * int64 m and v; the far node's share of q is q*F/65,536 rounded to nearest
 * (ties to even), the near node gets the rest, split along x then y (then z);
 * the page's bounds line (count * max m * max |v| must fit int64, positions on
 * the grid) runs before any scatter and on failure nothing is scattered
 * (MPM_E_BOUND / MPM_E_DOMAIN in the status).  That mode needs no mpm_bin:
 * `bins` (from mpm_bins_init for this descriptor) only carries the status words.
 */
mpm_status mpm_p2g(const mpm_grid_desc *desc, const mpm_particles *parts, mpm_bins *bins, void *grid_acc,
                   float dt, void *stream);

/*
 * mpm_grid_update -- for each node of the tiles that hold particles (and their
 * neighbours): v = (float)P / (float)M (zero where M == 0), v += dtg, then the
 * velocity-form boundary sign test: within `boundary_nodes` of a wall a
 * component pointing into the wall becomes zero (implementation guide 2.1 and
 * 3.3.2).  dtg = dt*g rounded to fp32 per component, computed by the caller.
 * Reads each accumulator once and writes it back to zero (consume-and-zero,
 * implementation guide section 2.1 and rule 4).  `grid_vel`: dim fp32 planes;
 * with volume_channel one more, the node volume fraction phi = (float)V * 2^-scale_log2
 * (fixed point) or the fp32 sum (MPM_ACC_F32).
 */
mpm_status mpm_grid_update(const mpm_grid_desc *desc, void *grid_acc, float *grid_vel, const float dtg[3],
                           mpm_bins *bins, void *stream);

/*
 * mpm_g2p -- grid-to-particle gather for the in-domain particles:
 * v' = sum_a w v(a);  C'_kl = (sum_a w v_k(a) (a_l - f_l)) * (4*inv_dx)
 * (APIC, "gather d and D (= B*4)" in cell units); x' = fma(dt, v', x).
 * The stencil sums run axis by axis, innermost axis first, each three-term
 * sum as fma(w2,t2, fma(w1,t1, w0*t0)), the same order the oracle uses.
 * With volume_channel, phi_p = sum_a w phi(a) (the same nested order) is
 * written to parts->phi: the grid-recovered volume fraction, about one in a
 * rest packing and above one where the material is compressed (the guide
 * reciprocates it and blends it into a tracked density where it reads
 * compressed; that policy is left to the caller).
 * Elastic particles also get F' = (I + dt C') F, each entry as
 * fma(D_k2, F_2l, fma(D_k1, F_1l, fma(D_k0, F_0l, F_kl))) with D = dt*C'.
 * Particles outside the domain are left unchanged.  In place, the storage
 * order is kept: an interleave written by an earlier mpm_g2p_sorted carries
 * over, and particles that change tiles stay where they are stored, so the
 * next binning finds more index runs (an occasional mpm_g2p_sorted puts the
 * particles back in bin order).
 * MPM_ACC_EXACT_INT: `grid` is the int64 accumulator; each on-grid particle's v is set
 * to its cell's momentum over its cell's mass, rounded to nearest (ties to even).
 */
mpm_status mpm_g2p(const mpm_grid_desc *desc, const void *grid, mpm_particles *parts, mpm_bins *bins,
                   float dt, void *stream);

/*
 * mpm_g2p_sorted -- mpm_g2p that also moves the particles into bin order.
 * The in-domain particles (perm entries below MPM_ST_N_VALID) are written
 * tile by tile in bin order, each P2G work item (a slice of up to 1024
 * consecutive perm entries of one tile) to the same range of out, but with
 * the slice reordered: stably sorted by the bank class of the particle's base
 * cell (with in-tile cell coordinates lx, ly, lz from the key and H = tile + 2,
 * class = (lx + H*ly + H*H*lz) mod 32), then dealt out column by column over
 * rounds of 32 (lane l
 * of R = ceil(cnt/32) rounds holds sorted entries cum(l) .. cum(l+1) - 1 with
 * cum(l) = l*R - max(0, l - L), L = cnt - 32*(R - 1), and entry cum(l) + rho
 * goes to slice place rho*32 + l).  Particles 32 apart in a round then sit in
 * cells that use different shared-memory banks, which the next step's P2G
 * and G2P exploit.  A slice of at most 32 particles (one round) keeps bin
 * order.  The remaining particles (outside the domain) are copied
 * unchanged to out[j] = in[perm[j]].  m, id, vol and phi are carried along.  This is
 * the ping-pong buffer of "Particle Worlds, part 3", Step 4 ("the sort writes
 * into a second buffer"): the next step's binning then starts from almost
 * sorted particles, so its runs are long and every particle pass reads and
 * writes contiguous memory.  The bits of every particle's new state are those
 * of mpm_g2p.  `in` and `out` must not overlap, and both or neither carry an
 * elastic state.
 */
mpm_status mpm_g2p_sorted(const mpm_grid_desc *desc, const float *grid_vel, const mpm_particles *in,
                          mpm_particles *out, mpm_bins *bins, float dt, void *stream);

/*
 * mpm_g2p_binned -- mpm_g2p_sorted without the bank-class interleave: the
 * in-domain particles are written in bin order, out[j] = the new state of
 * in[perm[j]] for j below MPM_ST_N_VALID, the others copied as by
 * mpm_g2p_sorted; the same bits per particle.  One warp per work item and no
 * block barrier, so it is faster than mpm_g2p_sorted; the order inside a tile
 * is the input's, so an interleave written by an earlier mpm_g2p_sorted
 * carries over and wears down slowly as particles change cells (the next
 * P2G's shared-memory bank conflicts grow with it; an occasional
 * mpm_g2p_sorted restores it).  `in` and `out` must not overlap.
 */
mpm_status mpm_g2p_binned(const mpm_grid_desc *desc, const float *grid_vel, const mpm_particles *in,
                          mpm_particles *out, mpm_bins *bins, float dt, void *stream);

/*
 * mpm_g2p_update -- mpm_grid_update and mpm_g2p in one pass over the
 * particles, without a velocity grid (implementation guide, section 2.1, the
 * worked shape: each tile's nodes are loaded applying the grid update; "the
 * grid clear can ride along").  `grid_acc` holds mpm_p2g's accumulators at the
 * positions binned in `bins` (int32 or int64 modes).  Each G2P work item
 * loads its tile's halo of accumulators and computes every node's velocity as
 * mpm_grid_update would (v = (float)P / (float)M + dtg, zero where M == 0, the
 * boundary sign test; the volume fraction with volume_channel), then gathers
 * exactly as mpm_g2p.  The accumulators are consumed: a node block is read
 * only by the work items of the 2^dim tiles below it, which count themselves
 * in a per-block counter of the workspace once their halo is in shared
 * memory; the one that completes the count clears the block.  So the grid is
 * zero afterwards, as mpm_grid_update leaves it.  The bits of every particle
 * are those of mpm_grid_update followed by mpm_g2p.  The status words of
 * mpm_g2p (MPM_ST_MAX_SPEED, MPM_ST_G2P_RANGE) are written as it writes them.
 *
 * With bins->next_keys set (MPM_ACC_I64), the call also writes each moved
 * particle's key of its new position into bins->key and the tile histogram of
 * all the particles' next keys into the workspace (the particles outside the
 * domain keep their key and their count), which the next mpm_bin takes with
 * MPM_BIN_KEYS_FROM_G2P instead of computing them: the same keys and counts,
 * the key pass skipped.  The caller promises that the positions are those the
 * call wrote when it passes the flag; a particle whose position has left its
 * key's tile since is found by mpm_p2g's box test and counted as one above the
 * range (MPM_E_BOUND).  bins->key then holds the next keys, not those of the
 * binning the call gathered with.
 */
mpm_status mpm_g2p_update(const mpm_grid_desc *desc, void *grid_acc, const float dtg[3], mpm_particles *parts,
                          mpm_bins *bins, float dt, void *stream);

/*
 * mpm_g2p_sorted_update -- mpm_grid_update followed by mpm_g2p_sorted, in one
 * pass as mpm_g2p_update: the new state goes from `in` to `out` in bin order
 * with the bank-class interleave (see mpm_g2p_sorted), the accumulators are
 * consumed.  `in` and `out` must not overlap.
 */
mpm_status mpm_g2p_sorted_update(const mpm_grid_desc *desc, void *grid_acc, const float dtg[3],
                                 const mpm_particles *in, mpm_particles *out, mpm_bins *bins, float dt, void *stream);

/*
 * mpm_step -- mpm_bin, mpm_p2g, mpm_grid_update and mpm_g2p in sequence on one
 * stream (device pointers throughout; particles keep their index).
 */
mpm_status mpm_step(const mpm_grid_desc *desc, mpm_particles *parts, mpm_bins *bins, void *grid_acc,
                    float *grid_vel, float dt, const float dtg[3], void *stream);

/*
 * mpm_step_sorted -- mpm_bin, mpm_p2g and mpm_grid_update on `in`, then
 * mpm_g2p_sorted from `in` into `out` (the caller swaps the two between steps).
 */
mpm_status mpm_step_sorted(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                           void *grid_acc, float *grid_vel, float dt, const float dtg[3], void *stream);

/*
 * mpm_step_binned -- mpm_bin, mpm_p2g and mpm_grid_update on `in`, then
 * mpm_g2p_binned from `in` into `out` (the caller swaps the two).
 */
mpm_status mpm_step_binned(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                           void *grid_acc, float *grid_vel, float dt, const float dtg[3], void *stream);

/*
 * mpm_step_host -- one step from and back to HOST particle arrays: copies the
 * host SoA (`host`: x, v, C, m, and id, F, vol and phi if given) into the
 * device arrays `dev_in`, runs mpm_step_sorted into `dev_out`, and copies the
 * same arrays of `dev_out` back into `host`, so the host arrays hold the new
 * state in the order mpm_g2p_sorted writes.  Asynchronous on `stream`; the
 * host arrays must stay valid until it completes.  When every host array is
 * pinned (page-locked, so the device can address it) the copies are made by a
 * kernel that issues the loads and stores from every SM, which moves data
 * over the CPU-GPU link faster than the copy engines do; otherwise by one
 * cudaMemcpyAsync per array.  Either way everything is ordered on `stream`.
 */
mpm_status mpm_step_host(const mpm_grid_desc *desc, mpm_particles *host, mpm_particles *dev_in,
                         mpm_particles *dev_out, mpm_bins *bins, void *grid_acc, float *grid_vel, float dt,
                         const float dtg[3], void *stream);

/*
 * mpm_step_fused -- one step as the fused gather-scatter kernel of the
 * implementation guide, section 2.1 (one kernel per step: load the tile's
 * nodes applying the grid update, gather each particle, scatter it back into
 * shared-memory accumulators, flush them once).  `acc_read` must hold the
 * accumulators of mpm_p2g at the positions of `in` (the first step: mpm_bin
 * and mpm_p2g on `in`; later steps: the previous call's `acc_write`);
 * `acc_write` must be zero.  The call bins `in`, gathers as mpm_grid_update +
 * mpm_g2p would (the same bits) and writes the new state to `out` in bin
 * order, out[j] = new state of in[perm[j]]: the order inside a tile is the
 * input's, so the bank-class interleave mpm_step_sorted writes carries over
 * (particles drifting between cells wear it down slowly; an occasional
 * sorted step restores it).  It scatters the new state into `acc_write` as
 * mpm_p2g on `out` would (the same integers), and clears `acc_read` (a second
 * kernel, after the reads); the caller then swaps in/out and the two grids.  One
 * warp per work item: a particle's new state is scattered into the warp's
 * tile accumulator while its base cell stays in the tile; a particle whose
 * base cell left the tile is scattered straight into the global grid and
 * counted in MPM_ST_N_ESCAPED; those leaving the domain are not scattered.
 * The new state is formed in the same kernel that scatters it, so no bound can
 * run before this scatter: the kernel forms 22-bit shares only and tests each
 * particle as mpm_p2g's fast path requires (wmax*|m S|*max(1, r_k) within
 * 2^22 - 4096, with int64 grids no node can then overflow); a particle beyond
 * it is counted in MPM_ST_N_OUT_OF_RANGE, MPM_E_BOUND is set and the step's
 * scatter is undone (acc_write left zero; `out` still holds the new state).
 * Where that happens the separate calls take mpm_p2g's int64 shares instead.
 * MPM_ACC_I64 only, without the
 * elastic state or the volume channel (MPM_E_ARG otherwise): the int32 mode's
 * bound is checked by the binning of the positions it will scatter, which
 * this scatter runs ahead of.  No velocity grid is written.
 */
mpm_status mpm_step_fused(const mpm_grid_desc *desc, mpm_particles *in, mpm_particles *out, mpm_bins *bins,
                          void *acc_read, void *acc_write, float dt, const float dtg[3], void *stream);

/*
 * mpm_iterate -- the transfer loop at fixed positions of the implementation
 * guide's position-based solver (section 3.3.2: P2G -> grid update -> G2P,
 * iterationCount times per substep, the particles in place; v and C carry the
 * displacement d and its gradient D, with the same transfer arithmetic), one
 * fused kernel per iteration (section 2.1): the grid update is applied while
 * the tile's accumulators are loaded, without gravity (the loop adds none),
 * each particle's new v and C are gathered and written in place, and -- but
 * for the last iteration -- scattered at the same position into the other
 * grid.  `bins` must hold mpm_bin of the current positions and `acc_a` the
 * mpm_p2g of the current state; `acc_b` must be zero.  Both grids are zero
 * afterwards; x, m and every particle outside the domain are unchanged.  The
 * bits equal `iterations` rounds of mpm_grid_update (dtg = 0) + mpm_g2p
 * (dt = 0) + mpm_p2g.  The material projections the guide runs between the
 * transfers are not part of this call.  Like mpm_step_fused it forms 22-bit
 * shares only; a round whose state does not fit them counts the particles in
 * MPM_ST_N_OUT_OF_RANGE and sets MPM_E_BOUND, and the state the call leaves is
 * then not valid.  MPM_ACC_I64 only, without the elastic
 * state or the volume channel.  iterations >= 1.
 */
mpm_status mpm_iterate(const mpm_grid_desc *desc, mpm_particles *parts, mpm_bins *bins, void *acc_a, void *acc_b,
                       int iterations, void *stream);

/* Reorders a particle SoA by bins->perm: out[j] = in[perm[j]] for every
 * component (and id if both are non-NULL), all n entries.  `in` and `out`
 * must not overlap. */
mpm_status mpm_permute(const mpm_grid_desc *desc, const mpm_particles *in, mpm_particles *out,
                       const mpm_bins *bins, void *stream);

/*
 * mpm_bin_static -- mpm_bin for callers that cannot give the library a
 * workspace.  The method's pages have no counterpart of this call; it is a
 * convenience of this library.
 *
 * Some callers cannot allocate device memory at the point where they bin:
 * code embedded in a host application that owns every device allocation
 * under its own budget, or a loop that must not call cudaMalloc because it
 * may synchronise the device and stall work already in flight.  This call
 * bins into a workspace the library holds itself: a file-scope device array
 * of MPM_STATIC_WORKSPACE_BYTES (16 MiB) per device, created when the
 * library's device code is loaded.  It calls no allocator (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 * Arguments and results are those of mpm_bin with bins = `out`: the call
 * fills `out` (host struct) as mpm_bins_init would, with every device array
 * pointing into the static workspace, then runs mpm_bin.  `out` may then be
 * passed to mpm_p2g, mpm_grid_update, mpm_g2p, mpm_g2p_sorted, mpm_permute
 * and mpm_read_status like any other bins.
 *  - Size limit: mpm_workspace_bytes(desc, parts->n) must be at most
 *    MPM_STATIC_WORKSPACE_BYTES; a larger problem returns MPM_E_WORKSPACE at
 *    once and launches nothing.  Use mpm_bins_init with your own memory then.
 *  - Zero state: nothing in the static workspace has to be zero beforehand
 *    (every call clears the counters it uses).  The accumulator grid given to
 *    a later mpm_p2g must still be zero, as always.
 *  - Setup: every call looks up the array's device address with the
 *    current device (so no address outlives a device reset); the first call
 *    on each device may load the library's device code, so make it before
 *    any stream capture begins.
 *  - Sharing: there is ONE static workspace per device and process.  A call
 *    overwrites what the previous call left there, so calls (and the P2G,
 *    grid update and G2P calls that read their `out`) must not overlap in
 *    time: two calls in flight at once on different streams or host threads
 *    race on the same memory.  Order them on one stream.
 */
#define MPM_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)
mpm_status mpm_bin_static(const mpm_grid_desc *desc, const mpm_particles *parts, int flags, mpm_bins *out,
                          void *stream);

/* Asynchronous copy of the MPM_STATUS_WORDS status words to host memory. */
mpm_status mpm_read_status(const mpm_bins *bins, uint32_t *host_out, void *stream);

/* Static text for a status code. */
const char *mpm_strerror(mpm_status s);

/* Library version, (major << 16) | minor. */
int32_t mpm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MPM_GB300_H */
