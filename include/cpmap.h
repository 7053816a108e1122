/*
 * cpmap.h -- C ABI of the GB300 (sm_103a) electrostatic potential-map library
 * (libcpmap.so).
 *
 * What it computes
 *   The electrostatic potential on a regular 3-D grid,
 *       V(g) = sum_a q_a / |r_a - g|,
 *   as defined in the PMPP ch.18 study notes ("Case study -- electrostatic
 *   potential map", section 18.1; the pwwt.cn chapter-18 article, section 一,
 *   gives the same sum).  Two routes:
 *     cp_direct  direct Coulomb summation as a gather: a thread owns grid
 *                points and atom tiles stream past it, no atomics (notes,
 *                sections 18.2-18.4).
 *     cp_cutoff  cutoff summation of the switched term
 *                    q * (1/r - g(r)),  r < c,
 *                    g(r) = GC0 + GC1 r^2 + GC2 r^4
 *                         = (1/c)(15/8 - 5/4 (r/c)^2 + 3/8 (r/c)^4)
 *                over atoms binned into a uniform cell grid, visiting the
 *                bins of a precomputed neighbourhood offset list (Input
 *                Binning lecture, slides "Large Bin Cut-off Kernel Code" (24),
 *                "Neighborhood Offset List (Pre-calculated)" (27), "Pseudo
 *                Code of an Implementation" (28), "Details on Small Bin
 *                Design" (30)).
 *   There is no Coulomb constant: V is in units of charge / length.
 *
 * Conventions shared by every entry point
 *   atoms      float32 [n_atoms][4] = (x, y, z, q), the 16-byte atom record
 *              of the notes' section 18.2.  DEVICE pointer, 16-byte aligned.
 *   grid       nx * ny * nz points; point (i, j, k) sits at
 *              origin + (i*h, j*h, k*h).  1 <= nx, ny, nz <= 2^24 and
 *              nx*ny*nz < 2^31.
 *   V          float32 [nz][ny][nx], x fastest: V[(k*ny + j)*nx + i] (notes,
 *              section 18.4).  DEVICE pointer, 4-byte aligned (16-byte
 *              alignment and nx % 4 == 0 enable vector stores).  V is
 *              OVERWRITTEN, never accumulated into (the one exception is
 *              cp_msm_longrange with accumulate = 1).
 *   stream     a cudaStream_t passed as void* (NULL = the legacy default
 *              stream).  Compute calls are asynchronous on that stream; the
 *              caller keeps every buffer alive until the stream has passed
 *              the call.
 *   ownership  the caller allocates and frees every buffer (atoms, V and the
 *              cutoff workspace).  The library allocates no device memory.
 *   errors     every int-returning call returns CP_OK (0) or a negative
 *              cp_status.  Arguments are checked on the host before any
 *              launch; a rejected call launches nothing and touches no
 *              buffer.  Problems found on the device (a bounded wait that ran
 *              out, more atoms than a range allows) are never traps: kernels
 *              record them in a device status word that cp_device_status()
 *              reads.
 *   singular   an atom exactly on a grid point (r = 0) has no defined
 *              potential there; the value at that point is then inf/nan.
 */
#ifndef CPMAP_H
#define CPMAP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CP_API __attribute__((visibility("default")))
#else
#define CP_API
#endif

/* Return codes. */
typedef enum {
    CP_OK = 0,
    CP_ERR_INVALID_ARGUMENT = -1,  /* null pointer, non-positive size, non-finite value */
    CP_ERR_MISALIGNED = -2,        /* atoms or workspace not aligned as required */
    CP_ERR_TOO_LARGE = -3,         /* grid, bin grid or offset list beyond the library's limits */
    CP_ERR_WORKSPACE_TOO_SMALL = -4,
    CP_ERR_UNSUPPORTED = -5,       /* e.g. a bin capacity other than 0, 8 or 16 */
    CP_ERR_CUDA = -6,              /* a CUDA runtime call or launch failed */
    CP_ERR_DEVICE = -7             /* a kernel reported a problem (see cp_device_status) */
} cp_status;

/* Device status bits (cp_device_status). */
#define CP_DEVICE_WAIT_TIMEOUT 0x1u /* a bounded wait on a shared-memory barrier gave up */
#define CP_DEVICE_RANGE 0x2u        /* an index fell outside a buffer; the access was skipped */
#define CP_DEVICE_ATOMS_OUTSIDE 0x4u /* cp_msm_longrange: an atom lay outside the domain box and was left out */

/* A point or vector in Angstrom. */
typedef struct {
    float x, y, z;
} cp_vec3;

/* ------------------------------------------------------------------------ */
/* Direct Coulomb summation (notes, sections 18.1-18.4).
 *
 * V(g) = sum over all n_atoms atoms of q / r for every grid point, computed
 * in fp32 (rsqrt on the SFU for most pairs, on the FMA pipe for a fixed
 * share), atom tiles accumulated block-wise.  Point-atom differences are
 * rounded once wherever the grid sits (see cp_grid_points_exact).
 * n_atoms may be 0 (V is then all zero).  Atoms are used as given and
 * must be finite and within 1e18 A of the grid, so that r^2 fits fp32
 * (farther atoms contribute about q/r, i.e. nothing measurable, up to that
 * limit; beyond it the FMA-pipe route overflows to inf).  The cutoff map
 * drops non-finite and out-of-range atoms instead.  Needs no workspace.
 * Returns CP_OK, CP_ERR_INVALID_ARGUMENT, CP_ERR_MISALIGNED (atoms not
 * 16-byte aligned), CP_ERR_TOO_LARGE or CP_ERR_CUDA.                        */
CP_API int cp_direct(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float *V,
                     void *stream);

/* cp_direct with the per-thread point patch and the cluster split forced,
 * for tests and tuning sweeps.  variant: -1 = planner's choice, else a
 * patch of PX x-points times PY rows times PZ planes, of whose (PX/2)*PY*PZ
 * point pairs the first EMU take their rsqrt on the FMA pipe instead of the
 * SFU, shared by LS neighbouring lanes that take every LS-th atom each
 * ((PX, PY, PZ, EMU, LS)): 0 = (4,4,2,0,1), 1 = (4,2,2,0,1),
 * 2 = (4,4,1,0,1), 3 = (4,2,1,0,1), 4 = (4,1,1,0,1), 5 = (4,4,2,4,1),
 * 6 = (4,4,2,5,1), 7 = (4,2,2,2,1), 8 = (4,4,1,2,1), 9 = (4,2,1,1,1),
 * 10 = (2,1,1,0,1), 11 = (2,2,1,0,1), 12 = (4,1,1,0,4), 13 = (4,1,1,0,2),
 * 14 = (4,2,1,1,4), 15 = (4,2,1,1,2), 16 = (4,2,1,1,8), 17 = (4,2,2,2,4),
 * 18 = (4,4,1,2,4) (the 2-point and shared-patch shapes
 * serve grids too small for 4-point patches to fill the GPU).
 * split: 0 = planner's choice, else 1..16 CTAs of a
 * cluster share one tile of points and take 1/split of the atoms each
 * (their partial sums meet in distributed shared memory; sizes above 8 use
 * non-portable clusters).  Results agree with cp_direct up to fp32
 * rounding order.  Same errors as cp_direct, plus CP_ERR_INVALID_ARGUMENT
 * for an unknown variant or split and CP_ERR_UNSUPPORTED for a cluster size
 * the device cannot run.                                                    */
CP_API int cp_direct_config(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                            float *V, int variant, int split, void *stream);

/* The patch shape (variant index as for cp_direct_config) and cluster split
 * that cp_direct would use for this grid and atom count on the current
 * device (assuming 16-byte aligned output and grid points exact in fp32,
 * e.g. origin 0 and h 1).  Queries occupancy, launches nothing.  Returns CP_OK, CP_ERR_INVALID_ARGUMENT, CP_ERR_TOO_LARGE or
 * CP_ERR_CUDA.                                                              */
CP_API int cp_direct_plan(int n_atoms, int nx, int ny, int nz, int *variant, int *split);

/* Whether every grid coordinate origin_d + i*h (0 <= i < n_d, each axis) is
 * exactly representable in fp32: 1 if so, 0 if not (or not provably), or a
 * negative cp_status for an invalid grid.  Host only.  The direct and
 * cutoff kernels use it to choose how they form a point-atom difference:
 * for exact points as point - atom, rounded once; otherwise as
 * i*h + (origin - atom) with one fused multiply-add, so that the rounding
 * follows the atom's offset from the grid origin rather than the grid's
 * distance from the coordinate origin.  The test is sufficient: all o + i*h
 * are multiples of 2^q, q the lowest set bit of o or h, and are exact when
 * both ends of the axis are below 2^(24 + q) in magnitude.                  */
CP_API int cp_grid_points_exact(int nx, int ny, int nz, cp_vec3 origin, float h);

/* ------------------------------------------------------------------------ */
/* Cutoff summation (Input Binning lecture, slides 24-37).
 *
 * Bin geometry (m bins of margin so that every atom within c of the grid is
 * binned; the bin-grid origin is rounded to fp32 once):
 *     m    = ceil(c / b)
 *     bo_d = float(origin_d - m*b)                      (double, rounded once)
 *     nb_d = ceil(((N_d - 1)*h + 2*m*b) / b) + 1
 * An atom goes to bin (ux, uy, uz), u_d = floor(float(float(a_d - bo_d) / b))
 * (two IEEE fp32 roundings, no fused operations), linear index
 * (uz*nb_y + uy)*nb_x + ux, when every u_d is in [0, nb_d); other atoms
 * (and atoms with non-finite coordinates) are dropped and counted.
 *
 * Within a bin atoms keep ascending input order.  The first `capacity` atoms
 * of each bin fill its fixed-capacity slots (slide "Coalesced Global Memory
 * Access to Atom Data" (33)); unused slots hold the pad record
 * (1e18, 1e18, 1e18, 0).  Atoms past the capacity are the bin's overflow
 * ("extra atoms", slide "Handling Overfull Bins" (34)); they stay in the
 * bin-sorted array and are swept on the GPU, not on the CPU.
 *
 * A pair contributes iff r^2 < c^2 (strict).  capacity is 8 (the
 * lecture's 128-byte bins), 16 (256-byte bins) or 0.  With 0 there are no
 * fixed-capacity slots: the map streams each run of consecutive bins as one
 * contiguous range of the bin-sorted array (the fixed 128-byte bins were the
 * lecture's answer to a 64-byte coalescing rule; a TMA bulk copy moves any
 * 16-byte-aligned range), and every binned atom counts as "overflow" in the
 * stats.                                                                    */

/* Where each array lives inside a cutoff workspace (byte offsets from its
 * base, each a multiple of 256), for inspection and tests. */
typedef struct {
    int nb[3];                 /* bins per axis */
    float bo[3];               /* bin-grid origin */
    int margin_bins;           /* m */
    int capacity;              /* K */
    long long nbins;           /* nb[0]*nb[1]*nb[2] */
    size_t off_count;          /* int32 [nbins]        atoms per bin */
    size_t off_start;          /* int32 [nbins + 1]    exclusive prefix sum of count */
    size_t off_csr_index;      /* int32 [n_atoms]      input index, sorted by (bin, index) */
    size_t off_csr_atoms;      /* float32 [n_atoms][4] atoms in that order */
    size_t off_padded;         /* float32 [nbins][K][4] fixed-capacity slots */
    size_t off_stats;          /* int32 [8]            see cp_cutoff_stats */
    size_t off_scratch;        /* internal */
    size_t total_bytes;        /* workspace size needed */
} cp_cutoff_layout;

/* Host-only: fills *out for these arguments.  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT, CP_ERR_UNSUPPORTED or CP_ERR_TOO_LARGE. */
CP_API int cp_cutoff_layout_of(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                               float bin_size, int capacity, cp_cutoff_layout *out);

/* Host-only: workspace bytes cp_cutoff / cp_bin_atoms need (0 if the
 * arguments are invalid). */
CP_API size_t cp_cutoff_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                                        float bin_size, int capacity);

/* The whole cutoff map: bin the atoms on the device (count, scan, scatter,
 * per-bin sort and pack), then one CTA per 8x8x8-point brick sweeps the
 * neighbourhood offset list's bins and the overflow of those bins, and
 * writes V.  `workspace` is a DEVICE buffer of at least
 * cp_cutoff_workspace_bytes(...) bytes, 256-byte aligned, owned by the
 * caller; its contents on entry do not matter and on return it holds the
 * bins (see cp_cutoff_layout).  Calls sharing a workspace must not overlap
 * on the GPU.  Returns CP_OK, CP_ERR_INVALID_ARGUMENT, CP_ERR_MISALIGNED,
 * CP_ERR_UNSUPPORTED, CP_ERR_TOO_LARGE, CP_ERR_WORKSPACE_TOO_SMALL or
 * CP_ERR_CUDA.                                                              */
CP_API int cp_cutoff(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                     float bin_size, int capacity, void *workspace, size_t workspace_bytes, float *V, void *stream);

/* Only the binning stage of cp_cutoff (same arguments, no V): leaves count,
 * start, csr_index, csr_atoms, padded and the stats in the workspace. */
CP_API int cp_bin_atoms(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                        float cutoff, float bin_size, int capacity, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Only the map stage of cp_cutoff: the brick kernel and overflow sweep over
 * bins that a preceding cp_bin_atoms call with the same arguments left in
 * `workspace` (same stream, or otherwise ordered after it).  Lets a caller
 * bin once and time the two stages apart.  Same arguments and errors as
 * cp_cutoff.                                                                */
CP_API int cp_cutoff_map(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                         float cutoff, float bin_size, int capacity, void *workspace, size_t workspace_bytes, float *V,
                         void *stream);

/* Work accounting of the cutoff map (no V is written): bins the atoms like
 * cp_cutoff, then runs the brick traversal in a counting variant that adds
 * into counts[0..2] (a DEVICE array of 3 uint64, zeroed by the call):
 *   counts[0]  useful pairs: (grid point, atom) with r^2 < c^2
 *   counts[1]  pairs evaluated: atoms that passed a warp's sub-box test
 *              times the warp's 128 points
 *   counts[2]  pairs examined at bin level: real atoms in the loaded bins
 *              times the points of the warps that loaded them
 * counts[0] / counts[2] is the "share of examined atoms within the cutoff"
 * of slide "Details on Small Bin Design" (30).  Same arguments and errors
 * as cp_cutoff, with `counts` in place of V.                                */
CP_API int cp_cutoff_pair_counts(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                 float cutoff, float bin_size, int capacity, void *workspace, size_t workspace_bytes,
                                 unsigned long long *counts, void *stream);

/* The cutoff map with no workspace argument and no allocation, for callers
 * that cannot allocate device memory themselves: a program whose device
 * memory is wholly owned by another allocator, or code that may not
 * allocate once it is running (a fixed budget set at start-up, a plugin
 * limited to what its host hands it).  The pages have no counterpart; this
 * is an addition for such callers.
 *
 * The scratch that cp_cutoff takes as `workspace` is here a fixed 16 MiB
 * array inside the library, created on every device that loads the library
 * and held until the process exits.  Maps whose workspace
 * (cp_cutoff_workspace_bytes) exceeds 16 MiB are rejected with
 * CP_ERR_TOO_LARGE before anything runs; 100,000 atoms on a 200^3 grid at
 * c = 12, b = 4, capacity 16 need about 12 MiB.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *
 * All calls on a device share the one array and find the previous call's
 * bins in it; the binning stage clears what must start at zero, so no
 * result depends on an earlier call.  Calls that overlap on the GPU (on
 * different streams, or from different threads without ordering) race on
 * the array: order them, e.g. by issuing them on one stream.
 *
 * Arguments, results and the other errors are those of cp_cutoff, without
 * workspace and workspace_bytes; CP_ERR_CUDA also when the array's device
 * address cannot be looked up, for instance because the first call on a
 * device was made while its stream was being captured.                     */
CP_API int cp_cutoff_no_alloc(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                              float cutoff, float bin_size, int capacity, float *V, void *stream);

/* Counters a binning pass leaves in the workspace. */
typedef struct {
    int n_binned;          /* atoms placed in a bin */
    int n_dropped;         /* atoms outside the bin grid (or non-finite) */
    int n_overflow;        /* atoms past their bin's capacity */
    int max_bin_count;     /* most atoms in one bin */
} cp_cutoff_stats_t;

/* Synchronises `stream`, then copies the counters of the last binning pass
 * on this workspace to *out.  Returns CP_OK, CP_ERR_INVALID_ARGUMENT or
 * CP_ERR_CUDA. */
CP_API int cp_cutoff_stats(const void *workspace, size_t workspace_bytes, int n_atoms, int nx, int ny, int nz,
                           cp_vec3 origin, float h, float cutoff, float bin_size, int capacity,
                           cp_cutoff_stats_t *out, void *stream);

/* Host-only: the brick neighbourhood offset list (slide "Neighborhood
 * Offset List (Pre-calculated)" (27)) as x-runs.  Run r covers the bins
 * (home_x + dx_lo .. home_x + dx_hi, home_y + dy, home_z + dz) of a brick
 * whose home bin is `home`; a bin is listed iff its box can come within
 * c (+ a rounding margin) of some point of some brick (per-axis minimum gap
 * over all bricks, so one list serves every brick); there is one run per
 * (dy, dz).  runs_out receives
 * 4 ints per run (dy, dz, dx_lo, dx_hi); pass NULL to query the sizes.
 * *n_runs and *n_bins receive the list's size.  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT, CP_ERR_TOO_LARGE (list longer than the library
 * supports) or CP_ERR_WORKSPACE_TOO_SMALL (max_runs too small).            */
CP_API int cp_offset_list(int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff, float bin_size,
                          int *runs_out, int max_runs, int *n_runs, int *n_bins);

/* Host-only: the home bin of brick (bx, by, bz) (8x8x8 points each). */
CP_API int cp_brick_home(int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff, float bin_size, int bx,
                         int by, int bz, int home_out[3]);

/* ------------------------------------------------------------------------ */
/* Comparison kernels: the strategies the pages describe, rebuilt as plain
 * CUDA so the optimised path can be timed against them (the pwwt.cn
 * chapter-18 article's five-way benchmark; PMPP ch.18 notes sections
 * 18.2-18.5).  Not the fast path.
 *
 * cp_direct_variant computes the same map as cp_direct with
 *   variant 0  scatter: one thread per atom, atomicAdd into every grid point
 *              (notes 18.2; article 二).  V is zeroed first; the summation
 *              order depends on timing, so results vary in the last bits.
 *   variant 1  gather: one thread per point, atoms through __constant__
 *              memory in chunks of 4000, one launch per chunk (notes 18.2).
 *   variant 2  coarsened gather: 4 adjacent x points per thread (notes 18.3).
 *   variant 3  coarsened + coalesced: 4 points a block-width apart (article 三).
 * Variants 1-3 share one __constant__ chunk table per device: calls that
 * overlap on the GPU race.  nz <= 65535.  Same errors as cp_direct, plus
 * CP_ERR_INVALID_ARGUMENT for an unknown variant.                           */
CP_API int cp_direct_variant(int variant, const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin,
                             float h, float *V, void *stream);

/* The 27-bin hard-cutoff map of notes 18.5: bins of edge c; each point scans
 * its own bin and the 26 around it and adds q/r for r^2 < c^2 (no
 * switching).  Binning is cp_bin_atoms with bin size c and capacity 0 in a
 * caller-owned workspace of cp_cutoff27_workspace_bytes bytes.  nz <= 65535.
 * Same errors as cp_cutoff.                                                 */
CP_API size_t cp_cutoff27_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                          float cutoff);
CP_API int cp_cutoff27(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                       float cutoff, void *workspace, size_t workspace_bytes, float *V, void *stream);

/* ------------------------------------------------------------------------ */
/* Long-range part of a multilevel summation.
 *
 * The Input Binning lecture's slide "Large Bin Cut-off Kernel Code" (24)
 * names its cutoff kernel mgpot_shortrng_energy: the switched sum of
 * cp_cutoff is the SHORT-RANGE part of a multilevel summation of 1/r.  What
 * it leaves out is smooth,
 *     V_long(x) = sum_a q_a g_c(|x - r_a|),
 *     g_c(r) = (1/c)(15/8 - 5/4 (r/c)^2 + 3/8 (r/c)^4)  for r < c,
 *     g_c(r) = 1/r                                      for r >= c,
 * so that cp_cutoff + V_long = the direct sum exactly.  The pages do not
 * describe the long-range part; these calls approximate it the multilevel
 * way (R. D. Skeel, I. Tezcan, D. J. Hardy, J. Comput. Chem. 23 (2002);
 * D. J. Hardy, J. E. Stone, K. Schulten, Parallel Computing 35 (2009)):
 *   lattices       level l has spacing 2^l * lattice_h; node i of every
 *                  level sits at o + i * spacing, o = the domain's low corner;
 *   anterpolation  charges to level-0 nodes with the C1 cubic basis
 *                  phi(t) = (1-|t|)(1+|t|-3/2 t^2) (|t| <= 1),
 *                  -1/2 (|t|-1)(2-|t|)^2 (1 <= |t| <= 2), 0 beyond, in each
 *                  axis;
 *   restriction    level l to l+1 with weights phi(i/2 - J);
 *   lattice cutoff on level l < L, e_i = 2^-l sum_d W(d) q_{i+d} with
 *                  W(d) = g_c(|d| h0) - g_2c(|d| h0), zero for |d| h0 >= 2c;
 *                  on the top level L, all pairs with 2^-L g_c(|d| h0);
 *   prolongation   e_l += the level-(l+1) potentials interpolated with
 *                  phi(i/2 - J), from the top down;
 *   interpolation  V_long at the grid points from level 0 with phi.
 * Its error against the exact V_long falls like lattice_h^3 (about 1e-4 of
 * sum_a |q_a| g_c(r) at c / lattice_h = 6).
 *
 * Geometry, computed on the host in fp64 from the fp32 arguments: the
 * domain [domain_lo, domain_hi] (which must contain every atom) is widened
 * to contain the grid; o = its low corner; level 0 has
 * nc = floor((hi - o)/lattice_h) + 2 cells per axis (one more than the box
 * needs, so that fp32 rounding never pushes an atom out) and nodes
 * -1 .. nc + 1;
 * level l+1 spans floor(lo_l/2) - 1 .. ceil(hi_l/2) + 1; the top level L
 * is the first whose every axis has at most 12 nodes.  The stencil radius
 * R = ceil(2c / lattice_h) must be at most CP_MSM_MAX_RADIUS.
 *
 * Work per call, all on the device: a counting sort of the atoms into the
 * level-0 cells (as cp_bin_atoms), the stencil W in fp64 rounded to fp32,
 * anterpolation (each node gathers the atoms of the 4x4x4 cells around it,
 * in a fixed order), restriction, the lattice cutoffs of all levels in one
 * launch (tap rows split over `split[l]` CTAs, partial sums added in a fixed
 * order), the top level, prolongation and interpolation.  Results are
 * deterministic.                                                           */
#define CP_MSM_MAX_LEVELS 16
#define CP_MSM_MAX_RADIUS 24

typedef struct {
    int levels;                        /* L + 1; level L is the dense top level */
    int lo[CP_MSM_MAX_LEVELS][3];      /* lowest node index per axis (x, y, z) */
    int n[CP_MSM_MAX_LEVELS][3];       /* nodes per axis */
    int split[CP_MSM_MAX_LEVELS];      /* CTAs sharing one tile's stencil rows (levels < L) */
    int radius;                        /* R */
    int taps;                          /* stencil points with |d| lattice_h < 2c */
    int cells[3];                      /* level-0 cells per axis */
    cp_vec3 lattice_origin;            /* o (fp32) */
    int q_dims[CP_MSM_MAX_LEVELS][3];  /* padded charge lattice: x + 2R, y rounded up to even + 2R,
                                        * z rounded up to a multiple of 8 + 2R */
    int q_plane[CP_MSM_MAX_LEVELS];    /* its z stride in entries: a power of two >= q_dims x * q_dims y */
    size_t off_q[CP_MSM_MAX_LEVELS];   /* float32 pairs [q_dims z][q_plane]: entry (x, y, z) at
                                        * z * q_plane + y * q_dims x + x holds (q(x, y, z), q(x, y+1, z));
                                        * node (i, j, k) of the level is entry (i - lo x + R, j - lo y + R,
                                        * k - lo z + R); zero padding */
    size_t off_e[CP_MSM_MAX_LEVELS];   /* lattice potentials, float32 [n z][n y][n x] */
    size_t off_cells;                  /* the cell sort's sections start here (a cp_cutoff_layout with
                                        * capacity 0, offsets relative to this one) */
    size_t off_stencil;                /* W as float32 pairs (w, w), [2R+1][2R+1][2R+1] */
    size_t off_partial;                /* partial lattice sums (internal) */
    size_t total_bytes;                /* workspace size needed */
} cp_msm_layout;

/* Host-only: fills *out for these arguments (n_atoms >= 0).  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT (non-finite or non-positive cutoff or lattice_h,
 * domain_hi < domain_lo) or CP_ERR_TOO_LARGE (R above CP_MSM_MAX_RADIUS,
 * more than CP_MSM_MAX_LEVELS levels, a lattice or cell grid beyond the
 * library's limits). */
CP_API int cp_msm_layout_of(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, cp_vec3 domain_lo,
                            cp_vec3 domain_hi, float cutoff, float lattice_h, cp_msm_layout *out);

/* Host-only: workspace bytes cp_msm_longrange needs (0 if invalid). */
CP_API size_t cp_msm_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                     cp_vec3 domain_lo, cp_vec3 domain_hi, float cutoff, float lattice_h);

/* V_long on the grid.  accumulate = 0 writes V = V_long; accumulate = 1
 * adds V_long to V (after cp_cutoff with the same cutoff on the same
 * stream, V becomes the multilevel approximation of the full direct sum).
 * `workspace` is a DEVICE buffer of at least cp_msm_workspace_bytes(...)
 * bytes, 256-byte aligned, owned by the caller; calls sharing it must not
 * overlap on the GPU.  An atom outside the domain box is left out and sets
 * CP_DEVICE_ATOMS_OUTSIDE.  Returns CP_OK, CP_ERR_INVALID_ARGUMENT,
 * CP_ERR_MISALIGNED, CP_ERR_TOO_LARGE, CP_ERR_WORKSPACE_TOO_SMALL or
 * CP_ERR_CUDA.                                                              */
CP_API int cp_msm_longrange(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                            cp_vec3 domain_lo, cp_vec3 domain_hi, float cutoff, float lattice_h, void *workspace,
                            size_t workspace_bytes, float *V, int accumulate, void *stream);

/* The atoms' bounding box, for the domain of cp_msm_longrange: writes
 * (min x, min y, min z, max x, max y, max z) as 6 floats to the DEVICE
 * array `bounds` (4-byte aligned).  n_atoms >= 1.  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT, CP_ERR_MISALIGNED or CP_ERR_CUDA. */
CP_API int cp_atom_bounds(const float *atoms, int n_atoms, float *bounds, void *stream);

/* ------------------------------------------------------------------------ */
/* Sharding a map over several GPUs by z-slabs (PMPP ch.18 notes, sections
 * 18.2 and 18.5: grid points are independent -- each is written only by the
 * thread that owns it -- so a map splits into slabs of planes that separate
 * GPUs compute with no exchange; the direct sum needs every atom on every
 * GPU, the cutoff sum only the atoms within c of a slab, which the bin rule
 * of the slab's own grid selects by itself).
 *
 * Host-only.  Rank `rank` of `world` owns planes z0 .. z0 + *nz_slab - 1 of
 * a grid of nz planes: the planes are cut into units of `align` planes (8
 * keeps the cutoff map's 8x8x8-point bricks whole), the units are shared
 * out as evenly as integer division allows, in rank order, and the last
 * unit may be cut short by nz.  A rank past the last unit gets
 * *nz_slab = 0.  *origin_z_slab = fmaf(z0, h, origin_z), the full grid's
 * plane z0 formed as the kernels form a grid coordinate, so that the slab
 * grid (nx, ny, *nz_slab; origin (x, y, *origin_z_slab); h) has exactly the
 * full grid's points when those are fp32 numbers (cp_grid_points_exact).
 * Calling cp_direct / cp_cutoff on the slab grid with V pointing at plane
 * z0 of the full map computes that slab.  Returns CP_OK or
 * CP_ERR_INVALID_ARGUMENT (nz, world or align below 1, rank outside
 * [0, world), a null pointer, non-finite origin_z or h <= 0).              */
CP_API int cp_slab(int nz, int world, int rank, int align, float origin_z, float h, int *z0, int *nz_slab,
                   float *origin_z_slab);

/* ------------------------------------------------------------------------ */
/* Status and measurement helpers. */

/* Reads and clears the device status word of the current device
 * (CP_DEVICE_* bits; 0 when every kernel finished cleanly).  Synchronises
 * `stream` first.  Returns CP_OK or CP_ERR_CUDA. */
CP_API int cp_device_status(unsigned int *bits_out, void *stream);

/* Number of kernels this library has launched in this process (all
 * devices), for accounting in benchmarks. */
CP_API unsigned long long cp_launch_count(void);

/* Static text for a cp_status value. */
CP_API const char *cp_status_string(int status);

/* Library ABI version (major*10000 + minor*100 + patch). */
CP_API int cp_version(void);

/* Evaluates n reciprocal square roots of the DEVICE array x into the DEVICE
 * array y with one of the kernels' two routes: kind 0 = the SFU
 * (rsqrt.approx.ftz.f32), kind 1 = the FMA-pipe route (magic-constant
 * estimate and two Newton steps on rsqrt(x)/sqrt(2), then times fp32
 * sqrt(2); relative error below 5e-6 for positive normal x).  For tests of those error bounds.  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT or CP_ERR_CUDA.                                    */
CP_API int cp_eval_rsqrt(int kind, const float *x, float *y, int n, void *stream);

/* Microbenchmark of one SM pipe: every SM runs `warps` warps, each thread
 * issuing `iters` x 8 independent dependent-chain operations of kind
 * `kind` (0 = MUFU rsqrt.approx.ftz.f32, 1 = FP32 FFMA): the two rates
 * behind the roofline of the direct and cutoff maps.  Writes the measured throughput in
 * operations per SM clock cycle (per-SM clock64 cycles, averaged over the
 * SMs) to *ops_per_clk and the kernel time to *ms.  Synchronous.
 * Returns CP_OK, CP_ERR_INVALID_ARGUMENT or CP_ERR_CUDA. */
CP_API int cp_probe_pipe_rate(int kind, int warps, int iters, double *ops_per_clk, double *ms, void *stream);

/* Failure-path check of the kernels' bounded waits (no page counterpart):
 * one thread waits on a shared-memory barrier that nothing arrives at, with
 * the wait limit cut to limit_ns (1 .. 2e9 ns); the wait gives up, sets
 * CP_DEVICE_WAIT_TIMEOUT in the device status word and the kernel returns,
 * writing 1 to the DEVICE int *gave_up (4-byte aligned).  Asynchronous on
 * `stream`; the GPU context stays usable.  Returns CP_OK,
 * CP_ERR_INVALID_ARGUMENT, CP_ERR_MISALIGNED or CP_ERR_CUDA. */
CP_API int cp_probe_wait_timeout(unsigned long long limit_ns, int *gave_up, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CPMAP_H */
