/*
 * oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, fp64 CPU reference for the electrostatic potential map.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or call it.  It shares no code, header, table or constant
 * generator with the CUDA library; it is written from the definitions on the
 * pages it cites and from the readings listed in the design notes.
 *
 * Conventions
 *   atoms   float32 [n][4] = (x, y, z, q), the 16-byte atom record
 *           (PMPP ch.18 notes "Case study -- electrostatic potential map",
 *           section 18.2, struct Atom).
 *   points  grid point (i, j, k) sits at origin + (i*h, j*h, k*h); origin and
 *           h arrive as float32 and are widened exactly to double.  A point
 *           list is int32 [m][3]; a NULL list means every point of the
 *           Nx x Ny x Nz grid in x-fastest order, i.e. flat index
 *           (k*Ny + j)*Nx + i (PMPP ch.18 notes, section 18.4).
 *   output  V[m] and B[m] in double, B = sum over the contributing atoms of
 *           |q_a| / r (the scale of the accuracy bound).
 *
 * Every function is single-pass, in atom index order, with no blocking or
 * reordering beyond what its definition states.  Threads split the points
 * into contiguous ranges only; a point's value never depends on the thread
 * count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Position given to the unused slots of a fixed-capacity bin.  It is far from
 * any grid, so a padded slot fails every cutoff test; its charge is 0.  (The
 * lecture's inner loop stops at the first slot whose charge is 0 -- Input
 * Binning lecture, slide "GPU Thread Inner Loop" (37); here the slot count
 * bounds the loop instead, so real atoms with q = 0 are kept.) */
#define OR_PAD_COORD 1.0e18f

/* ------------------------------------------------------------------------ */
/* threading: static contiguous split of [0, n) over n_threads workers       */

typedef void (*or_range_fn)(void *ctx, long begin, long end);

typedef struct {
    or_range_fn fn;
    void *ctx;
    long begin, end;
} or_job;

static void *or_job_main(void *p) {
    or_job *j = (or_job *)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

static void or_parallel_for(long n, int n_threads, or_range_fn fn, void *ctx) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long)n_threads > n) n_threads = (int)(n > 0 ? n : 1);
    if (n_threads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t tid[256];
    or_job job[256];
    int started[256];
    for (int t = 0; t < n_threads; ++t) {
        job[t].fn = fn;
        job[t].ctx = ctx;
        job[t].begin = n * t / n_threads;
        job[t].end = n * (t + 1) / n_threads;
        started[t] = pthread_create(&tid[t], NULL, or_job_main, &job[t]) == 0;
        if (!started[t]) or_job_main(&job[t]);
    }
    for (int t = 0; t < n_threads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* grid point coordinates                                                    */

typedef struct {
    const int *pts; /* NULL: all grid points, x fastest */
    int nx, ny, nz;
    double ox, oy, oz, h;
} or_grid;

static void or_point(const or_grid *g, long p, double *x, double *y, double *z) {
    long i, j, k;
    if (g->pts) {
        i = g->pts[3 * p + 0];
        j = g->pts[3 * p + 1];
        k = g->pts[3 * p + 2];
    } else {
        i = p % g->nx;
        j = (p / g->nx) % g->ny;
        k = p / ((long)g->nx * g->ny);
    }
    /* origin + index * spacing, in double */
    *x = g->ox + (double)i * g->h;
    *y = g->oy + (double)j * g->h;
    *z = g->oz + (double)k * g->h;
}

static or_grid or_make_grid(const int *pts, int nx, int ny, int nz, const float *origin, float h) {
    or_grid g;
    g.pts = pts;
    g.nx = nx;
    g.ny = ny;
    g.nz = nz;
    g.ox = (double)origin[0];
    g.oy = (double)origin[1];
    g.oz = (double)origin[2];
    g.h = (double)h;
    return g;
}

/* ------------------------------------------------------------------------ */
/* Direct Coulomb summation.
 * V(g) = sum_a q_a / r_{a,g}  (PMPP ch.18 notes, section 18.1; the pwwt.cn
 * chapter-18 article, section 一, states the same sum with r written as
 * sqrt(dx^2 + dy^2 + dz^2)).  No Coulomb constant: V is in charge/length.  */

typedef struct {
    const float *atoms;
    long n_atoms;
    or_grid grid;
    double *V, *B;
} or_direct_ctx;

static void or_direct_range(void *vctx, long begin, long end) {
    or_direct_ctx *c = (or_direct_ctx *)vctx;
    for (long p = begin; p < end; ++p) {
        double x, y, z;
        or_point(&c->grid, p, &x, &y, &z);
        double v = 0.0, b = 0.0;
        for (long a = 0; a < c->n_atoms; ++a) {
            const float *at = c->atoms + 4 * a;
            double dx = x - (double)at[0];
            double dy = y - (double)at[1];
            double dz = z - (double)at[2];
            double r = sqrt(dx * dx + dy * dy + dz * dz);
            double q = (double)at[3];
            v += q / r;
            b += fabs(q) / r;
        }
        c->V[p] = v;
        if (c->B) c->B[p] = b;
    }
}

int or_direct(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
              const float *origin, float h, double *V, double *B, int n_threads) {
    if (n_atoms < 0 || n_pts < 0 || !V || (n_atoms > 0 && !atoms)) return -1;
    or_direct_ctx c;
    c.atoms = atoms;
    c.n_atoms = n_atoms;
    c.grid = or_make_grid(pts, nx, ny, nz, origin, h);
    c.V = V;
    c.B = B;
    long m = pts ? n_pts : (long)nx * ny * nz;
    or_parallel_for(m, n_threads, or_direct_range, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Cutoff summation with the switched term.
 * A pair contributes iff r^2 < c^2 (strict, as in the cutoff tests of PMPP
 * ch.18 notes section 18.5 and of the Input Binning lecture slide "Large
 * Bin Cut-off Kernel Code" (24)), and contributes q * (1/r - g(r)) with the
 * even quartic g(r) = GC0 + GC1 r^2 + GC2 r^4 of that slide.  The
 * coefficients are those of
 *     g(r) = (1/c) * (15/8 - 5/4 (r/c)^2 + 3/8 (r/c)^4),
 * for which g, g' and g'' equal 1/r and its first two derivatives at r = c,
 * so each term vanishes smoothly at the cutoff.                            */

double or_switch_g(double r2, double c) {
    double s = r2 / (c * c);
    return (1.0 / c) * (15.0 / 8.0 - (5.0 / 4.0) * s + (3.0 / 8.0) * s * s);
}

/* 1/r - g(r) for r^2 = r2 (no cutoff test) */
double or_switched_term(double r2, double c) { return 1.0 / sqrt(r2) - or_switch_g(r2, c); }

typedef struct {
    const float *atoms;
    long n_atoms;
    or_grid grid;
    double c;
    double *V, *B;
} or_cut_ctx;

static void or_cutoff_range(void *vctx, long begin, long end) {
    or_cut_ctx *c = (or_cut_ctx *)vctx;
    const double c2 = c->c * c->c;
    for (long p = begin; p < end; ++p) {
        double x, y, z;
        or_point(&c->grid, p, &x, &y, &z);
        double v = 0.0, b = 0.0;
        for (long a = 0; a < c->n_atoms; ++a) {
            const float *at = c->atoms + 4 * a;
            double dx = x - (double)at[0];
            double dy = y - (double)at[1];
            double dz = z - (double)at[2];
            double r2 = dx * dx + dy * dy + dz * dz;
            if (r2 < c2) {
                double q = (double)at[3];
                v += q * or_switched_term(r2, c->c);
                b += fabs(q) / sqrt(r2);
            }
        }
        c->V[p] = v;
        if (c->B) c->B[p] = b;
    }
}

/* Hard cutoff without switching: sum of q / r over r^2 < c^2, the form of
 * the 27-bin kernel in PMPP ch.18 notes section 18.5. */
typedef struct {
    const float *atoms;
    long n_atoms;
    or_grid grid;
    double c;
    double *V, *B;
} or_hard_ctx;

static void or_hard_range(void *vctx, long begin, long end) {
    or_hard_ctx *c = (or_hard_ctx *)vctx;
    const double c2 = c->c * c->c;
    for (long p = begin; p < end; ++p) {
        double x, y, z;
        or_point(&c->grid, p, &x, &y, &z);
        double v = 0.0, b = 0.0;
        for (long a = 0; a < c->n_atoms; ++a) {
            const float *at = c->atoms + 4 * a;
            double dx = x - (double)at[0];
            double dy = y - (double)at[1];
            double dz = z - (double)at[2];
            double r2 = dx * dx + dy * dy + dz * dz;
            if (r2 < c2) {
                double q = (double)at[3];
                double r = sqrt(r2);
                v += q / r;
                b += fabs(q) / r;
            }
        }
        c->V[p] = v;
        if (c->B) c->B[p] = b;
    }
}

int or_cutoff_hard(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
                   const float *origin, float h, float cutoff, double *V, double *B, int n_threads) {
    if (n_atoms < 0 || n_pts < 0 || !V || !(cutoff > 0.0f) || (n_atoms > 0 && !atoms)) return -1;
    or_hard_ctx c;
    c.atoms = atoms;
    c.n_atoms = n_atoms;
    c.grid = or_make_grid(pts, nx, ny, nz, origin, h);
    c.c = (double)cutoff;
    c.V = V;
    c.B = B;
    long m = pts ? n_pts : (long)nx * ny * nz;
    or_parallel_for(m, n_threads, or_hard_range, &c);
    return 0;
}

int or_cutoff_brute(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
                    const float *origin, float h, float cutoff, double *V, double *B, int n_threads) {
    if (n_atoms < 0 || n_pts < 0 || !V || !(cutoff > 0.0f) || (n_atoms > 0 && !atoms)) return -1;
    or_cut_ctx c;
    c.atoms = atoms;
    c.n_atoms = n_atoms;
    c.grid = or_make_grid(pts, nx, ny, nz, origin, h);
    c.c = (double)cutoff;
    c.V = V;
    c.B = B;
    long m = pts ? n_pts : (long)nx * ny * nz;
    or_parallel_for(m, n_threads, or_cutoff_range, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Bin geometry and binning.
 *
 * The pages bin an atom by dividing its position by the bin size
 * (PMPP ch.18 notes, section 18.5: integer part of x / bsize; Input Binning
 * lecture, slide "Pseudo Code of an Implementation" (28)).  Made exactly
 * reproducible here:
 *   m      = ceil(c / b)                          bins of margin per side
 *   bo_d   = float(origin_d - m*b)                bin-grid origin (double, rounded once)
 *   nb_d   = ceil(((N_d - 1)*h + 2*m*b) / b) + 1  bins per axis
 *   u_d    = floor( float( float(a_d - bo_d) / b ) )   two IEEE fp32 roundings
 * An atom is binned iff all three u_d are finite and in [0, nb_d); else it is
 * dropped (it is then at least c away from every grid point, up to fp32
 * rounding of its coordinate).  Bin (ux, uy, uz) has linear index
 * (uz*nby + uy)*nbx + ux.  Within a bin atoms keep ascending input order; the
 * first K of a bin fill its fixed-capacity slots (Input Binning lecture,
 * slide "Coalesced Global Memory Access to Atom Data" (33): bins of fixed
 * size stored as a 3-D array) and the rest are that bin's overflow ("extra
 * atoms", slide "Handling Overfull Bins" (34)).  The sorted (CSR) array holds
 * all binned atoms; a bin's overflow is its CSR entries past the first K.   */

int or_bin_geometry(int nx, int ny, int nz, const float *origin, float h, float cutoff, float bin_size,
                    int *nb_out, float *bo_out, int *m_out) {
    if (nx <= 0 || ny <= 0 || nz <= 0 || !(h > 0.0f) || !(cutoff > 0.0f) || !(bin_size > 0.0f)) return -1;
    const double b = (double)bin_size;
    const double c = (double)cutoff;
    const int n[3] = {nx, ny, nz};
    double m = ceil(c / b);
    for (int d = 0; d < 3; ++d) {
        double span = (double)(n[d] - 1) * (double)h + 2.0 * m * b;
        double nb = ceil(span / b) + 1.0;
        if (nb > 1.0e6) return -2;
        nb_out[d] = (int)nb;
        bo_out[d] = (float)((double)origin[d] - m * b);
    }
    if (m_out) *m_out = (int)m;
    return 0;
}

/* fp32 bin coordinate of one atom coordinate; returns -1 if out of range */
static int or_bin_coord(float a, float bo, float b, int nb) {
    /* volatile pins each result to an fp32 rounding (no contraction, no
     * excess precision, whatever the compiler flags) */
    volatile float t = a - bo;
    volatile float u = t / b;
    float f = floorf(u);
    if (!(f >= 0.0f) || !(f < (float)nb)) return -1; /* also rejects NaN */
    return (int)f;
}

long or_atom_bin(const float *atom, const int *nb, const float *bo, float b) {
    int ux = or_bin_coord(atom[0], bo[0], b, nb[0]);
    int uy = or_bin_coord(atom[1], bo[1], b, nb[1]);
    int uz = or_bin_coord(atom[2], bo[2], b, nb[2]);
    if (ux < 0 || uy < 0 || uz < 0) return -1;
    return ((long)uz * nb[1] + uy) * nb[0] + ux;
}

/* Stable counting sort of atoms into bins.
 * outputs (caller-allocated; any may be NULL except count/start):
 *   bin_of_atom[n]        linear bin or -1 (dropped)
 *   count[nbins]          atoms per bin
 *   start[nbins+1]        exclusive prefix sum of count
 *   csr_index[n_binned]   original index, sorted by (bin, index)
 *   csr_atoms[n_binned*4] the atoms in that order
 *   padded[nbins*K*4]     first K atoms of each bin, unused slots
 *                         (PAD, PAD, PAD, 0)
 * returns the number of binned atoms, or < 0 on bad arguments.             */
long or_bin_atoms(const float *atoms, long n_atoms, const int *nb, const float *bo, float bin_size, int capacity,
                  int *bin_of_atom, int *count, int *start, int *csr_index, float *csr_atoms, float *padded,
                  long *n_dropped) {
    if (n_atoms < 0 || !nb || !bo || !count || !start || capacity < 0 || !(bin_size > 0.0f)) return -1;
    const long nbins = (long)nb[0] * nb[1] * nb[2];
    int *bins = (int *)malloc(sizeof(int) * (size_t)(n_atoms > 0 ? n_atoms : 1));
    int *fill = (int *)calloc((size_t)nbins, sizeof(int));
    if (!bins || !fill) {
        free(bins);
        free(fill);
        return -3;
    }
    memset(count, 0, sizeof(int) * (size_t)nbins);
    long dropped = 0;
    for (long a = 0; a < n_atoms; ++a) {
        long bi = or_atom_bin(atoms + 4 * a, nb, bo, bin_size);
        bins[a] = (int)bi;
        if (bi < 0)
            ++dropped;
        else
            ++count[bi];
        if (bin_of_atom) bin_of_atom[a] = (int)bi;
    }
    start[0] = 0;
    for (long i = 0; i < nbins; ++i) start[i + 1] = start[i] + count[i];
    for (long a = 0; a < n_atoms; ++a) { /* ascending index: stable */
        long bi = bins[a];
        if (bi < 0) continue;
        long pos = (long)start[bi] + fill[bi];
        if (csr_index) csr_index[pos] = (int)a;
        if (csr_atoms) memcpy(csr_atoms + 4 * pos, atoms + 4 * a, 4 * sizeof(float));
        if (padded && fill[bi] < capacity)
            memcpy(padded + 4 * ((size_t)bi * capacity + fill[bi]), atoms + 4 * a, 4 * sizeof(float));
        ++fill[bi];
    }
    if (padded) {
        for (long bi = 0; bi < nbins; ++bi)
            for (int s = count[bi]; s < capacity; ++s) {
                float *slot = padded + 4 * ((size_t)bi * capacity + s);
                slot[0] = OR_PAD_COORD;
                slot[1] = OR_PAD_COORD;
                slot[2] = OR_PAD_COORD;
                slot[3] = 0.0f;
            }
    }
    if (n_dropped) *n_dropped = dropped;
    free(bins);
    free(fill);
    return n_atoms - dropped;
}

/* ------------------------------------------------------------------------ */
/* Binned cutoff summation (the second, independent route to the cutoff sum).
 * Per grid point, visit the bins around the point's own bin whose box lies
 * within c (+ a rounding margin delta) of the point -- a per-point
 * neighbourhood offset list (Input Binning lecture, slides "Neighborhood
 * Offset List (Pre-calculated)" (27) and "Pseudo Code of an Implementation"
 * (28)) -- and test every atom they hold with r^2 < c^2.  The margin covers
 * atoms that the fp32 bin rule placed across a bin face from their exact
 * position; it only adds bins, never atoms, so the set of contributing pairs
 * equals the brute-force set.  Contributions are summed in ascending atom
 * index, the order the brute-force sum uses, so both give the same V.      */

typedef struct {
    const float *atoms;
    or_grid grid;
    double c, delta, b;
    int nb[3];
    double bo[3];
    const int *count, *start, *csr_index;
    double *V, *B;
} or_binned_ctx;

static int or_cmp_int(const void *a, const void *b) {
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

static double or_box_gap(double p, double lo, double hi) {
    if (p < lo) return lo - p;
    if (p > hi) return p - hi;
    return 0.0;
}

/* contributing atoms of one point, ascending index; returns count, *out malloc'd */
static int or_point_neighbours(const or_binned_ctx *c, double x, double y, double z, int **out) {
    const double pc[3] = {x, y, z};
    const double reach = c->c + c->delta;
    int lo[3], hi[3];
    for (int d = 0; d < 3; ++d) {
        double l = floor((pc[d] - reach - c->bo[d]) / c->b) - 1.0;
        double u = floor((pc[d] + reach - c->bo[d]) / c->b) + 1.0;
        if (l < 0.0) l = 0.0;
        if (u > (double)(c->nb[d] - 1)) u = (double)(c->nb[d] - 1);
        lo[d] = (int)l;
        hi[d] = (int)u;
    }
    int cap = 64, n = 0;
    int *list = (int *)malloc(sizeof(int) * (size_t)cap);
    const double c2 = c->c * c->c;
    for (int uz = lo[2]; uz <= hi[2]; ++uz)
        for (int uy = lo[1]; uy <= hi[1]; ++uy)
            for (int ux = lo[0]; ux <= hi[0]; ++ux) {
                const int u[3] = {ux, uy, uz};
                double g2 = 0.0;
                for (int d = 0; d < 3; ++d) {
                    double blo = c->bo[d] + (double)u[d] * c->b;
                    double g = or_box_gap(pc[d], blo, blo + c->b);
                    g2 += g * g;
                }
                if (!(g2 < reach * reach)) continue;
                long bi = ((long)uz * c->nb[1] + uy) * c->nb[0] + ux;
                for (int s = c->start[bi]; s < c->start[bi] + c->count[bi]; ++s) {
                    int a = c->csr_index[s];
                    const float *at = c->atoms + 4 * (long)a;
                    double dx = x - (double)at[0];
                    double dy = y - (double)at[1];
                    double dz = z - (double)at[2];
                    double r2 = dx * dx + dy * dy + dz * dz;
                    if (r2 < c2) {
                        if (n == cap) {
                            cap *= 2;
                            list = (int *)realloc(list, sizeof(int) * (size_t)cap);
                        }
                        list[n++] = a;
                    }
                }
            }
    qsort(list, (size_t)n, sizeof(int), or_cmp_int);
    *out = list;
    return n;
}

static void or_binned_range(void *vctx, long begin, long end) {
    or_binned_ctx *c = (or_binned_ctx *)vctx;
    for (long p = begin; p < end; ++p) {
        double x, y, z;
        or_point(&c->grid, p, &x, &y, &z);
        int *list = NULL;
        int n = or_point_neighbours(c, x, y, z, &list);
        double v = 0.0, b = 0.0;
        for (int t = 0; t < n; ++t) {
            const float *at = c->atoms + 4 * (long)list[t];
            double dx = x - (double)at[0];
            double dy = y - (double)at[1];
            double dz = z - (double)at[2];
            double r2 = dx * dx + dy * dy + dz * dz;
            double q = (double)at[3];
            v += q * or_switched_term(r2, c->c);
            b += fabs(q) / sqrt(r2);
        }
        free(list);
        c->V[p] = v;
        if (c->B) c->B[p] = b;
    }
}

static int or_binned_setup(or_binned_ctx *c, const float *atoms, long n_atoms, const int *pts, int nx, int ny,
                           int nz, const float *origin, float h, float cutoff, float bin_size, int **count_out,
                           int **start_out, int **csr_out) {
    float bo[3];
    int m;
    memset(c, 0, sizeof(*c));
    if (or_bin_geometry(nx, ny, nz, origin, h, cutoff, bin_size, c->nb, bo, &m) != 0) return -1;
    long nbins = (long)c->nb[0] * c->nb[1] * c->nb[2];
    int *count = (int *)malloc(sizeof(int) * (size_t)nbins);
    int *start = (int *)malloc(sizeof(int) * (size_t)(nbins + 1));
    int *csr = (int *)malloc(sizeof(int) * (size_t)(n_atoms > 0 ? n_atoms : 1));
    if (!count || !start || !csr) {
        free(count);
        free(start);
        free(csr);
        return -3;
    }
    or_bin_atoms(atoms, n_atoms, c->nb, bo, bin_size, 0, NULL, count, start, csr, NULL, NULL, NULL);
    c->atoms = atoms;
    c->grid = or_make_grid(pts, nx, ny, nz, origin, h);
    c->c = (double)cutoff;
    c->b = (double)bin_size;
    double extent = 0.0;
    for (int d = 0; d < 3; ++d) {
        c->bo[d] = (double)bo[d];
        double e = fabs((double)bo[d]) + (double)c->nb[d] * c->b;
        if (e > extent) extent = e;
    }
    c->delta = 1.0e-5 * (extent + c->c + c->b);
    c->count = count;
    c->start = start;
    c->csr_index = csr;
    *count_out = count;
    *start_out = start;
    *csr_out = csr;
    return 0;
}

int or_cutoff_binned(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
                     const float *origin, float h, float cutoff, float bin_size, double *V, double *B,
                     int n_threads) {
    if (n_atoms < 0 || n_pts < 0 || !V || (n_atoms > 0 && !atoms)) return -1;
    or_binned_ctx c;
    int *count, *start, *csr;
    int rc = or_binned_setup(&c, atoms, n_atoms, pts, nx, ny, nz, origin, h, cutoff, bin_size, &count, &start, &csr);
    if (rc) return rc;
    c.V = V;
    c.B = B;
    long m = pts ? n_pts : (long)nx * ny * nz;
    or_parallel_for(m, n_threads, or_binned_range, &c);
    free(count);
    free(start);
    free(csr);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Contributing (point, atom) pair sets, for the bit-exact comparison of the
 * brute-force and binned routes.  Pairs are written as (point ordinal, atom
 * index), sorted by point then atom.  Returns the number of pairs (which may
 * exceed cap; only the first cap are written), or < 0 on error.            */

long long or_pairs_brute(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
                         const float *origin, float h, float cutoff, long long *out, long long cap) {
    if (n_atoms < 0 || !(cutoff > 0.0f)) return -1;
    or_grid g = or_make_grid(pts, nx, ny, nz, origin, h);
    long m = pts ? n_pts : (long)nx * ny * nz;
    const double c2 = (double)cutoff * (double)cutoff;
    long long k = 0;
    for (long p = 0; p < m; ++p) {
        double x, y, z;
        or_point(&g, p, &x, &y, &z);
        for (long a = 0; a < n_atoms; ++a) {
            const float *at = atoms + 4 * a;
            double dx = x - (double)at[0];
            double dy = y - (double)at[1];
            double dz = z - (double)at[2];
            if (dx * dx + dy * dy + dz * dz < c2) {
                if (k < cap) {
                    out[2 * k] = p;
                    out[2 * k + 1] = a;
                }
                ++k;
            }
        }
    }
    return k;
}

long long or_pairs_binned(const float *atoms, long n_atoms, const int *pts, long n_pts, int nx, int ny, int nz,
                          const float *origin, float h, float cutoff, float bin_size, long long *out,
                          long long cap) {
    if (n_atoms < 0) return -1;
    or_binned_ctx c;
    int *count, *start, *csr;
    int rc = or_binned_setup(&c, atoms, n_atoms, pts, nx, ny, nz, origin, h, cutoff, bin_size, &count, &start, &csr);
    if (rc) return rc;
    long m = pts ? n_pts : (long)nx * ny * nz;
    long long k = 0;
    for (long p = 0; p < m; ++p) {
        double x, y, z;
        or_point(&c.grid, p, &x, &y, &z);
        int *list = NULL;
        int n = or_point_neighbours(&c, x, y, z, &list);
        for (int t = 0; t < n; ++t) {
            if (k < cap) {
                out[2 * k] = p;
                out[2 * k + 1] = list[t];
            }
            ++k;
        }
        free(list);
    }
    free(count);
    free(start);
    free(csr);
    return k;
}
