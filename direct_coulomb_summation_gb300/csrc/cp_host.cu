// cp_host.cu -- host logic of the library: argument checks, status strings,
// the bin geometry, the brick neighbourhood offset list, the cutoff
// workspace layout, per-device facts and the device status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "cp_internal.h"

namespace cpmap {

// ---------------------------------------------------------------------------
// argument checks

int check_grid(int nx, int ny, int nz, cp_vec3 origin, float h, Grid *g) {
    if (nx < 1 || ny < 1 || nz < 1) return CP_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(origin.x) || !std::isfinite(origin.y) || !std::isfinite(origin.z)) return CP_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(h) || !(h > 0.0f)) return CP_ERR_INVALID_ARGUMENT;
    const long long lim = 1ll << 24;  // grid indices convert to float exactly
    if (nx > lim || ny > lim || nz > lim) return CP_ERR_TOO_LARGE;
    const long long np = (long long)nx * ny * nz;
    if (np >= (1ll << 31)) return CP_ERR_TOO_LARGE;
    g->nx = nx;
    g->ny = ny;
    g->nz = nz;
    g->ox = origin.x;
    g->oy = origin.y;
    g->oz = origin.z;
    g->h = h;
    g->npoints = np;
    return CP_OK;
}

namespace {

// Exponent of the lowest set bit of a nonzero finite float: f is an odd
// integer times 2^low_bit(f).
int low_bit(float f) {
    int e = 0;
    const double m = std::frexp(std::fabs((double)f), &e);  // f = m 2^e, m in [0.5, 1)
    unsigned long long mant = (unsigned long long)std::ldexp(m, 53);  // exact: 53-bit integer
    int tz = 0;
    while ((mant & 1ull) == 0ull) {
        mant >>= 1;
        ++tz;
    }
    return e - 53 + tz;
}

bool axis_exact(float o, float h, int n) {
    int q = low_bit(h);
    if (o != 0.0f) q = std::min(q, low_bit(o));
    const double lim = std::ldexp(1.0, 24 + q);
    const double a = std::fabs((double)o), b = std::fabs((double)o + (double)(n - 1) * (double)h);
    return q >= -126 && a < lim && b < lim;  // no subnormal steps either
}

}  // namespace

bool grid_points_exact(const Grid &g) {
    return axis_exact(g.ox, g.h, g.nx) && axis_exact(g.oy, g.h, g.ny) && axis_exact(g.oz, g.h, g.nz);
}

int check_cutoff_args(const Grid &, float cutoff, float bin_size, int capacity) {
    if (!std::isfinite(cutoff) || !(cutoff > 0.0f)) return CP_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(bin_size) || !(bin_size > 0.0f)) return CP_ERR_INVALID_ARGUMENT;
    if (capacity != 0 && capacity != 8 && capacity != 16) return CP_ERR_UNSUPPORTED;
    return CP_OK;
}

// ---------------------------------------------------------------------------
// bin geometry: m = ceil(c/b) margin bins per side, bo = float(origin - m b),
// nb = ceil(((N-1) h + 2 m b) / b) + 1 bins per axis.

int make_bin_geometry(const Grid &g, float cutoff, float bin_size, BinGeom *out) {
    const double b = bin_size, c = cutoff, h = g.h;
    const double m = std::ceil(c / b);
    if (m > 127.0) return CP_ERR_TOO_LARGE;
    const int n[3] = {g.nx, g.ny, g.nz};
    const double o[3] = {g.ox, g.oy, g.oz};
    long long nbins = 1;
    for (int d = 0; d < 3; ++d) {
        const double span = (double)(n[d] - 1) * h + 2.0 * m * b;
        const double nb = std::ceil(span / b) + 1.0;
        if (!(nb <= (double)(1 << 20))) return CP_ERR_TOO_LARGE;
        out->nb[d] = (int)nb;
        out->bo[d] = (float)(o[d] - m * b);
        nbins *= (long long)nb;
    }
    if (nbins > (long long)kScanBlock * kMaxScanBlocks) return CP_ERR_TOO_LARGE;
    out->m = (int)m;
    out->nbins = nbins;
    out->b = bin_size;
    out->c = cutoff;
    return CP_OK;
}

int brick_home_axis(int brick, int m, double h, double b) {
    const double t = (8.0 * (double)brick) * h;  // 8*brick is exact
    return m + (int)std::floor(t / b);
}

// ---------------------------------------------------------------------------
// Neighbourhood offset list of the 8x8x8-point bricks (Input Binning
// lecture, slides "Neighborhood Offset List (Pre-calculated)" (27) and
// "Details on Small Bin Design" (30)).  The lecture lists the bins whose
// distance from a location is below the cutoff; for a brick the distance
// that matters is the smallest distance between the brick's point box and
// the bin's box.  Per axis, take the smallest gap over every brick of the
// grid, so the one list is a superset for each brick; a bin is listed iff
// the three per-axis gaps give a distance below c + delta, where delta covers
// fp32 rounding of bin assignment and point coordinates.

namespace {

struct AxisGaps {
    int lo, hi;               // offsets d in [lo, hi]
    std::vector<double> gap;  // gap[d - lo] (min over bricks), +inf if none
};

AxisGaps axis_gaps(int n, double origin, double h, double bo, double b, int m, int nb, double reach) {
    AxisGaps a;
    const int D = (int)std::ceil((reach + 7.0 * h) / b) + 3;
    a.lo = -D;
    a.hi = D;
    a.gap.assign(2 * D + 1, INFINITY);
    const int nbricks = (n + kBrick - 1) / kBrick;
    for (int B = 0; B < nbricks; ++B) {
        const int home = brick_home_axis(B, m, h, b);
        const int npts = std::min(kBrick, n - kBrick * B);
        const double plo = origin + (double)(kBrick * B) * h;
        const double phi = plo + (double)(npts - 1) * h;
        for (int d = -D; d <= D; ++d) {
            const int u = home + d;
            if (u < 0 || u >= nb) continue;  // no such bin
            const double blo = bo + (double)u * b, bhi = blo + b;
            const double gp = std::max(0.0, std::max(blo - phi, plo - bhi));
            double &slot = a.gap[d + D];
            slot = std::min(slot, gp);
        }
    }
    return a;
}

}  // namespace

int make_offset_list(const Grid &g, const BinGeom &bg, OffsetList *out) {
    const double b = bg.b, c = bg.c, h = g.h;
    double extent = 0.0;
    for (int d = 0; d < 3; ++d) extent = std::max(extent, std::fabs((double)bg.bo[d]) + bg.nb[d] * b);
    const double delta = 1.0e-5 * (extent + c + b);
    const double reach = c + delta;
    const int n[3] = {g.nx, g.ny, g.nz};
    const double o[3] = {g.ox, g.oy, g.oz};
    AxisGaps ax[3];
    for (int d = 0; d < 3; ++d) ax[d] = axis_gaps(n[d], o[d], h, bg.bo[d], b, bg.m, bg.nb[d], reach);
    if (ax[0].hi > 127 || ax[1].hi > 127 || ax[2].hi > 127) return CP_ERR_TOO_LARGE;
    const double r2 = reach * reach;
    int nr = 0, nbins = 0;
    for (int dz = ax[2].lo; dz <= ax[2].hi; ++dz) {
        const double gz = ax[2].gap[dz - ax[2].lo];
        if (!(gz * gz < r2)) continue;
        for (int dy = ax[1].lo; dy <= ax[1].hi; ++dy) {
            const double gy = ax[1].gap[dy - ax[1].lo];
            const double gyz = gy * gy + gz * gz;
            if (!(gyz < r2)) continue;
            // the listed dx of one (dy, dz) row form an interval (the per-axis
            // minimum gap falls and then rises with dx); one run covers it
            int run_lo = 0, run_hi = -1;
            for (int dx = ax[0].lo; dx <= ax[0].hi; ++dx) {
                const double gx = ax[0].gap[dx - ax[0].lo];
                if ((gx * gx + gyz) < r2) {
                    if (run_hi < run_lo) run_lo = dx;
                    run_hi = dx;
                }
            }
            if (run_hi < run_lo) continue;
            if (nr >= kMaxRuns) return CP_ERR_TOO_LARGE;
            out->run[nr][0] = (int8_t)dy;
            out->run[nr][1] = (int8_t)dz;
            out->run[nr][2] = (int8_t)run_lo;
            out->run[nr][3] = (int8_t)run_hi;
            ++nr;
            nbins += run_hi - run_lo + 1;
        }
    }
    out->n_runs = nr;
    out->n_bins = nbins;
    return CP_OK;
}

// ---------------------------------------------------------------------------
// workspace layout

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int make_layout(int n_atoms, const BinGeom &bg, int capacity, cp_cutoff_layout *out) {
    std::memset(out, 0, sizeof(*out));
    for (int d = 0; d < 3; ++d) {
        out->nb[d] = bg.nb[d];
        out->bo[d] = bg.bo[d];
    }
    out->margin_bins = bg.m;
    out->capacity = capacity;
    out->nbins = bg.nbins;
    const size_t n = (size_t)(n_atoms > 0 ? n_atoms : 0);
    const size_t nbins = (size_t)bg.nbins;
    const size_t nblk = (nbins + kScanBlock - 1) / kScanBlock;
    size_t off = 0;
    out->off_count = off;
    off = align256(off + 4 * nbins);
    out->off_start = off;
    off = align256(off + 4 * (nbins + 1));
    out->off_csr_index = off;
    off = align256(off + 4 * n);
    out->off_csr_atoms = off;
    off = align256(off + 16 * n);
    out->off_padded = off;
    off = align256(off + 16 * nbins * (size_t)capacity);
    out->off_stats = off;
    off = align256(off + 4 * 8);
    out->off_scratch = off;  // int2 bin/rank per atom, then block sums and block prefixes
    off = align256(off + 8 * n);
    off = align256(off + 4 * nblk);
    off = align256(off + 4 * nblk);
    out->total_bytes = off;
    return CP_OK;
}

// ---------------------------------------------------------------------------
// devices

namespace {
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];
unsigned int *g_status_ptr[kMaxDevices];
}  // namespace

__device__ unsigned int g_cp_device_status;

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void note_launches(unsigned long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

unsigned long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

int device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ok[dev]) {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return CP_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return CP_ERR_CUDA;
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return CP_OK;
}

unsigned int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cp_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace cpmap

// ---------------------------------------------------------------------------
// C ABI: host-only entry points and status helpers

using namespace cpmap;

extern "C" {

CP_API const char *cp_status_string(int status) {
    switch (status) {
        case CP_OK: return "ok";
        case CP_ERR_INVALID_ARGUMENT: return "invalid argument";
        case CP_ERR_MISALIGNED: return "misaligned pointer (atoms need 16 bytes, workspace 256 bytes)";
        case CP_ERR_TOO_LARGE: return "size beyond the library's limits";
        case CP_ERR_WORKSPACE_TOO_SMALL: return "workspace (or output buffer) too small";
        case CP_ERR_UNSUPPORTED: return "unsupported option";
        case CP_ERR_CUDA: return "CUDA runtime error";
        case CP_ERR_DEVICE: return "a kernel reported a problem (see cp_device_status)";
        default: return "unknown status";
    }
}

CP_API int cp_version(void) { return 100; }

CP_API int cp_slab(int nz, int world, int rank, int align, float origin_z, float h, int *z0, int *nz_slab,
                   float *origin_z_slab) {
    if (nz < 1 || world < 1 || rank < 0 || rank >= world || align < 1 || !z0 || !nz_slab || !origin_z_slab ||
        !std::isfinite(origin_z) || !std::isfinite(h) || !(h > 0.0f))
        return CP_ERR_INVALID_ARGUMENT;
    // whole units of `align` planes, split as evenly as integer division
    // allows, in rank order; the last unit may be cut short by nz
    const long long units = ((long long)nz + align - 1) / align;
    const long long u0 = units * rank / world, u1 = units * (rank + 1) / world;
    const long long p0 = std::min<long long>(u0 * align, nz), p1 = std::min<long long>(u1 * align, nz);
    *z0 = (int)p0;
    *nz_slab = (int)(p1 - p0);
    // the full grid's plane z0, formed as the kernels form a grid coordinate
    *origin_z_slab = fmaf((float)p0, h, origin_z);
    return CP_OK;
}

CP_API unsigned long long cp_launch_count(void) { return cpmap::launch_count(); }

CP_API int cp_cutoff_layout_of(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                               float bin_size, int capacity, cp_cutoff_layout *out) {
    if (!out || n_atoms < 0) return CP_ERR_INVALID_ARGUMENT;
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    rc = check_cutoff_args(g, cutoff, bin_size, capacity);
    if (rc) return rc;
    BinGeom bg;
    rc = make_bin_geometry(g, cutoff, bin_size, &bg);
    if (rc) return rc;
    return make_layout(n_atoms, bg, capacity, out);
}

CP_API size_t cp_cutoff_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                                        float bin_size, int capacity) {
    cp_cutoff_layout L;
    if (cp_cutoff_layout_of(n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, &L) != CP_OK) return 0;
    return L.total_bytes;
}

CP_API int cp_offset_list(int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff, float bin_size,
                          int *runs_out, int max_runs, int *n_runs, int *n_bins) {
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    if (!std::isfinite(cutoff) || !(cutoff > 0.0f) || !std::isfinite(bin_size) || !(bin_size > 0.0f))
        return CP_ERR_INVALID_ARGUMENT;
    BinGeom bg;
    rc = make_bin_geometry(g, cutoff, bin_size, &bg);
    if (rc) return rc;
    static thread_local OffsetList L;
    rc = make_offset_list(g, bg, &L);
    if (rc) return rc;
    if (n_runs) *n_runs = L.n_runs;
    if (n_bins) *n_bins = L.n_bins;
    if (runs_out) {
        if (max_runs < L.n_runs) return CP_ERR_WORKSPACE_TOO_SMALL;
        for (int r = 0; r < L.n_runs; ++r)
            for (int k = 0; k < 4; ++k) runs_out[4 * r + k] = L.run[r][k];
    }
    return CP_OK;
}

CP_API int cp_brick_home(int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff, float bin_size, int bx,
                         int by, int bz, int home_out[3]) {
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    if (!home_out || !std::isfinite(cutoff) || !(cutoff > 0.0f) || !std::isfinite(bin_size) || !(bin_size > 0.0f))
        return CP_ERR_INVALID_ARGUMENT;
    BinGeom bg;
    rc = make_bin_geometry(g, cutoff, bin_size, &bg);
    if (rc) return rc;
    const int B[3] = {bx, by, bz};
    for (int d = 0; d < 3; ++d) home_out[d] = brick_home_axis(B[d], bg.m, (double)h, (double)bin_size);
    return CP_OK;
}

CP_API int cp_device_status(unsigned int *bits_out, void *stream) {
    if (!bits_out) return CP_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return CP_ERR_CUDA;
    unsigned int *p = device_status_ptr();
    if (!p) return CP_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CP_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return CP_ERR_CUDA;
    *bits_out = v;
    return CP_OK;
}

}  // extern "C"
