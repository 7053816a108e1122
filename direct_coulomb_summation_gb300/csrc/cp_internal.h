// cp_internal.h -- host-side declarations shared by the library's translation
// units: argument checks, bin geometry, the brick offset list, the cutoff
// workspace layout, per-device properties and the device status word.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "cpmap.h"

namespace cpmap {

constexpr int kBrick = 8;            // brick edge in grid points (8x8x8 = 512 points)
constexpr int kMaxRuns = 1024;       // offset-list x-runs a brick kernel can take
constexpr float kPadCoord = 1.0e18f; // position of an unused bin slot
constexpr int kScanBlock = 2048;     // bins per block of the count scan
constexpr int kMaxScanBlocks = 8192; // so at most 16M bins

// Validated grid description.
struct Grid {
    int nx, ny, nz;
    float ox, oy, oz, h;
    long long npoints;
};

// True when every grid coordinate origin_d + i*h (0 <= i < n_d) is exactly
// representable in fp32, so that forming a point and subtracting an atom
// rounds only once.  Sufficient, not necessary: o + i*h are all multiples of
// 2^q, q the lowest set bit of o or h, and such a multiple is exact in fp32
// when its magnitude is below 2^(24 + q).
bool grid_points_exact(const Grid &g);

// Bin grid of the cutoff map (see cpmap.h for the definitions).
struct BinGeom {
    int nb[3];
    float bo[3];
    int m;
    long long nbins;
    float b;      // bin edge (fp32 as given)
    float c;      // cutoff (fp32 as given)
};

// Brick neighbourhood as x-runs: run r = (dy, dz, dx_lo, dx_hi) relative to
// the brick's home bin.
struct OffsetList {
    int n_runs;
    int n_bins;
    int8_t run[kMaxRuns][4];
};

int check_grid(int nx, int ny, int nz, cp_vec3 origin, float h, Grid *g);
int check_cutoff_args(const Grid &g, float cutoff, float bin_size, int capacity);
int make_bin_geometry(const Grid &g, float cutoff, float bin_size, BinGeom *out);
// Home bin of brick index `brick` along one axis: m + floor(8*brick*h / b),
// evaluated with IEEE double multiply and divide (the kernels do the same).
int brick_home_axis(int brick, int m, double h, double b);
int make_offset_list(const Grid &g, const BinGeom &bg, OffsetList *out);
int make_layout(int n_atoms, const BinGeom &bg, int capacity, cp_cutoff_layout *out);

// Per-device facts (cached after the first query on each device).
// Deterministic counting sort of atoms into the cells of `bg` (no fixed
// slots: L from make_layout(n, bg, 0, &L)), leaving count, start, the
// cell-sorted atoms and indices (ascending input index within a cell) and
// the stats in the sections of `workspace`.  Atoms outside the cell grid
// are dropped and counted in stats[1].
int sort_atoms_into_cells(const float4 *atoms, int n_atoms, const BinGeom &bg, const cp_cutoff_layout &L,
                          void *workspace, cudaStream_t stream);

// Devices the library keeps per-device state for (ordinals 0 .. kMaxDevices-1;
// calls on a device past that return CP_ERR_CUDA).
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
};
int device_info(DeviceInfo *out);

// Device address of the status word of the current device.
unsigned int *device_status_ptr();

// Adds n to the process-wide count of kernel launches (cp_launch_count).
void note_launches(unsigned long long n);
unsigned long long launch_count();

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launches kernel<<<grid, block, 0, stream>>>(args...) with programmatic
// stream serialization: it may be scheduled while the previous kernel on
// the stream drains, and it waits for that kernel (pdl_wait) before
// touching memory.
template <typename... KArgs, typename... Args>
bool launch_pdl(void (*kernel)(KArgs...), int grid, int block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess;
}


}  // namespace cpmap
