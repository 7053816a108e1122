// cp_variants.cu -- the pages' own strategies, rebuilt as plain CUDA for
// sm_103a so that the optimised kernels can be timed against them (the
// pwwt.cn chapter-18 article's five-way benchmark: sequential, scatter,
// gather, coarsening, coarsening + coalescing; PMPP ch.18 notes sections
// 18.2-18.5).  They compute the same maps as cp_direct (and, for the 27-bin
// kernel, the hard-cutoff map) and are parity-tested, but they are
// comparison baselines, not the fast path:
//   scatter    one thread per atom adds q/r into every grid point with
//              atomicAdd (notes 18.2, article 二);
//   gather     one thread per point; atoms pass through __constant__ memory
//              in chunks of 4000, one launch per chunk, V read and written
//              back each chunk (notes 18.2);
//   coarsen    the same with 4 adjacent x points per thread, dy^2 + dz^2
//              shared (notes 18.3);
//   coalesce   4 points per thread a block-width apart, so neighbouring
//              lanes write neighbouring addresses (article 三);
//   cutoff27   bins of edge c, each point scans its own bin and the 26
//              around it through the bin-sorted (CSR) atom array and adds
//              q/r for r < c, no switching (notes 18.5).
// Because the chunk table is one __constant__ array per device, calls of
// the gather-family variants that overlap on the GPU race.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "cp_device.cuh"
#include "cp_internal.h"

namespace cpmap {

constexpr int kChunkAtoms = 4000;  // 62.5 KiB of the 64 KiB constant bank
__constant__ float4 c_atoms[kChunkAtoms];

struct VariantGrid {
    int nx, ny, nz;
    float ox, oy, oz, h;
    float *V;
};

__global__ void zero_kernel(float *V, long long n) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) V[i] = 0.0f;
}

// one thread per atom, every grid point, atomicAdd
__global__ void scatter_kernel(const float4 *atoms, int n, VariantGrid g) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= n) return;
    const float4 at = atoms[a];
    for (int k = 0; k < g.nz; ++k) {
        const float dz = fmaf((float)k, g.h, g.oz) - at.z;
        for (int j = 0; j < g.ny; ++j) {
            const float dy = fmaf((float)j, g.h, g.oy) - at.y;
            const float dyz2 = fmaf(dy, dy, dz * dz);
            float *row = g.V + ((long long)k * g.ny + j) * g.nx;
            for (int i = 0; i < g.nx; ++i) {
                const float dx = fmaf((float)i, g.h, g.ox) - at.x;
                atomicAdd(&row[i], at.w * sfu_rsqrt(fmaf(dx, dx, dyz2)));
            }
        }
    }
}

// one thread per point over the chunk in constant memory
__global__ void gather_kernel(int n_chunk, VariantGrid g, int first) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = blockIdx.y * blockDim.y + threadIdx.y;
    const int k = blockIdx.z;
    if (i >= g.nx || j >= g.ny) return;
    const float x = fmaf((float)i, g.h, g.ox), y = fmaf((float)j, g.h, g.oy), z = fmaf((float)k, g.h, g.oz);
    float *out = g.V + ((long long)k * g.ny + j) * g.nx + i;
    float v = first ? 0.0f : *out;
    for (int a = 0; a < n_chunk; ++a) {
        const float dx = x - c_atoms[a].x, dy = y - c_atoms[a].y, dz = z - c_atoms[a].z;
        v += c_atoms[a].w * sfu_rsqrt(dx * dx + dy * dy + dz * dz);
    }
    *out = v;
}

// 4 adjacent x points per thread (STRIDE = 1) or 4 points a block-width
// apart (STRIDE = blockDim.x)
template <bool STRIDED>
__global__ void coarse_kernel(int n_chunk, VariantGrid g, int first) {
    const int t = threadIdx.x;
    const int base = STRIDED ? blockIdx.x * blockDim.x * 4 + t : (blockIdx.x * blockDim.x + t) * 4;
    const int step = STRIDED ? (int)blockDim.x : 1;
    const int j = blockIdx.y * blockDim.y + threadIdx.y;
    const int k = blockIdx.z;
    if (j >= g.ny) return;
    const float y = fmaf((float)j, g.h, g.oy), z = fmaf((float)k, g.h, g.oz);
    float *row = g.V + ((long long)k * g.ny + j) * g.nx;
    float x[4], v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int i = base + c * step;
        x[c] = fmaf((float)i, g.h, g.ox);
        v[c] = (first || i >= g.nx) ? 0.0f : row[i];
    }
    for (int a = 0; a < n_chunk; ++a) {
        const float4 at = c_atoms[a];
        const float dy = y - at.y, dz = z - at.z;
        const float dyz2 = dy * dy + dz * dz;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float dx = x[c] - at.x;
            v[c] += at.w * sfu_rsqrt(dx * dx + dyz2);
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int i = base + c * step;
        if (i < g.nx) row[i] = v[c];
    }
}

// one thread per point, 27 bins of edge c around the point's bin
struct Cut27 {
    VariantGrid g;
    float c2;
    int nb[3];
    float bo[3];
    float b;
    const int *start;
    const int *count;
    const float4 *csr;
};

__global__ void cutoff27_kernel(Cut27 p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = blockIdx.y * blockDim.y + threadIdx.y;
    const int k = blockIdx.z;
    if (i >= p.g.nx || j >= p.g.ny) return;
    const float x = fmaf((float)i, p.g.h, p.g.ox), y = fmaf((float)j, p.g.h, p.g.oy);
    const float z = fmaf((float)k, p.g.h, p.g.oz);
    const int bi = (int)floorf(__fdiv_rn(__fsub_rn(x, p.bo[0]), p.b));
    const int bj = (int)floorf(__fdiv_rn(__fsub_rn(y, p.bo[1]), p.b));
    const int bk = (int)floorf(__fdiv_rn(__fsub_rn(z, p.bo[2]), p.b));
    float v = 0.0f;
    for (int dk = -1; dk <= 1; ++dk)
        for (int dj = -1; dj <= 1; ++dj)
            for (int di = -1; di <= 1; ++di) {
                const int u = bi + di, w = bj + dj, s = bk + dk;
                if (u < 0 || w < 0 || s < 0 || u >= p.nb[0] || w >= p.nb[1] || s >= p.nb[2]) continue;
                const int bin = (s * p.nb[1] + w) * p.nb[0] + u;
                const int st = p.start[bin], cnt = p.count[bin];
                for (int t = 0; t < cnt; ++t) {
                    const float4 a = p.csr[st + t];
                    const float dx = x - a.x, dy = y - a.y, dz = z - a.z;
                    const float r2 = dx * dx + dy * dy + dz * dz;
                    if (r2 < p.c2) v += a.w * sfu_rsqrt(r2);
                }
            }
    p.g.V[((long long)k * p.g.ny + j) * p.g.nx + i] = v;
}

}  // namespace cpmap

using namespace cpmap;

extern "C" {

CP_API int cp_direct_variant(int variant, const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin,
                             float h, float *V, void *stream) {
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    if (variant < 0 || variant > 3) return CP_ERR_INVALID_ARGUMENT;
    if (n_atoms < 0 || !V || (n_atoms > 0 && !atoms)) return CP_ERR_INVALID_ARGUMENT;
    if (n_atoms > 0 && !aligned(atoms, 16)) return CP_ERR_MISALIGNED;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    if (nz > 65535) return CP_ERR_TOO_LARGE;  // grid z dimension of the launches
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const VariantGrid vg{g.nx, g.ny, g.nz, g.ox, g.oy, g.oz, g.h, V};
    const float4 *a4 = reinterpret_cast<const float4 *>(atoms);
    unsigned long long launches = 0;
    if (variant == 0 || n_atoms == 0) {
        zero_kernel<<<(unsigned)std::min<long long>((g.npoints + 255) / 256, 4096), 256, 0, s>>>(V, g.npoints);
        ++launches;
        if (variant == 0 && n_atoms > 0) {
            scatter_kernel<<<(n_atoms + 127) / 128, 128, 0, s>>>(a4, n_atoms, vg);
            ++launches;
        }
    } else {
        for (int off = 0; off < n_atoms; off += kChunkAtoms) {
            const int nch = std::min(kChunkAtoms, n_atoms - off);
            if (cudaMemcpyToSymbolAsync(c_atoms, a4 + off, (size_t)nch * 16, 0, cudaMemcpyDeviceToDevice, s) !=
                cudaSuccess)
                return CP_ERR_CUDA;
            const int first = off == 0;
            if (variant == 1) {
                const dim3 block(32, 4);
                const dim3 grid((nx + 31) / 32, (ny + 3) / 4, nz);
                gather_kernel<<<grid, block, 0, s>>>(nch, vg, first);
            } else {
                const dim3 block(32, 4);
                const dim3 grid((nx + 127) / 128, (ny + 3) / 4, nz);
                if (variant == 2)
                    coarse_kernel<false><<<grid, block, 0, s>>>(nch, vg, first);
                else
                    coarse_kernel<true><<<grid, block, 0, s>>>(nch, vg, first);
            }
            ++launches;
        }
    }
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(launches);
    return CP_OK;
}

CP_API size_t cp_cutoff27_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                          float cutoff) {
    return cp_cutoff_workspace_bytes(n_atoms, nx, ny, nz, origin, h, cutoff, cutoff, 0);
}

CP_API int cp_cutoff27(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                       float cutoff, void *workspace, size_t workspace_bytes, float *V, void *stream) {
    if (!V) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    if (nz > 65535) return CP_ERR_TOO_LARGE;
    cp_cutoff_layout L;
    int rc = cp_cutoff_layout_of(n_atoms, nx, ny, nz, origin, h, cutoff, cutoff, 0, &L);
    if (rc) return rc;
    rc = cp_bin_atoms(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, cutoff, 0, workspace, workspace_bytes, stream);
    if (rc) return rc;
    Grid g;
    check_grid(nx, ny, nz, origin, h, &g);
    const char *ws = static_cast<const char *>(workspace);
    Cut27 p;
    p.g = VariantGrid{g.nx, g.ny, g.nz, g.ox, g.oy, g.oz, g.h, V};
    p.c2 = (float)((double)cutoff * (double)cutoff);
    for (int d = 0; d < 3; ++d) {
        p.nb[d] = L.nb[d];
        p.bo[d] = L.bo[d];
    }
    p.b = cutoff;
    p.start = reinterpret_cast<const int *>(ws + L.off_start);
    p.count = reinterpret_cast<const int *>(ws + L.off_count);
    p.csr = reinterpret_cast<const float4 *>(ws + L.off_csr_atoms);
    const dim3 block(32, 4);
    const dim3 grid((nx + 31) / 32, (ny + 3) / 4, nz);
    cutoff27_kernel<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(p);
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

}  // extern "C"
