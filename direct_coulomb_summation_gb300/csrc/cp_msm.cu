// cp_msm.cu -- long-range part of a multilevel summation on sm_103a.
//
// The Input Binning lecture's slide "Large Bin Cut-off Kernel Code" (24)
// names its cutoff kernel mgpot_shortrng_energy: the switched sum that
// cp_cutoff computes is the short-range part of a multilevel summation of
// 1/r.  The smooth remainder V_long(x) = sum_a q_a g_c(|x - r_a|) (g_c = the
// switching polynomial inside c, 1/r beyond) is approximated here on nested
// lattices (R. D. Skeel, I. Tezcan, D. J. Hardy, "Multiple grid methods for
// classical molecular dynamics", J. Comput. Chem. 23 (2002); D. J. Hardy,
// J. E. Stone, K. Schulten, "Multilevel summation of electrostatic
// potentials using graphics processing units", Parallel Computing 35
// (2009)).  The pages do not describe this part.
//
// GPU mapping:
//   * anterpolation as a gather: the atoms are counting-sorted into the
//     level-0 lattice cells (the cutoff path's binning kernels), then every
//     node sums the atoms of the 4x4x4 cells its basis function covers, in
//     a fixed order -- no atomics, deterministic;
//   * charge lattices are stored with R zero nodes of padding on every side
//     (z rounded up to whole 8-node columns), so the lattice-cutoff stencil
//     reads them without bounds checks;
//   * lattice cutoff: a thread owns 8 nodes stacked in z in each of two
//     neighbouring y columns and walks the stencil column by column (fixed
//     dy, dx; dz innermost).  Charge lattices store each node with its +y
//     neighbour, (q(x,y,z), q(x,y+1,z)), and a power-of-two z stride that
//     is a compile-time constant, so each tap is one coalesced 8-byte load
//     at an immediate offset (the next pair of a sliding 8-node window),
//     one uniform load of the weight pair (w, w) and 8 f32x2 FMAs.  All levels below the top run in one
//     launch; the stencil columns of a tile are split over S CTAs whose
//     partial sums are added in a fixed order afterwards;
//   * top level: one warp per node, lanes split the other nodes, kernel
//     values from a table indexed by |d|^2, a fixed-order warp reduction;
//   * prolongation fused with that partial-sum reduction, level by level
//     from the top down;
//   * interpolation: a thread owns 4 consecutive x points of one row (a
//     float4 of V); it sums the lattice columns its points share once.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>

#include "cp_device.cuh"
#include "cp_internal.h"

namespace cpmap {

constexpr int kMsmMaxLevels = CP_MSM_MAX_LEVELS;
constexpr int kMsmMaxRadius = CP_MSM_MAX_RADIUS;
constexpr int kMsmSide = 2 * kMsmMaxRadius + 1;
constexpr int kMsmTopNodes = 12;                              // top level: at most 12 nodes per axis
constexpr int kMsmTopTable = 3 * (kMsmTopNodes - 1) * (kMsmTopNodes - 1) + 1;  // |d|^2 values
constexpr int kMsmZ = 8;                                      // nodes a lattice-cutoff thread stacks in z
constexpr long long kMsmTargetThreads = 1LL << 17;            // lattice-cutoff threads worth splitting for
constexpr int kMsmMaxSplit = 64;
constexpr int kMsmThreads = 128;
constexpr int kReduceGroup = 8;  // lanes per node in the partial-sum reduction of heavily split levels
constexpr long long kMsmMinPlane = 1024;     // z-plane strides of the charge lattices: powers of two
constexpr long long kMsmMaxPlane = 1 << 18;  // in this range, each a compile-time constant of the stencil loop

namespace {

// ---------------------------------------------------------------------------
// device helpers

// The C1 cubic interpolating basis function, support |t| < 2, without
// branches: both pieces are evaluated and the right one selected.
__device__ __forceinline__ float msm_phi(float t) {
    const float a = fabsf(t);
    const float b = 2.0f - a;
    const float inner = (1.0f - a) * fmaf(-1.5f * a, a, 1.0f + a);
    const float outer = -0.5f * (a - 1.0f) * b * b;
    return a <= 1.0f ? inner : (a <= 2.0f ? outer : 0.0f);
}

// phi(t) for |t| <= 2 (a node and an atom or point of one of the four cells
// around it): one cubic in a = |t| whose coefficients are chosen by a <= 1,
// 1 - 5a^2/2 + 3a^3/2 inside, 2 - 4a + 5a^2/2 - a^3/2 outside.
__device__ __forceinline__ float msm_phi_near(float t) {
    const float a = fabsf(t);
    const bool in = a <= 1.0f;
    const float c3 = in ? 1.5f : -0.5f, c2 = in ? -2.5f : 2.5f, c1 = in ? 0.0f : -4.0f, c0 = in ? 1.0f : 2.0f;
    return fmaf(fmaf(fmaf(c3, a, c2), a, c1), a, c0);
}

// g_c(r) = gamma(r/c)/c in fp64 with explicit roundings (no contraction).
__device__ double msm_g64(double r, double c) {
    const double s = __ddiv_rn(r, c);
    if (s < 1.0) {
        const double s2 = __dmul_rn(s, s);
        const double p = __dadd_rn(__dadd_rn(1.875, __dmul_rn(-1.25, s2)), __dmul_rn(0.375, __dmul_rn(s2, s2)));
        return __ddiv_rn(p, c);
    }
    return __ddiv_rn(1.0, r);
}

// Lattice coordinate of x relative to the lattice origin, in units of h0:
// the same fp32 expression the cell sort uses for the cell index.
__device__ __forceinline__ float msm_t(float x, float o, float h0) { return __fdiv_rn(__fsub_rn(x, o), h0); }

struct MsmLevelDev {
    int lo[3], n[3];
    int qd[3];              // padded charge lattice dims (x, y, z)
    float2 *q;              // padded charges as pairs (q(x,y,z), q(x,y+1,z)), [z][plane]
    int plane;              // entries per z plane: a power of two >= qd[0] * qd[1]
    float *e;               // potentials [n z][n y][n x]
    float *part;            // partial sums [split][n z][n y][n x]
    int split;
    long long cols;         // lattice-cutoff threads of this level (x * y * z-stacks)
    long long cta_begin;    // first lattice-cutoff CTA of this level
    float scale;            // 2^-l
};

struct MsmParams {
    int levels;  // L + 1
    MsmLevelDev lv[kMsmMaxLevels];
    int R;
    float2 *W;     // [2R+1]^3 stencil as pairs (w, w), symmetric in its three indices
    float *gtop;   // top-level kernel by |d|^2
    int cells[3];
    float o[3];
    float h0;
    const int *cell_start;
    const float4 *cell_atoms;
    float4 *cell_t;  // per cell-sorted atom: lattice coordinates (t x, t y, t z) and q
    long long ncells;
    int n_atoms;
    const int *cell_stats;
    unsigned int *status;
    double h0_64, a64, lim2;
    int8_t hw[kMsmSide * kMsmSide];  // stencil column (dy, dx) half height in dz, -1 if empty
};

// Writes charge q of padded entry (x, y, z): as the first half of its own
// pair and the second half of the pair of (x, y-1, z); the last row's
// second halves (beyond the lattice) are zero.
__device__ __forceinline__ void msm_store_pair(const MsmLevelDev &L, int x, int y, int z, float q,
                                               unsigned int *status) {
    const long long at = (long long)z * L.plane + (long long)y * L.qd[0] + x;
    if (!CP_IN(at, (long long)L.plane * L.qd[2], status) ||
        (y > 0 && !CP_IN(at - L.qd[0], (long long)L.plane * L.qd[2], status)))
        return;
    float2 *base = L.q + (long long)z * L.plane + x;
    float *own = reinterpret_cast<float *>(base + (long long)y * L.qd[0]);
    own[0] = q;
    if (y > 0) own[1 - 2 * L.qd[0]] = q;  // .y of the entry one row down
    if (y == L.qd[1] - 1) own[1] = 0.0f;
}

// ---------------------------------------------------------------------------
// kernels

// W(d) = g_c(|d| h0) - g_2c(|d| h0) for |d|^2 < (2c/h0)^2, else 0; and the
// top-level table 2^-L g_c(sqrt(s) h0) for s = 0 .. 3*11^2.
__global__ void msm_stencil_kernel(const __grid_constant__ MsmParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int side = 2 * p.R + 1;
    const int n = side * side * side;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n + kMsmTopTable; idx += stride) {
        if (idx < n) {
            const int dx = (int)(idx % side) - p.R;
            const int dy = (int)((idx / side) % side) - p.R;
            const int dz = (int)(idx / ((long long)side * side)) - p.R;
            const int s2 = dx * dx + dy * dy + dz * dz;
            float w = 0.0f;
            if ((double)s2 < p.lim2) {
                const double r = __dmul_rn(__dsqrt_rn((double)s2), p.h0_64);
                w = (float)__dsub_rn(msm_g64(r, p.a64), msm_g64(r, 2.0 * p.a64));
            }
            p.W[idx] = make_float2(w, w);
        } else {
            const int s2 = (int)(idx - n);
            const int L = p.levels - 1;
            const double r = __dmul_rn(__dsqrt_rn((double)s2), p.h0_64);
            p.gtop[s2] = (float)ldexp(msm_g64(r, p.a64), -L);
        }
    }
}

// Lattice coordinates t = (r - o)/h0 of every cell-sorted atom, once per
// atom (the same fp32 expression as the cell index), with its charge.
__global__ void __launch_bounds__(kMsmThreads) msm_tcoord_kernel(const __grid_constant__ MsmParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= p.cell_start[p.ncells]) return;
    const float4 a = p.cell_atoms[t];
    p.cell_t[t] = make_float4(msm_t(a.x, p.o[0], p.h0), msm_t(a.y, p.o[1], p.h0), msm_t(a.z, p.o[2], p.h0), a.w);
}

// q0 at every level-0 node (the padding was zeroed before): the sum over
// the atoms of the cells i-2 .. i+1 (per axis) of q Phi(t - i), in cell
// order.  One thread per node, nodes x fastest.
__global__ void __launch_bounds__(kMsmThreads) msm_anterp_kernel(const __grid_constant__ MsmParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const MsmLevelDev &L0 = p.lv[0];
    const long long total = (long long)L0.n[0] * L0.n[1] * L0.n[2];
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx == 0 && p.cell_stats[1] != 0) atomicOr(p.status, CP_DEVICE_ATOMS_OUTSIDE);  // dropped by the sort
    if (idx >= total) return;
    const int ax = (int)(idx % L0.n[0]);
    const int ay = (int)((idx / L0.n[0]) % L0.n[1]);
    const int az = (int)(idx / ((long long)L0.n[0] * L0.n[1]));
    const int i = ax + L0.lo[0], j = ay + L0.lo[1], k = az + L0.lo[2];  // node index
    const float fi = (float)i, fj = (float)j, fk = (float)k;
    const int cx0 = max(i - 2, 0), cx1 = min(i + 1, p.cells[0] - 1);
    const int cy0 = max(j - 2, 0), cy1 = min(j + 1, p.cells[1] - 1);
    const int cz0 = max(k - 2, 0), cz1 = min(k + 1, p.cells[2] - 1);
    float acc = 0.0f;
    if (cx0 <= cx1) {
        for (int cz = cz0; cz <= cz1; ++cz)
            for (int cy = cy0; cy <= cy1; ++cy) {
                const long long row = ((long long)cz * p.cells[1] + cy) * p.cells[0];
                const int b = p.cell_start[row + cx0], e = p.cell_start[row + cx1 + 1];
                if (e > b && !(CP_IN(b, p.n_atoms, p.status) && CP_IN(e - 1, p.n_atoms, p.status))) continue;
                for (int t = b; t < e; ++t) {
                    const float4 a = p.cell_t[t];
                    acc = fmaf(a.w, msm_phi_near(a.x - fi) * msm_phi_near(a.y - fj) * msm_phi_near(a.z - fk), acc);
                }
            }
    }
    msm_store_pair(L0, ax + p.R, ay + p.R, az + p.R, acc, p.status);
}

// Restriction weights phi(k/2) for fine offsets k = -3 .. 3 (k = +-2 weigh 0).
__device__ __forceinline__ float msm_rw(int k) {
    switch (k) {
        case 0: return 1.0f;
        case 1:
        case -1: return 0.5625f;
        case 3:
        case -3: return -0.0625f;
        default: return 0.0f;
    }
}

// q(l+1) at every padded entry: zero in the padding, else
// sum_k w(kx) w(ky) w(kz) q(l)[2J + k] over the fine nodes that exist.
__global__ void __launch_bounds__(kMsmThreads) msm_restrict_kernel(const __grid_constant__ MsmParams p, int l) {
    pdl_launch_dependents();
    pdl_wait();
    const MsmLevelDev &F = p.lv[l];
    const MsmLevelDev &C = p.lv[l + 1];
    const long long total = (long long)C.qd[0] * C.qd[1] * C.qd[2];
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int px = (int)(idx % C.qd[0]);
    const int py = (int)((idx / C.qd[0]) % C.qd[1]);
    const int pz = (int)(idx / ((long long)C.qd[0] * C.qd[1]));
    const int ax = px - p.R, ay = py - p.R, az = pz - p.R;
    float acc = 0.0f;
    if (ax >= 0 && ax < C.n[0] && ay >= 0 && ay < C.n[1] && az >= 0 && az < C.n[2]) {
        const int J[3] = {ax + C.lo[0], ay + C.lo[1], az + C.lo[2]};
        const int fx0 = 2 * J[0] - F.lo[0], fy0 = 2 * J[1] - F.lo[1], fz0 = 2 * J[2] - F.lo[2];
        constexpr int kOff[5] = {-3, -1, 0, 1, 3};
#pragma unroll
        for (int c = 0; c < 5; ++c) {
            const int fz = fz0 + kOff[c];
            float sz = 0.0f;
#pragma unroll
            for (int b = 0; b < 5; ++b) {
                const int fy = fy0 + kOff[b];
                const bool zy_in = fz >= 0 && fz < F.n[2] && fy >= 0 && fy < F.n[1];
                const float2 *row = F.q + (long long)(fz + p.R) * F.plane + (long long)(fy + p.R) * F.qd[0] + p.R;
                float sy = 0.0f;
#pragma unroll
                for (int a = 0; a < 5; ++a) {
                    const int fx = fx0 + kOff[a];
                    const float v = (zy_in && fx >= 0 && fx < F.n[0]) ? row[fx].x : 0.0f;
                    sy = fmaf(msm_rw(kOff[a]), v, sy);
                }
                sz = fmaf(msm_rw(kOff[b]), sy, sz);
            }
            acc = fmaf(msm_rw(kOff[c]), sz, acc);
        }
    }
    msm_store_pair(C, px, py, pz, acc, p.status);
}

// Lattice cutoff of every level below the top.  CTA -> (level, tile,
// split); thread -> node columns (x, y0) and (x, y0 + 1), 8 nodes z0 .. z0+7
// of each, the two columns' sums held as f32x2 pairs.  Split s of S takes
// the stencil columns c = s, s + S, ...; a column (dy, dx) covers
// dz = -hw .. hw.  Each charge entry holds the pair (q(x,y,z), q(x,y+1,z)),
// so a tap is one 8-byte load; PLANE (the z stride) is a compile-time
// constant, so the loads of an unrolled group of 8 taps use immediate
// offsets.  The padded charge lattice makes every read in range.
template <int PLANE>
__device__ __forceinline__ void msm_conv_tile(const MsmParams &p, const MsmLevelDev &Lv, int s, long long col) {
    const int ny2 = (Lv.n[1] + 1) / 2;
    const int x = (int)(col % Lv.n[0]);
    const int y0 = 2 * (int)((col / Lv.n[0]) % ny2);
    const int z0 = (int)(col / ((long long)Lv.n[0] * ny2)) * kMsmZ;
    const int R = p.R, side = 2 * R + 1;
    const int pitch = Lv.qd[0];
    const float2 *base = Lv.q + (long long)(z0 + R) * PLANE + (long long)(y0 + R) * pitch + (x + R);
    float2 acc[kMsmZ];
#pragma unroll
    for (int t = 0; t < kMsmZ; ++t) acc[t] = make_float2(0.0f, 0.0f);
    const int ncols = side * side;
    for (int c = s; c < ncols; c += Lv.split) {
        const int hw = p.hw[c];
        if (hw < 0) continue;
        const int dy = c / side - R, dx = c % side - R;
        const int taps = 2 * hw + 1;
        // q[m * PLANE] = node pair z0 + m - hw of column (x + dx, y0 + dy);
        // w[m] = (W, W) at dz = m - hw
        const float2 *q = base + dy * pitch + dx - hw * PLANE;
        const float2 *w = p.W + c * side + R - hw;
        if (!CP_IN(q - Lv.q, (long long)PLANE * Lv.qd[2], p.status) ||
            !CP_IN(q - Lv.q + (long long)(taps + kMsmZ - 2) * PLANE, (long long)PLANE * Lv.qd[2], p.status) ||
            !CP_IN(w - p.W + taps - 1, (long long)side * side * side, p.status))
            continue;
        // ring of 8 pairs: slot j holds the window node m' = j (mod 8), so
        // no register moves are needed
        float2 r[kMsmZ];
#pragma unroll
        for (int j = 0; j < kMsmZ - 1; ++j) r[j] = q[j * PLANE];
        q += (kMsmZ - 1) * PLANE;
        int m = 0;
        for (; m + kMsmZ <= taps; m += kMsmZ) {  // whole groups of 8 taps
#pragma unroll
            for (int k = 0; k < kMsmZ; ++k) {
                r[(k + kMsmZ - 1) & (kMsmZ - 1)] = q[k * PLANE];
                const float2 wd = __ldg(w + k);
#pragma unroll
                for (int t = 0; t < kMsmZ; ++t) acc[t] = __ffma2_rn(wd, r[(k + t) & (kMsmZ - 1)], acc[t]);
            }
            q += kMsmZ * PLANE;
            w += kMsmZ;
        }
#pragma unroll
        for (int k = 0; k < kMsmZ - 1; ++k) {  // the remaining taps - m < 8
            if (m + k < taps) {  // uniform across the warp
                r[(k + kMsmZ - 1) & (kMsmZ - 1)] = q[k * PLANE];
                const float2 wd = __ldg(w + k);
#pragma unroll
                for (int t = 0; t < kMsmZ; ++t) acc[t] = __ffma2_rn(wd, r[(k + t) & (kMsmZ - 1)], acc[t]);
            }
        }
    }
    const long long nodes = (long long)Lv.n[0] * Lv.n[1] * Lv.n[2];
    const long long zs = (long long)Lv.n[0] * Lv.n[1];
    float *out = Lv.part + (long long)s * nodes + (long long)y0 * Lv.n[0] + x;
    const bool y1 = y0 + 1 < Lv.n[1];
    if (!CP_IN(s, Lv.split, p.status)) return;
#pragma unroll
    for (int t = 0; t < kMsmZ; ++t)
        if (z0 + t < Lv.n[2]) {
            out[(long long)(z0 + t) * zs] = acc[t].x;
            if (y1) out[(long long)(z0 + t) * zs + Lv.n[0]] = acc[t].y;
        }
}

__global__ void __launch_bounds__(kMsmThreads) msm_conv_kernel(const __grid_constant__ MsmParams p) {
    pdl_launch_dependents();
    pdl_wait();
    int l = 0;
    while (l + 2 < p.levels && (long long)blockIdx.x >= p.lv[l + 1].cta_begin) ++l;
    const MsmLevelDev &Lv = p.lv[l];
    const long long local = (long long)blockIdx.x - Lv.cta_begin;
    const int s = (int)(local % Lv.split);
    const long long col = (local / Lv.split) * kMsmThreads + threadIdx.x;
    if (col >= Lv.cols) return;
    switch (Lv.plane) {
        case 1 << 10: msm_conv_tile<1 << 10>(p, Lv, s, col); break;
        case 1 << 11: msm_conv_tile<1 << 11>(p, Lv, s, col); break;
        case 1 << 12: msm_conv_tile<1 << 12>(p, Lv, s, col); break;
        case 1 << 13: msm_conv_tile<1 << 13>(p, Lv, s, col); break;
        case 1 << 14: msm_conv_tile<1 << 14>(p, Lv, s, col); break;
        case 1 << 15: msm_conv_tile<1 << 15>(p, Lv, s, col); break;
        case 1 << 16: msm_conv_tile<1 << 16>(p, Lv, s, col); break;
        case 1 << 17: msm_conv_tile<1 << 17>(p, Lv, s, col); break;
        default: msm_conv_tile<1 << 18>(p, Lv, s, col); break;
    }
}

// Top level: e_i = sum_j gtop[|i - j|^2] q_j over all top nodes; one warp
// per node, lanes take every 32nd node, fixed-order reduction.
__global__ void __launch_bounds__(kMsmThreads) msm_top_kernel(const __grid_constant__ MsmParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const MsmLevelDev &T = p.lv[p.levels - 1];
    const int nodes = T.n[0] * T.n[1] * T.n[2];
    const int node = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (node >= nodes) return;
    const int ix = node % T.n[0], iy = (node / T.n[0]) % T.n[1], iz = node / (T.n[0] * T.n[1]);
    float acc = 0.0f;
    // lane takes the top-level rows (jy, jz) = lane, lane + 32, ...; a row is
    // summed over jx in order
    const int rows = T.n[1] * T.n[2];
    for (int rj = lane; rj < rows; rj += 32) {
        const int jy = rj % T.n[1], jz = rj / T.n[1];
        const int dy = iy - jy, dz = iz - jz;
        const int d2 = dy * dy + dz * dz;
        const float2 *q = T.q + (long long)(jz + p.R) * T.plane + (long long)(jy + p.R) * T.qd[0] + p.R;
        if (!CP_IN(q - T.q + T.n[0] - 1, (long long)T.plane * T.qd[2], p.status)) continue;
        for (int jx = 0; jx < T.n[0]; ++jx) {
            const int dx = ix - jx;
            if (CP_IN(d2 + dx * dx, kMsmTopTable, p.status)) acc = fmaf(p.gtop[d2 + dx * dx], q[jx].x, acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
    if (lane == 0) T.e[node] = acc;
}

// Prolongation weight phi(i/2 - J) for fine index i and coarse index J.
__device__ __forceinline__ int msm_prolong_taps(int i, int J0[4], float w[4]) {
    if ((i & 1) == 0) {
        J0[0] = i / 2;
        w[0] = 1.0f;
        return 1;
    }
    const int h = (i - 1) >> 1;  // floor(i/2) for odd i, also negative
    J0[0] = h - 1;
    w[0] = -0.0625f;
    J0[1] = h;
    w[1] = 0.5625f;
    J0[2] = h + 1;
    w[2] = 0.5625f;
    J0[3] = h + 2;
    w[3] = -0.0625f;
    return 4;
}

// e(l) = 2^-l * (sum of the S partial sums, in split order) + the level-l+1
// potentials interpolated to the level-l nodes.
__global__ void __launch_bounds__(kMsmThreads) msm_reduce_prolong_kernel(const __grid_constant__ MsmParams p, int l) {
    pdl_launch_dependents();
    pdl_wait();
    const MsmLevelDev &F = p.lv[l];
    const MsmLevelDev &C = p.lv[l + 1];
    const long long nodes = (long long)F.n[0] * F.n[1] * F.n[2];
    // G consecutive lanes share a node when the split is large: lane g adds
    // partials g, g + G, ... and the G sums meet by a fixed shuffle tree
    const int G = F.split >= 16 ? kReduceGroup : 1;
    const long long gidx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long idx = gidx / G;
    const int g = (int)(gidx % G);
    float s = 0.0f;
    if (idx < nodes)
        for (int k = g; k < F.split; k += G) s += F.part[(long long)k * nodes + idx];
    if (G > 1) {
#pragma unroll
        for (int o = kReduceGroup / 2; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o, kReduceGroup);
    }
    if (idx >= nodes || g != 0) return;
    const int ax = (int)(idx % F.n[0]);
    const int ay = (int)((idx / F.n[0]) % F.n[1]);
    const int az = (int)(idx / ((long long)F.n[0] * F.n[1]));
    int Jx[4], Jy[4], Jz[4];
    float wx[4], wy[4], wz[4];
    const int nx = msm_prolong_taps(ax + F.lo[0], Jx, wx);
    const int ny = msm_prolong_taps(ay + F.lo[1], Jy, wy);
    const int nz = msm_prolong_taps(az + F.lo[2], Jz, wz);
    float pr = 0.0f;
    for (int c = 0; c < nz; ++c) {
        const int cz = Jz[c] - C.lo[2];
        if (cz < 0 || cz >= C.n[2]) continue;
        for (int b = 0; b < ny; ++b) {
            const int cy = Jy[b] - C.lo[1];
            if (cy < 0 || cy >= C.n[1]) continue;
            const float *row = C.e + ((long long)cz * C.n[1] + cy) * C.n[0];
            float r = 0.0f;
            for (int a = 0; a < nx; ++a) {
                const int cx = Jx[a] - C.lo[0];
                if (cx >= 0 && cx < C.n[0]) r = fmaf(wx[a], row[cx], r);
            }
            pr = fmaf(wz[c] * wy[b], r, pr);
        }
    }
    F.e[idx] = fmaf(F.scale, s, pr);
}

struct InterpParams {
    int nx, ny, nz;
    // grid origin minus lattice origin (rounded once on the host): a point's
    // offset from the lattice origin is i*h + this, formed with one fused
    // multiply-add, so its rounding follows the offset, not the distance of
    // the grid from the coordinate origin
    float dox, doy, doz, h;
    long long quads;
    int qx;
    float *V;
    int accumulate;
};

template <bool VEC>
__global__ void __launch_bounds__(kMsmThreads) msm_interp_kernel(const __grid_constant__ MsmParams p,
                                                                  const __grid_constant__ InterpParams g) {
    pdl_launch_dependents();
    pdl_wait();
    const long long quad = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (quad >= g.quads) return;
    const int qx = (int)(quad % g.qx);
    const int j = (int)((quad / g.qx) % g.ny);
    const int k = (int)(quad / ((long long)g.qx * g.ny));
    const int i0 = 4 * qx;
    const MsmLevelDev &L0 = p.lv[0];
    const float ty = __fdiv_rn(fmaf((float)j, g.h, g.doy), p.h0);
    const float tz = __fdiv_rn(fmaf((float)k, g.h, g.doz), p.h0);
    const int ky = (int)floorf(ty), kz = (int)floorf(tz);
    float wy[4], wz[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        wy[b] = msm_phi(ty - (float)(ky - 1 + b));
        wz[b] = msm_phi(tz - (float)(kz - 1 + b));
    }
    float tx[4];
    int kx[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        tx[c] = __fdiv_rn(fmaf((float)min(i0 + c, g.nx - 1), g.h, g.dox), p.h0);
        kx[c] = (int)floorf(tx[c]);
    }
    // node (i, j, k) of level 0 at e[(k - lo z) ...]
    const float *e = L0.e;
    const int n0 = L0.n[0], n1 = L0.n[1], n2 = L0.n[2];
    auto column = [&](int ix) {  // sum over the 4x4 (y, z) nodes of lattice column ix
        float s = 0.0f;
        const int ax = ix - L0.lo[0];
        if (ax < 0 || ax >= n0) return s;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int az = kz - 1 + c - L0.lo[2];
            if (az < 0 || az >= n2) continue;
            float r = 0.0f;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int ay = ky - 1 + b - L0.lo[1];
                if (ay >= 0 && ay < n1) r = fmaf(wy[b], e[((long long)az * n1 + ay) * n0 + ax], r);
            }
            s = fmaf(wz[c], r, s);
        }
        return s;
    };
    float v[4];
    const int kmin = kx[0], kmax = kx[3];
    if (kmax - kmin <= 3) {
        float cols[7];
#pragma unroll
        for (int m = 0; m < 7; ++m) cols[m] = (m <= kmax - kmin + 3) ? column(kmin - 1 + m) : 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float s = 0.0f;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int m = kx[c] - kmin + a;
                float cv = 0.0f;
#pragma unroll
                for (int mm = 0; mm < 7; ++mm) cv = (mm == m) ? cols[mm] : cv;
                s = fmaf(msm_phi(tx[c] - (float)(kx[c] - 1 + a)), cv, s);
            }
            v[c] = s;
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float s = 0.0f;
            for (int a = 0; a < 4; ++a) s = fmaf(msm_phi(tx[c] - (float)(kx[c] - 1 + a)), column(kx[c] - 1 + a), s);
            v[c] = s;
        }
    }
    float *row = g.V + ((long long)k * g.ny + j) * g.nx;
    if (VEC) {
        float4 *dst = reinterpret_cast<float4 *>(row + i0);
        float4 out = make_float4(v[0], v[1], v[2], v[3]);
        if (g.accumulate) {
            const float4 old = *dst;
            out.x += old.x;
            out.y += old.y;
            out.z += old.z;
            out.w += old.w;
        }
        *dst = out;
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (i0 + c < g.nx) row[i0 + c] = g.accumulate ? row[i0 + c] + v[c] : v[c];
    }
}

// Interpolation for grid spacings h <= h0: one CTA per 8x8x8-point brick.
// The brick's points need at most SPAN level-0 nodes per axis; those are
// staged in shared memory and the tensor-product sum is done one axis at a
// time (z, then y, then x), so a point costs about 12 FMAs instead of 64.
// SPAN is a compile-time bound (6, 8 or 12) so that the staging loops index
// with constant divisors.
template <int SPAN>
__global__ void __launch_bounds__(kMsmThreads) msm_interp_brick_kernel(const __grid_constant__ MsmParams p,
                                                                        const __grid_constant__ InterpParams g) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float E[SPAN][SPAN][SPAN];     // [z][y][x] nodes around the brick
    __shared__ float S1[kBrick][SPAN][SPAN];  // [point z][node y][node x]
    __shared__ float S2[kBrick][kBrick][SPAN];  // [point z][point y][node x]
    __shared__ float wgt[3][kBrick][4];
    __shared__ int off[3][kBrick];
    __shared__ int base[3], cnt[3];
    __shared__ int bad;

    const int tid = threadIdx.x;
    const int nbx = (g.nx + kBrick - 1) / kBrick, nby = (g.ny + kBrick - 1) / kBrick;
    const int bx = blockIdx.x % nbx, by = (blockIdx.x / nbx) % nby, bz = blockIdx.x / (nbx * nby);
    const MsmLevelDev &L0 = p.lv[0];
    if (tid == 0) bad = 0;
    __syncthreads();
    if (tid < 3 * kBrick) {
        // per axis d and point pt of the brick: node offset and the 4 weights
        const int d = tid / kBrick, pt = tid % kBrick;
        const int n = d == 0 ? g.nx : (d == 1 ? g.ny : g.nz);
        const int b = d == 0 ? bx : (d == 1 ? by : bz);
        const float o = d == 0 ? g.dox : (d == 1 ? g.doy : g.doz);
        const int idx = min(kBrick * b + pt, n - 1);  // points past the edge repeat the last one
        // lattice coordinate of the point: weights only, so a reciprocal
        // multiply suffices (the cell sort's exact division is for atoms)
        const float inv_h0 = 1.0f / p.h0;
        const float t = fmaf((float)idx, g.h, o) * inv_h0;
        const int k = min(max((int)floorf(t), 0), p.cells[d] - 1);
        const float t0 = fmaf((float)(kBrick * b), g.h, o) * inv_h0;
        const int k0 = min(max((int)floorf(t0), 0), p.cells[d] - 1);
        off[d][pt] = k - k0;
        for (int a = 0; a < 4; ++a) wgt[d][pt][a] = msm_phi(t - (float)(k - 1 + a));
        if (pt == kBrick - 1) {
            base[d] = k0 - 1 - L0.lo[d];  // array index of the first node
            cnt[d] = k - k0 + 4;
            if (k - k0 + 4 > SPAN || k < k0) atomicOr(&bad, 1);
        }
    }
    __syncthreads();
    if (bad) {  // the host picks SPAN from h/h0; recorded rather than trusted
        if (tid == 0) atomicOr(p.status, CP_DEVICE_RANGE);
        return;
    }
    const int cx = cnt[0], cy = cnt[1], cz = cnt[2];
    for (int e = tid; e < SPAN * SPAN * SPAN; e += kMsmThreads) {
        const int ex = e % SPAN, ey = (e / SPAN) % SPAN, ez = e / (SPAN * SPAN);
        if (ex < cx && ey < cy && ez < cz) {
            const int gx = base[0] + ex, gy = base[1] + ey, gz = base[2] + ez;
            const bool in = gx >= 0 && gx < L0.n[0] && gy >= 0 && gy < L0.n[1] && gz >= 0 && gz < L0.n[2];
            E[ez][ey][ex] = in ? L0.e[((long long)gz * L0.n[1] + gy) * L0.n[0] + gx] : 0.0f;
        }
    }
    __syncthreads();
    for (int e = tid; e < kBrick * SPAN * SPAN; e += kMsmThreads) {  // along z
        const int ex = e % SPAN, ey = (e / SPAN) % SPAN, pz = e / (SPAN * SPAN);
        if (ex < cx && ey < cy) {
            const int o = off[2][pz];
            float v = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) v = fmaf(wgt[2][pz][c], E[o + c][ey][ex], v);
            S1[pz][ey][ex] = v;
        }
    }
    __syncthreads();
    for (int e = tid; e < kBrick * kBrick * SPAN; e += kMsmThreads) {  // along y
        const int ex = e % SPAN, py = (e / SPAN) % kBrick, pz = e / (SPAN * kBrick);
        if (ex < cx) {
            const int o = off[1][py];
            float v = 0.0f;
#pragma unroll
            for (int b = 0; b < 4; ++b) v = fmaf(wgt[1][py][b], S1[pz][o + b][ex], v);
            S2[pz][py][ex] = v;
        }
    }
    __syncthreads();
    // along x: thread -> 4 consecutive points of one brick row
    const int half = tid & 1, py = (tid >> 1) & (kBrick - 1), pz = tid >> 4;
    float v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int px = 4 * half + c;
        const int o = off[0][px];
        float s = 0.0f;
#pragma unroll
        for (int a = 0; a < 4; ++a) s = fmaf(wgt[0][px][a], S2[pz][py][o + a], s);
        v[c] = s;
    }
    const int i0 = kBrick * bx + 4 * half, j = kBrick * by + py, k = kBrick * bz + pz;
    if (i0 >= g.nx || j >= g.ny || k >= g.nz) return;  // half-rows past the grid store nothing
    if (!CP_IN(((long long)k * g.ny + j) * g.nx + i0, (long long)g.nx * g.ny * g.nz, p.status)) return;
    float *row = g.V + ((long long)k * g.ny + j) * g.nx;
    if (i0 + 3 < g.nx && (g.nx % 4 == 0) && ((reinterpret_cast<uintptr_t>(g.V) & 15) == 0)) {
        float4 *dst = reinterpret_cast<float4 *>(row + i0);
        float4 out = make_float4(v[0], v[1], v[2], v[3]);
        if (g.accumulate) {
            const float4 old = *dst;
            out.x += old.x;
            out.y += old.y;
            out.z += old.z;
            out.w += old.w;
        }
        *dst = out;
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (i0 + c < g.nx) row[i0 + c] = g.accumulate ? row[i0 + c] + v[c] : v[c];
    }
}

// Bounding box of the atoms, one CTA: per-thread min/max, then a tree
// reduction in shared memory (min and max do not depend on the order).
__global__ void __launch_bounds__(1024) atom_bounds_kernel(const float4 *atoms, int n, float *out) {
    __shared__ float red[6][1024];
    float lo[3] = {INFINITY, INFINITY, INFINITY}, hi[3] = {-INFINITY, -INFINITY, -INFINITY};
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float4 a = atoms[i];
        lo[0] = fminf(lo[0], a.x);
        lo[1] = fminf(lo[1], a.y);
        lo[2] = fminf(lo[2], a.z);
        hi[0] = fmaxf(hi[0], a.x);
        hi[1] = fmaxf(hi[1], a.y);
        hi[2] = fmaxf(hi[2], a.z);
    }
    for (int d = 0; d < 3; ++d) {
        red[d][threadIdx.x] = lo[d];
        red[3 + d][threadIdx.x] = hi[d];
    }
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w)
            for (int d = 0; d < 3; ++d) {
                red[d][threadIdx.x] = fminf(red[d][threadIdx.x], red[d][threadIdx.x + w]);
                red[3 + d][threadIdx.x] = fmaxf(red[3 + d][threadIdx.x], red[3 + d][threadIdx.x + w]);
            }
        __syncthreads();
    }
    if (threadIdx.x < 6) out[threadIdx.x] = red[threadIdx.x][0];
}

// ---------------------------------------------------------------------------
// host side

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct MsmGeom {
    cp_msm_layout lay;
    double o[3], h0, a, lim2;
    BinGeom cells;
    cp_cutoff_layout sortL;
    size_t off_gtop;
    size_t off_part[kMsmMaxLevels];
    size_t off_tcoord;
    int8_t hw[kMsmSide * kMsmSide];
};

int make_msm_geometry(int n_atoms, const Grid &g, cp_vec3 dlo, cp_vec3 dhi, float cutoff, float lattice_h,
                      MsmGeom *out) {
    std::memset(out, 0, sizeof(*out));
    const float dl[3] = {dlo.x, dlo.y, dlo.z}, dh[3] = {dhi.x, dhi.y, dhi.z};
    for (int d = 0; d < 3; ++d)
        if (!std::isfinite(dl[d]) || !std::isfinite(dh[d]) || dh[d] < dl[d]) return CP_ERR_INVALID_ARGUMENT;
    if (n_atoms < 0 || !std::isfinite(cutoff) || !(cutoff > 0.0f) || !std::isfinite(lattice_h) ||
        !(lattice_h > 0.0f))
        return CP_ERR_INVALID_ARGUMENT;
    const double h0 = lattice_h, a = cutoff;
    const double ratio = 2.0 * a / h0;
    if (!(ratio <= (double)kMsmMaxRadius)) return CP_ERR_TOO_LARGE;
    const int R = std::max(1, (int)std::ceil(ratio));
    const double go[3] = {g.ox, g.oy, g.oz};
    const int gn[3] = {g.nx, g.ny, g.nz};
    double hi[3];
    long long ncells = 1;
    cp_msm_layout &L = out->lay;
    for (int d = 0; d < 3; ++d) {
        const double lo = std::min((double)dl[d], go[d]);
        hi[d] = std::max((double)dh[d], go[d] + (double)(gn[d] - 1) * (double)g.h);
        out->o[d] = lo;
        const double T = std::floor((hi[d] - lo) / h0);
        if (!(T < 1.0e6)) return CP_ERR_TOO_LARGE;
        L.cells[d] = (int)T + 2;
        ncells *= L.cells[d];
    }
    if (ncells > (long long)kMaxScanBlocks * kScanBlock) return CP_ERR_TOO_LARGE;
    L.lattice_origin = cp_vec3{(float)out->o[0], (float)out->o[1], (float)out->o[2]};
    out->h0 = h0;
    out->a = a;
    out->lim2 = ratio * ratio;
    L.radius = R;
    // stencil columns and taps
    const int side = 2 * R + 1;
    int taps = 0, ncols = 0;
    for (int c = 0; c < side * side; ++c) {
        const int dy = c / side - R, dx = c % side - R;
        int hwv = -1;
        for (int dz = 0; dz <= R; ++dz)
            if ((double)(dx * dx + dy * dy + dz * dz) < out->lim2) hwv = dz;
        out->hw[c] = (int8_t)hwv;
        if (hwv >= 0) {
            taps += 2 * hwv + 1;
            ++ncols;
        }
    }
    L.taps = taps;
    // levels
    int lo[3] = {-1, -1, -1}, hiI[3] = {L.cells[0] + 1, L.cells[1] + 1, L.cells[2] + 1};
    int levels = 0;
    for (;;) {
        if (levels == kMsmMaxLevels) return CP_ERR_TOO_LARGE;
        int mx = 0;
        for (int d = 0; d < 3; ++d) {
            L.lo[levels][d] = lo[d];
            L.n[levels][d] = hiI[d] - lo[d] + 1;
            mx = std::max(mx, L.n[levels][d]);
        }
        ++levels;
        if (mx <= kMsmTopNodes) break;
        for (int d = 0; d < 3; ++d) {
            lo[d] = (int)std::floor(lo[d] / 2.0) - 1;
            hiI[d] = (int)std::ceil(hiI[d] / 2.0) + 1;
        }
    }
    L.levels = levels;
    // layout
    size_t off = 0;
    out->cells.nb[0] = L.cells[0];
    out->cells.nb[1] = L.cells[1];
    out->cells.nb[2] = L.cells[2];
    for (int d = 0; d < 3; ++d) out->cells.bo[d] = (&L.lattice_origin.x)[d];
    out->cells.nbins = ncells;
    out->cells.b = lattice_h;
    out->cells.c = cutoff;
    out->cells.m = 0;
    int rc = make_layout(n_atoms, out->cells, 0, &out->sortL);
    if (rc) return rc;
    L.off_cells = off;
    off = align256(off + out->sortL.total_bytes);
    L.off_stencil = off;
    off = align256(off + 8 * (size_t)side * side * side);
    out->off_gtop = off;
    off = align256(off + 4 * (size_t)kMsmTopTable);
    for (int l = 0; l < levels; ++l) {
        const long long n0 = L.n[l][0], n1 = L.n[l][1], n2 = L.n[l][2];
        L.q_dims[l][0] = (int)n0 + 2 * R;
        L.q_dims[l][1] = (int)(2 * ((n1 + 1) / 2)) + 2 * R;
        L.q_dims[l][2] = (int)(kMsmZ * ((n2 + kMsmZ - 1) / kMsmZ)) + 2 * R;
        long long plane = kMsmMinPlane;
        while (plane < (long long)L.q_dims[l][0] * L.q_dims[l][1]) plane *= 2;
        if (plane > kMsmMaxPlane) return CP_ERR_TOO_LARGE;
        L.q_plane[l] = (int)plane;
        const long long qn = plane * L.q_dims[l][2];
        if (qn > INT_MAX) return CP_ERR_TOO_LARGE;
        L.off_q[l] = off;
        off = align256(off + 8 * (size_t)qn);
        L.off_e[l] = off;
        off = align256(off + 4 * (size_t)(n0 * n1 * n2));
    }
    L.off_partial = off;
    for (int l = 0; l + 1 < levels; ++l) {
        const long long cols = (long long)L.n[l][0] * ((L.n[l][1] + 1) / 2) * ((L.n[l][2] + kMsmZ - 1) / kMsmZ);
        const long long want = (kMsmTargetThreads + cols - 1) / cols;
        L.split[l] = (int)std::max(1LL, std::min<long long>({want, (long long)kMsmMaxSplit, (long long)ncols}));
        out->off_part[l] = off;
        off = align256(off + 4 * (size_t)L.split[l] * (size_t)(L.n[l][0] * L.n[l][1] * L.n[l][2]));
    }
    out->off_tcoord = off;
    off = align256(off + 16 * (size_t)n_atoms);
    L.total_bytes = off;
    return CP_OK;
}

int prepare_msm(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, cp_vec3 dlo, cp_vec3 dhi,
                float cutoff, float lattice_h, Grid *g, MsmGeom *geo) {
    int rc = check_grid(nx, ny, nz, origin, h, g);
    if (rc) return rc;
    return make_msm_geometry(n_atoms, *g, dlo, dhi, cutoff, lattice_h, geo);
}

}  // namespace

}  // namespace cpmap

using namespace cpmap;

extern "C" {

CP_API int cp_msm_layout_of(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, cp_vec3 domain_lo,
                            cp_vec3 domain_hi, float cutoff, float lattice_h, cp_msm_layout *out) {
    if (!out) return CP_ERR_INVALID_ARGUMENT;
    Grid g;
    static thread_local MsmGeom geo;
    const int rc = prepare_msm(n_atoms, nx, ny, nz, origin, h, domain_lo, domain_hi, cutoff, lattice_h, &g, &geo);
    if (rc) return rc;
    *out = geo.lay;
    return CP_OK;
}

CP_API size_t cp_msm_workspace_bytes(int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                     cp_vec3 domain_lo, cp_vec3 domain_hi, float cutoff, float lattice_h) {
    cp_msm_layout L;
    if (cp_msm_layout_of(n_atoms, nx, ny, nz, origin, h, domain_lo, domain_hi, cutoff, lattice_h, &L) != CP_OK)
        return 0;
    return L.total_bytes;
}

CP_API int cp_msm_longrange(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                            cp_vec3 domain_lo, cp_vec3 domain_hi, float cutoff, float lattice_h, void *workspace,
                            size_t workspace_bytes, float *V, int accumulate, void *stream) {
    if (!V || !workspace || (n_atoms > 0 && !atoms) || (accumulate != 0 && accumulate != 1))
        return CP_ERR_INVALID_ARGUMENT;
    Grid g;
    static thread_local MsmGeom geo;
    int rc = prepare_msm(n_atoms, nx, ny, nz, origin, h, domain_lo, domain_hi, cutoff, lattice_h, &g, &geo);
    if (rc) return rc;
    if (n_atoms > 0 && !aligned(atoms, 16)) return CP_ERR_MISALIGNED;
    if (!aligned(workspace, 256) || !aligned(V, 4)) return CP_ERR_MISALIGNED;
    if (workspace_bytes < geo.lay.total_bytes) return CP_ERR_WORKSPACE_TOO_SMALL;
    const cp_msm_layout &L = geo.lay;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    char *cells_ws = ws + L.off_cells;

    rc = sort_atoms_into_cells(reinterpret_cast<const float4 *>(atoms), n_atoms, geo.cells, geo.sortL, cells_ws, st);
    if (rc) return rc;

    MsmParams p;
    std::memset(&p, 0, sizeof(p));
    p.levels = L.levels;
    p.R = L.radius;
    p.W = reinterpret_cast<float2 *>(ws + L.off_stencil);
    p.gtop = reinterpret_cast<float *>(ws + geo.off_gtop);
    for (int d = 0; d < 3; ++d) {
        p.cells[d] = L.cells[d];
        p.o[d] = (&L.lattice_origin.x)[d];
    }
    p.h0 = lattice_h;
    p.cell_start = reinterpret_cast<const int *>(cells_ws + geo.sortL.off_start);
    p.cell_atoms = reinterpret_cast<const float4 *>(cells_ws + geo.sortL.off_csr_atoms);
    p.cell_stats = reinterpret_cast<const int *>(cells_ws + geo.sortL.off_stats);
    p.cell_t = reinterpret_cast<float4 *>(ws + geo.off_tcoord);
    p.ncells = geo.cells.nbins;
    p.n_atoms = n_atoms;
    p.status = device_status_ptr();
    if (!p.status) return CP_ERR_CUDA;
    p.h0_64 = geo.h0;
    p.a64 = geo.a;
    p.lim2 = geo.lim2;
    std::memcpy(p.hw, geo.hw, sizeof(p.hw));
    long long cta = 0;
    for (int l = 0; l < L.levels; ++l) {
        MsmLevelDev &v = p.lv[l];
        for (int d = 0; d < 3; ++d) {
            v.lo[d] = L.lo[l][d];
            v.n[d] = L.n[l][d];
            v.qd[d] = L.q_dims[l][d];
        }
        v.q = reinterpret_cast<float2 *>(ws + L.off_q[l]);
        v.plane = L.q_plane[l];
        v.e = reinterpret_cast<float *>(ws + L.off_e[l]);
        v.scale = (float)std::ldexp(1.0, -l);
        if (l + 1 < L.levels) {
            v.part = reinterpret_cast<float *>(ws + geo.off_part[l]);
            v.split = L.split[l];
            v.cols = (long long)v.n[0] * ((v.n[1] + 1) / 2) * ((v.n[2] + kMsmZ - 1) / kMsmZ);
            v.cta_begin = cta;
            cta += ((v.cols + kMsmThreads - 1) / kMsmThreads) * v.split;
        }
    }
    if (cta > 0x7fffffffLL) return CP_ERR_TOO_LARGE;
    unsigned long long launches = 0;
    const int side = 2 * L.radius + 1;
    const long long nst = (long long)side * side * side + kMsmTopTable;
    bool ok = launch_pdl(msm_stencil_kernel, (int)std::min<long long>((nst + 255) / 256, 1024), 256, st, p);
    const MsmLevelDev &L0 = p.lv[0];
    const long long q0n = (long long)L0.n[0] * L0.n[1] * L0.n[2];
    // the charge lattice's padding must be zero: clear it all, nodes follow
    if (cudaMemsetAsync(L0.q, 0, (size_t)8 * L0.plane * L0.qd[2], st) != cudaSuccess) return CP_ERR_CUDA;
    if (n_atoms > 0) {
        ok = ok && launch_pdl(msm_tcoord_kernel, (int)((n_atoms + kMsmThreads - 1) / kMsmThreads), kMsmThreads, st, p);
        ++launches;
    }
    ok = ok && launch_pdl(msm_anterp_kernel, (int)((q0n + kMsmThreads - 1) / kMsmThreads), kMsmThreads, st, p);
    launches += 2;
    for (int l = 0; l + 1 < L.levels; ++l) {
        const MsmLevelDev &C = p.lv[l + 1];
        const long long qn = (long long)C.qd[0] * C.qd[1] * C.qd[2];
        ok = ok && launch_pdl(msm_restrict_kernel, (int)((qn + kMsmThreads - 1) / kMsmThreads), kMsmThreads, st, p, l);
        ++launches;
    }
    if (cta > 0) {
        ok = ok && launch_pdl(msm_conv_kernel, (int)cta, kMsmThreads, st, p);
        ++launches;
    }
    const MsmLevelDev &T = p.lv[L.levels - 1];
    const long long tn = (long long)T.n[0] * T.n[1] * T.n[2];
    ok = ok && launch_pdl(msm_top_kernel, (int)((tn * 32 + kMsmThreads - 1) / kMsmThreads), kMsmThreads, st, p);
    ++launches;
    for (int l = L.levels - 2; l >= 0; --l) {
        const MsmLevelDev &F = p.lv[l];
        const long long fn = (long long)F.n[0] * F.n[1] * F.n[2] * (F.split >= 16 ? kReduceGroup : 1);
        ok = ok && launch_pdl(msm_reduce_prolong_kernel, (int)((fn + kMsmThreads - 1) / kMsmThreads), kMsmThreads, st, p, l);
        ++launches;
    }
    InterpParams ip;
    ip.nx = g.nx;
    ip.ny = g.ny;
    ip.nz = g.nz;
    ip.dox = (float)((double)g.ox - (double)p.o[0]);
    ip.doy = (float)((double)g.oy - (double)p.o[1]);
    ip.doz = (float)((double)g.oz - (double)p.o[2]);
    ip.h = g.h;
    ip.qx = (g.nx + 3) / 4;
    ip.quads = (long long)ip.qx * g.ny * g.nz;
    ip.V = V;
    ip.accumulate = accumulate;
    const unsigned iblocks = (unsigned)((ip.quads + kMsmThreads - 1) / kMsmThreads);
    const long long nbricks = (long long)((g.nx + kBrick - 1) / kBrick) * ((g.ny + kBrick - 1) / kBrick) *
                              ((g.nz + kBrick - 1) / kBrick);
    // nodes a brick's 8 points need per axis: at most ceil(7 h / h0) + 4
    const int span = (int)std::ceil(7.0 * (double)g.h / (double)lattice_h + 1e-4) + 4;
    if (g.h <= lattice_h && span <= 6 && nbricks <= 0x7fffffffLL)
        ok = ok && launch_pdl(msm_interp_brick_kernel<6>, (int)nbricks, kMsmThreads, st, p, ip);
    else if (g.h <= lattice_h && span <= 8 && nbricks <= 0x7fffffffLL)
        ok = ok && launch_pdl(msm_interp_brick_kernel<8>, (int)nbricks, kMsmThreads, st, p, ip);
    else if (g.h <= lattice_h && span <= 12 && nbricks <= 0x7fffffffLL)
        ok = ok && launch_pdl(msm_interp_brick_kernel<12>, (int)nbricks, kMsmThreads, st, p, ip);
    else if ((g.nx % 4 == 0) && aligned(V, 16))
        ok = ok && launch_pdl(msm_interp_kernel<true>, (int)iblocks, kMsmThreads, st, p, ip);
    else
        ok = ok && launch_pdl(msm_interp_kernel<false>, (int)iblocks, kMsmThreads, st, p, ip);
    ++launches;
    if (!ok || cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(launches);
    return CP_OK;
}

CP_API int cp_atom_bounds(const float *atoms, int n_atoms, float *bounds, void *stream) {
    if (!atoms || !bounds || n_atoms < 1) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(atoms, 16) || !aligned(bounds, 4)) return CP_ERR_MISALIGNED;
    atom_bounds_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<const float4 *>(atoms),
                                                                          n_atoms, bounds);
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

}  // extern "C"
