// cp_direct.cu -- direct Coulomb summation V(g) = sum_a q_a / r on sm_103a.
//
// Mapping (PMPP ch.18 notes "Case study -- electrostatic potential map",
// sections 18.2-18.4, rebuilt for GB300):
//   * gather: a thread owns grid points and every atom streams past it, so
//     each thread writes only its own points and no atomics are needed
//     (section 18.2);
//   * coarsening: a thread owns a patch of PX = 4 (or, for grids too small
//     to fill the GPU otherwise, 2) consecutive x points (one float4 or
//     float2 of the x-fastest output) times PY rows in y times PZ planes in z;
//     per atom the x differences are computed once per patch column and
//     dy^2 + dz^2 once per row, so a pair costs FFMA (r^2), MUFU (rsqrt) and
//     FFMA (accumulate) (section 18.3; the pwwt.cn article's section 三 does
//     the same with 8 points per thread);
//   * coalescing: neighbouring lanes own neighbouring x groups, so a warp
//     stores 32 consecutive float4s (float2s) of a row (section 18.4 and the article's
//     coarsen-plus-coalesce kernel, section 三);
//   * atom tiles: instead of 4K-atom chunks in constant memory re-launched
//     per chunk (section 18.2), one launch streams 512-atom tiles from global
//     memory into a 2-stage shared-memory ring with 1-D TMA bulk copies; all
//     threads read the same atom (a shared-memory broadcast);
//   * f32x2: a thread's x points are register pairs, so r^2, the
//     accumulate and the FMA-pipe rsqrt are paired Blackwell instructions;
//   * rsqrt on two pipes: a compile-time share of each thread's point pairs
//     takes its rsqrt on the FMA pipe (fma_rsqrt2_scaled) and the rest on the SFU,
//     so that neither unit alone limits the pair rate;
//   * accuracy: each tile's contribution is summed in separate registers and
//     then added to a running total kept in shared memory, so the fp32
//     rounding error grows like (tile + n_atoms / tile) instead of n_atoms;
//   * small grids: when there are too few point patches to fill the GPU,
//     LS = 2, 4 or 8 neighbouring lanes share a patch and take every LS-th
//     atom of each tile (a fixed xor-shuffle tree adds their sums), and S
//     CTAs of a thread-block cluster share one tile of points and take 1/S
//     of the atoms each; their partial sums meet in distributed shared
//     memory and are added in rank order (deterministic, no atomics, no
//     global scratch).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "cp_device.cuh"
#include "cp_internal.h"

namespace cg = cooperative_groups;

namespace cpmap {

constexpr int kDirectThreads = 128;
constexpr int kDirectTile = 512;  // atoms per shared-memory stage (8 KiB as loaded)
constexpr int kDirectStages = 2;
// dynamic shared memory: the TMA ring of atoms, then every thread's running
// totals (up to 16 point pairs of 8 bytes)
constexpr int kDirectRingBytes = kDirectStages * kDirectTile * 16;
constexpr int kDirectMaxPairs = 16;
constexpr int direct_smem_bytes(int px, int py, int pz) {
    return kDirectRingBytes + kDirectThreads * (px / 2 * py * pz) * 8;
}
constexpr int kMaxSplit = 16;       // cluster sizes above 8 are non-portable
constexpr int kPortableSplit = 8;

struct DirectParams {
    const float4 *atoms;
    int n_atoms;
    int split;  // CTAs per cluster sharing one tile of points
    int nx, ny, nz;
    float ox, oy, oz, h;
    int qx;         // x groups of PX points per row
    int yb;         // y blocks of PY rows
    long long npatch;
    float *V;
    unsigned int *status;
};


// Stores the PX x points from i0 of row (y, z): one float4 (PX = 4) or
// float2 (PX = 2) when the row is aligned and the group complete, else the
// in-range scalars.  v holds the points in x order (.z, .w unused for PX = 2).
template <int PX, bool VEC>
__device__ __forceinline__ void store_group(const DirectParams &p, int i0, int y, int z, float4 v) {
    if (y >= p.ny || z >= p.nz) return;
    const long long at = ((long long)z * p.ny + y) * p.nx + i0;
    if (!CP_IN(at, (long long)p.nx * p.ny * p.nz, p.status)) return;
    float *row = p.V + ((long long)z * p.ny + y) * p.nx;
    if (VEC) {
        if (!CP_IN(at + PX - 1, (long long)p.nx * p.ny * p.nz, p.status)) return;
        if (PX == 4)
            *reinterpret_cast<float4 *>(row + i0) = v;
        else
            *reinterpret_cast<float2 *>(row + i0) = make_float2(v.x, v.y);
    } else {
        if (i0 + 0 < p.nx) row[i0 + 0] = v.x;
        if (i0 + 1 < p.nx) row[i0 + 1] = v.y;
        if (PX == 4) {
            if (i0 + 2 < p.nx) row[i0 + 2] = v.z;
            if (i0 + 3 < p.nx) row[i0 + 3] = v.w;
        }
    }
}

// A patch is PX x points (PX/2 f32x2 pairs) x PY rows x PZ planes, i.e.
// (PX/2)*PY*PZ point pairs.  The first EMU pairs take their rsqrt on the FMA
// pipe (fma_rsqrt2_scaled), the others on the SFU, so that both units share the work.
// LS neighbouring lanes share a patch, each taking every LS-th atom of a tile
// (more warps for grids with few patches); their sums meet by a fixed
// xor-shuffle tree, so every lane of the group holds the same total.
// REL: the grid points are not all exact in fp32, so differences are formed
// relative to the grid origin (see below); otherwise point - atom, which
// then rounds only once.
template <int PX, int PY, int PZ, int EMU, int LS, bool VEC, bool REL>
__global__ void __launch_bounds__(kDirectThreads) direct_kernel(const __grid_constant__ DirectParams p) {
    static_assert(PX == 2 || PX == 4, "a thread owns one or two x pairs of each row");
    static_assert(LS == 1 || LS == 2 || LS == 4 || LS == 8, "lanes per patch");
    constexpr int PPC = kDirectThreads / LS;  // patches per CTA
    constexpr int HX = PX / 2;       // x pairs per row
    constexpr int NP = HX * PY * PZ;  // point pairs per thread
    static_assert(EMU >= 0 && EMU <= NP, "EMU counts point pairs");
    static_assert(NP <= kDirectMaxPairs, "running totals do not fit");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kDirectStages];
    float4 *ring = reinterpret_cast<float4 *>(smem);

    const int tid = threadIdx.x;
    const int split = p.split;
    const int rank = (int)(blockIdx.x % (unsigned)split);
    const long long ptile = blockIdx.x / (unsigned)split;
    const int slice = tid % LS;  // this lane's share of each atom tile
    const long long patch = ptile * PPC + tid / LS;

    // This CTA's slice of the atoms.
    const int a_begin = (int)((long long)p.n_atoms * rank / split);
    const int a_end = (int)((long long)p.n_atoms * (rank + 1) / split);
    const int n_local = a_end - a_begin;
    const int n_tiles = (n_local + kDirectTile - 1) / kDirectTile;

    // This thread's patch: x group qx, y block yb, z block zb (idle threads past
    // the last patch compute a copy of it and store nothing).
    const long long pc = patch < p.npatch ? patch : p.npatch - 1;
    const int qx = (int)(pc % p.qx);
    const long long t = pc / p.qx;
    const int yb = (int)(t % p.yb);
    const int zb = (int)(t / p.yb);
    const int i0 = PX * qx, j0 = PY * yb, k0 = PZ * zb;
    // REL: the points' grid indices, and a difference to an atom is formed
    // as index * h + (origin - atom) with one rounding (the fused multiply-add
    // keeps index * h exact), so its error follows the atom's offset from the
    // grid origin, not the grid's distance from the coordinate origin.
    // Otherwise the points' coordinates, exact in fp32, and point - atom.
    float x[PX], y[PY], z[PZ];
#pragma unroll
    for (int c = 0; c < PX; ++c) x[c] = REL ? (float)(i0 + c) : fmaf((float)(i0 + c), p.h, p.ox);
#pragma unroll
    for (int j = 0; j < PY; ++j) y[j] = REL ? (float)(j0 + j) : fmaf((float)(j0 + j), p.h, p.oy);
#pragma unroll
    for (int k = 0; k < PZ; ++k) z[k] = REL ? (float)(k0 + k) : fmaf((float)(k0 + k), p.h, p.oz);
    // difference of point coordinate (or index) u and the tile's atom
    // coordinate a (or origin - atom)
    auto diff = [&](float u, float a) { return REL ? fmaf(u, p.h, a) : u - a; };

    if (tid == 0) {
        for (int s = 0; s < kDirectStages; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
    }
    __syncthreads();

    auto issue = [&](int tl, int stage) {
        const int n = min(kDirectTile, n_local - tl * kDirectTile);
        const uint32_t bytes = (uint32_t)n * 16u;
        const long long first = a_begin + (long long)tl * kDirectTile;
        if (CP_IN(first, p.n_atoms, p.status) && CP_IN(first + n - 1, p.n_atoms, p.status)) {
            mbar_arrive_expect_tx(&full[stage], bytes);
            bulk_g2s(ring + stage * kDirectTile, p.atoms + first, bytes, &full[stage]);
        } else {
            mbar_arrive(&full[stage]);  // checked build only: no copy, the status says so
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kDirectStages && s < n_tiles; ++s) issue(s, s);
    }

    // Pair q = (k*PY + j)*HX + h is points (0,1) or (2,3) of row j, plane k.
    // Each tile is summed in registers (part); the running totals stay in
    // shared memory (tot[q][tid]), which keeps registers for the pair loop.
    float2 *tot = reinterpret_cast<float2 *>(smem + kDirectRingBytes);
#pragma unroll
    for (int q = 0; q < NP; ++q) tot[q * kDirectThreads + tid] = make_float2(0.f, 0.f);

    for (int it = 0; it < n_tiles; ++it) {
        const int stage = it % kDirectStages;
        mbar_wait(&full[stage], (uint32_t)((it / kDirectStages) & 1), p.status);
        const int n = min(kDirectTile, n_local - it * kDirectTile);
        float4 *tile = ring + stage * kDirectTile;
        if (REL) {
            // Once per tile and CTA, each atom becomes (origin - atom, q) in
            // place, so that every thread forms its differences with one
            // fused multiply-add each.  These plain stores precede the bulk
            // copy that later refills the stage, hence the proxy fence
            // before the barrier.
            for (int a = tid; a < n; a += kDirectThreads) {
                const float4 v = tile[a];
                tile[a] = make_float4(p.ox - v.x, p.oy - v.y, p.oz - v.z, v.w);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
        }

        float2 part[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) part[q] = make_float2(0.f, 0.f);

        // The per-atom differences are scalar FP32 operations written straight
        // into the register pairs the f32x2 instructions read (dx for points
        // 0,1 and 2,3; dy^2 + dz^2 duplicated per row), so only r^2, the
        // accumulate and the FMA-pipe rsqrt run as f32x2.
#pragma unroll 2
        for (int a = slice; a < n; a += LS) {
            const float4 at = tile[a];  // same address in the lanes of a slice: broadcast
            float2 dxp[HX];
#pragma unroll
            for (int hh = 0; hh < HX; ++hh) dxp[hh] = make_float2(diff(x[2 * hh], at.x), diff(x[2 * hh + 1], at.x));
            const float2 q2 = make_float2(at.w, at.w);
            // dy^2 + dz^2 per row: the square of the shorter axis is taken
            // once and the other axis fused into it (PY + PZ*PY operations
            // when PZ >= PY, PZ + PY*PZ otherwise)
            float dy[PY], dy2[PY];
#pragma unroll
            for (int j = 0; j < PY; ++j) {
                dy[j] = diff(y[j], at.y);
                dy2[j] = dy[j] * dy[j];
            }
#pragma unroll
            for (int k = 0; k < PZ; ++k) {
                const float dz = diff(z[k], at.z);
                const float dz2 = dz * dz;
#pragma unroll
                for (int j = 0; j < PY; ++j) {
                    const float d = PZ < PY ? fmaf(dy[j], dy[j], dz2) : fmaf(dz, dz, dy2[j]);
                    const float2 dyz2 = make_float2(d, d);
#pragma unroll
                    for (int hh = 0; hh < HX; ++hh) {
                        const int q = (k * PY + j) * HX + hh;
                        const float2 dx = dxp[hh];
                        const float2 r2 = __ffma2_rn(dx, dx, dyz2);
                        float2 rs;
                        if (q < EMU) {
                            rs = fma_rsqrt2_scaled(r2);  // rsqrt / sqrt(2): scaled back per tile
                        } else {
                            rs = make_float2(sfu_rsqrt(r2.x), sfu_rsqrt(r2.y));
                        }
                        part[q] = __ffma2_rn(q2, rs, part[q]);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            const float2 pq = q < EMU ? __fmul2_rn(part[q], make_float2(kSqrt2, kSqrt2)) : part[q];
            tot[q * kDirectThreads + tid] = __fadd2_rn(tot[q * kDirectThreads + tid], pq);
        }
        __syncthreads();  // every thread is done with this stage
        if (tid == 0 && it + kDirectStages < n_tiles) issue(it + kDirectStages, stage);
    }

    float2 acc[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) acc[q] = tot[q * kDirectThreads + tid];
    if (LS > 1) {
#pragma unroll
        for (int q = 0; q < NP; ++q)
#pragma unroll
            for (int o = 1; o < LS; o <<= 1) {
                acc[q].x += __shfl_xor_sync(0xffffffffu, acc[q].x, o);
                acc[q].y += __shfl_xor_sync(0xffffffffu, acc[q].y, o);
            }
    }
    if (split == 1) {
        if (patch < p.npatch && slice == 0) {
#pragma unroll
            for (int k = 0; k < PZ; ++k)
#pragma unroll
                for (int j = 0; j < PY; ++j) {
                    const float2 a01 = acc[(k * PY + j) * HX];
                    const float2 a23 = HX == 2 ? acc[(k * PY + j) * HX + HX - 1] : make_float2(0.f, 0.f);
                    store_group<PX, VEC>(p, i0, j0 + j, k0 + k, make_float4(a01.x, a01.y, a23.x, a23.y));
                }
        }
        return;
    }

    // Cluster reduction: each patch's partial sums replace the running
    // totals in this CTA's shared memory (a float4 (PX = 4) or float2
    // (PX = 2) per patch row, within the totals' space), then every element is
    // summed over ranks 0..S-1, in rank order, by the CTA that owns it.
    constexpr int R = PY * PZ;
    using Group = typename std::conditional<PX == 4, float4, float2>::type;
    Group *partial = reinterpret_cast<Group *>(tot);  // [R][PPC]
    __syncthreads();  // every thread has read its totals
    if (slice == 0) {
#pragma unroll
        for (int k = 0; k < PZ; ++k)
#pragma unroll
            for (int j = 0; j < PY; ++j) {
                if constexpr (PX == 4) {
                    const float2 a01 = acc[(k * PY + j) * 2], a23 = acc[(k * PY + j) * 2 + 1];
                    partial[(k * PY + j) * PPC + tid / LS] = make_float4(a01.x, a01.y, a23.x, a23.y);
                } else {
                    partial[(k * PY + j) * PPC + tid / LS] = acc[k * PY + j];
                }
            }
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int n_elem = R * PPC;
    const int e_begin = n_elem * rank / split;
    const int e_end = n_elem * (rank + 1) / split;
    for (int e = e_begin + tid; e < e_end; e += kDirectThreads) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < split; ++r) {
            const Group v = cluster.map_shared_rank(partial, r)[e];
            s.x += v.x;
            s.y += v.y;
            if constexpr (PX == 4) {
                s.z += v.z;
                s.w += v.w;
            }
        }
        const int row = e / PPC;
        const long long pe = ptile * PPC + (e % PPC);
        if (pe < p.npatch) {
            const int eqx = (int)(pe % p.qx);
            const long long et = pe / p.qx;
            const int eyb = (int)(et % p.yb);
            const int ezb = (int)(et / p.yb);
            store_group<PX, VEC>(p, PX * eqx, PY * eyb + row % PY, PZ * ezb + row / PY, s);
        }
    }
    cluster.sync();  // no CTA leaves while others still read its shared memory
}

// ---------------------------------------------------------------------------
// launch planning

namespace {

using KernelFn = void (*)(DirectParams);

// Patch shapes (PX x points, PY rows, PZ planes; EMU point pairs with rsqrt
// on the FMA pipe; LS lanes per patch).  `rate` is the pair rate per SM clock each one reached
// on a GB300 at full occupancy (best split on a 200^3 grid with 100k atoms,
// a run of about 0.13 s); the planner uses it to rank the shapes.  The
// 2-point and shared-patch (LS > 1) shapes exist for grids with too few
// 4-point patches to fill the GPU.
struct Variant {
    int px, py, pz, emu, ls;
    double rate;
    KernelFn fn[2][2];  // [vector stores][relative differences]
};

#define CP_VARIANT(PX, PY, PZ, EMU, LS, RATE)                                                              \
    {PX, PY, PZ, EMU, LS, RATE,                                                                            \
     {{direct_kernel<PX, PY, PZ, EMU, LS, false, false>, direct_kernel<PX, PY, PZ, EMU, LS, false, true>}, \
      {direct_kernel<PX, PY, PZ, EMU, LS, true, false>, direct_kernel<PX, PY, PZ, EMU, LS, true, true>}}}
const Variant kVariants[] = {
    CP_VARIANT(4, 4, 2, 0, 1, 15.48), CP_VARIANT(4, 2, 2, 0, 1, 15.47), CP_VARIANT(4, 4, 1, 0, 1, 15.41),
    CP_VARIANT(4, 2, 1, 0, 1, 15.58), CP_VARIANT(4, 1, 1, 0, 1, 15.31), CP_VARIANT(4, 4, 2, 4, 1, 18.96),
    CP_VARIANT(4, 4, 2, 5, 1, 19.40), CP_VARIANT(4, 2, 2, 2, 1, 19.28), CP_VARIANT(4, 4, 1, 2, 1, 19.39),
    CP_VARIANT(4, 2, 1, 1, 1, 18.81), CP_VARIANT(2, 1, 1, 0, 1, 14.57), CP_VARIANT(2, 2, 1, 0, 1, 15.32),
    CP_VARIANT(4, 1, 1, 0, 4, 15.35), CP_VARIANT(4, 1, 1, 0, 2, 15.36), CP_VARIANT(4, 2, 1, 1, 4, 18.87),
    CP_VARIANT(4, 2, 1, 1, 2, 18.94), CP_VARIANT(4, 2, 1, 1, 8, 18.73), CP_VARIANT(4, 2, 2, 2, 4, 19.69),
    CP_VARIANT(4, 4, 1, 2, 4, 19.89),
};
#undef CP_VARIANT
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

// Resident CTAs per GPU for variant v, store flavour and cluster size s,
// cached per device; 0 if the device cannot run that cluster size.  For
// sizes above 8 it also sets the non-portable cluster attribute of that
// exact kernel, which the launch needs.
std::mutex g_plan_mutex;
int g_slots[kMaxDevices][kNumVariants][2][2][kMaxSplit + 1];  // [device][variant][vector][relative][split]

int resident_ctas(int v, int s, bool vec, bool rel, const DeviceInfo &dev) {
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    int &cached = g_slots[dev.device][v][vec ? 1 : 0][rel ? 1 : 0][s];
    if (cached > 0) return cached;
    if (cached == -2) return 0;  // cluster size not available
    KernelFn fn = kVariants[v].fn[vec ? 1 : 0][rel ? 1 : 0];
    int slots = 0;
    if (s > kPortableSplit &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();  // not supported here: this split is never planned
        cached = -2;
        return 0;
    }
    if (s == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, fn, kDirectThreads, direct_smem_bytes(kVariants[v].px, kVariants[v].py, kVariants[v].pz)) !=
            cudaSuccess)
            return -1;
        slots = per_sm * dev.sm_count;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(s * 64, 1, 1);
        cfg.blockDim = dim3(kDirectThreads, 1, 1);
        cfg.dynamicSmemBytes = direct_smem_bytes(kVariants[v].px, kVariants[v].py, kVariants[v].pz);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = s;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            cached = -2;
            return 0;
        }
        slots = clusters * s;
    }
    if (slots <= 0) {
        cached = -2;
        return 0;
    }
    cached = slots;
    return cached;
}

struct Plan {
    int variant;
    int split;
    bool vec;  // whole-group vector stores
    long long ptiles;
    int qx, yb;
    long long npatch;
};

// Throughput of an SM relative to full occupancy when `warps` warps are
// resident: the pair loop needs about 24 warps per SM to hide the SFU and
// FMA latencies.
double occupancy_factor(double warps) { return std::sqrt(std::min(1.0, warps / 24.0)); }

// Whether variant v stores whole x groups as one vector: every row holds a
// whole number of groups and V is aligned to a group (v_align: the largest
// power of two, up to 16, dividing V's address).
bool vector_stores(int v, const Grid &g, int v_align) {
    const int px = kVariants[v].px;
    return g.nx % px == 0 && v_align >= 4 * px;
}

// Picks the patch shape and cluster split with the smallest modelled time.
// CTAs spread evenly over the SMs; the busiest SM runs ceil(CTAs / SMs) of
// them, at most `resident` at a time, at the shape's measured pair rate
// scaled by its occupancy; each split level adds a small reduction cost.
int plan_direct(const Grid &g, int n_atoms, int v_align, bool rel, const DeviceInfo &dev, Plan *out) {
    double best = INFINITY;
    for (int v = 0; v < kNumVariants; ++v) {
        const int px = kVariants[v].px, py = kVariants[v].py, pz = kVariants[v].pz;
        if (pz > 1 && g.nz < pz) continue;
        if (py > 1 && g.ny < py) continue;
        const bool vec = vector_stores(v, g, v_align);
        const long long qx = (g.nx + px - 1) / px, yb = (g.ny + py - 1) / py, zb = (g.nz + pz - 1) / pz;
        const long long npatch = qx * yb * zb;
        const int ppc = kDirectThreads / kVariants[v].ls;  // patches per CTA
        const long long ctas = (npatch + ppc - 1) / ppc;
        const double pts = (double)ppc * px * py * pz;
        for (int s = 1; s <= kMaxSplit; ++s) {
            if (s == 5 || s == 7 || (s > 8 && s != 12 && s != 16)) continue;
            if (s > 1 && (long long)n_atoms < (long long)s * 64) break;
            if (ctas * s > 0x7fffffffll) break;
            const int slots = resident_ctas(v, s, vec, rel, dev);
            if (slots < 0) return CP_ERR_CUDA;
            if (slots == 0) continue;  // cluster size not available on this device
            const double resident = std::max(1.0, (double)slots / dev.sm_count);
            const double per_sm = std::ceil((double)(ctas * s) / dev.sm_count);
            const double warps = 4.0 * std::min(per_sm, resident);
            const double work = pts * std::max(1.0, (double)n_atoms / s);  // pairs per CTA
            const double t = per_sm * work / (kVariants[v].rate * occupancy_factor(warps)) * (1.0 + 0.005 * s) +
                             2000.0 * std::ceil(per_sm / resident);
            if (t < best) {
                best = t;
                out->variant = v;
                out->split = s;
                out->vec = vec;
                out->ptiles = ctas;
                out->qx = (int)qx;
                out->yb = (int)yb;
                out->npatch = npatch;
            }
        }
    }
    return std::isfinite(best) ? CP_OK : CP_ERR_INVALID_ARGUMENT;
}

}  // namespace

int launch_direct(const float *atoms, int n_atoms, const Grid &g, float *V, cudaStream_t stream,
                  int force_variant, int force_split) {
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc) return rc;
    const int v_align = aligned(V, 16) ? 16 : aligned(V, 8) ? 8 : 4;
    const bool rel = !grid_points_exact(g);
    Plan plan;
    rc = plan_direct(g, n_atoms, v_align, rel, dev, &plan);
    if (rc) return rc;
    if (force_variant >= 0 && force_variant < kNumVariants) {
        const int v = force_variant;
        const int px = kVariants[v].px, py = kVariants[v].py, pz = kVariants[v].pz;
        plan.variant = v;
        plan.vec = vector_stores(v, g, v_align);
        plan.qx = (g.nx + px - 1) / px;
        plan.yb = (g.ny + py - 1) / py;
        plan.npatch = (long long)plan.qx * plan.yb * ((g.nz + pz - 1) / pz);
        const int ppc = kDirectThreads / kVariants[v].ls;
        plan.ptiles = (plan.npatch + ppc - 1) / ppc;
    }
    if (force_split >= 1 && force_split <= kMaxSplit) plan.split = force_split;
    if (plan.split > kPortableSplit) {  // sets the non-portable cluster attribute, checks support
        const int slots = resident_ctas(plan.variant, plan.split, plan.vec, rel, dev);
        if (slots < 0) return CP_ERR_CUDA;
        if (slots == 0) return CP_ERR_UNSUPPORTED;
    }

    DirectParams p;
    p.atoms = reinterpret_cast<const float4 *>(atoms);
    p.n_atoms = n_atoms;
    p.split = plan.split;
    p.nx = g.nx;
    p.ny = g.ny;
    p.nz = g.nz;
    p.ox = g.ox;
    p.oy = g.oy;
    p.oz = g.oz;
    p.h = g.h;
    p.qx = plan.qx;
    p.yb = plan.yb;
    p.npatch = plan.npatch;
    p.V = V;
    p.status = device_status_ptr();
    if (!p.status) return CP_ERR_CUDA;

    KernelFn fn = kVariants[plan.variant].fn[plan.vec ? 1 : 0][rel ? 1 : 0];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(plan.ptiles * plan.split), 1, 1);
    cfg.blockDim = dim3(kDirectThreads, 1, 1);
    cfg.dynamicSmemBytes =
        direct_smem_bytes(kVariants[plan.variant].px, kVariants[plan.variant].py, kVariants[plan.variant].pz);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = plan.split;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = plan.split > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, fn, p) != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

}  // namespace cpmap

using namespace cpmap;

extern "C" {

CP_API int cp_direct(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float *V,
                     void *stream) {
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    if (n_atoms < 0 || !V || (n_atoms > 0 && !atoms)) return CP_ERR_INVALID_ARGUMENT;
    if (n_atoms > 0 && !aligned(atoms, 16)) return CP_ERR_MISALIGNED;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    return launch_direct(atoms, n_atoms, g, V, static_cast<cudaStream_t>(stream), -1, 0);
}

CP_API int cp_direct_plan(int n_atoms, int nx, int ny, int nz, int *variant, int *split) {
    Grid g;
    int rc = check_grid(nx, ny, nz, cp_vec3{0.f, 0.f, 0.f}, 1.0f, &g);
    if (rc) return rc;
    if (n_atoms < 0 || !variant || !split) return CP_ERR_INVALID_ARGUMENT;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc) return rc;
    Plan plan;
    rc = plan_direct(g, n_atoms, 16, !grid_points_exact(g), dev, &plan);
    if (rc) return rc;
    *variant = plan.variant;
    *split = plan.split;
    return CP_OK;
}

CP_API int cp_grid_points_exact(int nx, int ny, int nz, cp_vec3 origin, float h) {
    Grid g;
    const int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    return grid_points_exact(g) ? 1 : 0;
}

// Same as cp_direct with the patch shape (index into the variant table
// kVariants) and the cluster split forced (pass -1 / 0 to let the planner
// choose).  For tests and tuning sweeps.
CP_API int cp_direct_config(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                            float *V, int variant, int split, void *stream) {
    Grid g;
    int rc = check_grid(nx, ny, nz, origin, h, &g);
    if (rc) return rc;
    if (n_atoms < 0 || !V || (n_atoms > 0 && !atoms)) return CP_ERR_INVALID_ARGUMENT;
    if (n_atoms > 0 && !aligned(atoms, 16)) return CP_ERR_MISALIGNED;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    if (variant >= kNumVariants || split > kMaxSplit || split < 0) return CP_ERR_INVALID_ARGUMENT;
    return launch_direct(atoms, n_atoms, g, V, static_cast<cudaStream_t>(stream), variant, split);
}

}  // extern "C"
