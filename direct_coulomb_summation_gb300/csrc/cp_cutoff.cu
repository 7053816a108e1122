// cp_cutoff.cu -- cutoff summation of the switched term on sm_103a.
//
// Binning (Input Binning lecture, slides "Pseudo Code of an Implementation"
// (28), "Coalesced Global Memory Access to Atom Data" (33), "Handling
// Overfull Bins" (34); PMPP ch.18 notes section 18.5 BinTable) runs on the
// GPU as a counting sort:
//   clear -> count (atomic per-bin counters, each atom keeps its arrival
//   rank) -> exclusive scan (per-block scans; the scan of the block sums
//   runs in the scatter kernel's prologue when there are at most 1024
//   blocks, else in a launch of its own) -> scatter (input index to
//   bin-sorted position) -> per-bin sort by input index (one warp per bin,
//   rank by comparison) and pack: the first K atoms of each bin into its
//   fixed-capacity slots, every atom into the bin-sorted (CSR) array.
//   Results are deterministic: within a bin the order is ascending input
//   index whatever order the atomics ran in.  Every launch, and the brick
//   kernel's after them, is a programmatic dependent launch: it may be
//   scheduled while the one before it drains, and waits for it
//   (griddepcontrol.wait) before touching memory.
//
// The map (slides "Details on Small Bin Design" (30), "Tiling Atom Data"
// (32), "GPU Thread Coarsening" (36), "GPU Thread Inner Loop" (37)): one CTA
// per 8x8x8-point brick, a producer warp and four consumer warps.
//   * The producer walks the brick's neighbourhood offset list (one x-run of
//     bins per (dy, dz), passed as a kernel parameter) and packs the atoms
//     into a ring of 8 shared-memory stages of 192 atoms with 1-D TMA bulk copies:
//     with capacity 0 each run is one contiguous range of the bin-sorted
//     array; with capacity 8 or 16 it is the run's fixed-capacity slots
//     (trimmed to its occupied bins), then the overflow of every bin holding
//     more than the capacity.
//   * Consumer warp w owns sub-box w of the brick (8 x 4 x 4 points; each
//     lane 4 consecutive x points as two f32x2 pairs).  For every stage each
//     consumer warp tests all the stage's atoms against its own sub-box,
//     copies those that can reach it into its own list (stage order),
//     releases the stage and runs the list through the pair loop.  An atom
//     inside c of every point of the sub-box by more than the rounding of
//     the test ("full") adds q * rsqrt(r^2)
//     per pair; its -q g(r) is a quartic polynomial in the point's position,
//     added once per point at the end from 15 charge moments of the full
//     atoms about the sub-box centre.  Any other listed atom adds the
//     switched term q * (rsqrt(r^2) - (GC0 + r^2 (GC1 + r^2 GC2))) for
//     r^2 < c^2.  The consumer warps never wait for one another: each may
//     run ahead of the others by up to the ring's depth.
//   * Unused fixed slots sit at 1e18 A and never pass the sub-box test,
//     which replaces the lecture's stop-at-the-first-empty-slot rule.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "cp_device.cuh"
#include "cp_internal.h"

namespace cpmap {

// ---------------------------------------------------------------------------
// binning kernels

struct BinParams {
    const float4 *atoms;
    int n;
    int nb[3];
    float bo[3];
    float b;
    int nbins;
    int K;
    int *count;
    int *start;
    int *csr_index;
    float4 *csr_atoms;
    float4 *padded;
    int *stats;  // [0] binned, [1] dropped, [2] overflow atoms, [3] max bin count
    int2 *bin_rank;
    int *block_sums;
    int *block_prefix;
    int prefix_inline;     // > 0: the scatter kernel scans this many block totals itself
    unsigned int *status;  // checked build: index checks record here
};

// Largest number of block totals the scatter kernel scans in its prologue
// (instead of a separate one-CTA launch).
constexpr int kInlinePrefixMax = 1024;

// fp32 bin coordinate: floor(float(float(a - bo) / b)), -1 outside [0, nb)
// (NaN fails both comparisons).
__device__ __forceinline__ int bin_axis(float a, float bo, float b, int nb) {
    const float t = __fsub_rn(a, bo);
    const float u = __fdiv_rn(t, b);
    const float f = floorf(u);
    return (f >= 0.0f && f < (float)nb) ? (int)f : -1;
}

__global__ void bin_clear_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.nbins; i += stride) p.count[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x < 8) p.stats[threadIdx.x] = 0;
}

__global__ void bin_count_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const float4 a = p.atoms[i];
    const int ux = bin_axis(a.x, p.bo[0], p.b, p.nb[0]);
    const int uy = bin_axis(a.y, p.bo[1], p.b, p.nb[1]);
    const int uz = bin_axis(a.z, p.bo[2], p.b, p.nb[2]);
    int bin = -1, rank = 0;
    if (ux >= 0 && uy >= 0 && uz >= 0 && CP_IN((uz * p.nb[1] + uy) * p.nb[0] + ux, p.nbins, p.status)) {
        bin = (uz * p.nb[1] + uy) * p.nb[0] + ux;
        rank = atomicAdd(&p.count[bin], 1);
    } else {
        atomicAdd(&p.stats[1], 1);
    }
    p.bin_rank[i] = make_int2(bin, rank);
}

// Exclusive scan of count within blocks of kScanBlock bins (256 threads x 8);
// local results go to start[], block totals to block_sums[].
__global__ void __launch_bounds__(256) bin_scan_local_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int warp_tot[8];
    const int base = blockIdx.x * kScanBlock + threadIdx.x * 8;
    int v[8];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = (base + k < p.nbins) ? p.count[base + k] : 0;
        sum += v[k];
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int warp_off = 0, block_tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        warp_off += (w < warp) ? warp_tot[w] : 0;
        block_tot += warp_tot[w];
    }
    int run = warp_off + incl - sum;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (base + k < p.nbins) p.start[base + k] = run;
        run += v[k];
    }
    if (threadIdx.x == 0) p.block_sums[blockIdx.x] = block_tot;
}

// One CTA: exclusive scan of the block totals; also start[nbins] and the
// binned-atom count.
__global__ void __launch_bounds__(1024) bin_scan_blocks_kernel(const __grid_constant__ BinParams p, int nblk) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int warp_tot[32];
    const int base = threadIdx.x * 8;
    int v[8];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[k] = (base + k < nblk) ? p.block_sums[base + k] : 0;
        sum += v[k];
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int warp_off = 0, total = 0;
    for (int w = 0; w < 32; ++w) {
        warp_off += (w < warp) ? warp_tot[w] : 0;
        total += warp_tot[w];
    }
    int run = warp_off + incl - sum;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (base + k < nblk) p.block_prefix[base + k] = run;
        run += v[k];
    }
    if (threadIdx.x == 0) {
        p.start[p.nbins] = total;
        p.stats[0] = total;
    }
}

__global__ void bin_scatter_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int pre[kInlinePrefixMax];
    const int nblk = p.prefix_inline;
    if (nblk > 0) {
        // the exclusive prefix of the block totals, by warp 0 (each lane a
        // run of consecutive totals, then a shuffle scan of the run sums);
        // block 0 also stores it, start[nbins] and the binned count
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            const int per = (nblk + 31) / 32;
            const int b0 = min(lane * per, nblk), b1 = min(b0 + per, nblk);
            int sum = 0;
            for (int b = b0; b < b1; ++b) sum += p.block_sums[b];
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            int run = incl - sum;
            for (int b = b0; b < b1; ++b) {
                pre[b] = run;
                if (blockIdx.x == 0) p.block_prefix[b] = run;
                run += p.block_sums[b];
            }
            if (blockIdx.x == 0 && lane == 31) {
                p.start[p.nbins] = incl;
                p.stats[0] = incl;
            }
        }
        __syncthreads();
    }
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const int2 br = p.bin_rank[i];
    if (br.x < 0) return;
    const int blk = br.x / kScanBlock;
    const int pos = p.start[br.x] + (nblk > 0 ? pre[blk] : p.block_prefix[blk]) + br.y;
    if (CP_IN(pos, p.n, p.status)) p.csr_index[pos] = i;
}

// One warp per bin: rank the bin's input indices by comparison, write the
// bin-sorted atoms and indices and the fixed-capacity slots (pads after the
// last atom), and the final start[] entry.  8 bins per 256-thread block.
__global__ void __launch_bounds__(256) bin_sort_pack_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int blk_overflow, blk_max;
    if (threadIdx.x == 0) {
        blk_overflow = 0;
        blk_max = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int bin = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nb_ = bin < p.nbins ? p.count[bin] : 0;
    const int sb_ = bin < p.nbins ? p.start[bin] + p.block_prefix[bin / kScanBlock] : 0;
    if (bin < p.nbins && (nb_ == 0 || (CP_IN(sb_, p.n, p.status) && CP_IN(sb_ + nb_ - 1, p.n, p.status)))) {
        const int n = nb_;
        const int s = sb_;
        int *tmp = reinterpret_cast<int *>(p.bin_rank);  // free after the scatter
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int e = (c0 + lane < n) ? p.csr_index[s + c0 + lane] : INT_MAX;
            int rank = 0;
            for (int c1 = 0; c1 < n; c1 += 32) {
                const int f = (c1 + lane < n) ? p.csr_index[s + c1 + lane] : INT_MAX;
                const int m = min(32, n - c1);
                for (int k = 0; k < m; ++k) rank += (__shfl_sync(0xffffffffu, f, k) < e) ? 1 : 0;
            }
            if (c0 + lane < n && CP_IN(e, p.n, p.status)) {
                const float4 a = p.atoms[e];
                tmp[s + rank] = e;
                p.csr_atoms[s + rank] = a;
                if (rank < p.K) p.padded[(long long)bin * p.K + rank] = a;
            }
        }
        __syncwarp();
        for (int k = lane; k < n; k += 32) p.csr_index[s + k] = tmp[s + k];
        for (int k = n + lane; k < p.K; k += 32)
            p.padded[(long long)bin * p.K + k] = make_float4(kPadCoord, kPadCoord, kPadCoord, 0.0f);
        __syncwarp();
        if (lane == 0) {
            p.start[bin] = s;
            if (n > p.K) atomicAdd(&blk_overflow, n - p.K);
            atomicMax(&blk_max, n);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (blk_overflow) atomicAdd(&p.stats[2], blk_overflow);
        atomicMax(&p.stats[3], blk_max);
    }
}

// The same per-bin sort and pack for bin grids whose bins hold few atoms
// (lattice cells): lane b of a warp owns bin 32*warp + b and ranks a bin of
// at most kLaneSortMax atoms by itself; larger bins are ranked by the whole
// warp, one after another.  Results are identical to bin_sort_pack_kernel.
constexpr int kLaneSortMax = 16;

__global__ void __launch_bounds__(256) bin_sort_pack_lane_kernel(const __grid_constant__ BinParams p) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int blk_overflow, blk_max;
    if (threadIdx.x == 0) {
        blk_overflow = 0;
        blk_max = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int bin0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * 32;
    const int bin = bin0 + lane;
    const int n0_ = bin < p.nbins ? p.count[bin] : 0;
    const int s0_ = bin < p.nbins ? p.start[bin] + p.block_prefix[bin / kScanBlock] : 0;
    const bool valid =
        bin < p.nbins && (n0_ == 0 || (CP_IN(s0_, p.n, p.status) && CP_IN(s0_ + n0_ - 1, p.n, p.status)));
    const int n = valid ? n0_ : 0;
    const int s = valid ? s0_ : 0;
    int *tmp = reinterpret_cast<int *>(p.bin_rank);  // free after the scatter
    const bool small = n <= kLaneSortMax;
    if (valid && small) {
        for (int c0 = 0; c0 < n; ++c0) {
            const int e = p.csr_index[s + c0];
            int rank = 0;
            for (int c1 = 0; c1 < n; ++c1) rank += (p.csr_index[s + c1] < e) ? 1 : 0;
            if (!CP_IN(e, p.n, p.status)) continue;
            const float4 a = p.atoms[e];
            tmp[s + rank] = e;
            p.csr_atoms[s + rank] = a;
            if (rank < p.K) p.padded[(long long)bin * p.K + rank] = a;
        }
    }
    unsigned big = __ballot_sync(0xffffffffu, valid && !small);
    while (big != 0u) {
        const int lb = __ffs(big) - 1;
        big &= big - 1u;
        const int bn = __shfl_sync(0xffffffffu, n, lb);
        const int bs = __shfl_sync(0xffffffffu, s, lb);
        const int bb = bin0 + lb;
        for (int c0 = 0; c0 < bn; c0 += 32) {
            const int e = (c0 + lane < bn) ? p.csr_index[bs + c0 + lane] : INT_MAX;
            int rank = 0;
            for (int c1 = 0; c1 < bn; c1 += 32) {
                const int f = (c1 + lane < bn) ? p.csr_index[bs + c1 + lane] : INT_MAX;
                const int m = min(32, bn - c1);
                for (int k = 0; k < m; ++k) rank += (__shfl_sync(0xffffffffu, f, k) < e) ? 1 : 0;
            }
            if (c0 + lane < bn && CP_IN(e, p.n, p.status)) {
                const float4 a = p.atoms[e];
                tmp[bs + rank] = e;
                p.csr_atoms[bs + rank] = a;
                if (rank < p.K) p.padded[(long long)bb * p.K + rank] = a;
            }
        }
        __syncwarp();
        for (int k = lane; k < bn; k += 32) p.csr_index[bs + k] = tmp[bs + k];
        __syncwarp();
    }
    if (valid) {
        if (small) {
            for (int k = 0; k < n; ++k) p.csr_index[s + k] = tmp[s + k];
            for (int k = n; k < p.K; ++k) p.padded[(long long)bin * p.K + k] = make_float4(kPadCoord, kPadCoord, kPadCoord, 0.0f);
        }
        p.start[bin] = s;
        if (n > p.K) atomicAdd(&blk_overflow, n - p.K);
        atomicMax(&blk_max, n);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (blk_overflow) atomicAdd(&p.stats[2], blk_overflow);
        atomicMax(&p.stats[3], blk_max);
    }
}

// ---------------------------------------------------------------------------
// brick kernel

constexpr int kBrickConsumerWarps = 4;
constexpr int kBrickThreads = 32 * (kBrickConsumerWarps + 1);  // + 1 producer warp
constexpr int kBrickStages = 8;

struct BrickParams {
    int nx, ny, nz;
    float ox, oy, oz, h;
    float c2, cull2, full2, gc0, gc1, gc2;
    int nb[3];
    int m;
    double h64, b64;
    int nbr[3];  // bricks per axis
    const float4 *padded;
    const int *count;
    const int *start;
    const float4 *csr_atoms;
    float *V;
    unsigned int *status;
    int n_csr;             // atoms in the bin-sorted array (checked build)
    long long n_padded;    // fixed slots in all bins (checked build)
    unsigned long long *counts;  // pair-counting variant only: [3] see cp_cutoff_pair_counts
    int n_runs;
    int runs[kMaxRuns];  // packed int8 (dy, dz, dx_lo, dx_hi)
};

__device__ __forceinline__ int brick_home_dev(int brick, int m, double h, double b) {
    const double t = __dmul_rn(8.0 * (double)brick, h);
    return m + (int)floor(__ddiv_rn(t, b));
}

// Atoms per shared-memory stage.  The producer packs as many bin runs (or
// pieces of runs) into a stage as fit, so a stage usually holds several
// runs; every consumer warp tests the whole stage against its own sub-box.
constexpr int kStageAtoms = 192;

// REL: the grid points are not all exact in fp32, so the lists hold
// origin - atom and differences are formed relative to the grid origin;
// otherwise the lists hold the atoms and differences are point - atom, which
// then rounds only once.
template <int K, bool VEC, bool COUNT, bool REL>
__global__ void __launch_bounds__(kBrickThreads, 6) cutoff_brick_kernel(const __grid_constant__ BrickParams p) {
    __shared__ __align__(128) float4 ring[kBrickStages][kStageAtoms];
    // each consumer warp's list of the stage's atoms that can reach its
    // sub-box, in stage order
    __shared__ __align__(16) float4 wlist[kBrickConsumerWarps][kStageAtoms];
    __shared__ uint64_t full[kBrickStages], empty[kBrickStages];
    __shared__ volatile int stage_n[kBrickStages];

    pdl_launch_dependents();
    pdl_wait();  // binning's results
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int brick = blockIdx.x;
    const int bx = brick % p.nbr[0];
    const int by = (brick / p.nbr[0]) % p.nbr[1];
    const int bz = brick / (p.nbr[0] * p.nbr[1]);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBrickStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBrickConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kBrickConsumerWarps) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues every copy; the other lanes load bin counts and
        // starts for it.  Stage s of use u is refilled only after the four
        // consumer warps released use u-1 (empty[s]); full[s] completes when
        // lane 0 has arrived and all bytes of the stage's copies landed.
        const int hx = brick_home_dev(bx, p.m, p.h64, p.b64);
        const int hy = brick_home_dev(by, p.m, p.h64, p.b64);
        const int hz = brick_home_dev(bz, p.m, p.h64, p.b64);
        int seq = 0, fill = 0, cur = 0;
        bool open = false, ok = true;
        auto open_stage = [&]() {
            cur = seq % kBrickStages;
            const int use = seq / kBrickStages;
            if (use > 0 && ok) ok = mbar_wait(&empty[cur], (uint32_t)((use - 1) & 1), p.status);
            fill = 0;
            open = true;
        };
        auto close_stage = [&]() {
            stage_n[cur] = fill;
            mbar_arrive(&full[cur]);
            ++seq;
            open = false;
        };
        // queue n atoms starting at src (lane 0 only)
        auto push = [&](const float4 *src, int n) {
            while (n > 0 && ok) {
                if (!open) open_stage();
                const int take = min(n, kStageAtoms - fill);
                mbar_expect_tx(&full[cur], (uint32_t)take * 16u);
                bulk_g2s(&ring[cur][fill], src, (uint32_t)take * 16u, &full[cur]);
                fill += take;
                src += take;
                n -= take;
                if (fill == kStageAtoms) close_stage();
            }
        };
        // bins of run r, clamped to the bin grid: first bin and count (0 if none)
        auto run_bins = [&](int r, int &first, int &nbin) {
            const int code = p.runs[r];
            const int dy = (int)(signed char)(code & 0xff);
            const int dz = (int)(signed char)((code >> 8) & 0xff);
            const int dxl = (int)(signed char)((code >> 16) & 0xff);
            const int dxh = (int)(signed char)((code >> 24) & 0xff);
            const int uy = hy + dy, uz = hz + dz;
            const int xlo = max(hx + dxl, 0), xhi = min(hx + dxh, p.nb[0] - 1);
            first = (uz * p.nb[1] + uy) * p.nb[0] + xlo;
            nbin = (uy < 0 || uy >= p.nb[1] || uz < 0 || uz >= p.nb[2] || xlo > xhi) ? 0 : xhi - xlo + 1;
        };
        if (K == 0) {
            // bin-sorted atoms of a run of consecutive bins are contiguous:
            // one copy of [start[first], start[first + nbin]) per run
            for (int r0 = 0; r0 < p.n_runs && ok; r0 += 32) {
                int lo = 0, hi = 0;
                if (r0 + lane < p.n_runs) {
                    int first, nbin;
                    run_bins(r0 + lane, first, nbin);
                    if (nbin > 0) {
                        lo = p.start[first];
                        hi = p.start[first + nbin];
                    }
                }
                const int nr = min(32, p.n_runs - r0);
                for (int t = 0; t < nr; ++t) {
                    const int l = __shfl_sync(0xffffffffu, lo, t);
                    const int h = __shfl_sync(0xffffffffu, hi, t);
                    if (lane == 0 && h > l && CP_IN(l, p.n_csr, p.status) && CP_IN(h - 1, p.n_csr, p.status))
                        push(p.csr_atoms + l, h - l);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        } else {
            // fixed-capacity slots of each run (trimmed to its occupied
            // bins), then the overflow of the bins holding more than K
            for (int pass = 0; pass < 2; ++pass) {
                for (int r = 0; r < p.n_runs && ok; ++r) {
                    int first, nbin;
                    run_bins(r, first, nbin);
                    for (int cb = 0; cb < nbin && ok; cb += 32) {  // 32 bins per step
                        const int nb32 = min(32, nbin - cb);
                        const int f32 = first + cb;
                        const int cnt = lane < nb32 ? p.count[f32 + lane] : 0;
                        if (pass == 0) {
                            const unsigned nz = __ballot_sync(0xffffffffu, cnt > 0);
                            if (nz != 0u && lane == 0) {
                                const int l0 = __ffs(nz) - 1, l1 = 31 - __clz(nz);
                                if (CP_IN((long long)(f32 + l0) * K, p.n_padded, p.status) &&
                                    CP_IN((long long)(f32 + l1 + 1) * K - 1, p.n_padded, p.status))
                                    push(p.padded + (long long)(f32 + l0) * K, (l1 - l0 + 1) * K);
                            }
                        } else {
                            const int st = lane < nb32 ? p.start[f32 + lane] : 0;
                            unsigned ov = __ballot_sync(0xffffffffu, cnt > K);
                            while (ov != 0u) {
                                const int jb = __ffs(ov) - 1;
                                ov &= ov - 1u;
                                const int cj = __shfl_sync(0xffffffffu, cnt, jb);
                                const int sj = __shfl_sync(0xffffffffu, st, jb);
                                if (lane == 0 && CP_IN(sj + K, p.n_csr, p.status) && CP_IN(sj + cj - 1, p.n_csr, p.status))
                                    push(p.csr_atoms + sj + K, cj - K);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                    }
                }
            }
        }
        if (lane == 0) {
            if (open) close_stage();
            open_stage();  // end of stream
            stage_n[cur] = -1;
            mbar_arrive(&full[cur]);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // A lane owns 4 consecutive x points (two f32x2 pairs) of one y row and z
    // plane: x = 8bx + xq .. +3, y = 8by + yy, z = 8bz + zz.  Warp w covers
    // sub-box w of the brick: all 8 x, y rows 4*(w & 1) .. +3, z planes
    // 4*(w >> 1) .. +3.
    const int xq = (lane & 1) * 4;
    const int yy = (warp & 1) * 4 + ((lane >> 1) & 3);
    const int zz = (warp >> 1) * 4 + (lane >> 3);
    const int i0 = kBrick * bx + xq, j = kBrick * by + yy, k = kBrick * bz + zz;
    // REL: the lane's grid indices, and a difference to a listed atom is
    // formed as index * h + (origin - atom) with one rounding (the list
    // holds origin - atom), so its error follows the atom's offset from the
    // grid origin, not the grid's distance from the coordinate origin.
    // Otherwise the points' coordinates, exact in fp32, and point - atom.
    float x[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) x[c] = REL ? (float)(i0 + c) : fmaf((float)(i0 + c), p.h, p.ox);
    const float y = REL ? (float)j : fmaf((float)j, p.h, p.oy);
    const float z = REL ? (float)k : fmaf((float)k, p.h, p.oz);
    auto diff = [&](float u, float a) { return REL ? fmaf(u, p.h, a) : u - a; };
    const float2 NG0 = make_float2(-p.gc0, -p.gc0), NG1 = make_float2(-p.gc1, -p.gc1);
    const float2 NG2 = make_float2(-p.gc2, -p.gc2);
    // this warp's sub-box: all 8 x, 4 y rows, 4 z planes
    const float lox = fmaf((float)(kBrick * bx), p.h, p.ox), hix = fmaf((float)(kBrick * bx + 7), p.h, p.ox);
    const int wy0 = kBrick * by + (warp & 1) * 4, wz0 = kBrick * bz + (warp >> 1) * 4;
    const float loy = fmaf((float)wy0, p.h, p.oy), hiy = fmaf((float)(wy0 + 3), p.h, p.oy);
    const float loz = fmaf((float)wz0, p.h, p.oz), hiz = fmaf((float)(wz0 + 3), p.h, p.oz);
    // Centre of the sub-box (its middle point, index 8bx + 3.5, wy0 + 1.5,
    // wz0 + 1.5), the expansion point of the full atoms' moments; REL:
    // relative to the grid origin, like the listed atoms.
    const float cxi = (float)(kBrick * bx) + 3.5f, cyi = (float)wy0 + 1.5f, czi = (float)wz0 + 1.5f;
    const float cx = REL ? cxi * p.h : fmaf(cxi, p.h, p.ox);
    const float cy = REL ? cyi * p.h : fmaf(cyi, p.h, p.oy);
    const float cz = REL ? czi * p.h : fmaf(czi, p.h, p.oz);
    const unsigned below = (1u << lane) - 1u;
    float4 *list = &wlist[warp][0];

    // Moments about the centre of the atoms within c of the whole sub-box
    // (w = atom - centre, m = |w|^2; this lane's share of them):
    // sum q, sum q w, sum q m, sum q m^2, sum q m w, sum q w w^T.
    float mq = 0.f, mqx = 0.f, mqy = 0.f, mqz = 0.f, mqm = 0.f, mqmm = 0.f;
    float mrx = 0.f, mry = 0.f, mrz = 0.f;
    float mtxx = 0.f, mtxy = 0.f, mtxz = 0.f, mtyy = 0.f, mtyz = 0.f, mtzz = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    unsigned long long n_real = 0, n_near = 0, n_useful = 0;  // COUNT only
    for (int seq = 0;; ++seq) {
        const int s = seq % kBrickStages;
        const bool got = mbar_wait(&full[s], (uint32_t)((seq / kBrickStages) & 1), p.status);
        const int n = got ? stage_n[s] : -1;
        if (n < 0) break;  // end of the stream (or a wait that ran out: recorded)
        // (1) every atom of the stage against this warp's sub-box.  An atom
        // within c of every point of it ("full") goes to the front of the
        // warp's list, one that can reach only some of its points
        // ("partial") to the back, both in stage order.
        int cnt_f = 0, cnt_p = 0;
        for (int i0s = 0; i0s < n; i0s += 32) {
            const int i = i0s + lane;
            const bool valid = i < n;
            const float4 a = valid ? ring[s][i] : make_float4(kPadCoord, kPadCoord, kPadCoord, 0.f);
            if (COUNT && warp == 0 && valid && a.x < 1.0e17f) ++n_real;
            const float ex = fmaxf(fmaxf(lox - a.x, a.x - hix), 0.0f);
            const float ey = fmaxf(fmaxf(loy - a.y, a.y - hiy), 0.0f);
            const float ez = fmaxf(fmaxf(loz - a.z, a.z - hiz), 0.0f);
            const bool near = fmaf(ez, ez, fmaf(ey, ey, ex * ex)) < p.cull2;
            // the sub-box's point farthest from the atom is one of its corners
            const float fx = fmaxf(a.x - lox, hix - a.x), fy = fmaxf(a.y - loy, hiy - a.y);
            const float fz = fmaxf(a.z - loz, hiz - a.z);
            const bool whole = near && fmaf(fz, fz, fmaf(fy, fy, fx * fx)) < p.full2;
            const unsigned mf = __ballot_sync(0xffffffffu, whole);
            const unsigned mp = __ballot_sync(0xffffffffu, near && !whole);
            const float4 entry = REL ? make_float4(p.ox - a.x, p.oy - a.y, p.oz - a.z, a.w) : a;
            if (whole && CP_IN(cnt_f + __popc(mf & below), kStageAtoms, p.status))
                list[cnt_f + __popc(mf & below)] = entry;
            if (near && !whole && CP_IN(kStageAtoms - 1 - cnt_p - __popc(mp & below), kStageAtoms, p.status))
                list[kStageAtoms - 1 - cnt_p - __popc(mp & below)] = entry;
            cnt_f += __popc(mf);
            cnt_p += __popc(mp);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage may be refilled: the list holds copies
        if (COUNT) n_near += (unsigned)(cnt_f + cnt_p);
        // (2) the full atoms' moments, lane t taking atoms t, t + 32, ...
        for (int t = lane; t < cnt_f && !COUNT; t += 32) {
            const float4 e = list[t];
            const float wx = REL ? -e.x - cx : e.x - cx;
            const float wy = REL ? -e.y - cy : e.y - cy;
            const float wz = REL ? -e.z - cz : e.z - cz;
            const float m = fmaf(wz, wz, fmaf(wy, wy, wx * wx));
            const float qm = e.w * m, qx = e.w * wx, qy = e.w * wy, qz = e.w * wz;
            mq += e.w;
            mqx += qx;
            mqy += qy;
            mqz += qz;
            mqm += qm;
            mqmm = fmaf(qm, m, mqmm);
            mrx = fmaf(qm, wx, mrx);
            mry = fmaf(qm, wy, mry);
            mrz = fmaf(qm, wz, mrz);
            mtxx = fmaf(qx, wx, mtxx);
            mtxy = fmaf(qx, wy, mtxy);
            mtxz = fmaf(qx, wz, mtxz);
            mtyy = fmaf(qy, wy, mtyy);
            mtyz = fmaf(qy, wz, mtyz);
            mtzz = fmaf(qz, wz, mtzz);
        }
        // (3) every listed atom against the lane's 4 points.  Full atoms add
        // q / r only (their -q g(r) is in the moments); partial atoms add the
        // switched term where r < c.
        // (both loops unrolled by 8: 4 % faster than by 2 on the 200^3 and
        // 400^3 maps, the most of 1, 2, 3, 4 and 8)
        float2 pf01 = make_float2(0.f, 0.f), pf23 = make_float2(0.f, 0.f);
#pragma unroll 8
        for (int t = 0; t < cnt_f; ++t) {
            const float4 a = list[t];  // broadcast
            const float dy = diff(y, a.y), dz = diff(z, a.z);
            const float d = fmaf(dy, dy, dz * dz);
            const float2 dyz2 = make_float2(d, d);
            const float2 dx01 = make_float2(diff(x[0], a.x), diff(x[1], a.x));
            const float2 dx23 = make_float2(diff(x[2], a.x), diff(x[3], a.x));
            const float2 r01 = __ffma2_rn(dx01, dx01, dyz2);
            const float2 r23 = __ffma2_rn(dx23, dx23, dyz2);
            const float2 rs01 = make_float2(sfu_rsqrt(r01.x), sfu_rsqrt(r01.y));
            const float2 rs23 = make_float2(sfu_rsqrt(r23.x), sfu_rsqrt(r23.y));
            const float2 qq = make_float2(a.w, a.w);
            pf01 = __ffma2_rn(qq, rs01, pf01);
            pf23 = __ffma2_rn(qq, rs23, pf23);
            if (COUNT) {
                const float r2c[4] = {r01.x, r01.y, r23.x, r23.y};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (r2c[c] < p.c2 && i0 + c < p.nx && j < p.ny && k < p.nz) ++n_useful;
            }
        }
#pragma unroll 8
        for (int t = kStageAtoms - cnt_p; t < kStageAtoms; ++t) {
            const float4 a = list[t];  // broadcast
            // differences as scalars (dy^2 + dz^2 is the same for the
            // lane's 4 points), written into the f32x2 operand pairs
            const float dy = diff(y, a.y), dz = diff(z, a.z);
            const float d = fmaf(dy, dy, dz * dz);
            const float2 dyz2 = make_float2(d, d);
            const float2 dx01 = make_float2(diff(x[0], a.x), diff(x[1], a.x));
            const float2 dx23 = make_float2(diff(x[2], a.x), diff(x[3], a.x));
            const float2 r01 = __ffma2_rn(dx01, dx01, dyz2);
            const float2 r23 = __ffma2_rn(dx23, dx23, dyz2);
            // e = rsqrt(r^2) - g(r^2), with -g by Horner on the negated coefficients
            const float2 rs01 = make_float2(sfu_rsqrt(r01.x), sfu_rsqrt(r01.y));
            const float2 rs23 = make_float2(sfu_rsqrt(r23.x), sfu_rsqrt(r23.y));
            const float2 e01 = __fadd2_rn(rs01, __ffma2_rn(__ffma2_rn(r01, NG2, NG1), r01, NG0));
            const float2 e23 = __fadd2_rn(rs23, __ffma2_rn(__ffma2_rn(r23, NG2, NG1), r23, NG0));
            if (r01.x < p.c2) pf01.x = fmaf(a.w, e01.x, pf01.x);
            if (r01.y < p.c2) pf01.y = fmaf(a.w, e01.y, pf01.y);
            if (r23.x < p.c2) pf23.x = fmaf(a.w, e23.x, pf23.x);
            if (r23.y < p.c2) pf23.y = fmaf(a.w, e23.y, pf23.y);
            if (COUNT) {
                const float r2c[4] = {r01.x, r01.y, r23.x, r23.y};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (r2c[c] < p.c2 && i0 + c < p.nx && j < p.ny && k < p.nz) ++n_useful;
            }
        }
        acc[0] += pf01.x;
        acc[1] += pf01.y;
        acc[2] += pf23.x;
        acc[3] += pf23.y;
        __syncwarp();  // the list is rewritten by the next stage
    }

    // -sum over the full atoms of q g(r) at each of the lane's points, from
    // the moments: with u = point - centre, r^2 = s - 2 u.w + m (s = |u|^2),
    //   sum q r^2 = s Q - 2 u.Q1 + M,
    //   sum q r^4 = s (s Q + 2 M - 4 u.Q1) + M2 - 4 u.R + 4 u^T T u,
    // and -g(r) = NG0 + NG1 r^2 + NG2 r^4.
#pragma unroll
    for (int o = 16; o > 0 && !COUNT; o >>= 1) {
        mq += __shfl_xor_sync(0xffffffffu, mq, o);
        mqx += __shfl_xor_sync(0xffffffffu, mqx, o);
        mqy += __shfl_xor_sync(0xffffffffu, mqy, o);
        mqz += __shfl_xor_sync(0xffffffffu, mqz, o);
        mqm += __shfl_xor_sync(0xffffffffu, mqm, o);
        mqmm += __shfl_xor_sync(0xffffffffu, mqmm, o);
        mrx += __shfl_xor_sync(0xffffffffu, mrx, o);
        mry += __shfl_xor_sync(0xffffffffu, mry, o);
        mrz += __shfl_xor_sync(0xffffffffu, mrz, o);
        mtxx += __shfl_xor_sync(0xffffffffu, mtxx, o);
        mtxy += __shfl_xor_sync(0xffffffffu, mtxy, o);
        mtxz += __shfl_xor_sync(0xffffffffu, mtxz, o);
        mtyy += __shfl_xor_sync(0xffffffffu, mtyy, o);
        mtyz += __shfl_xor_sync(0xffffffffu, mtyz, o);
        mtzz += __shfl_xor_sync(0xffffffffu, mtzz, o);
    }
    if (!COUNT) {
        const float uy = REL ? fmaf(y, p.h, -cy) : y - cy;
        const float uz = REL ? fmaf(z, p.h, -cz) : z - cz;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float ux = REL ? fmaf(x[c], p.h, -cx) : x[c] - cx;
            const float su = fmaf(uz, uz, fmaf(uy, uy, ux * ux));
            const float uq = fmaf(uz, mqz, fmaf(uy, mqy, ux * mqx));
            const float ur = fmaf(uz, mrz, fmaf(uy, mry, ux * mrx));
            const float tx = fmaf(uz, mtxz, fmaf(uy, mtxy, ux * mtxx));
            const float ty = fmaf(uz, mtyz, fmaf(uy, mtyy, ux * mtxy));
            const float tz = fmaf(uz, mtzz, fmaf(uy, mtyz, ux * mtxz));
            const float utu = fmaf(uz, tz, fmaf(uy, ty, ux * tx));
            const float s2 = fmaf(su, mq, fmaf(-2.f, uq, mqm));
            const float s4 = fmaf(su, fmaf(su, mq, fmaf(2.f, mqm, -4.f * uq)), fmaf(4.f, utu, fmaf(-4.f, ur, mqmm)));
            acc[c] += fmaf(NG2.x, s4, fmaf(NG1.x, s2, NG0.x * mq));
        }
    }

    if (COUNT) {
        // per warp: atoms listed for its sub-box, each evaluated against the
        // warp's 128 points; real atoms it sorted; useful = pairs with r < c
        // at stored points
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            n_real += __shfl_down_sync(0xffffffffu, n_real, o);
            n_useful += __shfl_down_sync(0xffffffffu, n_useful, o);
        }
        if (lane == 0) {
            atomicAdd(&p.counts[0], n_useful);
            atomicAdd(&p.counts[1], n_near * 128ull);
            // warp 0 counted every real atom of the stream once; each was
            // examined against all 512 points
            atomicAdd(&p.counts[2], n_real * 128ull * kBrickConsumerWarps);
        }
        return;
    }
    if (j < p.ny && k < p.nz) {
        float *row = p.V + ((long long)k * p.ny + j) * p.nx;
        const long long total = (long long)p.nx * p.ny * p.nz, at = ((long long)k * p.ny + j) * p.nx + i0;
        if (VEC) {
            if (i0 < p.nx && CP_IN(at + 3, total, p.status))
                *reinterpret_cast<float4 *>(row + i0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (i0 + c < p.nx) row[i0 + c] = acc[c];
        }
    }
}

// ---------------------------------------------------------------------------
// host side

namespace {

// Kernel arguments of the binning kernels for the sections of `L` at `ws`.
BinParams bin_params(const float4 *atoms, int n_atoms, const BinGeom &bg, const cp_cutoff_layout &L, void *workspace) {
    char *ws = static_cast<char *>(workspace);
    BinParams b;
    b.atoms = atoms;
    b.n = n_atoms;
    for (int d = 0; d < 3; ++d) {
        b.nb[d] = bg.nb[d];
        b.bo[d] = bg.bo[d];
    }
    b.b = bg.b;
    b.nbins = (int)bg.nbins;
    b.K = L.capacity;
    b.count = reinterpret_cast<int *>(ws + L.off_count);
    b.start = reinterpret_cast<int *>(ws + L.off_start);
    b.csr_index = reinterpret_cast<int *>(ws + L.off_csr_index);
    b.csr_atoms = reinterpret_cast<float4 *>(ws + L.off_csr_atoms);
    b.padded = reinterpret_cast<float4 *>(ws + L.off_padded);
    b.stats = reinterpret_cast<int *>(ws + L.off_stats);
    const size_t n = (size_t)(n_atoms > 0 ? n_atoms : 0);
    const size_t nblk = ((size_t)bg.nbins + kScanBlock - 1) / kScanBlock;
    size_t off = L.off_scratch;
    b.bin_rank = reinterpret_cast<int2 *>(ws + off);
    off += (8 * n + 255) & ~(size_t)255;
    b.block_sums = reinterpret_cast<int *>(ws + off);
    off += (4 * nblk + 255) & ~(size_t)255;
    b.block_prefix = reinterpret_cast<int *>(ws + off);
    b.prefix_inline = 0;
    b.status = device_status_ptr();
    return b;
}

int launch_binning_params(const BinParams &b, cudaStream_t stream, bool small_bins = false) {
    const int nblk = (int)(((long long)b.nbins + kScanBlock - 1) / kScanBlock);
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc) return rc;
    const int clear_blocks = (int)std::min<long long>((b.nbins + 255) / 256, 8LL * dev.sm_count);
    // each launch may be scheduled while the one before it drains (the
    // kernels wait for it before touching memory)
    bool ok = launch_pdl(bin_clear_kernel, std::max(clear_blocks, 1), 256, stream, b);
    if (b.n > 0) ok = ok && launch_pdl(bin_count_kernel, (b.n + 255) / 256, 256, stream, b);
    ok = ok && launch_pdl(bin_scan_local_kernel, nblk, 256, stream, b);
    // up to kInlinePrefixMax block totals the scatter kernel scans itself
    const bool inline_prefix = b.n > 0 && nblk <= kInlinePrefixMax;
    BinParams bs = b;
    bs.prefix_inline = inline_prefix ? nblk : 0;
    if (!inline_prefix) ok = ok && launch_pdl(bin_scan_blocks_kernel, 1, 1024, stream, b, nblk);
    if (b.n > 0) ok = ok && launch_pdl(bin_scatter_kernel, (b.n + 255) / 256, 256, stream, bs);
    if (small_bins)
        ok = ok && launch_pdl(bin_sort_pack_lane_kernel, (int)((b.nbins + 255) / 256), 256, stream, b);
    else
        ok = ok && launch_pdl(bin_sort_pack_kernel, (int)((b.nbins + 7) / 8), 256, stream, b);
    if (!ok) return CP_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(b.n > 0 ? (inline_prefix ? 5 : 6) : 4);
    return CP_OK;
}

struct Prepared {
    Grid g;
    BinGeom bg;
    cp_cutoff_layout L;
    BinParams bp;
};

// Host-only part of the set-up: arguments, bin geometry and workspace layout.
int plan(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
         float bin_size, int capacity, Prepared *out) {
    int rc = check_grid(nx, ny, nz, origin, h, &out->g);
    if (rc) return rc;
    if (n_atoms < 0 || (n_atoms > 0 && !atoms)) return CP_ERR_INVALID_ARGUMENT;
    rc = check_cutoff_args(out->g, cutoff, bin_size, capacity);
    if (rc) return rc;
    if (n_atoms > 0 && !aligned(atoms, 16)) return CP_ERR_MISALIGNED;
    rc = make_bin_geometry(out->g, cutoff, bin_size, &out->bg);
    if (rc) return rc;
    rc = make_layout(n_atoms, out->bg, capacity, &out->L);
    if (rc) return rc;
    if ((long long)out->bg.nbins * capacity > INT_MAX) return CP_ERR_TOO_LARGE;
    return CP_OK;
}

// Places the planned arrays in `workspace` (layout out->L).
int bind(const float *atoms, int n_atoms, void *workspace, size_t workspace_bytes, Prepared *out) {
    if (!workspace) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256)) return CP_ERR_MISALIGNED;
    if (workspace_bytes < out->L.total_bytes) return CP_ERR_WORKSPACE_TOO_SMALL;
    out->bp = bin_params(reinterpret_cast<const float4 *>(atoms), n_atoms, out->bg, out->L, workspace);
    return CP_OK;
}

int prepare(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
            float bin_size, int capacity, void *workspace, size_t workspace_bytes, Prepared *out) {
    if (!workspace) return CP_ERR_INVALID_ARGUMENT;
    int rc = plan(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, out);
    if (rc) return rc;
    return bind(atoms, n_atoms, workspace, workspace_bytes, out);
}

int launch_binning(const Prepared &P, cudaStream_t stream) { return launch_binning_params(P.bp, stream); }

template <int K>
int launch_bricks_k(const Prepared &P, const OffsetList &L, float *V, cudaStream_t stream,
                    unsigned long long *counts = nullptr) {
    const Grid &g = P.g;
    BrickParams p;
    p.nx = g.nx;
    p.ny = g.ny;
    p.nz = g.nz;
    p.ox = g.ox;
    p.oy = g.oy;
    p.oz = g.oz;
    p.h = g.h;
    const double c = P.bg.c;
    p.c2 = (float)(c * c);
    p.cull2 = (float)(c * c * (1.0 + 1.0e-5));
    // An atom is "full" (its pairs taken without the r < c test) only when
    // it is inside c of every point of a sub-box by more than the rounding
    // of the test: 1e-5 of c plus 8 ulps of the largest coordinate near the
    // grid (the sub-box corners and the atoms are fp32 numbers of that size).
    {
        double mag = 0.0;
        const double o[3] = {g.ox, g.oy, g.oz};
        const int n[3] = {g.nx, g.ny, g.nz};
        for (int d = 0; d < 3; ++d)
            mag = std::max(mag, std::max(std::fabs(o[d]), std::fabs(o[d] + (n[d] - 1) * (double)g.h)) + c);
        const double margin = 1.0e-5 * c + 8.0 * mag * std::ldexp(1.0, -24);
        p.full2 = margin < c ? (float)((c - margin) * (c - margin)) : 0.0f;
    }
    p.gc0 = (float)(15.0 / (8.0 * c));
    p.gc1 = (float)(-5.0 / (4.0 * c * c * c));
    p.gc2 = (float)(3.0 / (8.0 * c * c * c * c * c));
    for (int d = 0; d < 3; ++d) p.nb[d] = P.bg.nb[d];
    p.m = P.bg.m;
    p.h64 = (double)g.h;
    p.b64 = (double)P.bg.b;
    p.nbr[0] = (g.nx + kBrick - 1) / kBrick;
    p.nbr[1] = (g.ny + kBrick - 1) / kBrick;
    p.nbr[2] = (g.nz + kBrick - 1) / kBrick;
    p.padded = P.bp.padded;
    p.count = P.bp.count;
    p.start = P.bp.start;
    p.csr_atoms = P.bp.csr_atoms;
    p.n_csr = P.bp.n;
    p.n_padded = (long long)P.bg.nbins * P.bp.K;
    p.V = V;
    p.counts = counts;
    p.status = device_status_ptr();
    if (!p.status) return CP_ERR_CUDA;
    p.n_runs = L.n_runs;
    for (int r = 0; r < L.n_runs; ++r) {
        const unsigned u0 = (unsigned)(uint8_t)L.run[r][0], u1 = (unsigned)(uint8_t)L.run[r][1];
        const unsigned u2 = (unsigned)(uint8_t)L.run[r][2], u3 = (unsigned)(uint8_t)L.run[r][3];
        p.runs[r] = (int)(u0 | (u1 << 8) | (u2 << 16) | (u3 << 24));
    }
    const long long nbricks = (long long)p.nbr[0] * p.nbr[1] * p.nbr[2];
    if (nbricks > 0x7fffffffll) return CP_ERR_TOO_LARGE;
    const bool vec = V && (g.nx % 4 == 0) && aligned(V, 16);
    const bool rel = !grid_points_exact(g);
    const unsigned nb = (unsigned)nbricks;
    bool launched = false;
    if (counts && rel)
        launched = launch_pdl(cutoff_brick_kernel<K, false, true, true>, (int)nb, kBrickThreads, stream, p);
    else if (counts)
        launched = launch_pdl(cutoff_brick_kernel<K, false, true, false>, (int)nb, kBrickThreads, stream, p);
    else if (vec && rel)
        launched = launch_pdl(cutoff_brick_kernel<K, true, false, true>, (int)nb, kBrickThreads, stream, p);
    else if (vec)
        launched = launch_pdl(cutoff_brick_kernel<K, true, false, false>, (int)nb, kBrickThreads, stream, p);
    else if (rel)
        launched = launch_pdl(cutoff_brick_kernel<K, false, false, true>, (int)nb, kBrickThreads, stream, p);
    else
        launched = launch_pdl(cutoff_brick_kernel<K, false, false, false>, (int)nb, kBrickThreads, stream, p);
    if (!launched) return CP_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

int launch_bricks(const Prepared &P, const OffsetList &L, float *V, cudaStream_t stream,
                  unsigned long long *counts = nullptr) {
    switch (P.bp.K) {
        case 0: return launch_bricks_k<0>(P, L, V, stream, counts);
        case 8: return launch_bricks_k<8>(P, L, V, stream, counts);
        default: return launch_bricks_k<16>(P, L, V, stream, counts);
    }
}

}  // namespace

int sort_atoms_into_cells(const float4 *atoms, int n_atoms, const BinGeom &bg, const cp_cutoff_layout &L,
                          void *workspace, cudaStream_t stream) {
    if (L.capacity != 0 || L.nbins != bg.nbins) return CP_ERR_INVALID_ARGUMENT;
    return launch_binning_params(bin_params(atoms, n_atoms, bg, L, workspace), stream, true);
}

}  // namespace cpmap

using namespace cpmap;

extern "C" {

CP_API int cp_bin_atoms(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                        float cutoff, float bin_size, int capacity, void *workspace, size_t workspace_bytes,
                        void *stream) {
    Prepared P;
    int rc = prepare(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, workspace, workspace_bytes,
                     &P);
    if (rc) return rc;
    return launch_binning(P, static_cast<cudaStream_t>(stream));
}

CP_API int cp_cutoff(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h, float cutoff,
                     float bin_size, int capacity, void *workspace, size_t workspace_bytes, float *V, void *stream) {
    if (!V) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    Prepared P;
    int rc = prepare(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, workspace, workspace_bytes,
                     &P);
    if (rc) return rc;
    static thread_local OffsetList L;
    rc = make_offset_list(P.g, P.bg, &L);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_binning(P, s);
    if (rc) return rc;
    return launch_bricks(P, L, V, s);
}

CP_API int cp_cutoff_map(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                         float cutoff, float bin_size, int capacity, void *workspace, size_t workspace_bytes, float *V,
                         void *stream) {
    if (!V) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    Prepared P;
    int rc = prepare(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, workspace, workspace_bytes,
                     &P);
    if (rc) return rc;
    static thread_local OffsetList L;
    rc = make_offset_list(P.g, P.bg, &L);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return launch_bricks(P, L, V, s);
}

CP_API int cp_cutoff_pair_counts(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                                  float cutoff, float bin_size, int capacity, void *workspace,
                                  size_t workspace_bytes, unsigned long long *counts, void *stream) {
    if (!counts) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(counts, 8)) return CP_ERR_MISALIGNED;
    Prepared P;
    int rc = prepare(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, workspace, workspace_bytes,
                     &P);
    if (rc) return rc;
    static thread_local OffsetList L;
    rc = make_offset_list(P.g, P.bg, &L);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counts, 0, 3 * sizeof(unsigned long long), s) != cudaSuccess) return CP_ERR_CUDA;
    rc = launch_binning(P, s);
    if (rc) return rc;
    return launch_bricks(P, L, nullptr, s, counts);
}

CP_API int cp_cutoff_stats(const void *workspace, size_t workspace_bytes, int n_atoms, int nx, int ny, int nz,
                           cp_vec3 origin, float h, float cutoff, float bin_size, int capacity,
                           cp_cutoff_stats_t *out, void *stream) {
    if (!workspace || !out) return CP_ERR_INVALID_ARGUMENT;
    cp_cutoff_layout L;
    int rc = cp_cutoff_layout_of(n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, &L);
    if (rc) return rc;
    if (workspace_bytes < L.total_bytes) return CP_ERR_WORKSPACE_TOO_SMALL;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CP_ERR_CUDA;
    int v[8];
    if (cudaMemcpy(v, static_cast<const char *>(workspace) + L.off_stats, sizeof(v), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return CP_ERR_CUDA;
    out->n_binned = v[0];
    out->n_dropped = v[1];
    out->n_overflow = v[2];
    out->max_bin_count = v[3];
    return CP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free cutoff map.
//
// Some callers cannot hand the library a workspace: a host program whose
// device memory is wholly owned by another allocator (a framework's caching
// pool that has already reserved the device), or code that must not
// allocate once it is running (a fixed memory budget set at start-up, a
// plugin that may only use what its host gave it).  For them the cutoff
// map's scratch lives in a fixed array of this library's module, created
// when the module is loaded on a device and kept until the process exits.
// The caller passes only the atoms and V.

namespace cpmap {
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB per device

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: kernels get the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_static_ws_mutex;
void *g_static_ws_ptr[kMaxDevices];

// Device address of g_static_workspace on the current device, looked up
// once per device (the first call on each device does it).
void *static_workspace_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_ws_mutex);
    if (!g_static_ws_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return nullptr;
        g_static_ws_ptr[dev] = p;
    }
    return g_static_ws_ptr[dev];
}

}  // namespace
}  // namespace cpmap

extern "C" {

CP_API int cp_cutoff_no_alloc(const float *atoms, int n_atoms, int nx, int ny, int nz, cp_vec3 origin, float h,
                              float cutoff, float bin_size, int capacity, float *V, void *stream) {
    if (!V) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(V, 4)) return CP_ERR_MISALIGNED;
    // One layout, computed once: it decides both the size check and where
    // the arrays go in the fixed array.
    Prepared P;
    int rc = plan(atoms, n_atoms, nx, ny, nz, origin, h, cutoff, bin_size, capacity, &P);
    if (rc) return rc;
    if (P.L.total_bytes > kStaticWorkspaceBytes) return CP_ERR_TOO_LARGE;  // beyond the fixed 16 MiB
    void *ws = static_workspace_ptr();
    if (!ws) return CP_ERR_CUDA;
    // Every call reuses the same array and finds the previous call's bins in
    // it.  Nothing carries over: the binning stage zeroes the per-bin counters
    // and the counters block before counting, and every other array is
    // rewritten in full before it is read.
    rc = bind(atoms, n_atoms, ws, kStaticWorkspaceBytes, &P);
    if (rc) return rc;
    static thread_local OffsetList OL;
    rc = make_offset_list(P.g, P.bg, &OL);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_binning(P, s);
    if (rc) return rc;
    return launch_bricks(P, OL, V, s);
}

}  // extern "C"
