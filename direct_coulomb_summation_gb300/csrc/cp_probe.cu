// cp_probe.cu -- microbenchmarks of the SM pipes the potential map runs on:
// the SFU (MUFU) reciprocal square root and the FP32 FMA pipe.  They give
// the per-SM, per-clock
// throughputs that the roofline of the direct and cutoff kernels is built
// from.  One CTA per SM (a large shared-memory request keeps a second CTA
// off the SM); each CTA times itself with clock64, so the rate is per SM
// clock cycle whatever the clock frequency was.
#include <cuda_runtime.h>

#include <vector>

#include "cp_device.cuh"
#include "cp_internal.h"

namespace cpmap {

constexpr int kProbeChains = 8;
constexpr int kProbeSmem = 160 * 1024;

template <int KIND>
__global__ void probe_kernel(int iters, float seed, long long *cycles, float *sink) {
    float v[kProbeChains];
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) v[c] = seed + 0.001f * (float)(threadIdx.x + c);
    __syncthreads();
    long long t0 = 0;
    if (threadIdx.x == 0) t0 = clock64();
    __syncthreads();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kProbeChains; ++c) {
            if (KIND == 0) {
                v[c] = sfu_rsqrt(v[c]);
            } else if (KIND == 1) {
                v[c] = fmaf(v[c], 0.999f, 0.0013f);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) cycles[blockIdx.x] = clock64() - t0;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) s += v[c];
    if (s == 12345.678f) sink[threadIdx.x] = s;  // keeps the chains alive
}

template <int KIND>
__global__ void eval_rsqrt_kernel(const float *x, float *y, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float2 v = make_float2(x[i], i + 1 < n ? x[i + 1] : 1.0f);
    float2 r;
    if (KIND == 0)
        r = make_float2(sfu_rsqrt(v.x), sfu_rsqrt(v.y));
    else
        r = __fmul2_rn(fma_rsqrt2_scaled(v), make_float2(kSqrt2, kSqrt2));
    y[i] = r.x;
    if (i + 1 < n) y[i + 1] = r.y;
}

// One thread waits on a shared-memory barrier that nothing arrives at, with
// the kernels' bounded wait cut to limit_ns: the wait gives up, records
// CP_DEVICE_WAIT_TIMEOUT and the kernel returns.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, unsigned int *status, int *gave_up) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_init_fence();
    *gave_up = mbar_wait_limit(&bar, 0, status, limit_ns) ? 0 : 1;
}

}  // namespace cpmap

using namespace cpmap;

extern "C" {

CP_API int cp_eval_rsqrt(int kind, const float *x, float *y, int n, void *stream) {
    if ((kind != 0 && kind != 1) || n < 0 || (n > 0 && (!x || !y))) return CP_ERR_INVALID_ARGUMENT;
    if (n == 0) return CP_OK;
    const int threads = 256;
    const int blocks = (int)(((long long)(n + 1) / 2 + threads - 1) / threads);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kind == 0)
        eval_rsqrt_kernel<0><<<blocks, threads, 0, s>>>(x, y, n);
    else
        eval_rsqrt_kernel<1><<<blocks, threads, 0, s>>>(x, y, n);
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

CP_API int cp_probe_pipe_rate(int kind, int warps, int iters, double *ops_per_clk, double *ms, void *stream) {
    if (kind < 0 || kind > 1 || warps < 1 || warps > 32 || iters < 1 || !ops_per_clk) return CP_ERR_INVALID_ARGUMENT;
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    long long *cycles = nullptr;
    float *sink = nullptr;
    if (cudaMalloc(&cycles, sizeof(long long) * dev.sm_count) != cudaSuccess) return CP_ERR_CUDA;
    if (cudaMalloc(&sink, sizeof(float) * 1024) != cudaSuccess) {
        cudaFree(cycles);
        return CP_ERR_CUDA;
    }
    void (*fns[2])(int, float, long long *, float *) = {probe_kernel<0>, probe_kernel<1>};
    auto fn = fns[kind];
    rc = CP_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) != cudaSuccess ||
        cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        rc = CP_ERR_CUDA;
    } else {
        fn<<<dev.sm_count, warps * 32, kProbeSmem, s>>>(16, 0.75f, cycles, sink);  // warm-up
        cudaEventRecord(e0, s);
        fn<<<dev.sm_count, warps * 32, kProbeSmem, s>>>(iters, 0.75f, cycles, sink);
        cudaEventRecord(e1, s);
        if (cudaStreamSynchronize(s) != cudaSuccess) rc = CP_ERR_CUDA;
        note_launches(2);
    }
    if (rc == CP_OK) {
        std::vector<long long> cyc(dev.sm_count);
        float t = 0.f;
        if (cudaMemcpy(cyc.data(), cycles, sizeof(long long) * dev.sm_count, cudaMemcpyDeviceToHost) != cudaSuccess ||
            cudaEventElapsedTime(&t, e0, e1) != cudaSuccess) {
            rc = CP_ERR_CUDA;
        } else {
            const double ops = (double)warps * 32.0 * kProbeChains * (double)iters;
            double sum = 0.0;
            for (long long c : cyc) sum += ops / (double)(c > 0 ? c : 1);
            *ops_per_clk = sum / dev.sm_count;
            if (ms) *ms = t;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(cycles);
    cudaFree(sink);
    return rc;
}

CP_API int cp_probe_wait_timeout(unsigned long long limit_ns, int *gave_up, void *stream) {
    if (!gave_up || limit_ns == 0 || limit_ns > kWaitLimitNs) return CP_ERR_INVALID_ARGUMENT;
    if (!aligned(gave_up, 4)) return CP_ERR_MISALIGNED;
    unsigned int *status = device_status_ptr();
    if (!status) return CP_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status, gave_up);
    if (cudaGetLastError() != cudaSuccess) return CP_ERR_CUDA;
    note_launches(1);
    return CP_OK;
}

}  // extern "C"
