// probe.cu -- measurement utility: the GPU's sustained MUFU ex2 rate, which is
// the exponential roof of the scoring kernel (one ex2 per visible logit).  Not
// part of the method.
#include "../../include/up.h"
#include "common.cuh"
#include "sm100.cuh"

namespace up {

namespace {

constexpr int kProbeThreads = 1024;
constexpr int kChains = 8;
constexpr int kIters = 4096;

__device__ float g_probe_sink;

// Every thread runs kChains independent chains x <- 2^-x (the values stay in
// (0, 1)); at two CTAs of 1024 threads per SM there are 16 warps per SM
// sub-partition, enough to keep the MUFU busy.
__global__ void __launch_bounds__(kProbeThreads, 2) ex2_rate_kernel(int iters) {
    float a[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) a[j] = 0.125f * (float)(threadIdx.x & 7) + 0.01f * (float)j;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) a[j] = sm100::ex2_approx(-a[j]);
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += a[j];
    if (s == 12345.0f) g_probe_sink = s;  // keeps the chains alive
}

}  // namespace

}  // namespace up

extern "C" up_status up_measure_ex2_rate(double *ex2_per_second, up_stream_t stream) {
    if (!ex2_per_second) return UP_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return UP_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    up_status status = UP_ERR_CUDA;
    if (cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
        const dim3 grid(2 * sms), block(up::kProbeThreads);
        up::ex2_rate_kernel<<<grid, block, 0, st>>>(64);  // warm-up
        cudaEventRecord(e0, st);
        up::ex2_rate_kernel<<<grid, block, 0, st>>>(up::kIters);
        cudaEventRecord(e1, st);
        float ms = 0.f;
        if (cudaGetLastError() == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
            cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess && ms > 0.f) {
            const double n = (double)grid.x * up::kProbeThreads * up::kChains * up::kIters;
            *ex2_per_second = n / (ms * 1e-3);
            status = UP_OK;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return status;
}
