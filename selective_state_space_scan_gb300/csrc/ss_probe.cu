// Pipe-rate probe: how many results per clock one SM delivers for the operations the scan's
// roofline is built from.  The selective scan takes one exp2 per state update (the decay
// exp(Δ·A) = 2^(Δ·A·log2 e)) and about four fp32 multiply-adds, so its arithmetic floor is the
// slower of the SFU's ex2 rate and the FMA pipe's rate; neither is a documented constant on
// sm_103a, so the library measures them.
//
// Method: one CTA per SM (the dynamic shared memory asked for leaves room for one), 16 warps,
// each thread running 8 independent dependency chains of the probed operation, so the pipe,
// not latency, sets the pace.  Thread 0 reads the SM's cycle counter after a block barrier
// before and after the loop; results per clock = operations issued on the SM / elapsed cycles.
// Clock-independent, so the peak follows as SMs × rate × the SM clock.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "device_common.cuh"

namespace selscan {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeChains = 8;
constexpr int kProbeSmem = 150 * 1024;    // more than half an SM's shared memory: one CTA per SM

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// KIND 0: ex2 (x <- 2^-x stays in [0.5, 1]); 1: rcp (x <- 1/(1 + x)); 2: lg2 (x <- log2(1 + x));
// 3: tanh (x <- tanh(x + 0.5)); 4: scalar FFMA; 5: packed FFMA2 (two fp32 FMAs per result).
template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) ss_pipe_probe_kernel(int iters, float a, float b,
                                                                      long long* cycles, float* sink) {
    extern __shared__ float probe_smem[];
    float x[kProbeChains];
    float2 v[kProbeChains];
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) {
        x[k] = 0.5f + 0.01f * static_cast<float>((threadIdx.x + k) & 31);
        v[k] = make_float2(x[k], 1.f - x[k]);
    }
    __syncthreads();
    const long long t0 = clock64();
#pragma unroll 4
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kProbeChains; ++k) {
            if constexpr (KIND == 0) x[k] = ex2(-x[k]);
            if constexpr (KIND == 1) x[k] = rcp_approx(x[k] + 1.f);
            if constexpr (KIND == 2) x[k] = lg2_approx(x[k] + 1.f);
            if constexpr (KIND == 3) x[k] = tanh_approx(x[k] + 0.5f);
            if constexpr (KIND == 4) x[k] = fmaf(x[k], a, b);
            if constexpr (KIND == 5) v[k] = fma2(v[k], make_float2(a, a), make_float2(b, b));
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kProbeChains; ++k) s += x[k] + v[k].x + v[k].y;
    if (s == 12345.678f) sink[threadIdx.x] = s + probe_smem[threadIdx.x];   // keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND>
cudaError_t run_probe(int sms, int iters, long long* d_cycles, float* d_sink) {
    auto kern = ss_pipe_probe_kernel<KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
    if (e != cudaSuccess) return e;
    kern<<<sms, kProbeThreads, kProbeSmem>>>(iters, 0.999f, 1e-4f, d_cycles, d_sink);
    return cudaGetLastError();
}

}  // namespace
}  // namespace selscan

using namespace selscan;

// Internal measurement hook (not in the public header): runs the probe of `kind` (0 ex2,
// 1 rcp, 2 lg2, 3 tanh, 4 FFMA, 5 FFMA2) on the current device and returns in *per_clk_per_sm
// the results per clock per SM (for FFMA2: fp32 FMAs, two per instruction lane), the median
// over the SMs.  Synchronises the device.  Returns 0, or -1 on a bad argument or CUDA error.
extern "C" int ss__pipe_probe(int kind, int iters, double* per_clk_per_sm) {
    if (!per_clk_per_sm || kind < 0 || kind > 5 || iters < 16 || iters > (1 << 24)) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return -1;
    long long* d_cycles = nullptr;
    float* d_sink = nullptr;
    if (cudaMalloc(&d_cycles, sizeof(long long) * sms) != cudaSuccess) return -1;
    if (cudaMalloc(&d_sink, sizeof(float) * kProbeThreads) != cudaSuccess) {
        cudaFree(d_cycles);
        return -1;
    }
    cudaError_t e = cudaSuccess;
    switch (kind) {
        case 0: e = run_probe<0>(sms, iters, d_cycles, d_sink); break;
        case 1: e = run_probe<1>(sms, iters, d_cycles, d_sink); break;
        case 2: e = run_probe<2>(sms, iters, d_cycles, d_sink); break;
        case 3: e = run_probe<3>(sms, iters, d_cycles, d_sink); break;
        case 4: e = run_probe<4>(sms, iters, d_cycles, d_sink); break;
        default: e = run_probe<5>(sms, iters, d_cycles, d_sink); break;
    }
    std::vector<long long> cyc(sms, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(cyc.data(), d_cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
    cudaFree(d_cycles);
    cudaFree(d_sink);
    if (e != cudaSuccess) return -1;
    std::sort(cyc.begin(), cyc.end());
    const long long med = cyc[sms / 2];
    if (med <= 0) return -1;
    const double ops = static_cast<double>(kProbeThreads) * iters * kProbeChains * (kind == 5 ? 2.0 : 1.0);
    *per_clk_per_sm = ops / static_cast<double>(med);
    return 0;
}
