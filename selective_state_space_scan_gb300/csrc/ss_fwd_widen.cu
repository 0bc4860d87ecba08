// Widening pass of the workspace schedules for bf16 I/O: B and C [batch, L, N] bf16 (any strides
// the TMA path accepts) copied to fp32 [batch, L, N] contiguous in the workspace, four states per
// thread.  A bf16 value is the high half of the fp32 with the same value, so the copy is exact.
#include "device_common.cuh"
#include "internal.h"

namespace selscan {

__global__ void __launch_bounds__(256)
ss_widen_bc_kernel(const __nv_bfloat16* __restrict__ B, const __nv_bfloat16* __restrict__ C, int64_t B_b, int64_t B_l,
                   int64_t C_b, int64_t C_l, float* __restrict__ Bf, float* __restrict__ Cf, int64_t batch, int64_t L,
                   int N) {
    const int quads = N / 4;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= batch * L * quads) return;
    const int q = static_cast<int>(i % quads);
    const int64_t row = i / quads;
    const int64_t b = row / L, t = row - b * L;
    auto widen = [](uint2 v) {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    };
    const uint2 vb = *reinterpret_cast<const uint2*>(B + b * B_b + t * B_l + 4 * q);
    const uint2 vc = *reinterpret_cast<const uint2*>(C + b * C_b + t * C_l + 4 * q);
    reinterpret_cast<float4*>(Bf)[i] = widen(vb);
    reinterpret_cast<float4*>(Cf)[i] = widen(vc);
}

cudaError_t launch_widen_bc(const void* B, const void* C, int64_t B_b, int64_t B_l, int64_t C_b, int64_t C_l,
                            float* Bf, float* Cf, int64_t batch, int64_t L, int N, cudaStream_t stream) {
    const int64_t count = batch * L * (N / 4);
    if (count <= 0) return cudaSuccess;
    const int64_t blocks = (count + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    ss_widen_bc_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), B_b, B_l, C_b, C_l, Bf, Cf, batch,
        L, N);
    return cudaGetLastError();
}

}  // namespace selscan
