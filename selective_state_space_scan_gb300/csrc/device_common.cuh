// Device-side helpers shared by the selective-scan kernels: MUFU exponentials,
// the shared-memory swizzle that matches the TMA tile layout, mbarrier waits with a
// time limit, and TMA tile loads.  All hand-written inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace selscan {

constexpr float kLog2e = 1.4426950408889634f;

// Error bits written to the library's device error word.
enum : unsigned int {
    kErrWaitTimeout = 1u,   // an mbarrier wait for a TMA tile exceeded its limit
};

// 2^x on the SFU (ex2.approx.ftz: inputs below -126 flush to 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(x) = log(1 + exp(x)); the identity above x = 20 avoids exp overflow and is
// exact to fp32 precision there (log1p(e^-20) < 2^-24 · 20).
__device__ __forceinline__ float softplus(float x) {
    return x <= 20.f ? log1pf(expf(x)) : x;
}

// silu(z) = z · sigmoid(z) = z / (1 + e^{-z}).
__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.f + __expf(-z));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Byte offset inside a tile whose rows are RB bytes, after the TMA swizzle that a tensor
// map with CU_TENSOR_MAP_SWIZZLE_{128,64,32}B (chosen as RB) applies: address bits [4,7)
// (the 16-byte chunk) are XORed with bits [7,10) of the same offset, masked to the span.
template <int RB>
__device__ __forceinline__ uint32_t swz(uint32_t o) {
    constexpr uint32_t M = RB >= 128 ? 7u : RB == 64 ? 3u : RB == 32 ? 1u : 0u;
    return o ^ (((o >> 7) & M) << 4);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the barrier phase with the given parity.  Gives up after ~2^31 SM cycles
// (about a second at GB300 clocks), records kErrWaitTimeout, and raises the block's
// abort flag so that later waits return at once; the caller then finishes its loop
// without blocking, so no thread is left waiting on a barrier.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  unsigned int* err_word) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > (1ll << 31)) {
            *abort_flag = 1;
            if (err_word) atomicOr(err_word, kErrWaitTimeout);
            return false;
        }
    }
    return true;
}

// 3-D TMA tile load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads'.
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace selscan
