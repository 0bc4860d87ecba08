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
    kErrGeometry = 2u,      // launch geometry disagrees with the kernel's tile shape
};

// 2^x on the SFU (ex2.approx.ftz: inputs below -126 flush to 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the SFU (rcp.approx.ftz).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Coefficients of P(w) ~ 2·atanh(sqrt(w))/sqrt(w) on w in [0, 1/9], degree 4: fitted by
// iteratively reweighted least squares on the relative error (approaching the minimax fit);
// the approximation error is below 4e-9 relative, far under fp32 rounding.
constexpr float kLog1pP0 = 2.0f;
constexpr float kLog1pP1 = 0.6666631698608398f;
constexpr float kLog1pP2 = 0.40024885535240173f;
constexpr float kLog1pP3 = 0.27960675954818726f;
constexpr float kLog1pP4 = 0.28178852796554565f;

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e), e = e^{-|x|} in (0, 1].
// log1p(e) = 2·atanh(m) with m = e / (2 + e) in (0, 1/3] (the identity
// ln((1+m)/(1-m)) = 2·atanh(m) at (1+m)/(1-m) = 1+e), evaluated as m·P(m²).
// No branch and no overflow for any finite x; 13 instructions, 2 of them on the SFU.
// Relative error about 3e-7 at x ~ -5 (dominated by rounding x·log2(e)).
__device__ __forceinline__ float softplus(float x) {
    const float e = ex2(-fabsf(x) * kLog2e);
    const float m = e * rcp_approx(2.f + e);
    const float w = m * m;
    float p = fmaf(w, kLog1pP4, kLog1pP3);
    p = fmaf(w, p, kLog1pP2);
    p = fmaf(w, p, kLog1pP1);
    p = fmaf(w, p, kLog1pP0);
    return fmaf(m, p, fmaxf(x, 0.f));
}

// silu(z) = z · sigmoid(z) = z / (1 + e^{-z}); e^{-z} -> inf gives z · 0.
__device__ __forceinline__ float silu(float z) {
    return z * rcp_approx(1.f + ex2(-z * kLog2e));
}

// A run of steps of the recurrence acts on the state as the affine map h -> a·h + b, kept as the
// pair (a, b).  Running `earlier` and then `later` is again such a map, with
// a = a_later·a_earlier and b = a_later·b_earlier + b_later: the associative operator the scans
// combine with ("mamba-metal: Apple Silicon で Mamba を動かす", section "Selective scan の本質").
struct AffinePair {
    float a, b;
};
__device__ __forceinline__ AffinePair compose(AffinePair later, AffinePair earlier) {
    return AffinePair{later.a * earlier.a, fmaf(later.a, earlier.b, later.b)};
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic on sm_100+).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 ex2x2(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }
__device__ __forceinline__ float2 rcp2(float2 v) { return make_float2(rcp_approx(v.x), rcp_approx(v.y)); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// softplus of two independent values (two steps of one channel): the same arithmetic as
// softplus(), with the polynomial and the surrounding products on packed pairs, so one
// instruction serves both (the SFU operations stay one per value).
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 e = make_float2(ex2(-fabsf(x.x) * kLog2e), ex2(-fabsf(x.y) * kLog2e));
    const float2 m = mul2(e, rcp2(add2(splat2(2.f), e)));
    const float2 w = mul2(m, m);
    float2 p = fma2(w, splat2(kLog1pP4), splat2(kLog1pP3));
    p = fma2(w, p, splat2(kLog1pP2));
    p = fma2(w, p, splat2(kLog1pP1));
    p = fma2(w, p, splat2(kLog1pP0));
    return fma2(m, p, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

// log2(x) on the SFU (lg2.approx.ftz).
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLn2 = 0.6931471805599453f;

// softplus of two values for bf16 outputs: log(1 + e^x) = max(x, 0) + ln 2 · log2(1 + e^{-|x|})
// with the SFU's log2, 5 instructions a value against softplus2's 8.  Its relative error is
// about 2e-5 at x ~ -5 (the rounding of 1 + e^{-|x|} and lg2.approx's absolute error, over a
// result of ~e^x), two orders below bf16's own 2^-9 rounding of the output.
__device__ __forceinline__ float2 softplus2_lg2(float2 x) {
    const float2 e = make_float2(ex2(-fabsf(x.x) * kLog2e), ex2(-fabsf(x.y) * kLog2e));
    const float2 s = add2(splat2(1.f), e);
    return fma2(make_float2(lg2_approx(s.x), lg2_approx(s.y)), splat2(kLn2),
                make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

// silu of two independent values, as silu() with packed products.
__device__ __forceinline__ float2 silu2(float2 z) {
    const float2 e = ex2x2(mul2(z, splat2(-kLog2e)));
    return mul2(z, rcp2(add2(splat2(1.f), e)));
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

// The same with acquire at cluster scope, for a barrier that threads of other CTAs of the cluster
// arrive on (their stores before arriving are visible once the phase is seen complete).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the barrier phase with the given parity.  Gives up after ~2^31 SM cycles
// (about a second at GB300 clocks), records kErrWaitTimeout, and raises the block's
// abort flag so that later waits return at once; the caller then finishes its loop
// without blocking, so no thread is left waiting on a barrier.  CLUSTER_SCOPE: arrivals come
// from other CTAs of the cluster.
template <bool CLUSTER_SCOPE = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  unsigned int* err_word) {
    auto try_wait = [&]() { return CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (*abort_flag) return false;
    if (try_wait()) return true;
    const long long t0 = clock64();
    while (!try_wait()) {
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

// 3-D TMA tile store from shared memory (bulk async-group completion).  Rows and columns past
// the tensor's ends are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
        : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until the committed stores have read their shared-memory source.
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until the committed stores are complete.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Makes this thread's shared-memory writes visible to the async proxy (a later TMA store).
__device__ __forceinline__ void tma_store_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// into shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Thread-block clusters: this CTA's rank in its cluster, a barrier over every thread of the
// cluster (release/acquire: shared-memory writes before it are visible to the cluster's CTAs
// after it; a hardware barrier, so no wait to bound), and loads from a cluster peer's shared
// memory at the address that a local shared-memory pointer has in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_smem_addr(const void* local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_peer_f32x4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
// One arrival (release at cluster scope: this thread's earlier stores, to any CTA of the cluster,
// become visible to a thread that then sees the phase complete) on an mbarrier in a peer's shared
// memory, at the address peer_smem_addr gives.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads'.
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace selscan
