// Single-token decode update of the selective SSM (the O(1)-per-token step of
// "mamba-metal: Apple Silicon で Mamba を動かす", section "O(L) インクリメンタルデコード"):
//   Δ          = softplus(delta_raw[b,d] + delta_bias[d])
//   h[b,d,n]  <- exp(Δ A_n) h[b,d,n] + Δ x[b,d] B[b,n],    A_n = -exp(A_log[d,n])
//   y[b,d]     = (Σ_n C[b,n] h[b,d,n] + D[d] x[b,d]) · silu(z[b,d])
// The state is updated in place.  The step is elementwise over (b,d) and HBM-bound on the
// state read + write (16 states x 8 bytes per row against 16 bytes of x, Δ, z, y), so the
// kernel is a stream: LPR lanes per (b,d) row, each lane owning four consecutive states (one
// 16-byte load and store of h), RPT rows per thread with every load of all of them issued
// before any arithmetic (bytes in flight hide HBM latency), the partial C·h sums reduced
// across the row's lanes by shuffles.  Block x covers rows of batch row x / blocks_per_b: one
// 32-bit division per block, none per element.
// exp(A_log) is taken on the SFU (2^(A_log·log2 e)); its relative error (~1e-7) moves the
// decay exponent by as much, far below the fp32 tolerance.
#include "device_common.cuh"
#include "fwd_params.h"
#include "internal.h"

namespace selscan {

// Threads per block: small blocks (2 warps) measured 5% faster per layer than 256-thread ones
// (11.1 against 11.7 us on the 48-layer decode), 32 or 512 slower.
constexpr int kStepThreads = 64;

// Resident blocks per SM the many-layer kernel's registers are sized for: the step is bound by
// the state loads in flight, so occupancy pays.  At 24 blocks (at most 42 registers) the 48-layer
// launch measured 391 us against 455 us unbounded (56 registers, 52% occupancy) and 420 us at 32
// blocks (32 registers, with spills).  The single-layer kernel stays unbounded: its short
// launches measured 10.8 us a layer unbounded against 12.4 us at 24 blocks.
#ifndef SS_STEPL_MINB
#define SS_STEPL_MINB 24
#endif

template <typename TIO> struct Vec4;
template <> struct Vec4<float> {
    using T = float4;
    static __device__ __forceinline__ float4 get(const T& v) { return v; }
};
template <> struct Vec4<__nv_bfloat16> {
    using T = uint2;   // four bf16
    static __device__ __forceinline__ float4 get(const T& v) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// One row's decode update with the state already loaded (VEC path): returns this lane's C·h
// partial sum and writes the new state back.
__device__ __forceinline__ float step_quad(float4& hv, const float4& av, const float4& Bv,
                                           const float4& Cv, float dlt, float dx) {
    const float k = -dlt * kLog2e;
    const float h0 = fmaf(ex2(k * ex2(av.x * kLog2e)), hv.x, dx * Bv.x);
    const float h1 = fmaf(ex2(k * ex2(av.y * kLog2e)), hv.y, dx * Bv.y);
    const float h2 = fmaf(ex2(k * ex2(av.z * kLog2e)), hv.z, dx * Bv.z);
    const float h3 = fmaf(ex2(k * ex2(av.w * kLog2e)), hv.w, dx * Bv.w);
    hv = make_float4(h0, h1, h2, h3);
    return fmaf(Cv.x, h0, fmaf(Cv.y, h1, fmaf(Cv.z, h2, Cv.w * h3)));
}


// The work of block `block` of one layer's step (blocks_per_b row blocks per batch row).
template <typename TIO, int LPR, int RPT, bool VEC, int THREADS = kStepThreads>
__device__ __forceinline__ void step_block(const StepParams& p, int block, int blocks_per_b) {
    constexpr int ROWS_PASS = THREADS / LPR;         // rows one pass of the block covers
    const int b = block / blocks_per_b;
    const int blk = block - b * blocks_per_b;
    const int qd = threadIdx.x % LPR;
    const int d0 = blk * (ROWS_PASS * RPT) + threadIdx.x / LPR;
    const TIO* x = static_cast<const TIO*>(p.x) + static_cast<int64_t>(b) * p.x_b;
    const TIO* dr = static_cast<const TIO*>(p.delta) + static_cast<int64_t>(b) * p.d_b;
    const TIO* zz = p.z ? static_cast<const TIO*>(p.z) + static_cast<int64_t>(b) * p.z_b : nullptr;
    const TIO* Bm = static_cast<const TIO*>(p.Bm) + static_cast<int64_t>(b) * p.B_b;
    const TIO* Cm = static_cast<const TIO*>(p.Cm) + static_cast<int64_t>(b) * p.C_b;
    float* hb = p.state + static_cast<int64_t>(b) * p.s_b;

    if constexpr (VEC) {
        // B and C of this batch row, this lane's quad (shared by every row of the block)
        const int n0 = qd * 4;
        const bool q_ok = n0 < p.N;
        float4 Bv = make_float4(0.f, 0.f, 0.f, 0.f), Cv = Bv;
        if (q_ok) {
            Bv = Vec4<TIO>::get(*reinterpret_cast<const typename Vec4<TIO>::T*>(Bm + n0));
            Cv = Vec4<TIO>::get(*reinterpret_cast<const typename Vec4<TIO>::T*>(Cm + n0));
        }
        // issue every load of the RPT rows first
        float4 hv[RPT], av[RPT];
        float xv[RPT], dv[RPT], zv[RPT];
        bool ok[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int d = d0 + i * ROWS_PASS;
            ok[i] = d < p.Dm;
            hv[i] = av[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            xv[i] = dv[i] = zv[i] = 0.f;
            if (ok[i]) {
                xv[i] = to_f32<TIO>(x[d]);
                dv[i] = to_f32<TIO>(dr[d]) + (p.bias ? p.bias[d] : 0.f);
                if (zz) zv[i] = to_f32<TIO>(zz[d]);
                if (q_ok) {
                    hv[i] = *reinterpret_cast<const float4*>(hb + static_cast<int64_t>(d) * p.s_d + n0);
                    av[i] = *reinterpret_cast<const float4*>(p.A_log + static_cast<int64_t>(d) * p.N + n0);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int d = d0 + i * ROWS_PASS;
            const float dlt = softplus(dv[i]);
            float partial = 0.f;
            if (ok[i] && q_ok) {
                partial = step_quad(hv[i], av[i], Bv, Cv, dlt, dlt * xv[i]);
                *reinterpret_cast<float4*>(hb + static_cast<int64_t>(d) * p.s_d + n0) = hv[i];
            }
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) partial += __shfl_xor_sync(0xffffffffu, partial, off);
            if (ok[i] && qd == 0) {
                float v = fmaf(p.Dv ? p.Dv[d] : 0.f, xv[i], partial);
                if (zz) v *= silu(zv[i]);
                static_cast<TIO*>(p.y)[static_cast<int64_t>(b) * p.y_b + d] = from_f32<TIO>(v);
            }
        }
    } else {
        // any N, strides or alignment: scalar states
#pragma unroll 1
        for (int i = 0; i < RPT; ++i) {
            const int d = d0 + i * ROWS_PASS;
            const bool row_ok = d < p.Dm;
            float partial = 0.f, xv = 0.f, zv = 0.f;
            if (row_ok) {
                xv = to_f32<TIO>(x[d]);
                const float dlt = softplus(to_f32<TIO>(dr[d]) + (p.bias ? p.bias[d] : 0.f));
                const float dx = dlt * xv;
                if (zz) zv = to_f32<TIO>(zz[d]);
                float* h = hb + static_cast<int64_t>(d) * p.s_d;
                const float* al = p.A_log + static_cast<int64_t>(d) * p.N;
                for (int n0 = qd * 4; n0 < p.N; n0 += LPR * 4) {
                    for (int jj = 0; jj < 4 && n0 + jj < p.N; ++jj) {
                        const int n = n0 + jj;
                        const float a = ex2(-dlt * kLog2e * ex2(al[n] * kLog2e));
                        const float hn = fmaf(a, h[n], dx * to_f32<TIO>(Bm[n]));
                        h[n] = hn;
                        partial = fmaf(to_f32<TIO>(Cm[n]), hn, partial);
                    }
                }
            }
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) partial += __shfl_xor_sync(0xffffffffu, partial, off);
            if (row_ok && qd == 0) {
                float v = fmaf(p.Dv ? p.Dv[d] : 0.f, xv, partial);
                if (zz) v *= silu(zv);
                static_cast<TIO*>(p.y)[static_cast<int64_t>(b) * p.y_b + d] = from_f32<TIO>(v);
            }
        }
    }
}

template <int LPR, int RPT, int THREADS = kStepThreads>
__device__ __forceinline__ int step_blocks_per_b(int Dm) {
    constexpr int rows_block = (THREADS / LPR) * RPT;
    return static_cast<int>((static_cast<int64_t>(Dm) + rows_block - 1) / rows_block);
}

template <typename TIO, int LPR, int RPT, bool VEC>
__global__ void __launch_bounds__(kStepThreads) ss_step_kernel(const StepParams p) {
    step_block<TIO, LPR, RPT, VEC>(p, static_cast<int>(blockIdx.x), step_blocks_per_b<LPR, RPT>(p.Dm));
}

// Many layers' steps in one launch: block x works on layer x / blocks_per_layer.  The layers
// share sizes and strides; their pointers come from the parameter block.

template <typename TIO, int LPR, int RPT, bool VEC, int THREADS>
__global__ void __launch_bounds__(THREADS, SS_STEPL_MINB) ss_step_layers_kernel(const __grid_constant__ StepLayersParams q) {
    const int per_b = step_blocks_per_b<LPR, RPT, THREADS>(q.common.Dm);
    const int per_layer = per_b * q.common.batch;
    const int layer = static_cast<int>(blockIdx.x) / per_layer;
    if (layer >= q.n_layers) return;
    StepParams p = q.common;
    const StepLayerPtrs& L = q.layer[layer];
    p.state = L.state; p.x = L.x; p.delta = L.delta; p.z = L.z; p.Bm = L.Bm; p.Cm = L.Cm;
    p.bias = L.bias; p.A_log = L.A_log; p.Dv = L.Dv; p.y = L.y;
    step_block<TIO, LPR, RPT, VEC, THREADS>(p, static_cast<int>(blockIdx.x) - layer * per_layer, per_b);
}

template <typename TIO, int LPR, int THREADS, int RPT>
static cudaError_t launch_step_layers_s(const StepLayersParams& q, bool vec, cudaStream_t stream) {
    constexpr int rows_block = (THREADS / LPR) * RPT;
    const int64_t blocks = (static_cast<int64_t>(q.common.Dm) + rows_block - 1) / rows_block * q.common.batch *
                           q.n_layers;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (vec)
        ss_step_layers_kernel<TIO, LPR, RPT, true, THREADS><<<grid, THREADS, 0, stream>>>(q);
    else
        ss_step_layers_kernel<TIO, LPR, RPT, false, THREADS><<<grid, THREADS, 0, stream>>>(q);
    return cudaGetLastError();
}

// The same block shape as the single-layer launch: over the 48-layer decode workload it measured
// 426 us against 444-612 us for 128 or 256 threads and 2 or 4 rows per thread.
template <typename TIO, int LPR>
static cudaError_t launch_step_layers_t(const StepLayersParams& q, bool vec, cudaStream_t stream) {
    return launch_step_layers_s<TIO, LPR, kStepThreads, 2>(q, vec, stream);
}

template <typename TIO>
static cudaError_t launch_step_layers_dtype(const StepLayersParams& q, bool vec, cudaStream_t stream) {
    const int quads = (q.common.N + 3) / 4;
    if (quads <= 1) return launch_step_layers_t<TIO, 1>(q, vec, stream);
    if (quads <= 2) return launch_step_layers_t<TIO, 2>(q, vec, stream);
    return launch_step_layers_t<TIO, 4>(q, vec, stream);
}

template <typename TIO, int LPR>
static cudaError_t launch_step_t(const StepParams& p, bool vec, cudaStream_t stream) {
    constexpr int RPT = 2;
    constexpr int rows_block = (kStepThreads / LPR) * RPT;
    const int64_t blocks = (static_cast<int64_t>(p.Dm) + rows_block - 1) / rows_block * p.batch;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (vec)
        ss_step_kernel<TIO, LPR, RPT, true><<<grid, kStepThreads, 0, stream>>>(p);
    else
        ss_step_kernel<TIO, LPR, RPT, false><<<grid, kStepThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO>
static cudaError_t launch_step_dtype(const StepParams& p, bool vec, cudaStream_t stream) {
    const int quads = (p.N + 3) / 4;
    if (quads <= 1) return launch_step_t<TIO, 1>(p, vec, stream);
    if (quads <= 2) return launch_step_t<TIO, 2>(p, vec, stream);
    return launch_step_t<TIO, 4>(p, vec, stream);
}

cudaError_t launch_step(const StepParams& p, bool bf16, bool vec, cudaStream_t stream) {
    return bf16 ? launch_step_dtype<__nv_bfloat16>(p, vec, stream)
                : launch_step_dtype<float>(p, vec, stream);
}

cudaError_t launch_step_layers(const StepLayersParams& q, bool bf16, bool vec, cudaStream_t stream) {
    return bf16 ? launch_step_layers_dtype<__nv_bfloat16>(q, vec, stream)
                : launch_step_layers_dtype<float>(q, vec, stream);
}

}  // namespace selscan
