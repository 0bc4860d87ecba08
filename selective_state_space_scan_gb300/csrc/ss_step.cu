// Single-token decode update of the selective SSM (the O(1)-per-token step of
// "mamba-metal: Apple Silicon で Mamba を動かす", section "O(L) インクリメンタルデコード"):
//   Δ          = softplus(delta_raw[b,d] + delta_bias[d])
//   h[b,d,n]  <- exp(Δ A_n) h[b,d,n] + Δ x[b,d] B[b,n],    A_n = -exp(A_log[d,n])
//   y[b,d]     = (Σ_n C[b,n] h[b,d,n] + D[d] x[b,d]) · silu(z[b,d])
// The state is updated in place.  The step is elementwise over (b,d) and HBM-bound on the
// state read + write (16 states x 8 bytes per row against 16 bytes of x, Δ, z, y), so the
// kernels are streams with LPR lanes per (b,d) row, each lane owning four consecutive states,
// and the partial C·h sums reduced across the row's lanes by shuffles.  Two of them:
//   - the staged kernel (16 states, aligned rows: the usual case; see the section below): each
//     warp streams a contiguous range of 32-row units through its own ring of bulk-copied
//     shared-memory stages, so the bytes in flight are bound by shared memory, not registers;
//   - the per-block kernel (any N, strides or alignment): RPT rows per thread with every load of
//     all of them issued before any arithmetic, one 16-byte load and store of h per lane; block
//     x covers rows of batch row x / blocks_per_b (one 32-bit division per block).
// exp(A_log) is taken on the SFU (2^(A_log·log2 e)); its relative error (~1e-7) moves the
// decay exponent by as much, far below the fp32 tolerance.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "device_common.cuh"
#include "fwd_params.h"
#include "internal.h"

namespace selscan {

// Threads per block: small blocks (2 warps) measured 5% faster per layer than 256-thread ones
// (11.1 against 11.7 us on the 48-layer decode), 32 or 512 slower.
constexpr int kStepThreads = 64;

// Resident blocks per SM the per-block many-layer kernel's registers are sized for: it is bound
// by the state loads in flight, so occupancy pays.  At 24 blocks (at most 42 registers) the
// 48-layer launch measured 391 us against 455 us unbounded (56 registers, 52% occupancy) and
// 420 us at 32 blocks (32 registers, with spills).  The single-layer kernel stays unbounded: its short
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
// exp(A_log) of a quad (-A), on the SFU.
__device__ __forceinline__ float4 exp_quad(const float4& av) {
    return make_float4(ex2(av.x * kLog2e), ex2(av.y * kLog2e), ex2(av.z * kLog2e), ex2(av.w * kLog2e));
}

// The same with exp(A_log) already taken (ae = exp_quad(A_log quad)).
__device__ __forceinline__ float step_quad_e(float4& hv, const float4& ae, const float4& Bv,
                                             const float4& Cv, float dlt, float dx) {
    const float k = -dlt * kLog2e;
    const float h0 = fmaf(ex2(k * ae.x), hv.x, dx * Bv.x);
    const float h1 = fmaf(ex2(k * ae.y), hv.y, dx * Bv.y);
    const float h2 = fmaf(ex2(k * ae.z), hv.z, dx * Bv.z);
    const float h3 = fmaf(ex2(k * ae.w), hv.w, dx * Bv.w);
    hv = make_float4(h0, h1, h2, h3);
    return fmaf(Cv.x, h0, fmaf(Cv.y, h1, fmaf(Cv.z, h2, Cv.w * h3)));
}

__device__ __forceinline__ float step_quad(float4& hv, const float4& av, const float4& Bv,
                                           const float4& Cv, float dlt, float dx) {
    return step_quad_e(hv, exp_quad(av), Bv, Cv, dlt, dx);
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

// ---- Staged many-layer step (16 states, rows of whole 16-byte units) ----
// The rows of all layers form one sequence of units of kSlRows rows, ordered (layer, row block,
// batch row), split into equal contiguous ranges, one per warp of a persistent grid.  Each warp
// streams its range through its own ring of kSlStages shared-memory stages: one lane issues a
// unit's bulk copies (the state rows, x, Δ, z and the batch row's B and C) on the stage's
// mbarrier kSlStages - 1 units ahead, so that several units of every warp are in flight while it
// computes; the lanes then update the unit's rows in four passes of eight rows (four lanes of
// four states a row, the arithmetic of step_quad) and write the state back with 16-byte stores.
// Consecutive units of a warp share their row block, so exp(A_log), bias and D of the warp's
// rows stay in registers across the batch rows (reloaded when the block changes), and a stage
// holds only what changes with the batch row.  No block barrier: the warps run independently.
constexpr int kSlRows = 32;
#ifndef SS_STEPL_STAGES
#define SS_STEPL_STAGES 4
#endif
constexpr int kSlStages = SS_STEPL_STAGES;
#ifndef SS_STEPL_WARPS
#define SS_STEPL_WARPS 4
#endif
constexpr int kSlWarps = SS_STEPL_WARPS;

template <typename TIO>
struct SlStage {
    static constexpr int ES = static_cast<int>(sizeof(TIO));
    static constexpr int H = 0;                              // [32][16] fp32 state rows
    static constexpr int X = H + kSlRows * 16 * 4;           // [32] x
    static constexpr int DL = X + kSlRows * ES;              // [32] delta_raw
    static constexpr int Z = DL + kSlRows * ES;              // [32] z
    static constexpr int BR = Z + kSlRows * ES;              // [16] B of the batch row
    static constexpr int CR = BR + 16 * ES;                  // [16] C of the batch row
    static constexpr int BYTES = (CR + 16 * ES + 127) / 128 * 128;
    static constexpr int RING = kSlStages * BYTES;
    static constexpr int SMEM = kSlWarps * RING + kSlWarps * kSlStages * 8 + kSlWarps * 4;
    static_assert(X % 16 == 0 && DL % 16 == 0 && Z % 16 == 0 && BR % 16 == 0 && CR % 16 == 0,
                  "bulk copy destinations are 16-byte aligned");
};

template <typename TIO>
__global__ void __launch_bounds__(kSlWarps * 32) ss_step_layers_staged_kernel(const __grid_constant__ StepLayersParams q) {
    using St = SlStage<TIO>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* ring = smem + warp * St::RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSlWarps * St::RING) + warp * kSlStages;
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(smem + kSlWarps * St::RING + kSlWarps * kSlStages * 8) + warp;
    const StepParams& c = q.common;
    const int per_blk = c.batch;                             // units of one row block
    const int64_t per_layer = static_cast<int64_t>(c.Dm / kSlRows) * per_blk;
    const int64_t U = per_layer * q.n_layers;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * kSlWarps + warp;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kSlWarps;
    const int64_t u0 = U * wid / nw, u1 = U * (wid + 1) / nw;
    if (lane == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kSlStages; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncwarp();
    auto where = [&](int64_t u, int& layer, int& b, int& d0) {
        layer = static_cast<int>(u / per_layer);
        const int64_t rem = u - layer * per_layer;
        const int blk = static_cast<int>(rem / per_blk);
        b = static_cast<int>(rem - static_cast<int64_t>(blk) * per_blk);
        d0 = blk * kSlRows;
    };
    auto issue = [&](int64_t u, int s) {                     // lane 0
        int layer, b, d0;
        where(u, layer, b, d0);
        const StepLayerPtrs& L = q.layer[layer];
        uint8_t* st = ring + s * St::BYTES;
        const uint32_t rows_x = kSlRows * St::ES;
        const uint32_t bytes = kSlRows * 64u + 2u * rows_x + (L.z ? rows_x : 0u) + 2u * 16u * St::ES;
        mbar_expect_tx(&bars[s], bytes);
        bulk_load(st + St::H, L.state + static_cast<int64_t>(b) * c.s_b + static_cast<int64_t>(d0) * 16,
                  kSlRows * 64, &bars[s]);
        bulk_load(st + St::X, static_cast<const TIO*>(L.x) + static_cast<int64_t>(b) * c.x_b + d0, rows_x, &bars[s]);
        bulk_load(st + St::DL, static_cast<const TIO*>(L.delta) + static_cast<int64_t>(b) * c.d_b + d0, rows_x,
                  &bars[s]);
        if (L.z)
            bulk_load(st + St::Z, static_cast<const TIO*>(L.z) + static_cast<int64_t>(b) * c.z_b + d0, rows_x,
                      &bars[s]);
        bulk_load(st + St::BR, static_cast<const TIO*>(L.Bm) + static_cast<int64_t>(b) * c.B_b, 16 * St::ES, &bars[s]);
        bulk_load(st + St::CR, static_cast<const TIO*>(L.Cm) + static_cast<int64_t>(b) * c.C_b, 16 * St::ES, &bars[s]);
    };
    if (lane == 0)
        for (int k = 0; k < kSlStages && u0 + k < u1; ++k) issue(u0 + k, k);
    constexpr int PASSES = kSlRows / 8;
    const int qd = lane & 3, n0 = qd * 4;
    int cur_layer = -1, cur_d0 = -1;
    float4 ae[PASSES];                                       // exp(A_log) of this lane's quad of its rows
    float bias_r[PASSES], D_r[PASSES];
    int64_t k = 0;
    for (int64_t u = u0; u < u1; ++u, ++k) {
        const int s = static_cast<int>(k % kSlStages);
        int layer, b, d0;
        where(u, layer, b, d0);
        const StepLayerPtrs& L = q.layer[layer];
        if (layer != cur_layer || d0 != cur_d0) {            // a new row block: its parameters
            cur_layer = layer;
            cur_d0 = d0;
#pragma unroll
            for (int pass = 0; pass < PASSES; ++pass) {
                const int d = d0 + pass * 8 + (lane >> 2);
                ae[pass] = exp_quad(*reinterpret_cast<const float4*>(L.A_log + static_cast<int64_t>(d) * 16 + n0));
                bias_r[pass] = L.bias ? L.bias[d] : 0.f;
                D_r[pass] = L.Dv ? L.Dv[d] : 0.f;
            }
        }
        // every lane waits (a bounded wait: one lane's timeout raises the warp's abort flag, so
        // the others return too); the warp then leaves together or goes on together
        const bool got = mbar_wait_bounded(&bars[s], static_cast<uint32_t>((k / kSlStages) & 1), abort_flag, q.err);
        if (!__all_sync(0xffffffffu, got)) break;
        const uint8_t* st = ring + s * St::BYTES;
        const TIO* sx = reinterpret_cast<const TIO*>(st + St::X);
        const TIO* sdl = reinterpret_cast<const TIO*>(st + St::DL);
        const TIO* sz = reinterpret_cast<const TIO*>(st + St::Z);
        const float4 Bv = Vec4<TIO>::get(*reinterpret_cast<const typename Vec4<TIO>::T*>(st + St::BR + n0 * St::ES));
        const float4 Cv = Vec4<TIO>::get(*reinterpret_cast<const typename Vec4<TIO>::T*>(st + St::CR + n0 * St::ES));
        float* hrow = L.state + static_cast<int64_t>(b) * c.s_b;
        TIO* yrow = static_cast<TIO*>(L.y) + static_cast<int64_t>(b) * c.y_b;
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
            const int r = pass * 8 + (lane >> 2);
            const int d = d0 + r;
            float4 hv = *reinterpret_cast<const float4*>(st + St::H + r * 64 + qd * 16);
            const float xv = to_f32<TIO>(sx[r]);
            const float dv = to_f32<TIO>(sdl[r]) + bias_r[pass];
            const float dlt = softplus(dv);
            float partial = step_quad_e(hv, ae[pass], Bv, Cv, dlt, dlt * xv);
            *reinterpret_cast<float4*>(hrow + static_cast<int64_t>(d) * 16 + n0) = hv;
            partial += __shfl_xor_sync(0xffffffffu, partial, 1);
            partial += __shfl_xor_sync(0xffffffffu, partial, 2);
            if (qd == 0) {
                float v = fmaf(D_r[pass], xv, partial);
                if (L.z) v *= silu(to_f32<TIO>(sz[r]));
                yrow[d] = from_f32<TIO>(v);
            }
        }
        __syncwarp();                                        // every lane is done with stage s
        if (lane == 0 && u + kSlStages < u1) {
            tma_store_fence();                               // generic reads before the async refill
            issue(u + kSlStages, s);
        }
    }
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



// Test hook (ss_step and ss_step_layers): -1 automatic, 0 the per-block kernels, 1 the staged
// kernel (refused when it cannot be used).
static std::atomic<int> g_force_step_layers{-1};
// Which kernel the last ss_step or ss_step_layers call launched (0 per-block, 1 staged), for the
// benchmark's report.
static std::atomic<int> g_last_step_path{-1};

// Whether every layer's buffers suit the staged kernel: 16 states in rows of 64 bytes, row blocks
// of whole units, and every bulk-copied range (state rows, x, Δ, z, B and C rows) starting on a
// 16-byte boundary; A_log (16-byte rows), bias and D are read with plain loads.
static bool step_layers_staged_ok(const StepLayersParams& q, bool bf16) {
    const StepParams& c = q.common;
    const int64_t es = bf16 ? 2 : 4;
    if (c.N != 16 || c.s_d != 16 || c.Dm % kSlRows != 0) return false;
    if ((c.s_b * 4) % 16 || (c.x_b * es) % 16 || (c.d_b * es) % 16 || (c.z_b * es) % 16 || (c.B_b * es) % 16 ||
        (c.C_b * es) % 16)
        return false;
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    for (int l = 0; l < q.n_layers; ++l) {
        const StepLayerPtrs& L = q.layer[l];
        if (!al(L.state) || !al(L.A_log) || !al(L.x) || !al(L.delta) || (L.z && !al(L.z)) || !al(L.Bm) || !al(L.Cm))
            return false;
    }
    return true;
}

template <typename TIO>
static cudaError_t launch_step_layers_staged(const StepLayersParams& q, cudaStream_t stream) {
    using St = SlStage<TIO>;
    auto kern = ss_step_layers_staged_kernel<TIO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, St::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSlWarps * 32, St::SMEM)) != cudaSuccess)
        return e;
    const int64_t units = static_cast<int64_t>(q.n_layers) * q.common.batch * (q.common.Dm / kSlRows);
    const int64_t blocks = std::min<int64_t>(static_cast<int64_t>(std::max(per_sm, 1)) * sms,
                                             (units + kSlWarps - 1) / kSlWarps);
    if (blocks <= 0) return cudaSuccess;
    kern<<<static_cast<unsigned>(blocks), kSlWarps * 32, St::SMEM, stream>>>(q);
    return cudaGetLastError();
}

// One layer's step: the staged kernel over a table of one layer where it applies.
cudaError_t launch_step(const StepParams& p, bool bf16, bool vec, cudaStream_t stream) {
    const int force = g_force_step_layers.load();
    if (vec && force != 0) {
        StepLayersParams q;
        std::memset(&q, 0, sizeof(q));
        q.common = p;
        q.err = device_error_word();
        q.n_layers = 1;
        q.layer[0] = StepLayerPtrs{p.state, p.x, p.delta, p.z, p.Bm, p.Cm, p.bias, p.A_log, p.Dv, p.y};
        if (step_layers_staged_ok(q, bf16)) {
            g_last_step_path.store(1);
            return bf16 ? launch_step_layers_staged<__nv_bfloat16>(q, stream) : launch_step_layers_staged<float>(q, stream);
        }
    }
    if (force == 1) return cudaErrorInvalidValue;
    g_last_step_path.store(0);
    return bf16 ? launch_step_dtype<__nv_bfloat16>(p, vec, stream)
                : launch_step_dtype<float>(p, vec, stream);
}

cudaError_t launch_step_layers(const StepLayersParams& q, bool bf16, bool vec, cudaStream_t stream) {
    const int force = g_force_step_layers.load();
    const bool ok = vec && step_layers_staged_ok(q, bf16);
    if (force == 1 && !ok) return cudaErrorInvalidValue;
    if (ok && force != 0) {
        g_last_step_path.store(1);
        return bf16 ? launch_step_layers_staged<__nv_bfloat16>(q, stream) : launch_step_layers_staged<float>(q, stream);
    }
    g_last_step_path.store(0);
    return bf16 ? launch_step_layers_dtype<__nv_bfloat16>(q, vec, stream)
                : launch_step_layers_dtype<float>(q, vec, stream);
}

}  // namespace selscan

extern "C" int ss__force_step_layers_path(int v) {
    return selscan::g_force_step_layers.exchange(v < 0 ? -1 : v > 0 ? 1 : 0);
}
extern "C" int ss__last_step_path() { return selscan::g_last_step_path.load(); }

namespace selscan {

}  // namespace selscan
