// Causal depthwise conv1d (+ optional SiLU), the stage before the scan in a Mamba block
// ("mamba-metal: Apple Silicon で Mamba を動かす": MambaBlock = in_proj -> conv1d -> SiLU -> ...;
// SpeechLens docs/kernel-optimization.md, MetalCausalConv1d: depthwise, kernel 4, three zero
// samples on the causal left edge, output length L), with the sliding window the blog's section
// "O(L) インクリメンタルデコード" carries across calls:
//   out[b,t,d] = act(bias[d] + Σ_{k<4} w[d,k] · e[t + k]),   e = window[b,d,0..2] ++ x[b,:,d]
// and window_out[b,d,:] = the last three samples of e.
//
// The stage is a stream (4 multiply-adds per element against 8 bytes moved for fp32), so the
// kernel is laid out for bandwidth: a thread owns 4 adjacent channels (one 16-byte fp32 or
// 8-byte bf16 access per step, a warp covering 128 channels = 512 contiguous bytes) and a
// segment of seg steps (chosen per call so that the grid is whole waves of resident blocks); the three samples before the segment come from x itself (or, for the
// first segment, from the window), and kUnroll steps of loads are issued before their
// arithmetic.  The thread of a row's first segment is the only one that reads window_in and
// the only one that writes window_out (taking the last three samples from x), so the window
// may be updated in place.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/selscan.h"
#include "device_common.cuh"
#include "host_util.h"

namespace selscan {
namespace {

constexpr int kConvK = SS_CONV_WIDTH;   // 4
// Steps per thread: chosen per call (segment_steps) so that the grid fills whole waves of
// resident blocks; at least kSegMin, so that the three samples re-read before each segment stay
// a small part of its loads.
constexpr int kSegMin = 16;
constexpr int kSegMax = 128;
constexpr int kUnroll = 8;              // steps whose loads are issued together
constexpr int kThreads = 128;           // 512 channels per block

struct ConvParams {
    const void* x;
    void* out;
    const float* w;         // [Dm, 4]
    const float* bias;      // [Dm] or nullptr
    const float* win_in;    // [batch, Dm, 3] or nullptr
    float* win_out;         // [batch, Dm, 3] or nullptr
    int64_t x_b, x_l, o_b, o_l;
    int batch, L, Dm;
    int silu;
    int seg;                // steps per thread
};

template <typename TIO> struct Quad;
template <> struct Quad<float> {
    using T = float4;
    static __device__ __forceinline__ float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
    static __device__ __forceinline__ void store(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};
template <> struct Quad<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16* p) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float4 v) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p) = u;
    }
};

__device__ __forceinline__ float act(float v, int silu_on) { return silu_on ? silu(v) : v; }

// VEC: 4 channels per thread with quad loads (Dm % 4 == 0, aligned rows); else 4 channels
// per thread with scalar, bounds-checked loads.
template <typename TIO, bool VEC>
__global__ void __launch_bounds__(kThreads) ss_conv1d_kernel(const ConvParams p) {
    const int nbd = (p.Dm + 4 * kThreads - 1) / (4 * kThreads);   // channel blocks per row
    const int seg = static_cast<int>(blockIdx.x) / nbd, b = blockIdx.y;
    const int d0 = ((static_cast<int>(blockIdx.x) - seg * nbd) * kThreads + threadIdx.x) * 4;
    if (d0 >= p.Dm) return;
    const int t0 = seg * p.seg;
    const int nt = min(p.seg, p.L - t0);
    const TIO* x = static_cast<const TIO*>(p.x) + static_cast<int64_t>(b) * p.x_b;
    TIO* out = static_cast<TIO*>(p.out) + static_cast<int64_t>(b) * p.o_b;
    const int nc = min(4, p.Dm - d0);           // channels this thread owns (4 on the VEC path)

    float w[4][kConvK], bs[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const bool ok = c < nc;
#pragma unroll
        for (int k = 0; k < kConvK; ++k) w[c][k] = ok ? p.w[static_cast<int64_t>(d0 + c) * kConvK + k] : 0.f;
        bs[c] = (ok && p.bias) ? p.bias[d0 + c] : 0.f;
    }
    auto load4 = [&](int t) -> float4 {           // x[b, t, d0 .. d0+3], t >= 0
        const TIO* q = x + static_cast<int64_t>(t) * p.x_l + d0;
        if constexpr (VEC) {
            return Quad<TIO>::load(q);
        } else {
            float v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = c < nc ? to_f32<TIO>(q[c]) : 0.f;
            return make_float4(v[0], v[1], v[2], v[3]);
        }
    };
    auto store4 = [&](int t, float4 v) {
        TIO* q = out + static_cast<int64_t>(t) * p.o_l + d0;
        if constexpr (VEC) {
            Quad<TIO>::store(q, v);
        } else {
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (c < nc) q[c] = from_f32<TIO>(vv[c]);
        }
    };
    auto win = [&](int c, int k) -> float {       // window sample k (oldest first) of channel c
        return (p.win_in && c < nc) ? p.win_in[(static_cast<int64_t>(b) * p.Dm + d0 + c) * (kConvK - 1) + k] : 0.f;
    };

    // the three samples before the segment, per channel: e0 (oldest), e1, e2
    float e0[4], e1[4], e2[4];
    if (seg == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            e0[c] = win(c, 0);
            e1[c] = win(c, 1);
            e2[c] = win(c, 2);
        }
    } else {
        const float4 a = load4(t0 - 3), bq = load4(t0 - 2), cq = load4(t0 - 1);
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {bq.x, bq.y, bq.z, bq.w}, cv[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            e0[c] = av[c];
            e1[c] = bv[c];
            e2[c] = cv[c];
        }
    }
    // the new window (first segment's thread only): the last three samples of window ++ x,
    // read before anything is written so that window_out may be window_in
    float nw[4][3];
    const bool write_win = seg == 0 && p.win_out != nullptr;
    if (write_win) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int t = p.L - 3 + j;            // sample index in x; < 0: still in the old window
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (t >= 0) {
                const float4 q = load4(t);
                v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = win(c, 3 + t);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) nw[c][j] = v[c];
        }
    }

    for (int i0 = 0; i0 < nt; i0 += kUnroll) {
        float4 xs[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            xs[u] = (i0 + u < nt) ? load4(t0 + i0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (i0 + u < nt) {
                const float xv[4] = {xs[u].x, xs[u].y, xs[u].z, xs[u].w};
                float o[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float acc = fmaf(w[c][3], xv[c], fmaf(w[c][2], e2[c], fmaf(w[c][1], e1[c], fmaf(w[c][0], e0[c], bs[c]))));
                    o[c] = act(acc, p.silu);
                    e0[c] = e1[c];
                    e1[c] = e2[c];
                    e2[c] = xv[c];
                }
                store4(t0 + i0 + u, make_float4(o[0], o[1], o[2], o[3]));
            }
        }
    }
    if (write_win) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (c < nc)
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    p.win_out[(static_cast<int64_t>(b) * p.Dm + d0 + c) * (kConvK - 1) + j] = nw[c][j];
    }
}

// Steps per thread for a grid of batch x ceil(L / seg) x nbd blocks when `slots` blocks are
// resident at once: the length whose whole waves take the least time, modelling a wave as
// seg + 6 steps of one thread (the three re-read samples and the set-up).  On the 130m-shaped
// input (8 x 2048 x 1536, 760 resident blocks) it picks 33 steps: 1512 blocks in two full waves
// (38.8 us), where 32 steps gave 1536 blocks, two waves and 16 blocks more (42.9 us).
int segment_steps(int64_t batch, int64_t L, int64_t nbd, int64_t slots) {
    if (L <= kSegMin) return static_cast<int>(std::max<int64_t>(L, 1));
    int best = kSegMin;
    int64_t best_cost = -1;
    for (int seg = kSegMin; seg <= kSegMax; ++seg) {
        const int64_t blocks = batch * ((L + seg - 1) / seg) * nbd;
        const int64_t waves = (blocks + slots - 1) / slots;
        const int64_t cost = waves * (seg + 6);
        if (best_cost < 0 || cost <= best_cost) {
            best_cost = cost;
            best = seg;
        }
    }
    return best;
}

// Windows only (L == 0): window_out = window_in (or zeros).
__global__ void ss_conv1d_window_copy(const float* win_in, float* win_out, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) win_out[i] = win_in ? win_in[i] : 0.f;
}

}  // namespace
}  // namespace selscan

using namespace selscan;
using namespace selscan::host;

// Test hook: steps per thread, at least 3 (a later segment re-reads the three samples before it
// from x); anything else restores the choice per call.  Returns the previous value.
static std::atomic<int> g_force_conv_seg{0};
extern "C" int ss__force_conv_segment(int steps) { return g_force_conv_seg.exchange(steps >= 3 ? steps : 0); }

extern "C" ss_status ss_conv1d(const void* x, const float* weight, const float* bias, void* out,
                               const float* window_in, float* window_out, int64_t batch, int64_t L,
                               int64_t Dm, int32_t silu, const ss_conv_strides* strides, void* stream_ptr) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (batch < 0 || L < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    ss_conv_strides s;
    if (strides) {
        s = *strides;
    } else {
        std::memset(&s, 0, sizeof(s));
        s.io_dtype = SS_F32;
        s.x_b = s.out_b = L * Dm;
        s.x_l = s.out_l = Dm;
    }
    if (s.io_dtype != SS_F32 && s.io_dtype != SS_BF16) return SS_ERR_INVALID_ARG;
    if (batch == 0 || Dm == 0) return SS_OK;
    if (batch > 65535 || L > INT32_MAX || Dm > INT32_MAX) return SS_ERR_UNSUPPORTED;
    const bool bf16 = s.io_dtype == SS_BF16;
    const int64_t es = bf16 ? 2 : 4;
    if (!weight) return SS_ERR_INVALID_ARG;
    if (L > 0 && (!x || !out)) return SS_ERR_INVALID_ARG;
    if (s.x_b < 0 || s.x_l < 0 || s.out_b < 0 || s.out_l < 0) return SS_ERR_INVALID_ARG;
    if (L > 1 && (s.x_l < Dm || s.out_l < Dm)) return SS_ERR_INVALID_ARG;
    if (L > 0 && !distinct3(batch, s.out_b, L, s.out_l, Dm)) return SS_ERR_INVALID_ARG;   // out: one word each
    const void* f_ptrs[] = {weight, bias, window_in, window_out};
    for (const void* q : f_ptrs)
        if (q && !is_aligned(q, 4)) return SS_ERR_MISALIGNED;
    if ((x && !is_aligned(x, es)) || (out && !is_aligned(out, es))) return SS_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    const void* all[] = {x, out, weight, bias, window_in, window_out};
    for (const void* q : all)
        if (q && !dev_ptr(q, dev)) return SS_ERR_INVALID_ARG;
    // outputs: out must not meet any input or window; window_out may be window_in itself only
    const Range ro = range3(out, batch, L, Dm, s.out_b, s.out_l, es);
    const Range rwo = range3(window_out, batch, Dm, kConvK - 1, Dm * (kConvK - 1), kConvK - 1, 4);
    const Range rwi = range3(window_in, batch, Dm, kConvK - 1, Dm * (kConvK - 1), kConvK - 1, 4);
    const Range ins[] = {range3(x, batch, L, Dm, s.x_b, s.x_l, es), range3(weight, 1, Dm, kConvK, 0, kConvK, 4),
                         range3(bias, 1, 1, Dm, 0, 0, 4)};
    for (const Range& r : ins)
        if (meet(ro, r) || meet(rwo, r)) return SS_ERR_INVALID_ARG;
    if (meet(ro, rwi) || meet(ro, rwo)) return SS_ERR_INVALID_ARG;
    if (window_in != window_out && meet(rwo, rwi)) return SS_ERR_INVALID_ARG;

    if (L == 0) {
        if (!window_out || window_out == window_in) return SS_OK;
        const int64_t n = batch * Dm * (kConvK - 1);
        ss_conv1d_window_copy<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(window_in, window_out, n);
        return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
    }
    ConvParams p;
    p.x = x; p.out = out; p.w = weight; p.bias = bias; p.win_in = window_in; p.win_out = window_out;
    p.x_b = s.x_b; p.x_l = s.x_l; p.o_b = s.out_b; p.o_l = s.out_l;
    p.batch = static_cast<int>(batch); p.L = static_cast<int>(L); p.Dm = static_cast<int>(Dm);
    p.silu = silu ? 1 : 0;
    const int64_t va = 4 * es;   // quad access alignment
    const bool vec = Dm % 4 == 0 && is_aligned(x, va) && is_aligned(out, va) && (s.x_l * es) % va == 0 &&
                     (s.out_l * es) % va == 0 && (batch == 1 || ((s.x_b * es) % va == 0 && (s.out_b * es) % va == 0));
    const int64_t nbd = (Dm + 4 * kThreads - 1) / (4 * kThreads);
    void (*kern)(ConvParams) = bf16 ? (vec ? ss_conv1d_kernel<__nv_bfloat16, true> : ss_conv1d_kernel<__nv_bfloat16, false>)
                                    : (vec ? ss_conv1d_kernel<float, true> : ss_conv1d_kernel<float, false>);
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess)
        return SS_ERR_CUDA;
    const int forced = g_force_conv_seg.load();
    p.seg = forced > 0 ? forced : segment_steps(batch, L, nbd, static_cast<int64_t>(std::max(sms, 1)) * std::max(per_sm, 1));
    const int64_t segs = (L + p.seg - 1) / p.seg;
    if (segs * nbd > INT32_MAX) return SS_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(segs * nbd), static_cast<unsigned>(batch));   // x: (segment, channel block)
    kern<<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
