// Backward pass of the selective scan: the gradients of ss_fwd's outputs (y, last_state) with
// respect to every input.  No backward pass is implemented on the pages ("mamba-metal: Apple
// Silicon で Mamba を動かす" lists the backward kernel for training under "残り課題"); this is
// the derivative of the forward definition (same blog, section "Selective
// scan の本質": h_t = Ā_t h_{t-1} + B̄_t u_t, y_t = C_t h_t, with softplus on Δ, the D skip and
// the z gate of the blog's walkthrough of the official CUDA kernel, section "1チャンク内の処理
// フロー"), evaluated as the reverse (adjoint) recurrence of the same scan:
//   dŷ_t = dy_t g_t (g = silu(z)),  dz_t = dy_t ŷ_t silu'(z_t)
//   λ_t = C_t dŷ_t + a_{t+1} λ_{t+1}          (dlast joins at t = L-1)
//   dC_t += dŷ_t h_t,  dB_t += λ_t Δ_t u_t    (summed over the channels of a batch row)
//   du_t = D dŷ_t + Σ_n λ_t Δ_t B_t,   dΔ_t = Σ_n λ_t (A a_t h_{t-1} + B_t u_t),  dr_t = dΔ_t σ(r_t)
//   dA += λ_t Δ_t a_t h_{t-1} (then · A for A_log),  dD += dŷ_t u_t,  dbias += dr_t,  dh0 = a_0 λ_0
//
// Layout: the forward kernel's lanes (a channel's states split over NS/4 lanes of 4 states, a
// CTA = 32 channels of one batch row).  The reverse recurrence needs h_{t-1} at every step:
//   pass 1 folds the sequence forward and stores the state at every kBS-step sub-chunk start
//   (workspace);
//   pass 2 walks the chunks backwards; for each sub-chunk (last first) it refolds the sub-chunk's
//   kBS states into registers from its checkpoint and runs the adjoint backwards over them.
// The per-(step, channel) quantities (Δ, σ(r), dŷ, dy·silu'(z), u) and the chunk's B, C are
// staged in shared memory; dB, dC (sums over the CTA's channels) are reduced over a warp's
// channel lanes by shuffles, over the warps with shared atomics, and reach global memory with
// one 16-byte reduction per (step, four states) per CTA (scalar atomics when N is not a
// multiple of 4 or the sums are not 16-byte aligned); dA_log, dD and dbias are summed over
// batch rows with global atomics.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/selscan.h"
#include "device_common.cuh"
#include "host_util.h"
#include "internal.h"

namespace selscan {
namespace {

constexpr int kBT = 32;    // steps per chunk (the height of one staged tile)
constexpr int kBS = 16;    // steps per sub-chunk (their states are held in registers)
constexpr int kBW = 32;    // channels per CTA

// Test hook: -1 automatic, 0 plain-load staging, 1 TMA staging (refused when it cannot be used).
std::atomic<int> g_force_bwd_tma{-1};
// Test hook: -1 automatic time split, 0 never, n >= 2 always with up to n segments.
std::atomic<int> g_force_bwd_nseg{-1};

struct BwdParams {
    const void* u;
    const void* delta;
    const void* z;
    const void* Bm;
    const void* Cm;
    const float* bias;
    const float* A_log;
    const float* Dv;
    const float* h0;
    const void* dy;        // [batch, L, Dm] contiguous
    const float* dlast;    // [batch, Dm, N] or nullptr
    void* du;              // [batch, L, Dm] contiguous
    void* ddelta;
    void* dz;
    float* dB;             // [batch, L, N] contiguous (zeroed by the host)
    float* dC;
    float* dA_log;         // [Dm, N] (zeroed)
    float* dD;             // [Dm] or nullptr (zeroed)
    float* dbias;          // [Dm] or nullptr (zeroed)
    float* dh0;            // [batch, Dm, N] or nullptr
    float* ckpt;           // [tiles][nchunks][kBT / kBS][kBW][NS]: the state at every sub-chunk start
    int ckpt_given;        // the checkpoints came from the forward pass (ss_fwd_ckpt): no pass 1
    unsigned int* err;     // device error word
    // Time split (nseg > 1): CTA x takes segment x % nseg (chunks [seg·seg_chunks, ...)) of tile
    // x / nseg.  The local launch folds each segment from zero (end state into h_slots[seg + 1],
    // Σ Δ into dsum[seg]) and sweeps its adjoint from zero (the λ it hands to the segment on its
    // left into m_slots[seg - 1]); the carry passes turn the slots into each segment's entering
    // state (h_slots[seg]) and entering adjoint (m_slots[seg]); the main launch runs both passes
    // per segment from them.
    int nseg, seg_chunks;
    float* h_slots;        // [nseg][batch·Dm·N]
    float* m_slots;        // [nseg][batch·Dm·N]
    float* dsum;           // [nseg][batch·Dm]
    int64_t u_b, u_l, d_b, d_l, z_b, z_l, B_b, B_l, C_b, C_l;
    int batch, L, Dm, N, nchunks, tiles_per_batch;
    int bc_vec;            // N % 4 == 0 and dB, dC 16-byte aligned: vector reductions into them
};

// TMA descriptors: [T][W] boxes of u, δ, z, dy (loaded) and du, dδ, dz (stored); [T][NS] boxes
// of B, C (loaded).
struct BwdMaps {
    CUtensorMap u, delta, z, dy, B, C, du, ddelta, dz;
};

template <typename TIO, int NS_>
struct BwdCfg {
    static constexpr int NS = NS_;
    static constexpr int LPC = NS / 4;           // lanes per channel, four states each
    static constexpr int CPW = 32 / LPC;         // channels per warp
    static constexpr int WARPS = kBW / CPW;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int ES = static_cast<int>(sizeof(TIO));
    // staged input tiles, io dtype, as TMA writes them (bytes)
    static constexpr int RAW_X = kBT * kBW * ES;
    static constexpr int RAW_N = kBT * NS * ES;
    static constexpr int R_U = 0, R_D = RAW_X, R_Z = 2 * RAW_X, R_Y = 3 * RAW_X, R_B = 4 * RAW_X,
                         R_C = 4 * RAW_X + RAW_N;
    static constexpr int RAW_BYTES = 4 * RAW_X + 2 * RAW_N;
    // the chunk's du, dδ, dz tiles, io dtype, as a TMA store reads them (bytes after the staged tiles)
    static constexpr int O_DU = RAW_BYTES, O_DD = O_DU + RAW_X, O_DZ = O_DD + RAW_X;
    static constexpr int DER_BYTE = O_DZ + RAW_X;
    // fp32 arrays the chunk is processed from (float offsets from DER_BYTE); the chunk's dB and
    // dC sums interleaved per step ([T][2][NS]), so that one step's shared atomics of a warp hit
    // 2·NS consecutive words
    static constexpr int X = kBT * kBW, XN = kBT * NS;
    static constexpr int OFF_U = 0, OFF_DEL = X, OFF_SIG = 2 * X, OFF_DYH = 3 * X, OFF_DYG = 4 * X;
    static constexpr int OFF_B = 5 * X, OFF_C = OFF_B + XN, OFF_BC = OFF_C + XN;
    static constexpr int BAR_OFF = DER_BYTE + (OFF_BC + 2 * XN) * 4;
    static constexpr int SMEM = BAR_OFF + 16;    // the mbarrier, then the abort flag
    static_assert(RAW_X % 128 == 0 && RAW_N % 128 == 0, "TMA tiles stay 128-byte aligned");
};

__device__ __forceinline__ float sigmoid_f(float x) { return rcp_approx(1.f + ex2(-x * kLog2e)); }

// What a chunk's staging holds: the forward fold's inputs (u, δ, B), everything the reverse pass
// uses (u, δ, z, dy, B, C), or the adjoint sweep's alone (δ, z, dy, C: the time split's local launch).
enum StageKind { kStFwd = 0, kStFull = 1, kStLam = 2 };

// Build the chunk's fp32 arrays: Δ = softplus(δ + bias) always; u and B unless KIND is kStLam;
// σ(δ + bias) and dy·silu'(z) for kStFull; dŷ = dy·silu(z) and C unless KIND is kStFwd.  Inputs come
// from the staged tiles (TMA) or straight from global memory.  Steps past L and channels past Dm
// become zeros, which make those steps the identity of both recurrences.
template <class Cfg, typename TIO, bool TMA, int KIND>
__device__ __forceinline__ void bwd_prepare(float* sm, const uint8_t* raw, const BwdParams& p, int b, int d0,
                                            int chunk, float bias_c) {
    constexpr bool full = KIND != kStFwd;        // the reverse pass's inputs (dŷ, C)
    constexpr bool with_u = KIND != kStLam;      // u and B
    const int t0 = chunk * kBT;
    const int c = threadIdx.x % kBW;             // fixed per thread (THREADS is a multiple of kBW)
    const int d = d0 + c;
    const TIO* gu = static_cast<const TIO*>(p.u);
    const TIO* gd = static_cast<const TIO*>(p.delta);
    const TIO* gz = static_cast<const TIO*>(p.z);
    const TIO* gy = static_cast<const TIO*>(p.dy);
#pragma unroll 4
    for (int i = threadIdx.x; i < kBT * kBW; i += Cfg::THREADS) {
        const int t = t0 + i / kBW;
        const bool in = t < p.L && d < p.Dm;
        float uu = 0.f, rr = 0.f, zv = 0.f, dyv = 0.f;
        if constexpr (TMA) {
            if (with_u) uu = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_U)[i]);
            rr = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_D)[i]);
            if (full) {
                if (gz) zv = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_Z)[i]);
                dyv = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_Y)[i]);
            }
        } else if (in) {
            if (with_u) uu = to_f32<TIO>(gu[b * p.u_b + t * p.u_l + d]);
            rr = to_f32<TIO>(gd[b * p.d_b + t * p.d_l + d]);
            if (full) {
                if (gz) zv = to_f32<TIO>(gz[b * p.z_b + t * p.z_l + d]);
                dyv = to_f32<TIO>(gy[(static_cast<int64_t>(b) * p.L + t) * p.Dm + d]);
            }
        }
        rr += bias_c;
        if (with_u) sm[Cfg::OFF_U + i] = in ? uu : 0.f;
        sm[Cfg::OFF_DEL + i] = in ? softplus(rr) : 0.f;
        if (full) {
            float g = 1.f, dg = 0.f;
            if (gz) {
                const float s = sigmoid_f(zv);
                g = zv * s;
                dg = s * fmaf(zv, 1.f - s, 1.f);
            }
            sm[Cfg::OFF_DYH + i] = in ? dyv * g : 0.f;
            if (KIND == kStFull) {
                sm[Cfg::OFF_SIG + i] = in ? sigmoid_f(rr) : 0.f;
                sm[Cfg::OFF_DYG + i] = in ? dyv * dg : 0.f;
            }
        }
    }
    const TIO* gB = static_cast<const TIO*>(p.Bm);
    const TIO* gC = static_cast<const TIO*>(p.Cm);
#pragma unroll 2
    for (int i = threadIdx.x; i < kBT * Cfg::NS; i += Cfg::THREADS) {
        const int r = i / Cfg::NS, n = i % Cfg::NS;
        const int t = t0 + r;
        const bool in = t < p.L && n < p.N;
        float bv = 0.f, cv = 0.f;
        if constexpr (TMA) {
            if (with_u) bv = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_B)[i]);
            if (full) cv = to_f32<TIO>(reinterpret_cast<const TIO*>(raw + Cfg::R_C)[i]);
        } else if (in) {
            if (with_u) bv = to_f32<TIO>(gB[b * p.B_b + t * p.B_l + n]);
            if (full) cv = to_f32<TIO>(gC[b * p.C_b + t * p.C_l + n]);
        }
        if (with_u) sm[Cfg::OFF_B + i] = in ? bv : 0.f;
        if (full) sm[Cfg::OFF_C + i] = in ? cv : 0.f;
    }
}

// Sum over the LPC lanes of a channel (lanes c + CPW·j), every lane receiving the total.
template <int CPW>
__device__ __forceinline__ float channel_sum(float v) {
#pragma unroll
    for (int off = CPW; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Sum over the CPW channel lanes of a warp (lanes c + CPW·j, c = lane % CPW) of each of a
// lane's 8 values v[k] (dB of its 4 states, then dC of them), scattered: three halving rounds
// over the channel bits 2, 1, 0 leave value k = c & 7 in lane c; wider warps (CPW > 8) finish
// with plain add rounds, after which the lanes with c < 8 hold the sums.  Returns that value.
template <int CPW>
__device__ __forceinline__ float channel_reduce_scatter(const float (&v)[8], int c) {
    const bool b2 = (c & 4) != 0, b1 = (c & 2) != 0, b0 = (c & 1) != 0;
    float2 w4[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int lo = 2 * k, hi = 4 + 2 * k;
        const float2 keep = b2 ? make_float2(v[hi], v[hi + 1]) : make_float2(v[lo], v[lo + 1]);
        const float2 send = b2 ? make_float2(v[lo], v[lo + 1]) : make_float2(v[hi], v[hi + 1]);
        w4[k] = __fadd2_rn(keep, make_float2(__shfl_xor_sync(0xffffffffu, send.x, 4),
                                             __shfl_xor_sync(0xffffffffu, send.y, 4)));
    }
    const float2 keep = b1 ? w4[1] : w4[0], send = b1 ? w4[0] : w4[1];
    const float2 w2 = __fadd2_rn(keep, make_float2(__shfl_xor_sync(0xffffffffu, send.x, 2),
                                                   __shfl_xor_sync(0xffffffffu, send.y, 2)));
    float r = (b0 ? w2.y : w2.x) + __shfl_xor_sync(0xffffffffu, b0 ? w2.x : w2.y, 1);
#pragma unroll
    for (int off = 8; off < CPW; off <<= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }
__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

// LOCAL: the local launch of the time split (see BwdParams); otherwise both passes over this
// CTA's chunks from its entering state and adjoint (the whole sequence when nseg == 1).
template <typename TIO, int NS, bool TMA, bool LOCAL = false>
__global__ void __launch_bounds__(BwdCfg<TIO, NS>::THREADS)
ss_bwd_kernel(const BwdParams p, const __grid_constant__ BwdMaps maps) {
    using Cfg = BwdCfg<TIO, NS>;
    constexpr int CPW = Cfg::CPW;
    constexpr int NSUB = kBT / kBS;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* raw = smem;
    float* sm = reinterpret_cast<float*>(smem + Cfg::DER_BYTE);
    TIO* o_du = reinterpret_cast<TIO*>(smem + Cfg::O_DU);
    TIO* o_dd = reinterpret_cast<TIO*>(smem + Cfg::O_DD);
    TIO* o_dz = reinterpret_cast<TIO*>(smem + Cfg::O_DZ);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::BAR_OFF + 8);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = lane / CPW, c = lane % CPW;
    const int cw = warp * CPW + c;               // channel within the tile
    const int tile = static_cast<int>(blockIdx.x) / p.nseg;
    const int seg = static_cast<int>(blockIdx.x) - tile * p.nseg;
    const int c0 = seg * p.seg_chunks;                  // this CTA's chunks [c0, c1)
    const int c1 = min(p.nchunks, c0 + p.seg_chunks);
    const int b = tile / p.tiles_per_batch;
    const int d0 = (tile % p.tiles_per_batch) * kBW;
    const int d = d0 + cw;
    const bool d_ok = d < p.Dm;
    const int n0 = j * 4;
    const int dp = d0 + tid % kBW;               // the channel this thread prepares
    const float bias_c = (p.bias && dp < p.Dm) ? p.bias[dp] : 0.f;

    if (tid == 0) {
        *abort_flag = 0;
        if constexpr (TMA) {
            mbar_init(bar, 1);
            mbar_fence_init();
        }
    }
    for (int i = tid; i < 2 * Cfg::XN; i += Cfg::THREADS) sm[Cfg::OFF_BC + i] = 0.f;
    __syncthreads();
    // one TMA batch in flight at a time: the next chunk's tiles land while this chunk is processed
    auto issue = [&](int chunk, int kind) {     // a StageKind
        const int t0 = chunk * kBT;
        const bool full = kind != kStFwd, with_u = kind != kStLam;
        const bool hz = full && p.z != nullptr;
        const uint32_t nx = 1u + (with_u ? 1u : 0u) + (full ? 1u : 0u) + (hz ? 1u : 0u);
        const uint32_t nn = (with_u ? 1u : 0u) + (full ? 1u : 0u);
        mbar_expect_tx(bar, nx * Cfg::RAW_X + nn * Cfg::RAW_N);
        tma_load_3d(raw + Cfg::R_D, &maps.delta, bar, d0, t0, b);
        if (with_u) {
            tma_load_3d(raw + Cfg::R_U, &maps.u, bar, d0, t0, b);
            tma_load_3d(raw + Cfg::R_B, &maps.B, bar, 0, t0, b);
        }
        if (full) {
            if (hz) tma_load_3d(raw + Cfg::R_Z, &maps.z, bar, d0, t0, b);
            tma_load_3d(raw + Cfg::R_Y, &maps.dy, bar, d0, t0, b);
            tma_load_3d(raw + Cfg::R_C, &maps.C, bar, 0, t0, b);
        }
    };
    uint32_t phase = 0;
    auto wait_staged = [&]() {
        if constexpr (TMA) {
            mbar_wait_bounded(bar, phase, abort_flag, p.err);
            phase ^= 1u;
        }
    };
    // with the forward's checkpoints there is no forward pass here (the time split's local launch
    // then sums Δ during its adjoint sweep instead)
    const bool pass1 = !p.ckpt_given;
    if (TMA && tid == 0) {
        if (pass1) issue(c0, kStFwd);
        else issue(c1 - 1, LOCAL ? kStLam : kStFull);   // pass 2 starts from the last chunk
    }

    float2 A2[2], An[2];                         // A·log2(e) and A = -exp(A_log), state pairs
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float a[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = n0 + 2 * q + e;
            a[e] = (d_ok && n < p.N) ? -expf(p.A_log[static_cast<int64_t>(d) * p.N + n]) : 0.f;
        }
        An[q] = f2(a[0], a[1]);
        A2[q] = f2(a[0] * kLog2e, a[1] * kLog2e);
    }
    const float Dd = (d_ok && p.Dv) ? p.Dv[d] : 0.f;
    float* ck = p.ckpt + static_cast<int64_t>(tile) * p.nchunks * NSUB * kBW * NS;
    auto ckpt_at = [&](int ch, int k) {          // this lane's checkpoint slot: sub-chunk k of chunk ch
        return ck + ((static_cast<int64_t>(ch) * NSUB + k) * kBW + cw) * NS + n0;
    };
    const int64_t row = static_cast<int64_t>(b) * p.Dm + d;
    const int64_t count = static_cast<int64_t>(p.batch) * p.Dm * p.N;   // elements of one slot

    auto fold = [&](float2 (&h)[2], int r) {     // one step of the forward recurrence (chunk row r)
        const float del = sm[Cfg::OFF_DEL + r * kBW + cw];
        const float2 du = f2(del * sm[Cfg::OFF_U + r * kBW + cw]);
        const float4 Bv = *reinterpret_cast<const float4*>(&sm[Cfg::OFF_B + r * NS + n0]);
        const float2 e0 = mul2(f2(del), A2[0]), e1 = mul2(f2(del), A2[1]);
        h[0] = fma2(f2(ex2(e0.x), ex2(e0.y)), h[0], mul2(du, f2(Bv.x, Bv.y)));
        h[1] = fma2(f2(ex2(e1.x), ex2(e1.y)), h[1], mul2(du, f2(Bv.z, Bv.w)));
    };

    // this lane's four values of a [batch, Dm, N] state (zeros for none, or past Dm / N)
    auto load_quad = [&](const float* src, float2 (&q2)[2]) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = (src && d_ok && n0 + q < p.N) ? src[row * p.N + n0 + q] : 0.f;
        q2[0] = f2(v[0], v[1]);
        q2[1] = f2(v[2], v[3]);
    };
    auto store_quad = [&](float* dst, const float2 (&q2)[2]) {
        const float v[4] = {q2[0].x, q2[0].y, q2[1].x, q2[1].y};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (d_ok && n0 + q < p.N) dst[row * p.N + n0 + q] = v[q];
    };

    // ---- pass 1: forward, the state at every sub-chunk start (local launch: from zero, with Σ Δ)
    float2 h[2];
    float dsum = 0.f;
    if (LOCAL)
        h[0] = h[1] = f2(0.f);
    else
        load_quad(seg == 0 ? p.h0 : p.h_slots + seg * count, h);
    for (int ch = c0; pass1 && ch < c1; ++ch) {
        wait_staged();
        bwd_prepare<Cfg, TIO, TMA, kStFwd>(sm, raw, p, b, d0, ch, bias_c);
        __syncthreads();                         // staged tiles consumed; the chunk's arrays are ready
        if (TMA && tid == 0 && !*abort_flag) {
            if (ch + 1 < c1) issue(ch + 1, kStFwd);
            else issue(c1 - 1, LOCAL ? kStLam : kStFull);   // pass 2 starts from the last chunk
        }
#pragma unroll 1
        for (int k = 0; k < NSUB; ++k) {
            if constexpr (!LOCAL)
                __stcg(reinterpret_cast<float4*>(ckpt_at(ch, k)), make_float4(h[0].x, h[0].y, h[1].x, h[1].y));
#pragma unroll 4
            for (int r = k * kBS; r < (k + 1) * kBS; ++r) {
                if constexpr (LOCAL) dsum += sm[Cfg::OFF_DEL + r * kBW + cw];
                fold(h, r);
            }
        }
        __syncthreads();                         // the chunk's arrays are no longer read
    }
    if constexpr (LOCAL) {
        if (pass1) {
            if (seg + 1 < p.nseg) store_quad(p.h_slots + (seg + 1) * count, h);
            if (j == 0 && d_ok) p.dsum[seg * static_cast<int64_t>(p.batch) * p.Dm + row] = dsum;
        }
    }

    // ---- pass 2: reverse
    float2 mu[2];                                // a_{t+1} λ_{t+1}: what step t receives
    if (LOCAL)
        mu[0] = mu[1] = f2(0.f);
    else
        load_quad(seg + 1 == p.nseg ? p.dlast : p.m_slots + seg * count, mu);
    if constexpr (LOCAL) {
        // the adjoint alone, λ = C·dŷ + μ, μ ← a·λ, from zero at the segment's end
        for (int ch = c1 - 1; ch >= c0; --ch) {
            wait_staged();
            bwd_prepare<Cfg, TIO, TMA, kStLam>(sm, raw, p, b, d0, ch, bias_c);
            __syncthreads();
            if (TMA && tid == 0 && ch > c0 && !*abort_flag) issue(ch - 1, kStLam);
#pragma unroll 4
            for (int r = kBT - 1; r >= 0; --r) {
                const float del = sm[Cfg::OFF_DEL + r * kBW + cw];
                const float dyh = sm[Cfg::OFF_DYH + r * kBW + cw];
                const float4 Cv = *reinterpret_cast<const float4*>(&sm[Cfg::OFF_C + r * NS + n0]);
                const float2 C2[2] = {f2(Cv.x, Cv.y), f2(Cv.z, Cv.w)};
                if (!pass1) dsum += del;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 e = mul2(f2(del), A2[q]);
                    mu[q] = mul2(f2(ex2(e.x), ex2(e.y)), fma2(C2[q], f2(dyh), mu[q]));
                }
            }
            __syncthreads();
        }
        if (seg > 0) store_quad(p.m_slots + (seg - 1) * count, mu);
        if (!pass1 && j == 0 && d_ok) p.dsum[seg * static_cast<int64_t>(p.batch) * p.Dm + row] = dsum;
        return;
    }
    float2 dA[2] = {f2(0.f), f2(0.f)};
    float dDacc = 0.f, dbacc = 0.f;
    TIO* g_du = static_cast<TIO*>(p.du);
    TIO* g_dd = static_cast<TIO*>(p.ddelta);
    TIO* g_dz = static_cast<TIO*>(p.dz);
    for (int ch = c1 - 1; ch >= c0; --ch) {
        wait_staged();
        bwd_prepare<Cfg, TIO, TMA, kStFull>(sm, raw, p, b, d0, ch, bias_c);
        if (TMA && tid == 0) tma_store_wait_read();   // the previous chunk's gradient tiles are read out
        __syncthreads();
        if (TMA && tid == 0 && ch > c0 && !*abort_flag) issue(ch - 1, kStFull);
#pragma unroll 1
        for (int k = NSUB - 1; k >= 0; --k) {
            float2 H[kBS][2], hb0[2];
            float yh[kBS];
            {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(ckpt_at(ch, k)));
                hb0[0] = f2(v.x, v.y);
                hb0[1] = f2(v.z, v.w);
            }
            h[0] = hb0[0];
            h[1] = hb0[1];
            // refold the sub-chunk's states from its checkpoint, with ŷ = Σ C h + D u
#pragma unroll
            for (int i = 0; i < kBS; ++i) {
                const int r = k * kBS + i;
                fold(h, r);
                H[i][0] = h[0];
                H[i][1] = h[1];
                const float4 Cv = *reinterpret_cast<const float4*>(&sm[Cfg::OFF_C + r * NS + n0]);
                const float2 yp = fma2(h[1], f2(Cv.z, Cv.w), mul2(h[0], f2(Cv.x, Cv.y)));
                yh[i] = fmaf(Dd, sm[Cfg::OFF_U + r * kBW + cw], channel_sum<CPW>(yp.x + yp.y));
            }
            // the adjoint recurrence backwards over them
#pragma unroll
            for (int i = kBS - 1; i >= 0; --i) {
                const int r = k * kBS + i;
                const int t = ch * kBT + r;
                const float del = sm[Cfg::OFF_DEL + r * kBW + cw];
                const float ut = sm[Cfg::OFF_U + r * kBW + cw];
                const float dyh = sm[Cfg::OFF_DYH + r * kBW + cw];
                const float4 Bv = *reinterpret_cast<const float4*>(&sm[Cfg::OFF_B + r * NS + n0]);
                const float4 Cv = *reinterpret_cast<const float4*>(&sm[Cfg::OFF_C + r * NS + n0]);
                const float2 B2[2] = {f2(Bv.x, Bv.y), f2(Bv.z, Bv.w)};
                const float2 C2[2] = {f2(Cv.x, Cv.y), f2(Cv.z, Cv.w)};
                const float2 dut = f2(del * ut);
                float2 s1 = f2(0.f), slb = f2(0.f), bcB[2], bcC[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 l = fma2(C2[q], f2(dyh), mu[q]);          // λ_t
                    const float2 e = mul2(f2(del), A2[q]);
                    const float2 a = f2(ex2(e.x), ex2(e.y));             // a_t
                    const float2 hp = i > 0 ? H[i - 1][q] : hb0[q];       // h_{t-1}
                    mu[q] = mul2(a, l);
                    const float2 w = mul2(mu[q], hp);                    // λ_t a_t h_{t-1}
                    dA[q] = fma2(f2(del), w, dA[q]);
                    s1 = fma2(An[q], w, s1);
                    slb = fma2(l, B2[q], slb);
                    bcB[q] = mul2(l, dut);                               // dB of the pair
                    bcC[q] = mul2(f2(dyh), H[i][q]);                     // dC of the pair
                }
                {
                    // the tile's sums over channels: reduce over the warp's channel lanes,
                    // then one shared atomic per lane (the warps of the tile add up there)
                    const float bc[8] = {bcB[0].x, bcB[0].y, bcB[1].x, bcB[1].y,
                                         bcC[0].x, bcC[0].y, bcC[1].x, bcC[1].y};
                    const float sum = channel_reduce_scatter<CPW>(bc, c);
                    if (c < 8) {
                        const int kk = c & 7;
                        atomicAdd(&sm[Cfg::OFF_BC + r * 2 * NS + (kk < 4 ? 0 : NS) + n0 + (kk & 3)], sum);
                    }
                }
                const float S1 = channel_sum<CPW>(s1.x + s1.y);          // Σ_n A λ a h_{t-1}
                const float SLB = channel_sum<CPW>(slb.x + slb.y);       // Σ_n λ B
                // (steps past L and channels past Dm contribute zeros to the sums)
                const float ddel = fmaf(ut, SLB, S1) * sm[Cfg::OFF_SIG + r * kBW + cw];
                const float duv = fmaf(Dd, dyh, del * SLB);
                const float dzv = p.z ? sm[Cfg::OFF_DYG + r * kBW + cw] * yh[i] : 0.f;
                dDacc = fmaf(dyh, ut, dDacc);
                dbacc += ddel;
                if constexpr (TMA) {
                    // into the chunk's gradient tiles (the channel's LPC lanes write the same value)
                    o_du[r * kBW + cw] = from_f32<TIO>(duv);
                    o_dd[r * kBW + cw] = from_f32<TIO>(ddel);
                    if (p.z) o_dz[r * kBW + cw] = from_f32<TIO>(dzv);
                } else if (j == 0 && d_ok && t < p.L) {
                    const int64_t o = (static_cast<int64_t>(b) * p.L + t) * p.Dm + d;
                    g_du[o] = from_f32<TIO>(duv);
                    g_dd[o] = from_f32<TIO>(ddel);
                    if (p.z) g_dz[o] = from_f32<TIO>(dzv);
                }
            }
        }
        if constexpr (TMA) tma_store_fence();    // the gradient tiles' writes, before the TMA store
        __syncthreads();                         // every shared atomic and read of the chunk is done
        if (TMA && tid == 0) {
            const int t0 = ch * kBT;
            tma_store_3d(&maps.du, o_du, d0, t0, b);
            tma_store_3d(&maps.ddelta, o_dd, d0, t0, b);
            if (p.z) tma_store_3d(&maps.dz, o_dz, d0, t0, b);
            tma_store_commit();
        }
        // four states per thread: one 16-byte reduction each into dB and dC (scalar atomics
        // when N is not a multiple of 4 or the sums are not 16-byte aligned)
        for (int i = tid; i < Cfg::XN / 4; i += Cfg::THREADS) {
            const int r = i / (NS / 4), n = (i % (NS / 4)) * 4;
            const int t = ch * kBT + r;
            float4* bc = reinterpret_cast<float4*>(&sm[Cfg::OFF_BC + r * 2 * NS + n]);
            const float4 vb = bc[0], vc = bc[NS / 4];
            bc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            bc[NS / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < p.L && n < p.N) {
                const int64_t o = (static_cast<int64_t>(b) * p.L + t) * p.N + n;
                if (p.bc_vec) {
                    atomicAdd(reinterpret_cast<float4*>(p.dB + o), vb);
                    atomicAdd(reinterpret_cast<float4*>(p.dC + o), vc);
                } else {
                    const float b4[4] = {vb.x, vb.y, vb.z, vb.w}, c4[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (n + q < p.N) {
                            atomicAdd(p.dB + o + q, b4[q]);
                            atomicAdd(p.dC + o + q, c4[q]);
                        }
                }
            }
        }
    }
    if (TMA && tid == 0) tma_store_wait_all();
    if (d_ok) {
        const float m4[4] = {mu[0].x, mu[0].y, mu[1].x, mu[1].y};
        const float a4[4] = {dA[0].x * An[0].x, dA[0].y * An[0].y, dA[1].x * An[1].x, dA[1].y * An[1].y};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = n0 + q;
            if (n < p.N) {
                if (p.dh0 && seg == 0) p.dh0[row * p.N + n] = m4[q];
                atomicAdd(p.dA_log + static_cast<int64_t>(d) * p.N + n, a4[q]);
            }
        }
        if (j == 0) {
            if (p.dD) atomicAdd(p.dD + d, dDacc);
            if (p.dbias) atomicAdd(p.dbias + d, dbacc);
        }
    }
}

template <typename TIO, int NS, bool TMA, bool LOCAL>
cudaError_t launch_bwd_t(const BwdParams& p, const BwdMaps& m, cudaStream_t stream) {
    using Cfg = BwdCfg<TIO, NS>;
    cudaError_t e = cudaFuncSetAttribute(ss_bwd_kernel<TIO, NS, TMA, LOCAL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.batch) * static_cast<unsigned>(p.tiles_per_batch) *
                          static_cast<unsigned>(p.nseg);
    ss_bwd_kernel<TIO, NS, TMA, LOCAL><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(p, m);
    return cudaGetLastError();
}

template <typename TIO, bool LOCAL>
cudaError_t launch_bwd(const BwdParams& p, const BwdMaps& m, int ns, bool tma, cudaStream_t stream) {
    if (tma) {
        if (ns == 4) return launch_bwd_t<TIO, 4, true, LOCAL>(p, m, stream);
        if (ns == 8) return launch_bwd_t<TIO, 8, true, LOCAL>(p, m, stream);
        return launch_bwd_t<TIO, 16, true, LOCAL>(p, m, stream);
    }
    if (ns == 4) return launch_bwd_t<TIO, 4, false, LOCAL>(p, m, stream);
    if (ns == 8) return launch_bwd_t<TIO, 8, false, LOCAL>(p, m, stream);
    return launch_bwd_t<TIO, 16, false, LOCAL>(p, m, stream);
}

// Adjoint carry of the time split: slot s ends as the adjoint entering segment s from the right,
//   M_{nseg-1} = dlast,   M_s = exp(A ΣΔ_{s+1}) M_{s+1} + local_{s+1},
// where the local launch left local_{s+1} (the adjoint segment s + 1 hands on when swept from
// zero) in slot s; the mirror image of the forward carry (ss_fwd_carry.cu), right to left.
__global__ void __launch_bounds__(256)
ss_bwd_carry_kernel(const float* __restrict__ A_log, const float* __restrict__ dlast, float* __restrict__ slots,
                    const float* __restrict__ dsum, int64_t rows, int Dm, int N, int nseg) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t count = rows * N;
    if (i >= count) return;
    const int64_t row = i / N;
    const int n = static_cast<int>(i - row * N);
    const int d = static_cast<int>(row % Dm);
    const float a2 = -expf(A_log[static_cast<int64_t>(d) * N + n]) * kLog2e;
    float m = dlast ? dlast[i] : 0.f;
    slots[static_cast<int64_t>(nseg - 1) * count + i] = m;
    for (int s = nseg - 2; s >= 0; --s) {
        const float decay = ex2(a2 * dsum[static_cast<int64_t>(s + 1) * rows + row]);
        float* slot = slots + static_cast<int64_t>(s) * count + i;
        m = fmaf(decay, m, *slot);
        *slot = m;
    }
}

int bwd_ns(int64_t N) { return N <= 4 ? 4 : N <= 8 ? 8 : 16; }

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// CTAs of the backward kernel (fp32, 16 states, TMA: the representative instantiation) that the
// current device holds at once; 0 if it cannot be queried.
int64_t bwd_resident_ctas() {
    using Cfg = BwdCfg<float, 16>;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(ss_bwd_kernel<float, 16, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ss_bwd_kernel<float, 16, true, false>, Cfg::THREADS,
                                                      Cfg::SMEM) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return static_cast<int64_t>(sms) * per_sm;
}

// Schedule and workspace: one CTA per tile, or (when the tiles alone cannot fill the GPU, or
// when forced) the time split into nseg segments of seg_chunks chunks, as many as fill it once
// (at most one per chunk and 64).
struct BwdPlan {
    int nseg = 1, seg_chunks = 0;
    size_t ckpt = 0, slots = 0, dsum = 0, total = 0;
};

BwdPlan bwd_plan(int64_t batch, int64_t L, int64_t Dm, int64_t N) {
    BwdPlan pl;
    const int64_t tiles = batch * ((Dm + kBW - 1) / kBW);
    const int64_t nch = (L + kBT - 1) / kBT;
    const int forced = g_force_bwd_nseg.load();
    int64_t want = 1;
    if (forced >= 2) {
        want = forced;
    } else if (forced < 0) {
        const int64_t resident = bwd_resident_ctas();
        if (tiles > 0 && resident >= 2 * tiles) want = resident / tiles;
    }
    want = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(want, nch), 64));
    pl.seg_chunks = static_cast<int>((nch + want - 1) / want);
    pl.nseg = static_cast<int>((nch + pl.seg_chunks - 1) / pl.seg_chunks);
    pl.ckpt = up256(static_cast<size_t>(tiles) * nch * (kBT / kBS) * kBW * bwd_ns(N) * 4);
    if (pl.nseg > 1) {
        pl.slots = up256(static_cast<size_t>(pl.nseg) * batch * Dm * N * 4);
        pl.dsum = up256(static_cast<size_t>(pl.nseg) * batch * Dm * 4);
    }
    pl.total = pl.ckpt + 2 * pl.slots + pl.dsum;
    return pl;
}

}  // namespace
}  // namespace selscan

using namespace selscan;
using namespace selscan::host;

extern "C" size_t ss_bwd_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N) {
    if (batch <= 0 || L <= 0 || Dm <= 0 || N < 1 || N > 16) return 0;
    if (L > INT32_MAX || Dm > INT32_MAX || batch > INT32_MAX) return 0;
    return bwd_plan(batch, L, Dm, N).total;
}

// ckpt_in: the forward's checkpoints (ss_fwd_ckpt), used when the backward runs unsplit.
static ss_status bwd_impl(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                          const void* B, const void* C, const float* D, const void* z, const float* h0,
                          const void* dy, const float* dlast, void* du, void* ddelta_raw, void* dz,
                          float* dB, float* dC, float* dA_log, float* dD, float* ddelta_bias, float* dh0,
                          int64_t batch, int64_t L, int64_t Dm, int64_t N, const ss_fwd_strides* strides,
                          void* workspace, size_t workspace_bytes, void* stream_ptr, const float* ckpt_in) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (batch < 0 || L < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    ss_fwd_strides s;
    if (strides) {
        s = *strides;
    } else {
        std::memset(&s, 0, sizeof(s));
        s.io_dtype = SS_F32;
        s.u_b = s.delta_b = s.z_b = s.y_b = L * Dm;
        s.u_l = s.delta_l = s.z_l = s.y_l = Dm;
        s.B_b = s.C_b = L * N;
        s.B_l = s.C_l = N;
    }
    if (s.io_dtype != SS_F32 && s.io_dtype != SS_BF16) return SS_ERR_INVALID_ARG;
    const bool bf16 = s.io_dtype == SS_BF16;
    const int64_t es = bf16 ? 2 : 4;
    if (batch == 0 || Dm == 0) return SS_OK;
    if (!A_log || !dA_log) return SS_ERR_INVALID_ARG;
    if (L > INT32_MAX || Dm > INT32_MAX || batch > INT32_MAX) return SS_ERR_UNSUPPORTED;
    // alignment to the element type, checked before anything touches a device
    const void* io_ptrs[] = {u, delta_raw, B, C, z, dy, du, ddelta_raw, dz};
    for (const void* q : io_ptrs)
        if (q && !is_aligned(q, es)) return SS_ERR_MISALIGNED;
    const void* f_ptrs[] = {A_log, D, delta_bias, h0, dlast, dB, dC, dA_log, dD, ddelta_bias, dh0};
    for (const void* q : f_ptrs)
        if (q && !is_aligned(q, 4)) return SS_ERR_MISALIGNED;
    if (ckpt_in && (N != 16)) return SS_ERR_UNSUPPORTED;
    if (ckpt_in && !is_aligned(ckpt_in, 16)) return SS_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    // the sums are accumulated: clear them (also the whole answer when L == 0)
    auto clear = [&](float* q, int64_t n) { return q ? cudaMemsetAsync(q, 0, sizeof(float) * n, stream) : cudaSuccess; };
    if (L == 0) {
        const void* small[] = {A_log, dA_log, dD, ddelta_bias, dh0, dlast};
        for (const void* q : small)
            if (q && !dev_ptr(q, dev)) return SS_ERR_INVALID_ARG;
        if (clear(dA_log, Dm * N) != cudaSuccess || clear(dD, Dm) != cudaSuccess ||
            clear(ddelta_bias, Dm) != cudaSuccess)
            return SS_ERR_CUDA;
        if (dh0) {   // no steps: the gradient of h0 is dlast
            if (dlast) return cudaMemcpyAsync(dh0, dlast, sizeof(float) * batch * Dm * N, cudaMemcpyDeviceToDevice,
                                              stream) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
            return clear(dh0, batch * Dm * N) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
        }
        return SS_OK;
    }
    if (!u || !delta_raw || !B || !C || !dy || !du || !ddelta_raw || !dB || !dC) return SS_ERR_INVALID_ARG;
    if (z && !dz) return SS_ERR_INVALID_ARG;
    const int64_t st[] = {s.u_b, s.u_l, s.delta_b, s.delta_l, s.B_b, s.B_l, s.C_b, s.C_l,
                          z ? s.z_b : 0, z ? s.z_l : 0};
    for (int64_t v : st)
        if (v < 0) return SS_ERR_INVALID_ARG;
    // B, C rows at least N apart, or step stride 0 (time-invariant; dB, dC still come per step)
    if ((s.u_l < Dm || s.delta_l < Dm || (z && s.z_l < Dm) || (s.B_l < N && s.B_l != 0) ||
         (s.C_l < N && s.C_l != 0)) && L > 1)
        return SS_ERR_INVALID_ARG;
    const void* all[] = {u, delta_raw, B, C, z, dy, du, ddelta_raw, dz, A_log, D, delta_bias, h0, dlast,
                         dB, dC, dA_log, dD, ddelta_bias, dh0, ckpt_in};
    for (const void* q : all)
        if (q && !dev_ptr(q, dev)) return SS_ERR_INVALID_ARG;
    // outputs: pairwise disjoint and disjoint from every input
    const Range outs[] = {range3(du, batch, L, Dm, L * Dm, Dm, es), range3(ddelta_raw, batch, L, Dm, L * Dm, Dm, es),
                          range3(dz, batch, L, Dm, L * Dm, Dm, es), range3(dB, batch, L, N, L * N, N, 4),
                          range3(dC, batch, L, N, L * N, N, 4), range3(dA_log, 1, Dm, N, 0, N, 4),
                          range3(dD, 1, 1, Dm, 0, 0, 4), range3(ddelta_bias, 1, 1, Dm, 0, 0, 4),
                          range3(dh0, batch, Dm, N, Dm * N, N, 4)};
    const Range ins[] = {range3(u, batch, L, Dm, s.u_b, s.u_l, es), range3(delta_raw, batch, L, Dm, s.delta_b, s.delta_l, es),
                         range3(z, batch, L, Dm, s.z_b, s.z_l, es), range3(B, batch, L, N, s.B_b, s.B_l, es),
                         range3(C, batch, L, N, s.C_b, s.C_l, es), range3(dy, batch, L, Dm, L * Dm, Dm, es),
                         range3(A_log, 1, Dm, N, 0, N, 4), range3(D, 1, 1, Dm, 0, 0, 4),
                         range3(delta_bias, 1, 1, Dm, 0, 0, 4), range3(h0, batch, Dm, N, Dm * N, N, 4),
                         range3(dlast, batch, Dm, N, Dm * N, N, 4),
                         range3(ckpt_in, 1, 1, batch * ((Dm + kBW - 1) / kBW) * ((L + kBT - 1) / kBT) * 2 * kBW * 16,
                                0, 0, 4)};
    const int nouts = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < nouts; ++i) {
        for (const Range& r : ins)
            if (meet(outs[i], r)) return SS_ERR_INVALID_ARG;
        for (int k = i + 1; k < nouts; ++k)
            if (meet(outs[i], outs[k])) return SS_ERR_INVALID_ARG;
    }
    const BwdPlan plan = bwd_plan(batch, L, Dm, N);
    if (!workspace || workspace_bytes < plan.total) return SS_ERR_INVALID_ARG;
    if (!is_aligned(workspace, 256)) return SS_ERR_MISALIGNED;
    if (!dev_ptr(workspace, dev)) return SS_ERR_INVALID_ARG;
    if (clear(dB, batch * L * N) != cudaSuccess || clear(dC, batch * L * N) != cudaSuccess ||
        clear(dA_log, Dm * N) != cudaSuccess || clear(dD, Dm) != cudaSuccess ||
        clear(ddelta_bias, Dm) != cudaSuccess)
        return SS_ERR_CUDA;

    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.u = u; p.delta = delta_raw; p.z = z; p.Bm = B; p.Cm = C; p.bias = delta_bias; p.A_log = A_log; p.Dv = D;
    p.h0 = h0; p.dy = dy; p.dlast = dlast; p.du = du; p.ddelta = ddelta_raw; p.dz = dz; p.dB = dB; p.dC = dC;
    p.dA_log = dA_log; p.dD = dD; p.dbias = ddelta_bias; p.dh0 = dh0;
    p.ckpt = static_cast<float*>(workspace);
    if (ckpt_in) {                                // the forward's checkpoints: no pass 1
        p.ckpt = const_cast<float*>(ckpt_in);
        p.ckpt_given = 1;
    }
    p.u_b = s.u_b; p.u_l = s.u_l; p.d_b = s.delta_b; p.d_l = s.delta_l; p.z_b = s.z_b; p.z_l = s.z_l;
    p.B_b = s.B_b; p.B_l = s.B_l; p.C_b = s.C_b; p.C_l = s.C_l;
    p.batch = static_cast<int>(batch); p.L = static_cast<int>(L); p.Dm = static_cast<int>(Dm);
    p.N = static_cast<int>(N);
    p.nchunks = static_cast<int>((L + kBT - 1) / kBT);
    p.tiles_per_batch = static_cast<int>((Dm + kBW - 1) / kBW);
    p.bc_vec = (N % 4 == 0 && is_aligned(dB, 16) && is_aligned(dC, 16)) ? 1 : 0;
    if (static_cast<int64_t>(p.batch) * p.tiles_per_batch * plan.nseg > INT32_MAX) return SS_ERR_UNSUPPORTED;
    p.nseg = plan.nseg;
    p.seg_chunks = plan.nseg > 1 ? plan.seg_chunks : p.nchunks;
    if (plan.nseg > 1) {
        char* ws = static_cast<char*>(workspace);
        p.h_slots = reinterpret_cast<float*>(ws + plan.ckpt);
        p.m_slots = reinterpret_cast<float*>(ws + plan.ckpt + plan.slots);
        p.dsum = reinterpret_cast<float*>(ws + plan.ckpt + 2 * plan.slots);
    }
    p.err = device_error_word();
    // staged by TMA when every tensor allows it, else by plain loads
    const int ns = bwd_ns(N);
    const int ft = g_force_bwd_tma.load();
    BwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    bool tma = ft != 0 && (ns * es) % 16 == 0;
    if (tma) {
        tma = make_tile_map(&maps.u, u, bf16, Dm, L, batch, s.u_l, s.u_b, kBW, kBT) &&
              make_tile_map(&maps.delta, delta_raw, bf16, Dm, L, batch, s.delta_l, s.delta_b, kBW, kBT) &&
              (!z || make_tile_map(&maps.z, z, bf16, Dm, L, batch, s.z_l, s.z_b, kBW, kBT)) &&
              make_tile_map(&maps.dy, dy, bf16, Dm, L, batch, Dm, L * Dm, kBW, kBT) &&
              make_tile_map(&maps.B, B, bf16, N, L, batch, s.B_l, s.B_b, ns, kBT) &&
              make_tile_map(&maps.C, C, bf16, N, L, batch, s.C_l, s.C_b, ns, kBT) &&
              make_tile_map(&maps.du, du, bf16, Dm, L, batch, Dm, L * Dm, kBW, kBT) &&
              make_tile_map(&maps.ddelta, ddelta_raw, bf16, Dm, L, batch, Dm, L * Dm, kBW, kBT) &&
              (!z || make_tile_map(&maps.dz, dz, bf16, Dm, L, batch, Dm, L * Dm, kBW, kBT));
    }
    if (ft == 1 && !tma) return SS_ERR_UNSUPPORTED;
    cudaError_t e = cudaSuccess;
    if (plan.nseg > 1) {
        // local sweeps of every segment, then the two carries
        e = bf16 ? launch_bwd<__nv_bfloat16, true>(p, maps, ns, tma, stream)
                 : launch_bwd<float, true>(p, maps, ns, tma, stream);
        if (e != cudaSuccess) return SS_ERR_CUDA;
        if (!p.ckpt_given) {                     // (the checkpoints hold the entering states)
            FwdParams fp;
            std::memset(&fp, 0, sizeof(fp));
            fp.A_log = A_log; fp.h0 = h0; fp.seg_slots = p.h_slots; fp.seg_dsum = p.dsum;
            fp.batch = p.batch; fp.Dm = p.Dm; fp.N = p.N; fp.nseg = p.nseg;
            if (launch_fwd_carry(fp, stream) != cudaSuccess) return SS_ERR_CUDA;
        }
        const int64_t count = batch * Dm * N;
        ss_bwd_carry_kernel<<<static_cast<unsigned>((count + 255) / 256), 256, 0, stream>>>(
            A_log, dlast, p.m_slots, p.dsum, batch * Dm, p.Dm, p.N, p.nseg);
        if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
    }
    e = bf16 ? launch_bwd<__nv_bfloat16, false>(p, maps, ns, tma, stream)
             : launch_bwd<float, false>(p, maps, ns, tma, stream);
    return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

extern "C" ss_status ss_bwd(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                            const void* B, const void* C, const float* D, const void* z, const float* h0,
                            const void* dy, const float* dlast, void* du, void* ddelta_raw, void* dz,
                            float* dB, float* dC, float* dA_log, float* dD, float* ddelta_bias, float* dh0,
                            int64_t batch, int64_t L, int64_t Dm, int64_t N, const ss_fwd_strides* strides,
                            void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, h0, dy, dlast, du, ddelta_raw, dz, dB, dC, dA_log,
                    dD, ddelta_bias, dh0, batch, L, Dm, N, strides, workspace, workspace_bytes, stream, nullptr);
}

extern "C" ss_status ss_bwd_ckpt(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                                 const void* B, const void* C, const float* D, const void* z, const float* h0,
                                 const float* ckpt, const void* dy, const float* dlast, void* du, void* ddelta_raw,
                                 void* dz, float* dB, float* dC, float* dA_log, float* dD, float* ddelta_bias,
                                 float* dh0, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                                 const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream) {
    if (!ckpt && batch > 0 && L > 0 && Dm > 0) return SS_ERR_INVALID_ARG;
    return bwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, h0, dy, dlast, du, ddelta_raw, dz, dB, dC, dA_log,
                    dD, ddelta_bias, dh0, batch, L, Dm, N, strides, workspace, workspace_bytes, stream, ckpt);
}

// Internal test hook (not in the public header): -1 automatic time split, 0 (or 1) never,
// n >= 2 always with up to n segments.  Returns the previous setting.
extern "C" int ss__force_bwd_nseg(int n) { return g_force_bwd_nseg.exchange(n < 0 ? -1 : n <= 1 ? 0 : n); }

// Internal test hook (not in the public header): -1 automatic, 0 plain-load staging, 1 TMA
// staging (SS_ERR_UNSUPPORTED where the tensors rule it out).  Returns the previous setting.
extern "C" int ss__force_bwd_tma(int v) { return g_force_bwd_tma.exchange(v < 0 ? -1 : v > 0 ? 1 : 0); }
