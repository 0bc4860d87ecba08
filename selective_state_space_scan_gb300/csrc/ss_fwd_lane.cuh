// Selective-scan forward kernel, state-split lane layout, for sm_103a.
//
// Computes exactly what ss_fwd specifies (include/selscan.h): per batch row b, channel d,
// state n and step t, with h_{-1} = 0,
//   Δ_t = softplus(delta_raw + bias),  h_t = exp(Δ_t A_n) h_{t-1} + Δ_t B_t,n u_t,
//   y_t = (Σ_n C_t,n h_t[n] + D u_t) · silu(z_t),   last_state = h_{L-1},
// i.e. the recurrence of "mamba-metal: Apple Silicon で Mamba を動かす" (section "Selective
// scan の本質") folded over the pairs (a, b) = (exp2(Δ·A·log2 e), Δ B u) left to right (the
// sequential schedule of the associative scan: the state after step t is the inclusive prefix
// of the pairs applied to h_{-1} = 0), chunk by chunk with the state carried across chunks
// (section "チャンク間 running prefix"); softplus, D·u skip and z gate as in the blog's
// walkthrough of the official CUDA kernel (section "1チャンク内の処理フロー"); raw A_log
// turned into -exp(A_log) once per channel as in SpeechLens kernel-optimization.md
// (MetalSelectiveScan).
//
// Why this layout: every (channel, state) chain is independent, and the sequential fold is
// the cheapest evaluation there is (no second pass, no aggregates).  To give the GPU enough
// independent warps when there are fewer than ~40k channels, a channel's NS states are split
// over LPC lanes (LPC = 1, 2 or 4), each lane folding NS/LPC states with its slice of the state
// in registers across the whole sequence.  A warp covers CPW = 32/LPC channels; a CTA is LPC
// warps covering 32 channels, which share one B/C tile.
//   * per group of LPC steps, lane (c, j) computes Δ, Δ·u for step j of the group and channel
//     c (one warp instruction covers 32 (step, channel) pairs, as when a lane owns a whole
//     channel), and the LPC lanes of a channel exchange them by shuffles;
//   * each lane folds its states over the LPC steps; B, C are read as 16-byte broadcasts;
//   * the C·h partial sums of the LPC lanes of a channel are combined by a shuffle
//     reduce-scatter, after which lane (c, j) owns step j's output: D·u skip, z gate, store.
// u/Δ/z arrive by TMA as one [T × CPW] tile per warp (rows of CPW channels), B/C as one
// [T × NS] tile per CTA, in a STAGES-deep ring of mbarrier-completed stages.  Packed fp32x2
// instructions carry pairs of states.  Steps past L are identity pairs (Δ = 0).
#pragma once

#include "device_common.cuh"
#include "fwd_params.h"

namespace selscan {

template <typename TIO_, int NS_, int LPC_, int T_, int STAGES_, int MINB_>
struct LaneCfg {
    using TIO = TIO_;
    static constexpr int NS = NS_;            // states handled (4, 8 or 16; N <= NS)
    static constexpr int LPC = LPC_;          // lanes per channel
    static constexpr int T = T_;              // steps per chunk
    static constexpr int STAGES = STAGES_;
    static constexpr int MINB = MINB_;
    static constexpr int CPW = 32 / LPC;      // channels per warp
    static constexpr int WARPS = LPC;         // warps per CTA
    static constexpr int W = CPW * WARPS;     // channels per CTA (32)
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int SPL = NS / LPC;      // states per lane
    static constexpr int QPL = SPL / 4;       // state quads per lane
    static constexpr int ES = sizeof(TIO);
    static constexpr bool CONVERT_BC = ES == 2;
    static constexpr int up128(int x) { return (x + 127) / 128 * 128; }
    static constexpr int SUB = T * CPW * ES;                  // one warp's u/Δ/z sub-tile
    static constexpr int TILE_X = WARPS * up128(SUB);          // one tensor, all warps
    static constexpr int TILE_N = T * NS * ES;
    static constexpr int OFF_U = 0;
    static constexpr int OFF_D = TILE_X;
    static constexpr int OFF_Z = 2 * TILE_X;
    static constexpr int OFF_B = 3 * TILE_X;
    static constexpr int OFF_C = OFF_B + up128(TILE_N);
    static constexpr int STAGE_BYTES = OFF_C + up128(TILE_N);
    static constexpr int AUX_BC = 0;                                       // fp32 B,C [2][T][NS]
    static constexpr int AUX_XBUF = AUX_BC + (CONVERT_BC ? 2 * T * NS * 4 : 0);  // [WARPS][32][4] floats
    static constexpr int AUX_FLAG = AUX_XBUF + WARPS * 32 * 16;
    static constexpr int AUX_DONE = AUX_FLAG + 16;                        // per-stage warp counters
    static constexpr int AUX_BAR = AUX_DONE + ((STAGES * 4 + 15) / 16) * 16;
    static constexpr int AUX_BYTES = AUX_BAR + STAGES * 8;
    static constexpr int SMEM_BYTES = 128 + STAGES * STAGE_BYTES + AUX_BYTES;
    static_assert(NS % (4 * LPC) == 0, "each lane must hold whole state quads");
    static_assert(T % LPC == 0 && T <= 256, "chunk must be whole groups and one TMA box");
};

// Plain-load fill of one stage with the TMA layout (per-warp sub-tiles, zeros outside).
template <class Cfg>
__device__ void lane_fill_generic(uint8_t* st, const FwdParams& p, int b, int d0, int chunk) {
    using TIO = typename Cfg::TIO;
    const int64_t t0 = static_cast<int64_t>(chunk) * Cfg::T;
    const TIO zero = from_f32<TIO>(0.f);
    const TIO* u = static_cast<const TIO*>(p.u);
    const TIO* dl = static_cast<const TIO*>(p.delta);
    const TIO* z = static_cast<const TIO*>(p.z);
    for (int idx = threadIdx.x; idx < Cfg::T * Cfg::W; idx += Cfg::THREADS) {
        const int w = idx / (Cfg::T * Cfg::CPW);             // warp sub-tile
        const int rem = idx % (Cfg::T * Cfg::CPW);
        const int r = rem / Cfg::CPW, c = rem % Cfg::CPW;
        const int64_t t = t0 + r;
        const int d = d0 + w * Cfg::CPW + c;
        const bool in = t < p.L && d < p.Dm;
        const int o = w * Cfg::up128(Cfg::SUB) / Cfg::ES + rem;
        reinterpret_cast<TIO*>(st + Cfg::OFF_U)[o] = in ? u[b * p.u_b + t * p.u_l + d] : zero;
        reinterpret_cast<TIO*>(st + Cfg::OFF_D)[o] = in ? dl[b * p.d_b + t * p.d_l + d] : zero;
        if (z) reinterpret_cast<TIO*>(st + Cfg::OFF_Z)[o] = in ? z[b * p.z_b + t * p.z_l + d] : zero;
    }
    const TIO* Bm = static_cast<const TIO*>(p.Bm);
    const TIO* Cm = static_cast<const TIO*>(p.Cm);
    for (int idx = threadIdx.x; idx < Cfg::T * Cfg::NS; idx += Cfg::THREADS) {
        const int r = idx / Cfg::NS, n = idx % Cfg::NS;
        const int64_t t = t0 + r;
        const bool in = t < p.L && n < p.N;
        reinterpret_cast<TIO*>(st + Cfg::OFF_B)[idx] = in ? Bm[b * p.B_b + t * p.B_l + n] : zero;
        reinterpret_cast<TIO*>(st + Cfg::OFF_C)[idx] = in ? Cm[b * p.C_b + t * p.C_l + n] : zero;
    }
}

template <class Cfg>
__device__ __forceinline__ void lane_issue_tma(uint8_t* st, uint64_t* bar, const FwdMaps& m,
                                               bool has_z, int b, int d0, int chunk) {
    const uint32_t bytes = (has_z ? 3u : 2u) * Cfg::WARPS * Cfg::SUB + 2u * Cfg::TILE_N;
    mbar_expect_tx(bar, bytes);
    const int t0 = chunk * Cfg::T;
#pragma unroll
    for (int w = 0; w < Cfg::WARPS; ++w) {
        const int o = w * Cfg::up128(Cfg::SUB);
        const int dw = d0 + w * Cfg::CPW;
        tma_load_3d(st + Cfg::OFF_U + o, &m.u, bar, dw, t0, b);
        tma_load_3d(st + Cfg::OFF_D + o, &m.delta, bar, dw, t0, b);
        if (has_z) tma_load_3d(st + Cfg::OFF_Z + o, &m.z, bar, dw, t0, b);
    }
    tma_load_3d(st + Cfg::OFF_B, &m.B, bar, 0, t0, b);
    tma_load_3d(st + Cfg::OFF_C, &m.C, bar, 0, t0, b);
}

template <class Cfg, bool USE_TMA>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
ss_fwd_lane_kernel(const FwdParams p, const __grid_constant__ FwdMaps maps) {
    using TIO = typename Cfg::TIO;
    constexpr int LPC = Cfg::LPC, CPW = Cfg::CPW, NS = Cfg::NS, QPL = Cfg::QPL, T = Cfg::T;
    constexpr int STAGES = USE_TMA ? Cfg::STAGES : 1;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    uint8_t* aux = smem + STAGES * Cfg::STAGE_BYTES;
    float* bcf = reinterpret_cast<float*>(aux + Cfg::AUX_BC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + Cfg::AUX_FLAG);
    int* done = reinterpret_cast<int*>(aux + Cfg::AUX_DONE);
    float* xbuf = reinterpret_cast<float*>(aux + Cfg::AUX_XBUF) + (threadIdx.x >> 5) * 32 * 4;
    uint64_t* full = reinterpret_cast<uint64_t*>(aux + Cfg::AUX_BAR);

    // A grid or TMA box sized for another tile shape would never complete the stage
    // barriers: refuse to run, and say so.
    if (p.chunk_steps != T || p.tile_channels != Cfg::W) {
        if (threadIdx.x == 0 && p.err) atomicOr(p.err, kErrGeometry);
        return;
    }
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int j = lane / CPW;            // state slice of this lane / step within a group
    const int c = lane % CPW;            // channel within the warp
    const int tile = blockIdx.x;
    const int b = tile / p.tiles_per_batch;
    const int d0 = (tile % p.tiles_per_batch) * Cfg::W;
    const int d = d0 + warp * CPW + c;
    const bool d_ok = d < p.Dm;
    const int nchunks = p.nchunks;
    const bool has_z = p.z != nullptr;
    const int64_t L = p.L;
    const int n0 = j * Cfg::SPL;         // first state of this lane's slice

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) done[s] = 0;
        if (USE_TMA) {
            for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
            mbar_fence_init();
            tma_prefetch_desc(&maps.u);
            tma_prefetch_desc(&maps.delta);
            if (has_z) tma_prefetch_desc(&maps.z);
            tma_prefetch_desc(&maps.B);
            tma_prefetch_desc(&maps.C);
        }
    }
    __syncthreads();
    if (USE_TMA && tid == 0) {
        const int pre = nchunks < STAGES ? nchunks : STAGES;
        for (int ch = 0; ch < pre; ++ch)
            lane_issue_tma<Cfg>(smem + ch * Cfg::STAGE_BYTES, &full[ch], maps, has_z, b, d0, ch);
    }

    // A'[n] = -exp(A_log[d,n]) · log2(e) for this lane's states, hoisted out of the scan.
    float2 A2[QPL][2];
#pragma unroll
    for (int qq = 0; qq < QPL; ++qq) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int n = n0 + 4 * qq + k;
            v[k] = (d_ok && n < p.N) ? -expf(p.A_log[static_cast<int64_t>(d) * p.N + n]) * kLog2e : 0.f;
        }
        A2[qq][0] = make_float2(v[0], v[1]);
        A2[qq][1] = make_float2(v[2], v[3]);
    }
    const float bias_w = (p.bias && d_ok) ? p.bias[d] : 0.f;
    const float D_w = (p.Dv && d_ok) ? p.Dv[d] : 0.f;
    const int64_t ystride = p.y_l * static_cast<int64_t>(sizeof(TIO));   // bytes between steps of y

    float2 h[QPL][2];                    // this lane's slice of the state, kept across chunks
#pragma unroll
    for (int qq = 0; qq < QPL; ++qq) h[qq][0] = h[qq][1] = make_float2(0.f, 0.f);

    for (int ch = 0; ch < nchunks; ++ch) {
        const int stage = ch % STAGES;
        uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
        if (USE_TMA) {
            mbar_wait_bounded(&full[stage], static_cast<uint32_t>((ch / STAGES) & 1), abort_flag, p.err);
        } else {
            lane_fill_generic<Cfg>(st, p, b, d0, ch);
            __syncthreads();
        }
        const int sub = warp * Cfg::up128(Cfg::SUB) / Cfg::ES;   // element offset of this warp's sub-tile
        const TIO* tu = reinterpret_cast<const TIO*>(st + Cfg::OFF_U) + sub;
        const TIO* td = reinterpret_cast<const TIO*>(st + Cfg::OFF_D) + sub;
        const TIO* tz = reinterpret_cast<const TIO*>(st + Cfg::OFF_Z) + sub;
        const float* tB;
        const float* tC;
        if constexpr (Cfg::CONVERT_BC) {
            const TIO* rb = reinterpret_cast<const TIO*>(st + Cfg::OFF_B);
            const TIO* rc = reinterpret_cast<const TIO*>(st + Cfg::OFF_C);
            for (int i = tid; i < T * NS; i += Cfg::THREADS) {
                bcf[i] = to_f32<TIO>(rb[i]);
                bcf[T * NS + i] = to_f32<TIO>(rc[i]);
            }
            __syncthreads();
            tB = bcf;
            tC = bcf + T * NS;
        } else {
            tB = reinterpret_cast<const float*>(st + Cfg::OFF_B);
            tC = reinterpret_cast<const float*>(st + Cfg::OFF_C);
        }
        const int64_t tbase = static_cast<int64_t>(ch) * T;
        const int64_t left = L - tbase;                     // steps of this chunk before L
        const bool whole = left >= T;
        constexpr int GT = T / LPC;                         // step groups in the chunk
        constexpr int G = GT > 16 ? 16 : GT;                // groups per sub-block (register budget)
        static_assert(GT % G == 0, "chunk must be whole sub-blocks");
#pragma unroll 1
        for (int g0 = 0; g0 < GT; g0 += G) {

            // Phase 1: Δ and Δ·u of the steps this lane prepares (step g·LPC + j of each group;
            // zero past L, i.e. identity pairs).  G independent softplus chains.
            float dd[G], du[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int r = (g0 + g) * LPC + j;
                const float x = softplus(to_f32<TIO>(td[r * CPW + c]) + bias_w);
                dd[g] = x;
                du[g] = x * to_f32<TIO>(tu[r * CPW + c]);
            }
            if (!whole) {
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if ((g0 + g) * LPC + j >= left) dd[g] = du[g] = 0.f;
            }
            // Phase 2: the sequential fold.  Step g·LPC + k takes its Δ, Δ·u from lane (c, k);
            // the C·h partial sums of the channel's LPC lanes are reduce-scattered so that lane
            // (c, j) ends with the sum of step g·LPC + j.
            float yv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float dk[LPC], uk[LPC];
#pragma unroll
                for (int k = 0; k < LPC; ++k) {
                    dk[k] = LPC == 1 ? dd[g] : __shfl_sync(0xffffffffu, dd[g], k * CPW + c);
                    uk[k] = LPC == 1 ? du[g] : __shfl_sync(0xffffffffu, du[g], k * CPW + c);
                }
                float yp[LPC];
#pragma unroll
                for (int k = 0; k < LPC; ++k) {
                    const float2 dl2 = make_float2(dk[k], dk[k]), du2 = make_float2(uk[k], uk[k]);
                    const int row = (g0 + g) * LPC + k;
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int qq = 0; qq < QPL; ++qq) {
                        const float4 B4 = *reinterpret_cast<const float4*>(tB + row * NS + n0 + 4 * qq);
                        const float4 C4 = *reinterpret_cast<const float4*>(tC + row * NS + n0 + 4 * qq);
                        const float2 a01 = ex2x2(mul2(dl2, A2[qq][0]));
                        const float2 a23 = ex2x2(mul2(dl2, A2[qq][1]));
                        h[qq][0] = fma2(a01, h[qq][0], mul2(du2, make_float2(B4.x, B4.y)));
                        h[qq][1] = fma2(a23, h[qq][1], mul2(du2, make_float2(B4.z, B4.w)));
                        acc = fma2(make_float2(C4.x, C4.y), h[qq][0], acc);
                        acc = fma2(make_float2(C4.z, C4.w), h[qq][1], acc);
                    }
                    yp[k] = acc.x + acc.y;
                }
                if constexpr (LPC == 1) {
                    yv[g] = yp[0];
                } else if constexpr (LPC == 2) {
                    const bool hi = j & 1;
                    const float send = hi ? yp[0] : yp[1];
                    const float keep = hi ? yp[1] : yp[0];
                    yv[g] = keep + __shfl_xor_sync(0xffffffffu, send, CPW);
                } else {
                    // transpose through this warp's shared scratch: lane (c, j) stores its four
                    // partials, then reads the four slices' partials of step j
                    *reinterpret_cast<float4*>(xbuf + lane * 4) = make_float4(yp[0], yp[1], yp[2], yp[3]);
                    __syncwarp();
                    float sum = 0.f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) sum += xbuf[(k * CPW + c) * 4 + j];
                    yv[g] = sum;
                    __syncwarp();
                }
            }
            // Phase 3: D skip, z gate, store (G independent chains).
            if (d_ok) {
                char* yrow = reinterpret_cast<char*>(static_cast<TIO*>(p.y) + b * p.y_b + (tbase + g0 * LPC + j) * p.y_l + d);
                const int64_t rem = left - g0 * LPC - j;          // steps of this lane's column before L
                const int nst = whole ? G : (rem <= 0 ? 0 : rem >= int64_t(G) * LPC ? G : static_cast<int>((rem + LPC - 1) / LPC));
                if (has_z && nst == G) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int r = (g0 + g) * LPC + j;
                        const float v = fmaf(D_w, to_f32<TIO>(tu[r * CPW + c]), yv[g]) * silu(to_f32<TIO>(tz[r * CPW + c]));
                        *reinterpret_cast<TIO*>(yrow + g * LPC * ystride) = from_f32<TIO>(v);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if (g < nst) {
                            const int r = (g0 + g) * LPC + j;
                            float v = fmaf(D_w, to_f32<TIO>(tu[r * CPW + c]), yv[g]);
                            if (has_z) v *= silu(to_f32<TIO>(tz[r * CPW + c]));
                            *reinterpret_cast<TIO*>(yrow + g * LPC * ystride) = from_f32<TIO>(v);
                        }
                    }
                }
            }
        }
        if (USE_TMA && !Cfg::CONVERT_BC) {
            // Release the stage without a block-wide barrier: the warp that finishes it last
            // refills it, so warps that are ahead run on into the stages already loaded.
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&done[stage], 1) == Cfg::WARPS - 1) {
                    done[stage] = 0;
                    if (ch + STAGES < nchunks && !*abort_flag)
                        lane_issue_tma<Cfg>(st, &full[stage], maps, has_z, b, d0, ch + STAGES);
                }
            }
        } else {
            __syncthreads();   // stage (and the widened B/C) consumed by every warp
            if (USE_TMA && tid == 0 && ch + STAGES < nchunks && !*abort_flag)
                lane_issue_tma<Cfg>(st, &full[stage], maps, has_z, b, d0, ch + STAGES);
        }
    }

    if (p.last_state && d_ok) {
        float* out = p.last_state + (static_cast<int64_t>(b) * p.Dm + d) * p.N;
#pragma unroll
        for (int qq = 0; qq < QPL; ++qq) {
            const float v[4] = {h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (n0 + 4 * qq + k < p.N) out[n0 + 4 * qq + k] = v[k];
        }
    }
}

}  // namespace selscan
