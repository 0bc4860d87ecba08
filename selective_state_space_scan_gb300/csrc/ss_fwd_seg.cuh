// Selective-scan forward kernel, segment-lane layout (time-parallel inside a warp), for sm_103a.
//
// What it computes (per batch row b, channel d, state n, step t; h_{-1} = h0, or 0):
//   Δ_t   = softplus(delta_raw[b,t,d] + delta_bias[d])
//   h_t   = exp(Δ_t A_n) h_{t-1} + Δ_t B[b,t,n] u[b,t,d],   A_n = -exp(A_log[d,n])
//   y_t   = (Σ_n C[b,t,n] h_t[n] + D[d] u[b,t,d]) · silu(z[b,t,d])
//   last_state[b,d,n] = h_{L-1}[n]
// following "mamba-metal: Apple Silicon で Mamba を動かす" (section "Selective scan の本質"
// for the recurrence, "チャンク間 running prefix" for the carry) and the blog's walkthrough of
// the official CUDA kernel (section "1チャンク内の処理フロー": softplus, D·u skip, the
// (exp2(Δ·A·log2e), Δ B u) pair per state, scan, out += h·C, z gate), with the tensor
// contract of SpeechLens kernel-optimization.md (MetalSelectiveScan: [B,L,D] streams,
// [B,L,N] B/C shared by all channels, raw A_log turned into -exp(A_log) in registers).
//
// GB300 design (not the pages' design):
//   * One CTA owns a tile of W = 8·G consecutive channels of one batch row and walks
//     the whole sequence in chunks of T = 4·Q·K steps.  Every chunk's u, Δ, z tiles
//     ([T rows × W channels]) and B, C tiles ([T × N], shared by all W channels) arrive
//     by TMA into a STAGES-deep ring of shared-memory buffers, each stage completing on
//     its own mbarrier; the tiles use the hardware swizzle, and the reads below apply
//     the same XOR, which puts a warp's B/C quad reads on different banks.
//   * A warp's 32 lanes are 8 channels × 4 time segments; the warps of a channel group g
//     are Q consecutive groups of 4 segments.  Each thread runs K consecutive steps of
//     one channel sequentially (pass 1, folding the (a,b) pairs into a segment
//     aggregate), the segment aggregates are combined by an intra-warp (a,b) shuffle
//     scan, then across the Q warps through shared memory, and left-combined with the
//     per-(channel,state) carry left by the previous chunk; pass 2 replays the thread's
//     K pairs from its exclusive prefix and accumulates C·h.  States are processed four
//     at a time so that B and C come in as one 16-byte shared load per step.
//   * Rows past L are identity pairs (a = 1, b = 0), so the carry after the last chunk
//     is h_{L-1}.  Channels past Dm read zeros and store nothing.
#pragma once

#include "device_common.cuh"
#include "fwd_params.h"

namespace selscan {

template <typename TIO_, int NS_, int G_, int Q_, int K_, int STAGES_>
struct FwdCfg {
    using TIO = TIO_;
    static constexpr int NS = NS_;            // states handled (N rounded up to 4, 8 or 16)
    static constexpr int G = G_;              // channel groups of 8 per CTA
    static constexpr int Q = Q_;              // warps (4 segments each) per channel group
    static constexpr int K = K_;              // steps per thread per chunk
    static constexpr int STAGES = STAGES_;    // TMA ring depth
    static constexpr int W = 8 * G;           // channels per CTA
    static constexpr int S = 4 * Q;           // segments per chunk
    static constexpr int T = S * K;           // steps per chunk
    static constexpr int THREADS = 32 * G * Q;
    static constexpr int NQ = NS / 4;         // state quads
    static constexpr int ES = sizeof(TIO);
    static constexpr int RB = W * ES;         // bytes in one u/Δ/z tile row
    static constexpr int RBC = NS * ES;       // bytes in one B/C tile row
    static constexpr int TILE_X = T * RB;
    static constexpr int TILE_N = T * RBC;
    static constexpr int up1k(int x) { return (x + 1023) / 1024 * 1024; }
    static constexpr int OFF_U = 0;
    static constexpr int OFF_D = up1k(TILE_X);
    static constexpr int OFF_Z = 2 * up1k(TILE_X);
    static constexpr int OFF_B = 3 * up1k(TILE_X);
    static constexpr int OFF_C = OFF_B + up1k(TILE_N);
    static constexpr int STAGE_BYTES = OFF_C + up1k(TILE_N);
    // auxiliary shared memory after the stages (floats)
    // A' and the carry are read as one state quad per channel by the warp's 8 channel lanes: a
    // channel pitch of an odd number of 16-byte units (NSP floats) puts them on different banks
    static constexpr int NSP = (NS / 4) % 2 == 1 ? NS : NS + 4;
    static constexpr int AUX_A = 0;                       // A'[W][NSP] = -exp(A_log)·log2(e)
    static constexpr int AUX_CARRY = AUX_A + W * NSP;     // carry[2][W][NSP]
    static constexpr int AUX_AGGA = AUX_CARRY + 2 * W * NSP;  // aggA[2][Q][W][4]
    static constexpr int AUX_AGGH = AUX_AGGA + 2 * Q * W * 4; // aggH[2][Q][W][4]
    static constexpr int AUX_FLOATS = AUX_AGGH + 2 * Q * W * 4;
    static constexpr int AUX_BYTES = AUX_FLOATS * 4 + 64 + STAGES * 8;   // + abort flag + mbarriers
    static constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + AUX_BYTES;
    static_assert(NS % 4 == 0 && NS <= 16, "NS must be 4, 8 or 16");
    static_assert(T <= 256, "a TMA box row count is at most 256");
    static_assert(RB % 16 == 0 && RBC % 16 == 0 || true, "");
};

// Shared-memory element read from a swizzled tile with RB-byte rows.
template <typename TIO, int RB>
__device__ __forceinline__ float ld_elem(const uint8_t* tile, int row, int col) {
    const uint32_t o = swz<RB>(static_cast<uint32_t>(row * RB + col * (int)sizeof(TIO)));
    return to_f32<TIO>(*reinterpret_cast<const TIO*>(tile + o));
}

// Four consecutive states (one quad) of a B/C tile row, converted to fp32.
template <typename TIO, int RBC>
__device__ __forceinline__ float4 ld_quad(const uint8_t* tile, int row, int quad);

template <>
__device__ __forceinline__ float4 ld_quad<float, 64>(const uint8_t* tile, int row, int quad) {
    return *reinterpret_cast<const float4*>(tile + swz<64>(row * 64 + quad * 16));
}
template <>
__device__ __forceinline__ float4 ld_quad<float, 32>(const uint8_t* tile, int row, int quad) {
    return *reinterpret_cast<const float4*>(tile + swz<32>(row * 32 + quad * 16));
}
template <>
__device__ __forceinline__ float4 ld_quad<float, 16>(const uint8_t* tile, int row, int quad) {
    return *reinterpret_cast<const float4*>(tile + row * 16 + quad * 16);
}
template <int RBC>
__device__ __forceinline__ float4 ld_quad_bf16(const uint8_t* tile, int row, int quad) {
    const uint2 raw = *reinterpret_cast<const uint2*>(tile + swz<RBC>(row * RBC + quad * 8));
    float4 r;
    r.x = __uint_as_float(raw.x << 16);
    r.y = __uint_as_float(raw.x & 0xffff0000u);
    r.z = __uint_as_float(raw.y << 16);
    r.w = __uint_as_float(raw.y & 0xffff0000u);
    return r;
}
template <>
__device__ __forceinline__ float4 ld_quad<__nv_bfloat16, 32>(const uint8_t* t, int r, int q) {
    return ld_quad_bf16<32>(t, r, q);
}
template <>
__device__ __forceinline__ float4 ld_quad<__nv_bfloat16, 16>(const uint8_t* t, int r, int q) {
    return ld_quad_bf16<16>(t, r, q);
}
template <>
__device__ __forceinline__ float4 ld_quad<__nv_bfloat16, 8>(const uint8_t* t, int r, int q) {
    return ld_quad_bf16<8>(t, r, q);
}

__device__ __forceinline__ float f4get(const float4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Plain-load fill of one stage (the path for strides or sizes TMA cannot describe).
// Produces exactly the layout (including swizzle and zero fill) a TMA fill would.
template <class Cfg>
__device__ void fill_stage_generic(uint8_t* st, const FwdParams& p, int b, int d0, int chunk) {
    using TIO = typename Cfg::TIO;
    const int t0 = chunk * Cfg::T;
    for (int idx = threadIdx.x; idx < Cfg::T * Cfg::W; idx += Cfg::THREADS) {
        const int r = idx / Cfg::W, w = idx % Cfg::W;
        const int64_t t = t0 + r;
        const int d = d0 + w;
        const bool in = t < p.L && d < p.Dm;
        const uint32_t o = swz<Cfg::RB>(static_cast<uint32_t>(r * Cfg::RB + w * Cfg::ES));
        const TIO zero = from_f32<TIO>(0.f);
        const TIO* u = static_cast<const TIO*>(p.u);
        const TIO* dl = static_cast<const TIO*>(p.delta);
        *reinterpret_cast<TIO*>(st + Cfg::OFF_U + o) = in ? u[b * p.u_b + t * p.u_l + d] : zero;
        *reinterpret_cast<TIO*>(st + Cfg::OFF_D + o) = in ? dl[b * p.d_b + t * p.d_l + d] : zero;
        if (p.z) {
            const TIO* z = static_cast<const TIO*>(p.z);
            *reinterpret_cast<TIO*>(st + Cfg::OFF_Z + o) = in ? z[b * p.z_b + t * p.z_l + d] : zero;
        }
    }
    for (int idx = threadIdx.x; idx < Cfg::T * Cfg::NS; idx += Cfg::THREADS) {
        const int r = idx / Cfg::NS, n = idx % Cfg::NS;
        const int64_t t = t0 + r;
        const bool in = t < p.L && n < p.N;
        const uint32_t o = swz<Cfg::RBC>(static_cast<uint32_t>(r * Cfg::RBC + n * Cfg::ES));
        const TIO zero = from_f32<TIO>(0.f);
        const TIO* Bm = static_cast<const TIO*>(p.Bm);
        const TIO* Cm = static_cast<const TIO*>(p.Cm);
        *reinterpret_cast<TIO*>(st + Cfg::OFF_B + o) = in ? Bm[b * p.B_b + t * p.B_l + n] : zero;
        *reinterpret_cast<TIO*>(st + Cfg::OFF_C + o) = in ? Cm[b * p.C_b + t * p.C_l + n] : zero;
    }
}

template <class Cfg>
__device__ __forceinline__ void issue_stage_tma(uint8_t* st, uint64_t* bar, const FwdMaps& m,
                                                bool has_z, int b, int d0, int chunk) {
    const uint32_t bytes = (has_z ? 3u : 2u) * Cfg::TILE_X + 2u * Cfg::TILE_N;
    mbar_expect_tx(bar, bytes);
    const int t0 = chunk * Cfg::T;
    tma_load_3d(st + Cfg::OFF_U, &m.u, bar, d0, t0, b);
    tma_load_3d(st + Cfg::OFF_D, &m.delta, bar, d0, t0, b);
    if (has_z) tma_load_3d(st + Cfg::OFF_Z, &m.z, bar, d0, t0, b);
    tma_load_3d(st + Cfg::OFF_B, &m.B, bar, 0, t0, b);
    tma_load_3d(st + Cfg::OFF_C, &m.C, bar, 0, t0, b);
}

template <class Cfg, bool USE_TMA>
__global__ void __launch_bounds__(Cfg::THREADS, 2)   // two CTAs per SM: the few-rows grid is one wave
ss_fwd_seg_kernel(const FwdParams p, const __grid_constant__ FwdMaps maps) {
    using TIO = typename Cfg::TIO;
    constexpr int W = Cfg::W, K = Cfg::K, Q = Cfg::Q, NS = Cfg::NS, NQ = Cfg::NQ, T = Cfg::T;
    constexpr int STAGES = USE_TMA ? Cfg::STAGES : 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Round up to 1024 bytes (the swizzle period) by pointer arithmetic on the shared array,
    // keeping every pointer visibly in the shared window.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* aux = reinterpret_cast<float*>(smem + STAGES * Cfg::STAGE_BYTES);
    float* sA = aux + Cfg::AUX_A;
    float* carry = aux + Cfg::AUX_CARRY;
    float* aggA = aux + Cfg::AUX_AGGA;
    float* aggH = aux + Cfg::AUX_AGGH;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + Cfg::AUX_FLOATS);
    uint64_t* full = reinterpret_cast<uint64_t*>(aux + Cfg::AUX_FLOATS + 16);

    // A grid or TMA box sized for another tile shape would never complete the stage
    // barriers: refuse to run, and say so.
    if (p.chunk_steps != Cfg::T || p.tile_channels != Cfg::W) {
        if (threadIdx.x == 0 && p.err) atomicOr(p.err, kErrGeometry);
        return;
    }
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int w_lo = lane & 7, s_lo = lane >> 3;
    const int g = warp % Cfg::G, q = warp / Cfg::G;
    const int w = g * 8 + w_lo;                 // channel within the tile
    const int seg = q * 4 + s_lo;               // time segment within the chunk
    const int row0 = seg * K;

    const int tile = blockIdx.x;
    const int b = tile / p.tiles_per_batch;
    const int d0 = (tile % p.tiles_per_batch) * W;
    const int d = d0 + w;
    const bool d_ok = d < p.Dm;
    const int nchunks = p.nchunks;
    const bool has_z = p.z != nullptr;

    if (USE_TMA && tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        tma_prefetch_desc(&maps.u);
        tma_prefetch_desc(&maps.delta);
        if (has_z) tma_prefetch_desc(&maps.z);
        tma_prefetch_desc(&maps.B);
        tma_prefetch_desc(&maps.C);
    }
    if (!USE_TMA && tid == 0) *abort_flag = 0;
    // A'[w][n] = -exp(A_log[d,n]) · log2(e): hoisted out of the sequence loop.
    for (int i = tid; i < W * NS; i += Cfg::THREADS) {
        const int ww = i / NS, n = i % NS;
        const int dd = d0 + ww;
        sA[ww * Cfg::NSP + n] = (dd < p.Dm && n < p.N) ? -expf(p.A_log[static_cast<int64_t>(dd) * p.N + n]) * kLog2e
                                                      : 0.f;
        // the state before the first chunk: h0, or zeros
        carry[ww * Cfg::NSP + n] = (p.h0 && dd < p.Dm && n < p.N)
                                       ? p.h0[(static_cast<int64_t>(b) * p.Dm + dd) * p.N + n] : 0.f;
    }
    __syncthreads();
    if (USE_TMA && tid == 0) {
        const int pre = nchunks < STAGES ? nchunks : STAGES;
        for (int c = 0; c < pre; ++c)
            issue_stage_tma<Cfg>(smem + c * Cfg::STAGE_BYTES, &full[c], maps, has_z, b, d0, c);
    }

    const float bias_w = (p.bias && d_ok) ? p.bias[d] : 0.f;
    const float D_w = (p.Dv && d_ok) ? p.Dv[d] : 0.f;

    for (int c = 0; c < nchunks; ++c) {
        const int stage = c % STAGES;
        uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
        if (USE_TMA) {
            mbar_wait_bounded(&full[stage], static_cast<uint32_t>((c / STAGES) & 1), abort_flag,
                              p.err);
        } else {
            fill_stage_generic<Cfg>(st, p, b, d0, c);
            __syncthreads();
        }
        const uint8_t* tu = st + Cfg::OFF_U;
        const uint8_t* td = st + Cfg::OFF_D;
        const uint8_t* tB = st + Cfg::OFF_B;
        const uint8_t* tC = st + Cfg::OFF_C;
        const int64_t tbase = static_cast<int64_t>(c) * T;

        // Δ and Δ·u for this thread's K steps (rows past L become identity pairs).
        float dl[K], du[K];
        float sumd = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int r = row0 + i;
            const float x = ld_elem<TIO, Cfg::RB>(td, r, w) + bias_w;
            const float uu = ld_elem<TIO, Cfg::RB>(tu, r, w);
            const float dd = (tbase + r < p.L) ? softplus(x) : 0.f;
            dl[i] = dd;
            du[i] = dd * uu;
            sumd += dd;
        }
        // C·h partial sums of each step, over even and odd states (packed fp32x2 arithmetic)
        float2 yacc[K];
#pragma unroll
        for (int i = 0; i < K; ++i) yacc[i] = make_float2(0.f, 0.f);

        const float* carry_in = carry + (c & 1) * W * Cfg::NSP;
        float* carry_out = carry + ((c & 1) ^ 1) * W * Cfg::NSP;

#pragma unroll 1
        for (int qd = 0; qd < NQ; ++qd) {
            const float4 A4 = *reinterpret_cast<const float4*>(sA + w * Cfg::NSP + qd * 4);
            const float2 A2[2] = {make_float2(A4.x, A4.y), make_float2(A4.z, A4.w)};
            // the quad's states as two pairs: (a, b) of every step, and the local fold
            float2 a[K][2], bb[K][2];
            float2 H2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            // pass 1: pairs and the thread-local fold over K steps
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float4 Bq = ld_quad<TIO, Cfg::RBC>(tB, row0 + i, qd);
                const float2 Bp[2] = {make_float2(Bq.x, Bq.y), make_float2(Bq.z, Bq.w)};
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const float2 e = mul2(make_float2(dl[i], dl[i]), A2[pr]);
                    a[i][pr] = make_float2(ex2(e.x), ex2(e.y));
                    bb[i][pr] = mul2(make_float2(du[i], du[i]), Bp[pr]);
                    H2[pr] = fma2(a[i][pr], H2[pr], bb[i][pr]);
                }
            }
            float H[4] = {H2[0].x, H2[0].y, H2[1].x, H2[1].y};
            float Ag[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) Ag[j] = ex2(sumd * f4get(A4, j));
            // Inclusive scan of the segment maps across this warp's 4 segments (lanes 8 apart): in
            // two doubling rounds each lane composes its map with the one `off` segments earlier,
            // so that it ends with the map of every segment up to its own.
#pragma unroll
            for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const AffinePair earlier{__shfl_up_sync(0xffffffffu, Ag[j], off),
                                             __shfl_up_sync(0xffffffffu, H[j], off)};
                    if (lane >= off) {
                        const AffinePair upto = compose(AffinePair{Ag[j], H[j]}, earlier);
                        Ag[j] = upto.a;
                        H[j] = upto.b;
                    }
                }
            }
            float Ae[4], He[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                Ae[j] = __shfl_up_sync(0xffffffffu, Ag[j], 8);
                He[j] = __shfl_up_sync(0xffffffffu, H[j], 8);
                if (s_lo == 0) { Ae[j] = 1.f; He[j] = 0.f; }
            }
            // block level: aggregates of the earlier warps of this channel group
            const int par = (c * NQ + qd) & 1;
            if constexpr (Q > 1) {
                if (s_lo == 3) {
                    const int slot = ((par * Q + q) * W + w) * 4;
                    *reinterpret_cast<float4*>(aggA + slot) = make_float4(Ag[0], Ag[1], Ag[2], Ag[3]);
                    *reinterpret_cast<float4*>(aggH + slot) = make_float4(H[0], H[1], H[2], H[3]);
                }
                named_barrier(1 + g, Q * 32);
            }
            float4 hin4 = *reinterpret_cast<const float4*>(carry_in + w * Cfg::NSP + qd * 4);
            float hin[4] = {hin4.x, hin4.y, hin4.z, hin4.w};
            if constexpr (Q > 1) {
                for (int qq = 0; qq < q; ++qq) {
                    const int slot = ((par * Q + qq) * W + w) * 4;
                    const float4 pa = *reinterpret_cast<const float4*>(aggA + slot);
                    const float4 ph = *reinterpret_cast<const float4*>(aggH + slot);
#pragma unroll
                    for (int j = 0; j < 4; ++j) hin[j] = fmaf(f4get(pa, j), hin[j], f4get(ph, j));
                }
            }
            if (q == Q - 1 && s_lo == 3) {
                *reinterpret_cast<float4*>(carry_out + w * Cfg::NSP + qd * 4) =
                    make_float4(fmaf(Ag[0], hin[0], H[0]), fmaf(Ag[1], hin[1], H[1]),
                                fmaf(Ag[2], hin[2], H[2]), fmaf(Ag[3], hin[3], H[3]));
            }
            // pass 2: replay the K pairs from the exclusive prefix, accumulate C·h
            float2 h[2] = {make_float2(fmaf(Ae[0], hin[0], He[0]), fmaf(Ae[1], hin[1], He[1])),
                           make_float2(fmaf(Ae[2], hin[2], He[2]), fmaf(Ae[3], hin[3], He[3]))};
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float4 Cq = ld_quad<TIO, Cfg::RBC>(tC, row0 + i, qd);
                const float2 Cp[2] = {make_float2(Cq.x, Cq.y), make_float2(Cq.z, Cq.w)};
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    h[pr] = fma2(a[i][pr], h[pr], bb[i][pr]);
                    yacc[i] = fma2(Cp[pr], h[pr], yacc[i]);
                }
            }
        }

        // epilogue: D skip, z gate, store
        if (d_ok) {
            TIO* y = static_cast<TIO*>(p.y);
            const uint8_t* tz = st + Cfg::OFF_Z;
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const int r = row0 + i;
                const int64_t t = tbase + r;
                if (t < p.L) {
                    float v = fmaf(D_w, ld_elem<TIO, Cfg::RB>(tu, r, w), yacc[i].x + yacc[i].y);
                    if (has_z) v *= silu(ld_elem<TIO, Cfg::RB>(tz, r, w));
                    y[b * p.y_b + t * p.y_l + d] = from_f32<TIO>(v);
                }
            }
        }
        __syncthreads();   // stage consumed; carry_out visible to the next chunk
        if (USE_TMA && tid == 0 && c + STAGES < nchunks && !*abort_flag)
            issue_stage_tma<Cfg>(st, &full[stage], maps, has_z, b, d0, c + STAGES);
    }

    if (p.last_state && d_ok) {
        const float* fin = carry + (nchunks & 1) * W * Cfg::NSP;
        for (int n = seg; n < p.N; n += Cfg::S)
            p.last_state[(static_cast<int64_t>(b) * p.Dm + d) * p.N + n] = fin[w * Cfg::NSP + n];
    }
}

}  // namespace selscan
