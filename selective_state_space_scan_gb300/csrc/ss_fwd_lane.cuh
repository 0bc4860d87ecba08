// Selective-scan forward kernel, state-split lane layout, for sm_103a.
//
// Computes exactly what ss_fwd specifies (include/selscan.h): per batch row b, channel d,
// state n and step t, with h_{-1} = h0 (zeros when none is given),
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
// in registers.  A warp covers CPW = 32/LPC channels; a CTA covers a tile of W channels
// (W/CPW warps), which share one B/C tile.  Each chunk of T steps runs in three phases per warp:
//   1. lane (c, j) computes Δ, Δ·u for step j of every group of LPC steps (one warp
//      instruction covers 32 (step, channel) pairs; independent softplus chains);
//   2. the fold: step g·LPC + k takes Δ, Δ·u from lane (c, k) by shuffle, B and C are 16-byte
//      shared-memory broadcasts, packed fp32x2 instructions carry pairs of states; the C·h
//      partial sums of a channel's LPC lanes are reduce-scattered by shuffles so that lane
//      (c, j) owns step j's sum;
//   3. D·u skip, z gate, store (one row of the warp's channels per step).
// u/Δ/z arrive by TMA as one [T × W] tile per stream (rows of W channels, hardware swizzle:
// few, long rows keep the TMA engine's row count low), B/C as one [T × NS] tile, in a
// STAGES-deep ring of mbarrier-completed stages.  Steps past L are identity pairs (Δ = 0).
//
// Schedules.  Without a workspace each CTA owns one tile and walks its whole sequence.  With
// one (FwdParams::ws_flag), the grid is the number of CTAs that fit on the GPU at once and each
// CTA takes an equal contiguous range of the (tile, chunk) units, so every SM gets the same
// work.  A range may start inside a tile: the previous CTA folds that tile's head first and
// publishes the state where it stops; this CTA folds that piece last, after waiting (with a
// time limit) for the publication.  In the time-split schedule (FwdParams::seg_launch) CTA x
// folds one segment of one tile: pass A (STATE_ONLY) from a zero state, keeping only the end
// state and Σ Δ; pass C from the segment's start state that the carry kernel composed.
#pragma once

#include <type_traits>

#include "device_common.cuh"
#include "fwd_params.h"

namespace selscan {

// DTR > 0: the low-rank time-step projection is folded in; the Δ tile's place holds a
// [T][DTR-float-pitch] dt_low tile instead.
// BCF32: B and C arrive as fp32 tiles (a widened copy of bf16 B, C that the workspace schedules
// make before the scan), so bf16 streams need no per-chunk widening in shared memory.
// XCH: room for this CTA's segment summary (end state [W][NS] and Σ Δ [W]) that the CTAs of a
// cluster read from each other (the single-launch time split).
// DX4: at 4 lanes per channel (fp32), the prepared (Δ, Δ·u) go through shared memory as at 2
// (see DXS); its rows take 16.5 KB a CTA, which leaves room for two CTAs per SM, so only the
// balanced schedule on 32-channel tiles uses it, where the grid is two CTAs per SM anyway
// (130m-shaped layer: 133.5 -> 129.7 us; one CTA per tile, which needs three per SM, 141 -> 168).
template <typename TIO_, int NS_, int LPC_, int W_, int T_, int STAGES_, int MINB_, int DTR_ = 0, bool BCF32_ = false,
          bool XCH_ = false, bool DX4_ = false>
struct LaneCfg {
    using TIO = TIO_;
    static constexpr int NS = NS_;            // states handled (4, 8 or 16; N <= NS)
    static constexpr int LPC = LPC_;          // lanes per channel
    static constexpr int W = W_;              // channels per CTA (tile)
    static constexpr int T = T_;              // steps per chunk
    static constexpr int STAGES = STAGES_;
    static constexpr int MINB = MINB_;
    static constexpr int DTR = DTR_;          // dt_low row pitch bound (floats); 0: Δ tile
    static constexpr int CPW = 32 / LPC;      // channels per warp
    static constexpr int WARPS = W / CPW;     // warps per CTA
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int SPL = NS / LPC;      // states per lane
    static constexpr int QPL = SPL / 4;       // state quads per lane
    static constexpr int ES = sizeof(TIO);
    static constexpr bool BCF32 = BCF32_;
    static constexpr bool XCH = XCH_;
    static constexpr int ES_BC = BCF32_ ? 4 : ES;             // bytes per staged B/C element
    static constexpr bool CONVERT_BC = ES_BC == 2;
    static constexpr int up128(int x) { return (x + 127) / 128 * 128; }
    static constexpr int up1024(int x) { return (x + 1023) / 1024 * 1024; }
    static constexpr int RB = W * ES;                         // bytes of one tile row (W channels)
    static constexpr int TILE_X = T * RB;                     // one tensor's [T][W] tile, swizzled
    static constexpr int TILE_N = T * NS * ES_BC;
    static constexpr int TILE_D = DTR > 0 ? up1024(T * DTR * 4) : TILE_X;
    static constexpr int OFF_U = 0;
    static constexpr int OFF_D = TILE_X;
    static constexpr int OFF_Z = OFF_D + TILE_D;
    static constexpr int OFF_B = OFF_Z + TILE_X;
    static constexpr int OFF_C = OFF_B + up128(TILE_N);
    static constexpr int STAGE_BYTES = up1024(OFF_C + up128(TILE_N));   // keeps every tile 1 KB aligned
    static constexpr int AUX_BC = 0;                                       // fp32 B,C [2][T][NS]
    static constexpr int AUX_FLAG = AUX_BC + (CONVERT_BC ? 2 * T * NS * 4 : 0);
    static constexpr int AUX_DONE = AUX_FLAG + 16;                        // per-stage warp counters
    static constexpr int AUX_BAR = AUX_DONE + ((STAGES * 4 + 15) / 16) * 16;
    static constexpr int AUX_W = AUX_BAR + ((STAGES * 8 + 15) / 16) * 16;   // DTR > 0: W_dt rows [W][DTR]
    // Step groups per sub-block (register budget): at most 16, a divisor of the chunk's groups.
    static constexpr int GT = T / LPC;
// (At most 16 groups: at 8 the 2.8b-shaped layer measured 717 against 677 us.)
#ifndef SS_LANE_GMAX
#define SS_LANE_GMAX 16
#endif
    static constexpr int G = GT <= SS_LANE_GMAX ? GT : GT % SS_LANE_GMAX == 0 ? SS_LANE_GMAX : GT % 12 == 0 ? 12 : 8;
    // DXS: the prepared (Δ, Δ·u) of a sub-block go through shared memory, [CPW][G·LPC + 2] float2
    // per warp (rows padded so that a warp's 16-byte reads of its channels spread over the banks),
    // read back two steps per 16-byte load, instead of two shuffles per step.  fp32 only: at 2
    // lanes per channel it measured 153 against 170 us on the 130m-shaped layer, while on the
    // 2.8b-shaped bf16 layer the shuffles were faster (694 against 724 us).
    // (At 2 lanes with bf16 streams and fp32 B/C tiles it measured 701 against 667 us.)
    static constexpr bool DXS = ES == 4 && ((LPC == 2 && SS_DX_SMEM) || (LPC == 4 && DX4_));
    static constexpr int NDX = LPC > 1 ? LPC / 2 : 1;                     // 16-byte reads per group
    static constexpr int DX_PITCH = G * LPC + 2;                          // float2 per channel row
    static constexpr int AUX_DX = AUX_W + (DTR > 0 ? W * DTR * 4 : 0);
    static constexpr int AUX_XCH = AUX_DX + (DXS ? WARPS * CPW * DX_PITCH * 8 : 0);
    static constexpr int AUX_BYTES = AUX_XCH + (XCH_ ? W * NS * 4 + W * 4 : 0);
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + AUX_BYTES;
    static_assert(RB == 128 || RB == 64 || RB == 32, "a tile row must be one TMA swizzle span");
    static_assert(NS % (4 * LPC) == 0, "each lane must hold whole state quads");
    static_assert(W % CPW == 0 && WARPS >= 1, "a tile is whole warps");
    static_assert(T % LPC == 0 && T <= 256, "chunk must be whole groups and one TMA box");
    static_assert(DTR == 0 || ES == 4, "the folded projection is built for fp32 I/O");
    static_assert(!BCF32_ || (ES == 2 && DTR == 0), "widened B/C tiles serve bf16 streams");
    static_assert(!DX4_ || (LPC == 4 && ES == 4), "the 4-lane shared-memory hand-over is built for fp32");
};

// A CTA's work in processing order: up to three runs of (tile, chunk) units.
//   run 0: the head (chunks [0, c_end)) of the last tile of the range, if the range ends
//          inside it; its final state is published for the next CTA;
//   run 1: whole tiles;
//   run 2: the tail (chunks [c_start, nchunks)) of the first tile of the range, if the range
//          starts inside it; its initial state comes from the previous CTA.
struct LaneWork {
    int t0, n0;          // run 0: tile, chunk count (chunks 0 .. n0-1)
    int t1, n1;          // run 1: first whole tile, unit count (whole tiles × nchunks)
    int t2, c2, n2;      // run 2: tile, first chunk, count
    __device__ __forceinline__ int total() const { return n0 + n1 + n2; }
    __device__ __forceinline__ void unit(int k, int nchunks, int& tile, int& chunk) const {
        if (k < n0) { tile = t0; chunk = k; return; }
        k -= n0;
        if (k < n1) { tile = t1 + k / nchunks; chunk = k % nchunks; return; }
        k -= n1;
        tile = t2;
        chunk = c2 + k;
    }
};

__device__ __forceinline__ LaneWork lane_work(const FwdParams& p, int tiles_total) {
    LaneWork w{0, 0, 0, 0, 0, 0, 0};
    const int nch = p.nchunks;
    if (p.seg_launch > 0) {                   // time-split: one segment of one tile
        const int s = static_cast<int>(blockIdx.x) % p.seg_launch;
        const int c0 = s * p.seg_chunks;
        const int cnt = nch - c0 < p.seg_chunks ? nch - c0 : p.seg_chunks;
        w.t2 = static_cast<int>(blockIdx.x) / p.seg_launch;
        w.c2 = c0;
        w.n2 = cnt > 0 ? cnt : 0;
        return w;
    }
    int64_t U, u0, u1, tbase = 0;
    if (p.cbal > 0) {                         // cluster-balanced: this cluster's whole tiles, split S ways
        const int S = p.cbal, Q = p.grid / p.cbal;
        const int q = static_cast<int>(blockIdx.x) / S, r = static_cast<int>(cluster_ctarank());
        tbase = static_cast<int64_t>(tiles_total) * q / Q;
        U = (static_cast<int64_t>(tiles_total) * (q + 1) / Q - tbase) * nch;
        u0 = U * r / S;
        u1 = U * (r + 1) / S;
    } else if (p.ws_flag == nullptr) {        // one whole tile per CTA
        w.t1 = blockIdx.x;
        w.n1 = nch;
        return w;
    } else {
        U = static_cast<int64_t>(tiles_total) * nch;
        u0 = U * blockIdx.x / p.grid;
        u1 = U * (blockIdx.x + 1) / p.grid;
    }
    if (u1 <= u0) return w;
    const int tf = static_cast<int>(tbase + u0 / nch), cf = static_cast<int>(u0 % nch);
    const int tl = static_cast<int>(tbase + (u1 - 1) / nch), ce = static_cast<int>((u1 - 1) % nch) + 1;
    if (tf == tl) {                           // the whole of one tile (a range spans at least one tile)
        w.t1 = tf;
        w.n1 = nch;
        return w;
    }
    if (ce < nch) { w.t0 = tl; w.n0 = ce; }
    if (cf > 0) { w.t2 = tf; w.c2 = cf; w.n2 = nch - cf; }
    const int first_whole = cf > 0 ? tf + 1 : tf;
    const int last_whole = ce < nch ? tl - 1 : tl;
    w.t1 = first_whole;
    w.n1 = last_whole >= first_whole ? (last_whole - first_whole + 1) * nch : 0;
    return w;
}

// Plain-load fill of one stage with the TMA layout (swizzled [T][W] tiles, zeros outside).
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
        const uint32_t o = swz<Cfg::RB>(static_cast<uint32_t>(r * Cfg::RB + (w * Cfg::CPW + c) * Cfg::ES));
        *reinterpret_cast<TIO*>(st + Cfg::OFF_U + o) = in ? u[b * p.u_b + t * p.u_l + d] : zero;
        *reinterpret_cast<TIO*>(st + Cfg::OFF_D + o) = in ? dl[b * p.d_b + t * p.d_l + d] : zero;
        if (z) *reinterpret_cast<TIO*>(st + Cfg::OFF_Z + o) = in ? z[b * p.z_b + t * p.z_l + d] : zero;
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

// WITH_C = false (pass A of the time split) skips the C tile; has_z = false the z tile; LTI
// (time-invariant B and C, held in registers) both B/C tiles.
// With the projection folded in (Cfg::DTR > 0) the Δ box is the chunk's [T][dt_pitch] dt_low
// rows (shared by all channels, x = 0).
template <class Cfg, bool WITH_C, bool LTI = false>
__device__ __forceinline__ void lane_issue_tma(uint8_t* st, uint64_t* bar, const FwdMaps& m,
                                               bool has_z, int b, int d0, int chunk, int dt_pitch) {
    const uint32_t d_bytes = Cfg::DTR > 0 ? static_cast<uint32_t>(Cfg::T * dt_pitch * 4) : Cfg::TILE_X;
    const uint32_t bytes = (has_z ? 2u : 1u) * Cfg::TILE_X + d_bytes + (LTI ? 0u : (WITH_C ? 2u : 1u) * Cfg::TILE_N);
    mbar_expect_tx(bar, bytes);
    const int t0 = chunk * Cfg::T;
    // one [T][W] box per stream (rows of W channels, hardware swizzle), one [T][NS] box for B, C.
    // (L2 eviction hints were measured: evict-first on the streams re-fetched lines that a
    // neighbouring tile still needed, evict-last on B/C changed nothing; none are used.)
    tma_load_3d(st + Cfg::OFF_U, &m.u, bar, d0, t0, b);
    tma_load_3d(st + Cfg::OFF_D, &m.delta, bar, Cfg::DTR > 0 ? 0 : d0, t0, b);
    if (has_z) tma_load_3d(st + Cfg::OFF_Z, &m.z, bar, d0, t0, b);
    if (!LTI) {
        tma_load_3d(st + Cfg::OFF_B, &m.B, bar, 0, t0, b);
        if (WITH_C) tma_load_3d(st + Cfg::OFF_C, &m.C, bar, 0, t0, b);
    }
}

// Wait (thread 0 only) until another CTA has published with this call's epoch; gives up
// after ~2^31 SM cycles, recording kErrWaitTimeout.
__device__ __forceinline__ void wait_published(const unsigned int* flag, unsigned int epoch,
                                               unsigned int* err) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == epoch) return;
    const long long t0 = clock64();
    while (true) {
        __nanosleep(64);
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v == epoch) return;
        if (clock64() - t0 > (1ll << 31)) {
            if (err) atomicOr(err, kErrWaitTimeout);
            return;
        }
    }
}

// STATE_ONLY: pass A of the time-split schedule.  The same fold from a zero state, without
// C, y or the z gate: it writes the segment's end state and its Σ Δ.
// LTI: B and C do not vary with the step (the linear time-invariant case, step stride 0): each
// lane holds its states' B and C in registers and no B/C tiles are staged.
// CLUSTER: the single-launch time split.  The grid is tiles × p.seg_launch CTAs in clusters of
// p.seg_launch; CTA rank r of a cluster folds segment r of the cluster's tile twice: first from a
// zero state keeping only its end state and Σ Δ (as STATE_ONLY), which it leaves in its shared
// memory; after a cluster barrier it reads the summaries of ranks 0 .. r-1 from their shared
// memory and composes the state entering its segment, H_0 = h0, H_{s+1} = 2^(A'·ΣΔ_s)·H_s + end_s;
// then it folds the segment again from that state with every output.
// CKPT: also write the backward pass's checkpoints (FwdParams::ckpt): one CTA per 32-channel tile,
// or (CLUSTER) from the full fold of each time segment.
// CBAL: the cluster-balanced schedule (FwdParams::cbal; no workspace).  The CTAs of a cluster split
// its tiles' (tile, chunk) units into equal ranges as the balanced schedule does, and a tile split
// between two of them is handed over through distributed shared memory: the CTA that folds the
// head of the tile (its first piece) stores its final state into the exchange area of the next
// CTA of the cluster and arrives on that CTA's hand-over mbarrier; the next CTA waits (bounded)
// on it before the tail (its last piece).  Only neighbours wait for each other; cluster barriers
// at the start (every hand-over mbarrier initialised) and the end (no CTA leaves while its
// neighbour may still write to it) bracket the work.
template <class Cfg, bool USE_TMA, bool STATE_ONLY = false, bool LTI = false, bool CLUSTER = false, bool CKPT = false,
          bool CBAL = false>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
ss_fwd_lane_kernel(const FwdParams p, const __grid_constant__ FwdMaps maps) {
    static_assert(!Cfg::BCF32 || (USE_TMA && !LTI), "widened B/C tiles come by TMA");
    static_assert(!CLUSTER || (USE_TMA && !STATE_ONLY && !LTI && Cfg::DTR == 0), "the cluster split is TMA-fed");
    static_assert(!CBAL || (USE_TMA && Cfg::XCH && !STATE_ONLY && !LTI && !CLUSTER && !CKPT && Cfg::DTR == 0),
                  "the cluster-balanced schedule is TMA-fed and hands states over in the exchange area");
    static_assert(!CKPT || (Cfg::NS == 16 && Cfg::W == 32 && Cfg::LPC > 1 && Cfg::G * Cfg::LPC % 16 == 0 &&
                            !STATE_ONLY && Cfg::DTR == 0),
                  "checkpoints: 16 states, 32-channel tiles, sub-blocks of whole 16-step pieces");
    using TIO = typename Cfg::TIO;
    constexpr int LPC = Cfg::LPC, CPW = Cfg::CPW, NS = Cfg::NS, QPL = Cfg::QPL, T = Cfg::T;
    constexpr int STAGES = USE_TMA ? Cfg::STAGES : 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1 KB alignment (the 128-byte swizzle's period) by pointer arithmetic on the shared array
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* aux = smem + STAGES * Cfg::STAGE_BYTES;
    float* bcf = reinterpret_cast<float*>(aux + Cfg::AUX_BC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + Cfg::AUX_FLAG);
    int* done = reinterpret_cast<int*>(aux + Cfg::AUX_DONE);
    uint64_t* full = reinterpret_cast<uint64_t*>(aux + Cfg::AUX_BAR);

    // A grid or TMA box sized for another tile shape would never complete the stage
    // barriers: refuse to run, and say so.
    if (p.chunk_steps != T || p.tile_channels != Cfg::W || (USE_TMA && p.box_channels != Cfg::W)) {
        if (threadIdx.x == 0 && p.err) atomicOr(p.err, kErrGeometry);
        return;
    }
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int j = lane / CPW;            // state slice of this lane / step within a group
    const int c = lane % CPW;            // channel slot within the warp
    // Channel of this lane within the tile.  fp32: a warp's channels are the 16-byte chunks
    // w, w + WARPS, w + 2·WARPS, ... of the tile row (4 channels each), so that the LPC rows
    // one load touches land on different banks of the swizzled tile; bf16 (8 channels per chunk)
    // is conflict-free with consecutive channels.
    const int cw = Cfg::ES == 4 ? 4 * (warp + Cfg::WARPS * (c >> 2)) + (c & 3) : warp * CPW + c;
    const int nchunks = p.nchunks;
    const bool has_z = p.z != nullptr;
    const int64_t L = p.L;
    const int n0 = j * Cfg::SPL;         // first state of this lane's slice
    const int64_t ystride = p.y_l * static_cast<int64_t>(sizeof(TIO));   // bytes between steps of y
    const LaneWork work = lane_work(p, p.batch * p.tiles_per_batch);
    // CLUSTER: the segment's chunks are staged twice (the summary fold, then the full fold)
    const int total = CLUSTER ? 2 * work.total() : work.total();
    // Byte offset of this lane's element in a swizzled [T][W] tile, for rows j + q·LPC (row
    // offset included).  A sub-block's rows g·LPC + j fall in NCX classes mod 8, and the
    // swizzle depends on the row only mod 8.
    constexpr int NCX = LPC == 4 ? 2 : LPC == 2 ? 4 : 8;
    uint32_t cx[NCX];
#pragma unroll
    for (int q = 0; q < NCX; ++q)
        cx[q] = swz<Cfg::RB>(static_cast<uint32_t>((q * LPC + j) * Cfg::RB + cw * Cfg::ES));

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) done[s] = 0;
        if (USE_TMA) {
            for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
            // the hand-over barrier: one arrival per thread of the previous CTA of the cluster
            if (CBAL) mbar_init(reinterpret_cast<uint64_t*>(aux + Cfg::AUX_XCH + Cfg::W * NS * 4), Cfg::THREADS);
            mbar_fence_init();
            tma_prefetch_desc(&maps.u);
            tma_prefetch_desc(&maps.delta);
            if (has_z) tma_prefetch_desc(&maps.z);
            if (!LTI) {
                tma_prefetch_desc(&maps.B);
                tma_prefetch_desc(&maps.C);
            }
        }
    }
    __syncthreads();
    auto issue = [&](int k, uint8_t* st, uint64_t* bar) {
        int tl, chk;
        if constexpr (CLUSTER) {
            // units 0 .. n-1: the summary fold (u, Δ, B only); n .. 2n-1: the full fold
            const int n = work.n2;
            tl = work.t2;
            chk = work.c2 + (k < n ? k : k - n);
            if (k < n)
                lane_issue_tma<Cfg, false, LTI>(st, bar, maps, false, tl / p.tiles_per_batch,
                                                (tl % p.tiles_per_batch) * Cfg::W, chk, p.dt_pitch);
            else
                lane_issue_tma<Cfg, true, LTI>(st, bar, maps, has_z, tl / p.tiles_per_batch,
                                               (tl % p.tiles_per_batch) * Cfg::W, chk, p.dt_pitch);
            return;
        }
        work.unit(k, nchunks, tl, chk);
        lane_issue_tma<Cfg, !STATE_ONLY, LTI>(st, bar, maps, has_z, tl / p.tiles_per_batch,
                            (tl % p.tiles_per_batch) * Cfg::W, chk, p.dt_pitch);
    };
    if (USE_TMA && tid == 0) {
        const int pre = total < STAGES ? total : STAGES;
        for (int k = 0; k < pre; ++k) issue(k, smem + k * Cfg::STAGE_BYTES, &full[k]);
    }

    // per-tile state of this lane (set when a piece enters a tile)
    int b = 0, d = 0;
    bool d_ok = false;
    float bias_w = 0.f, D_w = 0.f;
    float2 A2[QPL][2];                   // A'[n] = -exp(A_log[d,n])·log2(e), hoisted out of the scan
    float2 h[QPL][2];                    // this lane's slice of the state
    float dsum = 0.f;                    // STATE_ONLY: Σ Δ over this lane's steps
    float4 bL[QPL], cL[QPL];             // LTI: this lane's B and C
#pragma unroll
    for (int qq = 0; qq < QPL; ++qq) {
        A2[qq][0] = A2[qq][1] = make_float2(0.f, 0.f);
        h[qq][0] = h[qq][1] = make_float2(0.f, 0.f);
        bL[qq] = cL[qq] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // The work is a list of pieces, each chunks [c0, c0 + cnt) of one tile, in the order the
    // unit index k (the stage ring position) runs through them.  Entering a piece (tile
    // constants, initial state) and leaving it (final or handed-over state) stay outside the
    // chunk loop, which keeps that loop's body the fold alone.
    const int whole_tiles = work.n1 / nchunks;
    const int npieces = (work.n0 > 0 ? 1 : 0) + whole_tiles + (work.n2 > 0 ? 1 : 0);
    int k = 0;
    // One piece; SO: the state-only fold (pass A of the time split, or the summary fold of the
    // cluster split), known at compile time.
    auto run_piece = [&](auto so_tag, int piece) {
        constexpr bool SO = decltype(so_tag)::value;
        constexpr bool KEEP_H = CLUSTER && !SO;     // the cluster's full fold starts from the composed state
        int tile, c0, cnt;
        const int q = piece - (work.n0 > 0 ? 1 : 0);
        if (q < 0) {
            tile = work.t0; c0 = 0; cnt = work.n0;            // head, handed over at its end
        } else if (q < whole_tiles) {
            tile = work.t1 + q; c0 = 0; cnt = nchunks;        // whole tile
        } else {
            tile = work.t2; c0 = work.c2; cnt = work.n2;      // tail, or a time-split segment
        }
        b = tile / p.tiles_per_batch;
        d = (tile % p.tiles_per_batch) * Cfg::W + cw;
        d_ok = d < p.Dm;
        bias_w = (p.bias && d_ok) ? p.bias[d] : 0.f;
        D_w = (p.Dv && d_ok) ? p.Dv[d] : 0.f;
#pragma unroll
        for (int qq = 0; qq < QPL; ++qq) {
            float v[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int n = n0 + 4 * qq + q4;
                v[q4] = (d_ok && n < p.N) ? -expf(p.A_log[static_cast<int64_t>(d) * p.N + n]) * kLog2e : 0.f;
            }
            A2[qq][0] = make_float2(v[0], v[1]);
            A2[qq][1] = make_float2(v[2], v[3]);
            if constexpr (!KEEP_H) h[qq][0] = h[qq][1] = make_float2(0.f, 0.f);
            if constexpr (LTI) {
                const TIO* Bb = static_cast<const TIO*>(p.Bm) + b * p.B_b;
                const TIO* Cb = static_cast<const TIO*>(p.Cm) + b * p.C_b;
                float w[8];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int n = n0 + 4 * qq + q4;
                    w[q4] = n < p.N ? to_f32<TIO>(Bb[n]) : 0.f;
                    w[4 + q4] = n < p.N ? to_f32<TIO>(Cb[n]) : 0.f;
                }
                bL[qq] = make_float4(w[0], w[1], w[2], w[3]);
                cL[qq] = make_float4(w[4], w[5], w[6], w[7]);
            }
        }
        dsum = 0.f;
        if constexpr (Cfg::DTR > 0) {
            // the tile's W_dt rows, [W][dt_pitch] (zeros past Dm); one piece per CTA on this path
            float* sW = reinterpret_cast<float*>(aux + Cfg::AUX_W);
            const int d0 = (tile % p.tiles_per_batch) * Cfg::W;
            for (int i = tid; i < Cfg::W * p.dt_rank; i += Cfg::THREADS) {
                const int r = i / p.dt_rank, k = i % p.dt_rank;
                sW[r * p.dt_pitch + k] = d0 + r < p.Dm ? p.W_dt[static_cast<int64_t>(d0 + r) * p.dt_rank + k] : 0.f;
            }
            __syncthreads();
        }
        if constexpr (!SO && !CLUSTER) {
            const float* src = nullptr;    // the state before this unit's first chunk
            if (p.seg_launch > 0) {
                // time-split pass C: the carry the carry kernel left for this segment
                src = p.seg_slots +
                      ((static_cast<int64_t>(c0 / p.seg_chunks) * p.batch + b) * p.Dm + d) * p.N;
            } else if (c0 == 0) {
                if (p.h0) src = p.h0 + (static_cast<int64_t>(b) * p.Dm + d) * p.N;
            } else if constexpr (CBAL) {
                // the tail of a tile whose head the previous CTA of the cluster folded: its state,
                // which that CTA stored into this CTA's exchange area before arriving
                const float* xh = reinterpret_cast<const float*>(aux + Cfg::AUX_XCH);
                mbar_wait_bounded<true>(reinterpret_cast<uint64_t*>(aux + Cfg::AUX_XCH + Cfg::W * NS * 4), 0u,
                                        abort_flag, p.err);
#pragma unroll
                for (int qq = 0; qq < QPL; ++qq) {
                    const float4 v = *reinterpret_cast<const float4*>(xh + cw * NS + n0 + 4 * qq);
                    h[qq][0] = make_float2(v.x, v.y);
                    h[qq][1] = make_float2(v.z, v.w);
                }
            } else {
                // balanced: the tail of a tile whose head the previous CTA folded
                if (tid == 0) wait_published(p.ws_flag + blockIdx.x - 1, p.epoch, p.err);
                __syncthreads();
                const float* ws = p.ws_state + (static_cast<int64_t>(blockIdx.x - 1) * Cfg::W +
                                                 cw) * NS + n0;
#pragma unroll
                for (int qq = 0; qq < QPL; ++qq) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(ws + 4 * qq));
                    h[qq][0] = make_float2(v.x, v.y);
                    h[qq][1] = make_float2(v.z, v.w);
                }
            }
            if (src && d_ok) {
#pragma unroll
                for (int qq = 0; qq < QPL; ++qq) {
                    float v[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int n = n0 + 4 * qq + q4;
                        v[q4] = n < p.N ? __ldcg(src + n) : 0.f;
                    }
                    h[qq][0] = make_float2(v[0], v[1]);
                    h[qq][1] = make_float2(v[2], v[3]);
                }
            }
        }

        for (int i = 0; i < cnt; ++i, ++k) {
            const int ch = c0 + i;
            const int stage = k % STAGES;
            uint8_t* st = smem + stage * Cfg::STAGE_BYTES;
            if (USE_TMA) {
                mbar_wait_bounded(&full[stage], static_cast<uint32_t>((k / STAGES) & 1), abort_flag, p.err);
            } else {
                lane_fill_generic<Cfg>(st, p, b, (tile % p.tiles_per_batch) * Cfg::W, ch);
                __syncthreads();
            }
            const uint8_t* tu = st + Cfg::OFF_U;
            const uint8_t* td = st + Cfg::OFF_D;
            const uint8_t* tz = st + Cfg::OFF_Z;
            // this lane's element of row (g0 + g)·LPC + j (g0 a multiple of G, hence of NCX)
            auto at = [&](const uint8_t* tile, int g0, int g) -> float {
                return to_f32<TIO>(*reinterpret_cast<const TIO*>(tile + (g0 + g - g % NCX) * LPC * Cfg::RB +
                                                                 cx[g % NCX]));
            };
            const float* tB;
            const float* tC;
            if constexpr (Cfg::CONVERT_BC && !LTI) {
                // widen four bf16 at a time (a bf16 is the high half of its fp32)
                const uint2* rb = reinterpret_cast<const uint2*>(st + Cfg::OFF_B);
                const uint2* rc = reinterpret_cast<const uint2*>(st + Cfg::OFF_C);
                float4* wb = reinterpret_cast<float4*>(bcf);
                auto widen = [](uint2 v) {
                    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                };
                for (int i = tid; i < T * NS / 4; i += Cfg::THREADS) {
                    wb[i] = widen(rb[i]);
                    if constexpr (!SO) wb[T * NS / 4 + i] = widen(rc[i]);
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
            constexpr int GT = Cfg::GT;                         // step groups in the chunk
            constexpr int G = Cfg::G;                           // groups per sub-block
            static_assert(GT % G == 0, "chunk must be whole sub-blocks");
            static_assert(G % NCX == 0, "sub-blocks start on a swizzle row class");
            static_assert(G % 2 == 0, "phases 1 and 3 take the steps in pairs");
#pragma unroll (kLaneUnrollSub)
            for (int g0 = 0; g0 < GT; g0 += G) {
                // Phase 1: Δ and Δ·u of the steps this lane prepares (step g·LPC + j of each group;
                // zero past L, i.e. identity pairs).  G independent softplus chains.
                // u of this lane's steps, read once here and kept for phase 3's D·u skip
                float dd[G], du[G], uv[G];
                if constexpr (Cfg::DTR > 0) {
                    // delta_raw = Σ_k W_dt[d,k] · dt_low[t,k] for this lane's G steps, four ranks at a
                    // time: the W row from the tile's shared copy, the dt_low rows broadcast from
                    // the staged tile; packed pairs carry the even- and odd-rank partial sums
                    const float* trow = reinterpret_cast<const float*>(td) + (g0 * LPC + j) * p.dt_pitch;
                    const float4* wrow = reinterpret_cast<const float4*>(
                        reinterpret_cast<const float*>(aux + Cfg::AUX_W) + cw * p.dt_pitch);
                    float2 xr[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) xr[g] = make_float2(0.f, 0.f);
#pragma unroll 2
                    for (int k4 = 0; k4 < p.dt_rank / 4; ++k4) {
                        const float4 w4 = wrow[k4];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float4 x4 = *reinterpret_cast<const float4*>(trow + g * LPC * p.dt_pitch + 4 * k4);
                            xr[g] = fma2(make_float2(w4.x, w4.y), make_float2(x4.x, x4.y), xr[g]);
                            xr[g] = fma2(make_float2(w4.z, w4.w), make_float2(x4.z, x4.w), xr[g]);
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; g += 2) {
                        const float2 x = add2(make_float2(xr[g].x + xr[g].y, xr[g + 1].x + xr[g + 1].y),
                                              splat2(bias_w));
                        const float2 dl = softplus2(x);
                        uv[g] = at(tu, g0, g);
                        uv[g + 1] = at(tu, g0, g + 1);
                        const float2 uu = mul2(dl, make_float2(uv[g], uv[g + 1]));
                        dd[g] = dl.x; dd[g + 1] = dl.y;
                        du[g] = uu.x; du[g + 1] = uu.y;
                    }
                } else {
                    // two steps per pass: the polynomial and the products on packed pairs (bf16
                    // outputs: the SFU's log2, whose error is far below the output's rounding)
#pragma unroll
                    for (int g = 0; g < G; g += 2) {
                        const float2 x = add2(make_float2(at(td, g0, g), at(td, g0, g + 1)), splat2(bias_w));
                        const float2 dl = (Cfg::ES == 2 && SS_BF16_LG2_SOFTPLUS) ? softplus2_lg2(x) : softplus2(x);
                        uv[g] = at(tu, g0, g);
                        uv[g + 1] = at(tu, g0, g + 1);
                        const float2 uu = mul2(dl, make_float2(uv[g], uv[g + 1]));
                        dd[g] = dl.x; dd[g + 1] = dl.y;
                        du[g] = uu.x; du[g + 1] = uu.y;
                    }
                }
                if (!whole) {
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        if ((g0 + g) * LPC + j >= left) dd[g] = du[g] = 0.f;
                }
                if constexpr (SO) {
#pragma unroll
                    for (int g = 0; g < G; ++g) dsum += dd[g];
                }
                float2* dxrow = nullptr;
                (void)dxrow;                                    // used by the DXS hand-over only
                if constexpr (Cfg::DXS) {
                    // this warp's rows; the previous sub-block's reads are done once every lane is here
                    dxrow = reinterpret_cast<float2*>(aux + Cfg::AUX_DX) + (warp * CPW + c) * Cfg::DX_PITCH;
                    __syncwarp();
#pragma unroll
                    for (int g = 0; g < G; ++g) dxrow[g * LPC + j] = make_float2(dd[g], du[g]);
                    __syncwarp();
                }
                // Phase 2: the sequential fold.  Step g·LPC + k takes its Δ, Δ·u from lane (c, k);
                // the C·h partial sums of the channel's LPC lanes are reduce-scattered so that lane
                // (c, j) ends with the sum of step g·LPC + j.
                float yv[G];
                {
                    // The decays a = 2^(Δ·A') and inputs b = Δu·B of group g + 1 are formed (shuffle,
                    // B load, SFU) while group g's recurrence runs, so their latency overlaps it; the
                    // source interleaves them state pair by state pair (two decays on the SFU beside
                    // two FMA-pipe updates; about 1% faster than issuing them as one block first).
                    float2 an[LPC][QPL][2], bn[LPC][QPL][2];
                    // Δ and Δ·u of step kk of group g (dxq: the group's pairs when DXS)
                    auto step_in = [&](int g, int kk, const float4 (&dxq)[Cfg::NDX], float& dk, float& uk) {
                        if constexpr (LPC == 1) {
                            dk = dd[g];
                            uk = du[g];
                        } else if constexpr (Cfg::DXS) {
                            dk = (kk & 1) == 0 ? dxq[kk >> 1].x : dxq[kk >> 1].z;
                            uk = (kk & 1) == 0 ? dxq[kk >> 1].y : dxq[kk >> 1].w;
                        } else {
                            dk = __shfl_sync(0xffffffffu, dd[g], kk * CPW + c);
                            uk = __shfl_sync(0xffffffffu, du[g], kk * CPW + c);
                        }
                    };
                    auto prep = [&](int g, float2 (&a)[LPC][QPL][2], float2 (&bb)[LPC][QPL][2]) {
                        float4 dxq[Cfg::NDX];
#pragma unroll
                        for (int x = 0; x < Cfg::NDX; ++x)
                            dxq[x] = Cfg::DXS ? *reinterpret_cast<const float4*>(dxrow + g * LPC + 2 * x)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int kk = 0; kk < LPC; ++kk) {
                            float dk, uk;
                            step_in(g, kk, dxq, dk, uk);
                            const float2 dl2 = make_float2(dk, dk), du2 = make_float2(uk, uk);
                            const float* rowB = tB + ((g0 + g) * LPC + kk) * NS + n0;
#pragma unroll
                            for (int qq = 0; qq < QPL; ++qq) {
                                const float4 B4 = LTI ? bL[qq]
                                                      : *reinterpret_cast<const float4*>(rowB + 4 * qq);
                                a[kk][qq][0] = ex2x2(mul2(dl2, A2[qq][0]));
                                a[kk][qq][1] = ex2x2(mul2(dl2, A2[qq][1]));
                                bb[kk][qq][0] = mul2(du2, make_float2(B4.x, B4.y));
                                bb[kk][qq][1] = mul2(du2, make_float2(B4.z, B4.w));
                            }
                        }
                    };
                    // The channel's LPC partial sums of one step group, reduce-scattered so that lane
                    // (c, j) ends with step j's sum.  LPC = 2: one exchange.  LPC = 4: a butterfly over
                    // the four slices (lanes c + CPW·s), first across slice bit 1 (each side keeps two
                    // steps), then across bit 0.  Only shuffles, no shared-memory round trip or warp
                    // barrier.  (The fold must visit the steps in time order, so the slots cannot be
                    // renumbered per lane to spare the selects.)
                    auto reduce_scatter = [&](const float (&v)[LPC]) -> float {
                        if constexpr (LPC == 2) {
                            const bool hi = j & 1;
                            const float send = hi ? v[0] : v[1];
                            const float keep = hi ? v[1] : v[0];
                            return keep + __shfl_xor_sync(0xffffffffu, send, CPW);
                        } else if constexpr (LPC == 4) {
                            const bool b1 = (j & 2) != 0, b0 = (j & 1) != 0;
                            const float s0 = b1 ? v[0] : v[2], s1 = b1 ? v[1] : v[3];
                            const float k0 = b1 ? v[2] : v[0], k1 = b1 ? v[3] : v[1];
                            const float t0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 2 * CPW);
                            const float t1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 2 * CPW);
                            const float sd = b0 ? t0 : t1, kp = b0 ? t1 : t0;
                            return kp + __shfl_xor_sync(0xffffffffu, sd, CPW);
                        } else {
                            return v[0];
                        }
                    };
                    float ypp[LPC];                 // the previous group's partial sums (deferred reduce)
#pragma unroll
                    for (int kk = 0; kk < LPC; ++kk) ypp[kk] = 0.f;
                    prep(0, an, bn);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if constexpr (CKPT) {
                            // the state entering step t of every 16: the backward's checkpoint
                            if ((g * LPC) % 16 == 0) {
                                const int64_t t = tbase + (g0 + g) * LPC;
                                if (d_ok && t < static_cast<int64_t>(p.ckpt_chunks) * 32) {
                                    float* dst = p.ckpt + (((static_cast<int64_t>(tile) * p.ckpt_chunks + t / 32) * 2 +
                                                            (t / 16) % 2) * 32 + cw) * 16 + n0;
#pragma unroll
                                    for (int qq = 0; qq < QPL; ++qq)
                                        __stcg(reinterpret_cast<float4*>(dst + 4 * qq),
                                               make_float4(h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y));
                                }
                            }
                        }
                        float2 ac[LPC][QPL][2], bc[LPC][QPL][2];
#pragma unroll
                        for (int kk = 0; kk < LPC; ++kk)
#pragma unroll
                            for (int qq = 0; qq < QPL; ++qq) {
                                ac[kk][qq][0] = an[kk][qq][0]; ac[kk][qq][1] = an[kk][qq][1];
                                bc[kk][qq][0] = bn[kk][qq][0]; bc[kk][qq][1] = bn[kk][qq][1];
                            }
                        float yp[LPC];
                        if constexpr (LPC == 1) {
                            // one step per group: the next group's inputs as one block first
                            // (interleaving them costs this register-heavy layout spills)
                            if (g + 1 < G) prep(g + 1, an, bn);
                            const float* rowC = tC + (g0 + g) * NS + n0;
                            (void)rowC;                         // unread when C is in registers or unused
                            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                            for (int qq = 0; qq < QPL; ++qq) {
                                float4 C4 = make_float4(0.f, 0.f, 0.f, 0.f);
                                if constexpr (LTI)
                                    C4 = cL[qq];
                                else if constexpr (!SO)
                                    C4 = *reinterpret_cast<const float4*>(rowC + 4 * qq);
                                h[qq][0] = fma2(ac[0][qq][0], h[qq][0], bc[0][qq][0]);
                                h[qq][1] = fma2(ac[0][qq][1], h[qq][1], bc[0][qq][1]);
                                if constexpr (!SO) {
                                    acc = fma2(make_float2(C4.x, C4.y), h[qq][0], acc);
                                    acc = fma2(make_float2(C4.z, C4.w), h[qq][1], acc);
                                }
                            }
                            yp[0] = acc.x + acc.y;
                        } else {
                        const bool more = g + 1 < G;
                        const int gn = more ? g + 1 : g;
                        float4 dxq[Cfg::NDX];
#pragma unroll
                        for (int x = 0; x < Cfg::NDX; ++x)
                            dxq[x] = Cfg::DXS ? *reinterpret_cast<const float4*>(dxrow + gn * LPC + 2 * x)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int kk = 0; kk < LPC; ++kk) {
                            float dk = 0.f, uk = 0.f;
                            if (more) step_in(gn, kk, dxq, dk, uk);
                            const float2 dl2 = make_float2(dk, dk), du2 = make_float2(uk, uk);
                            const float* rowB = tB + ((g0 + gn) * LPC + kk) * NS + n0;
                            const float* rowC = tC + ((g0 + g) * LPC + kk) * NS + n0;
                            (void)rowC;
                            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                            for (int qq = 0; qq < QPL; ++qq) {
                                float4 C4 = make_float4(0.f, 0.f, 0.f, 0.f);
                                if constexpr (LTI)
                                    C4 = cL[qq];
                                else if constexpr (!SO)
                                    C4 = *reinterpret_cast<const float4*>(rowC + 4 * qq);
                                float4 B4 = make_float4(0.f, 0.f, 0.f, 0.f);
                                if (more) B4 = LTI ? bL[qq] : *reinterpret_cast<const float4*>(rowB + 4 * qq);
                                if (more) an[kk][qq][0] = ex2x2(mul2(dl2, A2[qq][0]));
                                h[qq][0] = fma2(ac[kk][qq][0], h[qq][0], bc[kk][qq][0]);
                                if constexpr (!SO) acc = fma2(make_float2(C4.x, C4.y), h[qq][0], acc);
                                if (more) an[kk][qq][1] = ex2x2(mul2(dl2, A2[qq][1]));
                                h[qq][1] = fma2(ac[kk][qq][1], h[qq][1], bc[kk][qq][1]);
                                if constexpr (!SO) acc = fma2(make_float2(C4.z, C4.w), h[qq][1], acc);
                                if (more) {
                                    bn[kk][qq][0] = mul2(du2, make_float2(B4.x, B4.y));
                                    bn[kk][qq][1] = mul2(du2, make_float2(B4.z, B4.w));
                                }
                            }
                            yp[kk] = acc.x + acc.y;
                        }
                        }
                        if constexpr (SO) {
                            (void)yp;
                        } else if constexpr (LPC == 1) {
                            yv[g] = yp[0];
                        } else if constexpr (kLaneDeferReduce) {
                            // reduce the previous group's partial sums now, after this group's
                            // arithmetic, so that the shuffles' latency overlaps it
                            if (g > 0) yv[g - 1] = reduce_scatter(ypp);
#pragma unroll
                            for (int kk = 0; kk < LPC; ++kk) ypp[kk] = yp[kk];
                            if (g + 1 == G) yv[g] = reduce_scatter(ypp);
                        } else {
                            yv[g] = reduce_scatter(yp);
                        }
                    }
                }
                // Phase 3: D skip, z gate, store (G independent chains).
                if (!SO && d_ok) {
                    char* yrow = reinterpret_cast<char*>(static_cast<TIO*>(p.y) + b * p.y_b + (tbase + g0 * LPC + j) * p.y_l + d);
                    const int64_t rem = left - g0 * LPC - j;          // steps of this lane's column before L
                    const int nst = whole ? G : (rem <= 0 ? 0 : rem >= int64_t(G) * LPC ? G : static_cast<int>((rem + LPC - 1) / LPC));
                    if (has_z && nst == G) {
#pragma unroll
                        for (int g = 0; g < G; g += 2) {
                            const float2 v = mul2(fma2(splat2(D_w), make_float2(uv[g], uv[g + 1]),
                                                       make_float2(yv[g], yv[g + 1])),
                                                  silu2(make_float2(at(tz, g0, g), at(tz, g0, g + 1))));
                            *reinterpret_cast<TIO*>(yrow + g * LPC * ystride) = from_f32<TIO>(v.x);
                            *reinterpret_cast<TIO*>(yrow + (g + 1) * LPC * ystride) = from_f32<TIO>(v.y);
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            if (g < nst) {
                                float v = fmaf(D_w, uv[g], yv[g]);
                                if (has_z) v *= silu(at(tz, g0, g));
                                *reinterpret_cast<TIO*>(yrow + g * LPC * ystride) = from_f32<TIO>(v);
                            }
                        }
                    }
                }
            }
            if (USE_TMA && !(Cfg::CONVERT_BC && !LTI)) {
                // Release the stage without a block-wide barrier: the warp that finishes it last
                // refills it, so warps that are ahead run on into the stages already loaded.
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    if (atomicAdd(&done[stage], 1) == Cfg::WARPS - 1) {
                        done[stage] = 0;
                        if (k + STAGES < total && !*abort_flag) issue(k + STAGES, st, &full[stage]);
                    }
                }
            } else {
                __syncthreads();   // stage (and the widened B/C) consumed by every warp
                if (USE_TMA && tid == 0 && k + STAGES < total && !*abort_flag) issue(k + STAGES, st, &full[stage]);
            }
        }

        // End of the piece: the sequence's final state, or (head of a tile another CTA
        // finishes) the state to hand over; for pass A, the segment's end state and Σ Δ.
        if constexpr (SO && CLUSTER) {
            // the summary stays on chip: the end state in h, the channel's Σ Δ (over its lanes) in dsum
            if constexpr (LPC >= 2) dsum += __shfl_xor_sync(0xffffffffu, dsum, CPW);
            if constexpr (LPC >= 4) dsum += __shfl_xor_sync(0xffffffffu, dsum, 2 * CPW);
        } else if constexpr (SO) {
            const int sg = c0 / p.seg_chunks;
            if (d_ok) {
                float* dst = p.seg_slots + ((static_cast<int64_t>(sg + p.seg_out0) * p.batch + b) * p.Dm + d) * p.N;
#pragma unroll
                for (int qq = 0; qq < QPL; ++qq) {
                    const float v[4] = {h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y};
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        if (n0 + 4 * qq + q4 < p.N) dst[n0 + 4 * qq + q4] = v[q4];
                }
            }
            float x = dsum;                 // Σ over the channel's LPC lanes
            if constexpr (LPC >= 2) x += __shfl_xor_sync(0xffffffffu, x, CPW);
            if constexpr (LPC >= 4) x += __shfl_xor_sync(0xffffffffu, x, 2 * CPW);
            if (j == 0 && d_ok) p.seg_dsum[(static_cast<int64_t>(sg) * p.batch + b) * p.Dm + d] = x;
        } else if (c0 + cnt == nchunks) {
            if (p.last_state && d_ok) {
                float* out = p.last_state + (static_cast<int64_t>(b) * p.Dm + d) * p.N;
#pragma unroll
                for (int qq = 0; qq < QPL; ++qq) {
                    const float v[4] = {h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y};
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        if (n0 + 4 * qq + q4 < p.N) out[n0 + 4 * qq + q4] = v[q4];
                }
            }
        } else if (CBAL && work.n0 > 0 && piece == 0) {
            // the head of a tile the next CTA of the cluster finishes: the state into that CTA's
            // exchange area, then one arrival per thread on its hand-over barrier
            const float* xh = reinterpret_cast<const float*>(aux + Cfg::AUX_XCH);
            const uint32_t next = cluster_ctarank() + 1;
#pragma unroll
            for (int qq = 0; qq < QPL; ++qq)
                st_peer_f32x4(peer_smem_addr(xh + cw * NS + n0 + 4 * qq, next),
                              make_float4(h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y));
            mbar_arrive_peer(peer_smem_addr(aux + Cfg::AUX_XCH + Cfg::W * NS * 4, next));
        } else if (work.n0 > 0 && piece == 0) {
            float* dst = p.ws_state + (static_cast<int64_t>(blockIdx.x) * Cfg::W + cw) * NS + n0;
#pragma unroll
            for (int qq = 0; qq < QPL; ++qq)
                __stcg(reinterpret_cast<float4*>(dst + 4 * qq),
                       make_float4(h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y));
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.ws_flag + blockIdx.x), "r"(p.epoch)
                             : "memory");
            }
        }
    };

    if constexpr (CLUSTER) {
        // this CTA's segment: the summary fold, the exchange, the full fold (one piece; an empty
        // segment folds nothing and passes the state through)
        if (npieces > 0) run_piece(std::true_type{}, 0);
        float* xh = reinterpret_cast<float*>(aux + Cfg::AUX_XCH);   // [W][NS] end state from zero
        float* xd = xh + Cfg::W * NS;                                // [W] Σ Δ
#pragma unroll
        for (int qq = 0; qq < QPL; ++qq)
            *reinterpret_cast<float4*>(xh + cw * NS + n0 + 4 * qq) =
                make_float4(h[qq][0].x, h[qq][0].y, h[qq][1].x, h[qq][1].y);
        if (j == 0) xd[cw] = dsum;
        cluster_sync_all();                 // every summary of the cluster written
        const uint32_t rank = cluster_ctarank();
        float2 H[QPL][2];
#pragma unroll
        for (int qq = 0; qq < QPL; ++qq) H[qq][0] = H[qq][1] = make_float2(0.f, 0.f);
        if (p.h0 && d_ok) {
            const float* src = p.h0 + (static_cast<int64_t>(b) * p.Dm + d) * p.N;
#pragma unroll
            for (int qq = 0; qq < QPL; ++qq) {
                float v[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) v[q4] = n0 + 4 * qq + q4 < p.N ? __ldcg(src + n0 + 4 * qq + q4) : 0.f;
                H[qq][0] = make_float2(v[0], v[1]);
                H[qq][1] = make_float2(v[2], v[3]);
            }
        }
        for (uint32_t r = 0; r < rank; ++r) {
            const float ds = ld_peer_f32(peer_smem_addr(xd + cw, r));
            const float2 ds2 = make_float2(ds, ds);
#pragma unroll
            for (int qq = 0; qq < QPL; ++qq) {
                const float4 e = ld_peer_f32x4(peer_smem_addr(xh + cw * NS + n0 + 4 * qq, r));
                H[qq][0] = fma2(ex2x2(mul2(ds2, A2[qq][0])), H[qq][0], make_float2(e.x, e.y));
                H[qq][1] = fma2(ex2x2(mul2(ds2, A2[qq][1])), H[qq][1], make_float2(e.z, e.w));
            }
        }
        cluster_sync_all();                 // no CTA leaves while a peer may still read its summary
#pragma unroll
        for (int qq = 0; qq < QPL; ++qq) {
            h[qq][0] = H[qq][0];
            h[qq][1] = H[qq][1];
        }
        if (npieces > 0) run_piece(std::false_type{}, 0);
    } else if constexpr (CBAL) {
        // head (handed over at its end), whole tiles, tail (taken over at its start)
        cluster_sync_all();                 // every CTA's hand-over barrier is initialised
        for (int piece = 0; piece < npieces; ++piece) run_piece(std::false_type{}, piece);
        cluster_sync_all();                 // no CTA leaves while its neighbour may still write to it
    } else {
        for (int piece = 0; piece < npieces; ++piece) run_piece(std::integral_constant<bool, STATE_ONLY>{}, piece);
    }
}

}  // namespace selscan
