// Tile geometry of the forward-scan kernel instantiations, shared by the host dispatcher
// (grid sizing, TMA boxes) and the kernel translation units.
#pragma once

namespace selscan {

// State-split lane family: 32 channels per CTA; a channel's states are split over LPC lanes
// (1, 2 or 4), so a CTA is LPC warps of 32/LPC channels each; T steps per chunk.
#ifndef SS_LANE_T
#define SS_LANE_T 64
#endif
#ifndef SS_LANE_STAGES
#define SS_LANE_STAGES 2
#endif
constexpr int kLaneT = SS_LANE_T;
// Sub-blocks of a chunk unrolled together (1: a loop over the sub-blocks; 2 measured 842 against
// 677 us on the 2.8b-shaped layer).
#ifndef SS_UNROLL_SUB
#define SS_UNROLL_SUB 1
#endif
constexpr int kLaneUnrollSub = SS_UNROLL_SUB;
// The reduce-scatter of a step group's C·h partial sums issued after the next group's
// arithmetic (1) or right after its own (0).
#ifndef SS_DEFER_REDUCE
#define SS_DEFER_REDUCE 1
#endif
constexpr bool kLaneDeferReduce = SS_DEFER_REDUCE != 0;

// Lane kernel options (compile-time, for measurement): the (Δ, Δ·u) hand-over at 2 lanes per
// channel through shared memory instead of shuffles (fp32); softplus through the SFU's log2 for
// bf16 (742 -> 723 us on the 2.8b-shaped layer).
#ifndef SS_DX_SMEM
#define SS_DX_SMEM 1
#endif
#ifndef SS_BF16_LG2_SOFTPLUS
#define SS_BF16_LG2_SOFTPLUS 1
#endif
constexpr int kLaneStages = SS_LANE_STAGES;
#ifndef SS_LANE_MINB4
#define SS_LANE_MINB4 3
#endif
// Resident CTAs per SM the register budget is sized for: about 12 warps per SM with 2 or 4 lanes
// per channel, 8 with one (a CTA of a w-channel tile is w·lpc/32 warps).
constexpr int lane_minb(int lpc, int w) {
    return (lpc == 4 ? 4 * SS_LANE_MINB4 : lpc == 2 ? 12 : 8) / (w * lpc / 32 > 0 ? w * lpc / 32 : 1);
}
// bf16 streams with fp32 B/C tiles (the workspace schedules): shared memory holds five CTAs of a
// 32-channel tile per SM, and a 2-lane CTA sized for four per SM gets 176 registers per thread,
// which still lets five reside (126 before: 674 -> 667 us on the 2.8b-shaped layer).
constexpr int lane_minb_bcf32(int lpc, int w) { return lpc == 2 && w == 32 ? 4 : lane_minb(lpc, w); }
// Tile width: 32 channels for one CTA per tile.  The balanced schedule needs at least as many
// tiles as SMs times resident CTAs, so its fp32 tiles are 16 channels (64-byte rows) unless the
// 32-channel tiles alone give two CTAs per SM (FwdVariant::w32: the per-tile kernel itself, run
// balanced; 133 against 148 us on the 130m-shaped layer); its bf16 tiles stay at 32 (64-byte rows
// too: narrower rows would have each 64-byte DRAM access read by two CTAs at different times,
// which measured 1.8x the stream bytes in DRAM traffic).  A lane family tile is whole warps of
// 32/lpc channels.
constexpr int lane_w(int lpc, bool balanced, int es) { return balanced && lpc > 1 && es == 4 ? 16 : 32; }
// With the low-rank time-step projection folded in: 48-step chunks (the staged dt_low tile
// replaces the Δ tile and is wider), ranks up to 64, rows padded to an odd number of 16-byte
// chunks (at most 68 floats).
constexpr int kLaneTD = 48;
constexpr int kDtRankMax = 64;
constexpr int kDtPitchMax = 68;
constexpr int dt_pitch(int rank) { return (rank / 4) % 2 == 1 ? rank : rank + 4; }

// Segment-lane family (time-parallel; few channels, long sequences): 8 channels per CTA,
// each warp holds 4 time segments of those 8 channels, 4 warps of K = 14 steps per thread
// (224-step chunks).  Shared memory holds two CTAs per SM whatever the warp count, so each
// thread may use up to 255 registers: 14 steps per scan measured 791 us on long-32k against
// 837 us for 8 warps of 7.  The B/C quad reads of the 4 segments stay on different banks.
constexpr int kSegG = 1, kSegQ = 4, kSegK = 14, kSegStages = 2;

}  // namespace selscan
