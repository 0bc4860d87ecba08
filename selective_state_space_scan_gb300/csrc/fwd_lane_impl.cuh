// Instantiation of the state-split lane forward kernels for one I/O type.
#pragma once

#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {

// WIDE: the balanced schedule on the per-tile kernel's 32-channel tiles (the same instantiation).
// CKPT: the per-tile kernel that also writes the backward's checkpoints.
// DX4: (Δ, Δ·u) handed over through shared memory at 4 lanes per channel (fp32, two CTAs per SM).
template <typename TIO, int NS, int LPC, bool BAL, bool TMA, bool SO = false, bool LTI = false, bool BCF = false,
          bool WIDE = false, bool CKPT = false, bool DX4 = false>
cudaError_t launch_lane_cfg(const FwdParams& p, const FwdMaps& m, cudaStream_t stream, int* max_grid) {
    constexpr int W = WIDE ? 32 : lane_w(LPC, BAL, static_cast<int>(sizeof(TIO)));
    using Cfg = LaneCfg<TIO, NS, LPC, W, kLaneT, kLaneStages, BCF ? lane_minb_bcf32(LPC, W) : lane_minb(LPC, W), 0, BCF,
                        false, DX4>;
    constexpr int smem = TMA ? Cfg::SMEM_BYTES : Cfg::SMEM_BYTES - (Cfg::STAGES - 1) * Cfg::STAGE_BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget exceeded");
    return launch_with_smem<Cfg, TMA>(ss_fwd_lane_kernel<Cfg, TMA, SO, LTI, false, CKPT>, p, m, stream, smem, BAL,
                                      max_grid);
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_lane_v(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t s, int* mg) {
    if (v.ckpt) {
        // TMA-fed, 16 states at 4 lanes per channel on 32-channel tiles: per tile, or balanced
        if constexpr (NS == 16 && LPC == 4) {
            if (!v.tma || v.state_only || v.lti) return cudaErrorInvalidValue;
            if (v.balanced) {
                if (!v.w32) return cudaErrorInvalidValue;
                return launch_lane_cfg<TIO, NS, LPC, true, true, false, false, false, true, true>(p, m, s, mg);
            }
            return launch_lane_cfg<TIO, NS, LPC, false, true, false, false, false, false, true>(p, m, s, mg);
        } else {
            return cudaErrorInvalidValue;
        }
    }
    if (v.lti) {
        if (!v.tma || v.balanced || v.state_only) return cudaErrorInvalidValue;   // per-tile, TMA-fed only
        return launch_lane_cfg<TIO, NS, LPC, false, true, false, true>(p, m, s, mg);
    }
    if (v.state_only) {
        if (!v.tma || v.balanced) return cudaErrorInvalidValue;   // pass A is TMA-fed only
        return launch_lane_cfg<TIO, NS, LPC, false, true, true>(p, m, s, mg);
    }
    if (v.balanced) {
        if (!v.tma) return cudaErrorInvalidValue;   // the balanced schedule is TMA-fed only
        if (v.w32) {
            if constexpr (LPC == 4 && sizeof(TIO) == 4) {
                if (v.dx4) return launch_lane_cfg<TIO, NS, LPC, true, true, false, false, false, true, false, true>(p, m, s, mg);
            }
            if (v.dx4) return cudaErrorInvalidValue;
            return launch_lane_cfg<TIO, NS, LPC, true, true, false, false, false, true>(p, m, s, mg);
        }
        return launch_lane_cfg<TIO, NS, LPC, true, true>(p, m, s, mg);
    }
    return v.tma ? launch_lane_cfg<TIO, NS, LPC, false, true>(p, m, s, mg)
                 : launch_lane_cfg<TIO, NS, LPC, false, false>(p, m, s, mg);
}

template <typename TIO>
cudaError_t launch_lane_dtype(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t s, int* mg) {
    if (v.ns == 16) {
        if (v.lpc == 1) return launch_lane_v<TIO, 16, 1>(v, p, m, s, mg);
        if (v.lpc == 2) return launch_lane_v<TIO, 16, 2>(v, p, m, s, mg);
        if (v.lpc == 4) return launch_lane_v<TIO, 16, 4>(v, p, m, s, mg);
    } else if (v.ns == 8) {
        if (v.lpc == 1) return launch_lane_v<TIO, 8, 1>(v, p, m, s, mg);
        if (v.lpc == 2) return launch_lane_v<TIO, 8, 2>(v, p, m, s, mg);
    } else if (v.ns == 4) {
        if (v.lpc == 1) return launch_lane_v<TIO, 4, 1>(v, p, m, s, mg);
    }
    return cudaErrorInvalidValue;
}

}  // namespace selscan
