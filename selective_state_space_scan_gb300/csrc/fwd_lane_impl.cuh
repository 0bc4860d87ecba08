// Instantiation of the state-split lane forward kernels for one I/O type.
#pragma once

#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {

template <typename TIO, int NS, int LPC, bool TMA>
cudaError_t launch_lane_cfg(const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    using Cfg = LaneCfg<TIO, NS, LPC, kLaneT, kLaneStages, lane_minb(LPC)>;
    constexpr int smem = TMA ? Cfg::SMEM_BYTES : Cfg::SMEM_BYTES - (Cfg::STAGES - 1) * Cfg::STAGE_BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget exceeded");
    return launch_with_smem<Cfg, TMA>(ss_fwd_lane_kernel<Cfg, TMA>, p, m, stream, smem);
}

template <typename TIO, int NS, int LPC>
cudaError_t launch_lane_tma(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
    return v.tma ? launch_lane_cfg<TIO, NS, LPC, true>(p, m, s) : launch_lane_cfg<TIO, NS, LPC, false>(p, m, s);
}

template <typename TIO>
cudaError_t launch_lane_dtype(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t s) {
    if (v.ns == 16) {
        if (v.lpc == 1) return launch_lane_tma<TIO, 16, 1>(v, p, m, s);
        if (v.lpc == 2) return launch_lane_tma<TIO, 16, 2>(v, p, m, s);
        if (v.lpc == 4) return launch_lane_tma<TIO, 16, 4>(v, p, m, s);
    } else if (v.ns == 8) {
        if (v.lpc == 1) return launch_lane_tma<TIO, 8, 1>(v, p, m, s);
        if (v.lpc == 2) return launch_lane_tma<TIO, 8, 2>(v, p, m, s);
    } else if (v.ns == 4) {
        if (v.lpc == 1) return launch_lane_tma<TIO, 4, 1>(v, p, m, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace selscan
