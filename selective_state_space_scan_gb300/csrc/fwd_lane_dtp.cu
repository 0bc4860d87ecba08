// The state-split lane forward kernel with the low-rank time-step projection folded in
// (fp32 I/O, one CTA per tile, TMA-fed, 48-step chunks).
#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {
namespace {

template <int NS, int LPC>
cudaError_t launch_dtp(const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    using Cfg = LaneCfg<float, NS, LPC, 32, kLaneTD, kLaneStages, lane_minb(LPC, 32), kDtPitchMax>;
    static_assert(Cfg::SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    return launch_with_smem<Cfg, true>(ss_fwd_lane_kernel<Cfg, true, false, false>, p, m, stream, Cfg::SMEM_BYTES);
}

}  // namespace

cudaError_t launch_fwd_lane_dtp(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    if (!v.tma || v.balanced || v.state_only || v.lti || v.family != kFamLane) return cudaErrorInvalidValue;
    if (v.ns == 16) {
        if (v.lpc == 1) return launch_dtp<16, 1>(p, m, stream);
        if (v.lpc == 2) return launch_dtp<16, 2>(p, m, stream);
        if (v.lpc == 4) return launch_dtp<16, 4>(p, m, stream);
    } else if (v.ns == 8) {
        if (v.lpc == 1) return launch_dtp<8, 1>(p, m, stream);
        if (v.lpc == 2) return launch_dtp<8, 2>(p, m, stream);
    } else if (v.ns == 4) {
        if (v.lpc == 1) return launch_dtp<4, 1>(p, m, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace selscan
