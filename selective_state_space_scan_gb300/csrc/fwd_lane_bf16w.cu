// bf16-I/O state-split lane forward kernels that stage B and C as fp32 tiles: the workspace
// schedules (balanced, time split) widen bf16 B and C once into the workspace before the scan, so
// the kernel needs no per-chunk widening in shared memory and no block barrier for it.  16 states.
#include "fwd_lane_impl.cuh"

namespace selscan {

template <int LPC>
static cudaError_t launch_bf16w_lpc(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t s,
                                    int* mg) {
    using T = __nv_bfloat16;
    if (v.ckpt) {       // the balanced schedule that also writes the backward's checkpoints
        if constexpr (LPC == 2) {
            if (!v.balanced || v.state_only) return cudaErrorInvalidValue;
            return launch_lane_cfg<T, 16, LPC, true, true, false, false, true, false, true>(p, m, s, mg);
        } else {
            return cudaErrorInvalidValue;
        }
    }
    if (v.state_only) return launch_lane_cfg<T, 16, LPC, false, true, true, false, true>(p, m, s, mg);
    if (v.balanced) return launch_lane_cfg<T, 16, LPC, true, true, false, false, true>(p, m, s, mg);
    return launch_lane_cfg<T, 16, LPC, false, true, false, false, true>(p, m, s, mg);
}

cudaError_t launch_fwd_lane_bf16w(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t stream,
                                  int* max_grid) {
    if (v.ns != 16 || !v.tma || v.lti || v.dtp || v.family != kFamLane) return cudaErrorInvalidValue;
    if (v.lpc == 1) return launch_bf16w_lpc<1>(v, p, m, stream, max_grid);
    if (v.lpc == 2) return launch_bf16w_lpc<2>(v, p, m, stream, max_grid);
    if (v.lpc == 4) return launch_bf16w_lpc<4>(v, p, m, stream, max_grid);
    return cudaErrorInvalidValue;
}

}  // namespace selscan
