// Test instantiations of the state-split lane forward kernel at other chunk lengths: 16, 32 and
// 256 steps per chunk (the library's kernels use 64).  The carry across chunks must make the
// result independent of where the chunks fall ("mamba-metal: Apple Silicon で Mamba を動かす",
// section "チャンク間 running prefix"); these let a test check that on the GPU.  One
// configuration only: fp32 I/O, 16 states at 4 lanes per channel, one CTA per 32-channel tile,
// TMA-fed.  The 256-step chunk holds a whole sequence of up to 256 steps in one chunk, so no
// carry is crossed at all; its stage is 128 KB, so it runs with a single stage.
#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {
namespace {

template <int T, int STAGES>
cudaError_t launch_chunked(const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    using Cfg = LaneCfg<float, 16, 4, 32, T, STAGES, lane_minb(4, 32)>;
    static_assert(Cfg::SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    return launch_with_smem<Cfg, true>(ss_fwd_lane_kernel<Cfg, true, false, false>, p, m, stream, Cfg::SMEM_BYTES);
}

}  // namespace

bool chunk_override_ok(const FwdVariant& v) {
    return v.family == kFamLane && v.ns == 16 && v.lpc == 4 && v.tma && v.es == 4 && !v.balanced &&
           !v.state_only && !v.lti && !v.dtp && (v.chunk == 16 || v.chunk == 32 || v.chunk == 256);
}

cudaError_t launch_fwd_lane_chunked(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    if (!chunk_override_ok(v)) return cudaErrorInvalidValue;
    if (v.chunk == 16) return launch_chunked<16, 2>(p, m, stream);
    if (v.chunk == 32) return launch_chunked<32, 2>(p, m, stream);
    return launch_chunked<256, 1>(p, m, stream);
}

}  // namespace selscan
