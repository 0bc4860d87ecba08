// Segment-lane forward kernels (8-channel tiles, time segments inside each warp), both I/O types.
#include "fwd_launch_common.cuh"
#include "ss_fwd_seg.cuh"

namespace selscan {

template <typename TIO, int NS, bool TMA>
static cudaError_t launch_seg_cfg(const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    using Cfg = FwdCfg<TIO, NS, kSegG, kSegQ, kSegK, kSegStages>;
    constexpr int smem = TMA ? Cfg::SMEM_BYTES : Cfg::SMEM_BYTES - (Cfg::STAGES - 1) * Cfg::STAGE_BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget exceeded");
    return launch_with_smem<Cfg, TMA>(ss_fwd_seg_kernel<Cfg, TMA>, p, m, stream, smem);
}

template <typename TIO>
static cudaError_t launch_seg_dtype(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                    cudaStream_t s) {
    switch (v.ns) {
        case 4: return v.tma ? launch_seg_cfg<TIO, 4, true>(p, m, s) : launch_seg_cfg<TIO, 4, false>(p, m, s);
        case 8: return v.tma ? launch_seg_cfg<TIO, 8, true>(p, m, s) : launch_seg_cfg<TIO, 8, false>(p, m, s);
        case 16: return v.tma ? launch_seg_cfg<TIO, 16, true>(p, m, s) : launch_seg_cfg<TIO, 16, false>(p, m, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_seg(const FwdVariant& v, bool bf16, const FwdParams& p, const FwdMaps& m,
                           cudaStream_t stream) {
    return bf16 ? launch_seg_dtype<__nv_bfloat16>(v, p, m, stream) : launch_seg_dtype<float>(v, p, m, stream);
}

}  // namespace selscan
