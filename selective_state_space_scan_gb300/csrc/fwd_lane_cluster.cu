// The single-launch time split of the lane kernel (one CTA per (channel tile, time segment),
// the segments of a tile forming one thread-block cluster that exchanges segment summaries
// through distributed shared memory): fp32 and bf16 I/O, 16 states at 4 lanes per channel,
// 32-channel tiles, TMA-fed; with or without the backward's checkpoints.
#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {
namespace {

template <typename TIO, bool CKPT>
cudaError_t launch_cluster_t(const FwdParams& p, const FwdMaps& m, cudaStream_t stream, int cluster,
                             int* fit) {
    using Cfg = LaneCfg<TIO, 16, 4, 32, kLaneT, kLaneStages, lane_minb(4, 32), 0, false, true>;
    static_assert(Cfg::SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    auto kern = ss_fwd_lane_kernel<Cfg, true, false, false, true, CKPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid > 0 ? p.grid : cluster));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (fit) {
        // fit[0]: clusters of this size resident at once (0: the size cannot run); fit[1]: CTAs per SM
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::THREADS, Cfg::SMEM_BYTES)) !=
            cudaSuccess)
            return e;
        fit[1] = per_sm;
        return cudaOccupancyMaxActiveClusters(&fit[0], kern, &cfg);
    }
    e = cudaLaunchKernelEx(&cfg, kern, p, m);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_lane_cluster(bool bf16, const FwdParams& p, const FwdMaps& m, cudaStream_t stream, int cluster,
                                    int* fit) {
    if (cluster < 2 || cluster > 8) return cudaErrorInvalidValue;
    // with FwdParams::ckpt: the instantiation that also writes the backward's checkpoints
    if (p.ckpt)
        return bf16 ? launch_cluster_t<__nv_bfloat16, true>(p, m, stream, cluster, fit)
                    : launch_cluster_t<float, true>(p, m, stream, cluster, fit);
    return bf16 ? launch_cluster_t<__nv_bfloat16, false>(p, m, stream, cluster, fit)
                : launch_cluster_t<float, false>(p, m, stream, cluster, fit);
}

}  // namespace selscan
