// The cluster-balanced schedule of the lane kernel (ss_fwd without a workspace when one CTA per
// tile would need more than one wave): clusters of S CTAs, each cluster taking a contiguous run of
// whole channel tiles and splitting its (tile, chunk) units into S equal ranges; a tile split
// between two CTAs of a cluster hands its state over through distributed shared memory.  16
// states on 32-channel tiles, TMA-fed: bf16 at 2 lanes per channel, fp32 at 4 (the lanes the
// balanced schedule takes for each).
#include "fwd_launch_common.cuh"
#include "ss_fwd_lane.cuh"

namespace selscan {
namespace {

template <typename TIO, int LPC>
cudaError_t launch_cbal_t(const FwdParams& p, const FwdMaps& m, cudaStream_t stream, int cluster, int per_sm,
                          int* fit) {
    using Cfg = LaneCfg<TIO, 16, LPC, 32, kLaneT, kLaneStages, lane_minb(LPC, 32), 0, false, true>;
    static_assert(Cfg::SMEM_BYTES <= 227 * 1024, "shared memory budget exceeded");
    auto kern = ss_fwd_lane_kernel<Cfg, true, false, false, false, false, true>;
    // per_sm > 0: pad the shared memory so that one CTA more than per_sm does not fit an SM.  The
    // cluster scheduler may otherwise put more of a cluster's CTAs on one SM than the even share
    // the plan assumes (130m-shaped layer: 2 CTAs per SM planned, 3 fit, 184 us against 142 us for
    // one CTA per tile).
    int smem = Cfg::SMEM_BYTES;
    if (per_sm > 0) {
        int dev = 0, sm_smem = 0, reserved = 0;
        cudaError_t e0 = cudaGetDevice(&dev);
        if (e0 == cudaSuccess)
            e0 = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e0 != cudaSuccess) return e0;
        const int pad = sm_smem / (per_sm + 1) - reserved + 128;
        if (pad > smem) smem = pad < 227 * 1024 ? pad : 227 * 1024;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid > 0 ? p.grid : cluster));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (fit) {
        // fit[0]: clusters of this size resident at once (0: the size cannot run); fit[1]: CTAs per SM
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit[1], kern, Cfg::THREADS, smem)) !=
            cudaSuccess)
            return e;
        return cudaOccupancyMaxActiveClusters(&fit[0], kern, &cfg);
    }
    e = cudaLaunchKernelEx(&cfg, kern, p, m);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_lane_cbal(bool bf16, int lpc, const FwdParams& p, const FwdMaps& m, cudaStream_t stream,
                                 int cluster, int per_sm, int* fit) {
    if (cluster < 2 || cluster > 8) return cudaErrorInvalidValue;
    if (bf16 && lpc == 2) return launch_cbal_t<__nv_bfloat16, 2>(p, m, stream, cluster, per_sm, fit);
    if (!bf16 && lpc == 4) return launch_cbal_t<float, 4>(p, m, stream, cluster, per_sm, fit);
    return cudaErrorInvalidValue;
}

}  // namespace selscan
