// fp32-I/O state-split lane forward kernels.
#include "fwd_lane_impl.cuh"

namespace selscan {
cudaError_t launch_fwd_lane_f32(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                cudaStream_t stream, int* max_grid) {
    return launch_lane_dtype<float>(v, p, m, stream, max_grid);
}
}  // namespace selscan
