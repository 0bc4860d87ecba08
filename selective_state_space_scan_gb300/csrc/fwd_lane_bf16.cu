// bf16-I/O state-split lane forward kernels (fp32 state and arithmetic).
#include "fwd_lane_impl.cuh"

namespace selscan {
cudaError_t launch_fwd_lane_bf16(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                 cudaStream_t stream, int* max_grid) {
    return launch_lane_dtype<__nv_bfloat16>(v, p, m, stream, max_grid);
}
}  // namespace selscan
