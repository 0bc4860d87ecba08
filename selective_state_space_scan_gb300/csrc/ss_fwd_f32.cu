// fp32-I/O forward-scan kernels.
#include "ss_fwd_launch.cuh"

namespace selscan {

int fwd_tile_channels() { return 8 * kG; }
int fwd_chunk_steps() { return 4 * kQ * kK; }

cudaError_t launch_fwd_f32(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                           cudaStream_t stream) {
    return launch_fwd_dtype<float>(v, p, m, stream);
}

}  // namespace selscan
