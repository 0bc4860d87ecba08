// bf16-I/O forward-scan kernels (fp32 state and arithmetic).
#include "ss_fwd_launch.cuh"

namespace selscan {

cudaError_t launch_fwd_bf16(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                            cudaStream_t stream) {
    return launch_fwd_dtype<__nv_bfloat16>(v, p, m, stream);
}

}  // namespace selscan
