// Host-side entry points of the kernel translation units (internal to libselscan).
#pragma once

#include <cuda_runtime.h>

#include "fwd_params.h"

namespace selscan {

// Forward-scan kernel variants.  `ns` is the state count the kernel is built for (4, 8
// or 16, N <= ns); `tma` selects the TMA-fed variant (which needs N == ns and 16-byte
// aligned bases and row strides) over the plain-load variant.
struct FwdVariant {
    int ns;
    bool tma;
};

// Channels per CTA and steps per chunk of the forward kernels (for grid sizing).
int fwd_tile_channels();
int fwd_chunk_steps();

cudaError_t launch_fwd_f32(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                           cudaStream_t stream);
cudaError_t launch_fwd_bf16(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                            cudaStream_t stream);
cudaError_t launch_step(const StepParams& p, bool bf16, bool vec, cudaStream_t stream);

}  // namespace selscan
