// Instantiation and launch of the forward-scan kernel family for one I/O type.
#pragma once

#include "internal.h"
#include "ss_fwd_kernel.cuh"

namespace selscan {

// Tile shape used for every forward launch: 4 groups of 8 channels (32 channels), 2 warps
// of 4 segments per group (8 segments), 6 steps per thread -> 48 steps per chunk, 4-deep
// TMA ring.  6 steps per thread keeps both the u/Δ/z reads and the B/C quad reads free of
// shared-memory bank conflicts under the TMA swizzle.
constexpr int kG = 4, kQ = 2, kK = 6, kStages = 4;

template <typename TIO, int NS, bool TMA>
cudaError_t launch_fwd_cfg(const FwdParams& p, const FwdMaps& m, cudaStream_t stream) {
    using Cfg = FwdCfg<TIO, NS, kG, kQ, kK, kStages>;
    auto kern = ss_fwd_kernel<Cfg, TMA>;
    constexpr int smem = TMA ? Cfg::SMEM_BYTES : Cfg::SMEM_BYTES - (kStages - 1) * Cfg::STAGE_BYTES;
    static_assert(smem <= 227 * 1024, "shared memory budget exceeded");
    // Opting in to > 48 KB of dynamic shared memory is idempotent; done on every launch
    // so that each device the library runs on gets it.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.batch) * static_cast<unsigned>(p.tiles_per_batch);
    kern<<<grid, Cfg::THREADS, smem, stream>>>(p, m);
    return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_fwd_dtype(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                             cudaStream_t stream) {
    switch (v.ns) {
        case 4: return v.tma ? launch_fwd_cfg<TIO, 4, true>(p, m, stream)
                             : launch_fwd_cfg<TIO, 4, false>(p, m, stream);
        case 8: return v.tma ? launch_fwd_cfg<TIO, 8, true>(p, m, stream)
                             : launch_fwd_cfg<TIO, 8, false>(p, m, stream);
        case 16: return v.tma ? launch_fwd_cfg<TIO, 16, true>(p, m, stream)
                              : launch_fwd_cfg<TIO, 16, false>(p, m, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace selscan
