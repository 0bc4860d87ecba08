// Shared launch helper for the forward-scan kernel instantiations.
#pragma once

#include "internal.h"

namespace selscan {

template <class Cfg, bool TMA, class Kern>
cudaError_t launch_with_smem(Kern kern, const FwdParams& p, const FwdMaps& m, cudaStream_t stream,
                             int smem) {
    // Opting in to more than 48 KB of dynamic shared memory is idempotent; done on every
    // launch so that each device the library runs on gets it.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.batch) * static_cast<unsigned>(p.tiles_per_batch);
    kern<<<grid, Cfg::THREADS, smem, stream>>>(p, m);
    return cudaGetLastError();
}

}  // namespace selscan
