// Shared launch helper for the forward-scan kernel instantiations.
#pragma once

#include "internal.h"

namespace selscan {

template <class Cfg, bool TMA, class Kern>
cudaError_t launch_with_smem(Kern kern, const FwdParams& p, const FwdMaps& m, cudaStream_t stream,
                             int smem, bool cooperative = false, int* max_grid = nullptr) {
    // Opting in to more than 48 KB of dynamic shared memory is idempotent; done on every
    // launch so that each device the library runs on gets it.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (max_grid) {
        int dev = 0, sms = 0, per_sm = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::THREADS, smem)) != cudaSuccess)
            return e;
        *max_grid = sms * per_sm;
        return cudaSuccess;
    }
    const unsigned grid = p.grid > 0 ? static_cast<unsigned>(p.grid)
                                     : static_cast<unsigned>(p.batch) * static_cast<unsigned>(p.tiles_per_batch);
    if (cooperative) {
        // All CTAs must be resident together: a CTA may wait for another's published state.
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(Cfg::THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, p, m);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    kern<<<grid, Cfg::THREADS, smem, stream>>>(p, m);
    return cudaGetLastError();
}

}  // namespace selscan
