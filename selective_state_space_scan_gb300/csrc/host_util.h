// Host-side argument checks shared by every entry point (selscan_api.cu, ss_conv1d.cu, ss_bwd.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace selscan {
namespace host {

// Device memory of device `dev` (or managed memory).
inline bool dev_ptr(const void* q, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

inline bool is_aligned(const void* q, size_t a) { return reinterpret_cast<uintptr_t>(q) % a == 0; }

// Byte range touched by a [n0, n1, n2] tensor with element strides (s0, s1, 1).
struct Range {
    uintptr_t lo = 0, hi = 0;
};
inline Range range3(const void* q, int64_t n0, int64_t n1, int64_t n2, int64_t s0, int64_t s1, int64_t es) {
    Range r;
    if (!q || n0 <= 0 || n1 <= 0 || n2 <= 0) return r;
    r.lo = reinterpret_cast<uintptr_t>(q);
    r.hi = r.lo + static_cast<uintptr_t>(((n0 - 1) * s0 + (n1 - 1) * s1 + n2) * es);
    return r;
}
inline bool meet(const Range& a, const Range& b) {
    return a.hi > a.lo && b.hi > b.lo && a.lo < b.hi && b.lo < a.hi;
}

}  // namespace host
}  // namespace selscan
