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

// Whether a [n0, n1, n2] tensor with element strides (s0, s1, 1) puts every element at its own
// address, so that an output written through it has no two writers per word.  The dimensions
// of more than one element, taken in order of stride, must each step past the whole span of
// the smaller ones: a sufficient test, which accepts contiguous, strided-view and interleaved
// layouts and refuses a broadcast (stride 0) or rows that run into each other.  Strides are
// non-negative; a span beyond int64 counts as overlapping.
inline bool distinct3(int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t n2) {
    int64_t n[3] = {n2, n1, n0}, s[3] = {1, s1, s0};
    for (int i = 1; i < 3; ++i)                     // order by stride
        for (int j = i; j > 0 && s[j] < s[j - 1]; --j) {
            const int64_t tn = n[j], ts = s[j];
            n[j] = n[j - 1]; s[j] = s[j - 1];
            n[j - 1] = tn; s[j - 1] = ts;
        }
    int64_t span = 1;                               // one past the largest offset so far
    for (int i = 0; i < 3; ++i) {
        if (n[i] <= 1) continue;
        if (s[i] < span || s[i] > (INT64_MAX - span) / (n[i] - 1)) return false;
        span += (n[i] - 1) * s[i];
    }
    return true;
}

}  // namespace host
}  // namespace selscan
