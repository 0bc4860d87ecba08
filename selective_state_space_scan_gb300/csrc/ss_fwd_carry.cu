// Carry pass of the time-split forward schedule.
//
// The sequence of every (batch row, channel) is cut into segments.  Pass A folded each
// segment but the last from a zero state, leaving its end state in slot s + 1 and the sum of
// its Δ in seg_dsum[s].  Over one segment the pairs compose to (Π a_t, local end state) with
// Π a_t = exp(A Σ Δ_t) (the product of the per-step decays exp(Δ_t A)), so the state at the
// start of segment s is
//   H_0 = h0,   H_s = exp(A ΣΔ_{s-1}) H_{s-1} + local_{s-1},
// the carry combined from the left as in "mamba-metal: Apple Silicon で Mamba を動かす"
// (section "チャンク間 running prefix"), here across segments.  One thread per (row, state)
// walks the segments in order and overwrites slot s with H_s.
#include "device_common.cuh"
#include "internal.h"

namespace selscan {

__global__ void __launch_bounds__(256)
ss_fwd_carry_kernel(const float* __restrict__ A_log, const float* __restrict__ h0,
                    float* __restrict__ slots, const float* __restrict__ dsum,
                    int64_t rows, int Dm, int N, int nseg) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t count = rows * N;
    if (i >= count) return;
    const int64_t row = i / N;
    const int n = static_cast<int>(i - row * N);
    const int d = static_cast<int>(row % Dm);
    const float a2 = -expf(A_log[static_cast<int64_t>(d) * N + n]) * kLog2e;
    float h = h0 ? h0[i] : 0.f;
    slots[i] = h;
    for (int s = 1; s < nseg; ++s) {
        const float decay = ex2(a2 * dsum[static_cast<int64_t>(s - 1) * rows + row]);
        float* slot = slots + static_cast<int64_t>(s) * count + i;
        h = fmaf(decay, h, *slot);
        *slot = h;
    }
}

cudaError_t launch_fwd_carry(const FwdParams& p, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(p.batch) * p.Dm;
    const int64_t count = rows * p.N;
    const int64_t blocks = (count + 255) / 256;
    if (blocks <= 0) return cudaSuccess;
    ss_fwd_carry_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        p.A_log, p.h0, p.seg_slots, p.seg_dsum, rows, p.Dm, p.N, p.nseg);
    return cudaGetLastError();
}

}  // namespace selscan
