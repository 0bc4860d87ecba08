// Single-token decode update of the selective SSM (the O(1)-per-token step of
// "mamba-metal: Apple Silicon で Mamba を動かす", section "O(L) インクリメンタルデコード"):
//   Δ          = softplus(delta_raw[b,d] + delta_bias[d])
//   h[b,d,n]  <- exp(Δ A_n) h[b,d,n] + Δ x[b,d] B[b,n],    A_n = -exp(A_log[d,n])
//   y[b,d]     = (Σ_n C[b,n] h[b,d,n] + D[d] x[b,d]) · silu(z[b,d])
// The state is updated in place.  The step is elementwise over (b,d) and HBM-bound on the
// state read + write, so the mapping is: LPR lanes per (b,d) row, each lane owning four
// consecutive states (one 16-byte load and store of h), the partial C·h sums reduced across
// the row's lanes by shuffles.
#include "device_common.cuh"
#include "fwd_params.h"
#include "internal.h"

namespace selscan {

template <typename TIO, int LPR, bool VEC>
__global__ void __launch_bounds__(256) ss_step_kernel(const StepParams p) {
    const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = gt / LPR;
    const int qd = static_cast<int>(gt % LPR);
    const int64_t rows = static_cast<int64_t>(p.batch) * p.Dm;
    const bool row_ok = row < rows;
    const int64_t b = row_ok ? row / p.Dm : 0;
    const int64_t d = row_ok ? row % p.Dm : 0;

    float partial = 0.f, xv = 0.f, zv = 0.f;
    if (row_ok) {
        const TIO* x = static_cast<const TIO*>(p.x);
        const TIO* dr = static_cast<const TIO*>(p.delta);
        xv = to_f32<TIO>(x[b * p.x_b + d]);
        const float bias = p.bias ? p.bias[d] : 0.f;
        const float dlt = softplus(to_f32<TIO>(dr[b * p.d_b + d]) + bias);
        const float dx = dlt * xv;
        if (p.z) zv = to_f32<TIO>(static_cast<const TIO*>(p.z)[b * p.z_b + d]);
        float* h = p.state + b * p.s_b + d * p.s_d;
        const float* al = p.A_log + d * p.N;
        const TIO* Bm = static_cast<const TIO*>(p.Bm) + b * p.B_b;
        const TIO* Cm = static_cast<const TIO*>(p.Cm) + b * p.C_b;
        for (int n0 = qd * 4; n0 < p.N; n0 += LPR * 4) {
            if (VEC) {
                float4 hv = *reinterpret_cast<const float4*>(h + n0);
                const float4 av = *reinterpret_cast<const float4*>(al + n0);
                float hs[4] = {hv.x, hv.y, hv.z, hv.w};
                const float as[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float A2 = -expf(as[j]) * kLog2e;
                    hs[j] = fmaf(ex2(dlt * A2), hs[j], dx * to_f32<TIO>(Bm[n0 + j]));
                    partial = fmaf(to_f32<TIO>(Cm[n0 + j]), hs[j], partial);
                }
                *reinterpret_cast<float4*>(h + n0) = make_float4(hs[0], hs[1], hs[2], hs[3]);
            } else {
                for (int j = 0; j < 4 && n0 + j < p.N; ++j) {
                    const int n = n0 + j;
                    const float A2 = -expf(al[n]) * kLog2e;
                    const float hn = fmaf(ex2(dlt * A2), h[n], dx * to_f32<TIO>(Bm[n]));
                    h[n] = hn;
                    partial = fmaf(to_f32<TIO>(Cm[n]), hn, partial);
                }
            }
        }
    }
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) partial += __shfl_xor_sync(0xffffffffu, partial, off);
    if (row_ok && qd == 0) {
        float v = fmaf(p.Dv ? p.Dv[d] : 0.f, xv, partial);
        if (p.z) v *= silu(zv);
        static_cast<TIO*>(p.y)[b * p.y_b + d] = from_f32<TIO>(v);
    }
}

template <typename TIO, int LPR>
static cudaError_t launch_step_t(const StepParams& p, bool vec, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(p.batch) * p.Dm * LPR;
    const int64_t blocks = (threads + 255) / 256;
    if (vec)
        ss_step_kernel<TIO, LPR, true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        ss_step_kernel<TIO, LPR, false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIO>
static cudaError_t launch_step_dtype(const StepParams& p, bool vec, cudaStream_t stream) {
    const int quads = (p.N + 3) / 4;
    if (quads <= 1) return launch_step_t<TIO, 1>(p, vec, stream);
    if (quads <= 2) return launch_step_t<TIO, 2>(p, vec, stream);
    return launch_step_t<TIO, 4>(p, vec, stream);
}

cudaError_t launch_step(const StepParams& p, bool bf16, bool vec, cudaStream_t stream) {
    return bf16 ? launch_step_dtype<__nv_bfloat16>(p, vec, stream)
                : launch_step_dtype<float>(p, vec, stream);
}

}  // namespace selscan
