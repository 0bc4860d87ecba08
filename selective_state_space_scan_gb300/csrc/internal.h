// Host-side entry points of the kernel translation units (internal to libselscan).
#pragma once

#include <cuda_runtime.h>

#include "fwd_configs.h"
#include "fwd_params.h"

namespace selscan {

enum FwdFamily { kFamLane = 0, kFamSeg = 1 };

// One forward-scan kernel instantiation.  `ns` is the state count it is built for (4, 8
// or 16, with N <= ns); `lpc` the lane family's lanes per channel (1, 2 or 4, at most
// ns/4); `tma` selects TMA-fed tiles (needs N == ns, 16-byte aligned bases and row strides)
// over the plain-load fill.
struct FwdVariant {
    int family;
    int ns;
    int lpc;
    bool tma;
    bool balanced;   // lane family: equal (tile, chunk) ranges per CTA (needs a workspace, TMA)
    bool state_only; // lane family, TMA: pass A of the time-split schedule (end states only)
    bool lti;        // lane family, TMA, per tile: B and C constant over the steps (held in registers)
    bool dtp;        // lane family, TMA, per tile: the low-rank time-step projection folded in
    int es = 4;      // bytes per I/O element (4 fp32, 2 bf16)
    int chunk = 0;   // test override of the steps per chunk (16, 32 or 256; 0: the kernels' own)
    bool bcf32 = false;  // bf16 streams with B and C staged as fp32 (a widened copy in the workspace)
    int cluster = 0;     // > 0: the single-launch time split, segments per cluster
    bool w32 = false;    // balanced fp32 on 32-channel tiles (the per-tile kernel's own geometry)
    bool ckpt = false;   // per tile, LPC 4, 16 states: also write the backward's checkpoints
    bool dx4 = false;    // balanced fp32 32-channel tiles at LPC 4: (Δ, Δ·u) through shared memory
    int cbal = 0;        // > 0: the cluster-balanced schedule (no workspace), CTAs per cluster
};

struct FwdGeom {
    int tile_channels;   // channels per CTA
    int box_channels;    // width of one u/Δ/z TMA box
    int chunk_steps;     // steps per chunk (TMA box height)
};

inline FwdGeom fwd_geometry(const FwdVariant& v) {
    if (v.family == kFamSeg) return FwdGeom{8 * kSegG, 8 * kSegG, 4 * kSegQ * kSegK};
    if (v.dtp) return FwdGeom{32, 32, kLaneTD};
    const int w = v.w32 ? 32 : lane_w(v.lpc, v.balanced, v.es);
    return FwdGeom{w, w, v.chunk > 0 ? v.chunk : kLaneT};
}

// Launch (grid = p.grid CTAs; cooperative when v.balanced).  With `max_grid` non-null, launch
// nothing and return in it the number of CTAs of this kernel that fit on the current device.
cudaError_t launch_fwd_lane_f32(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                cudaStream_t stream, int* max_grid = nullptr);
cudaError_t launch_fwd_lane_bf16(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                 cudaStream_t stream, int* max_grid = nullptr);
// The bf16 lane kernels with widened (fp32) B/C tiles, 16 states (v.bcf32).
cudaError_t launch_fwd_lane_bf16w(const FwdVariant& v, const FwdParams& p, const FwdMaps& m,
                                  cudaStream_t stream, int* max_grid = nullptr);
// bf16 B and C [batch, L, N] (strides in elements) widened to fp32 [batch, L, N] contiguous; N a
// multiple of 4, rows 8-byte aligned.
cudaError_t launch_widen_bc(const void* B, const void* C, int64_t B_b, int64_t B_l, int64_t C_b, int64_t C_l,
                            float* Bf, float* Cf, int64_t batch, int64_t L, int N, cudaStream_t stream);
cudaError_t launch_fwd_seg(const FwdVariant& v, bool bf16, const FwdParams& p, const FwdMaps& m,
                           cudaStream_t stream);
cudaError_t launch_step(const StepParams& p, bool bf16, bool vec, cudaStream_t stream);
cudaError_t launch_step_layers(const StepLayersParams& q, bool bf16, bool vec, cudaStream_t stream);
// The lane kernel with the low-rank time-step projection folded in (fp32, per tile, TMA).
cudaError_t launch_fwd_lane_dtp(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t stream);
// The single-launch time split (fwd_lane_cluster.cu): p.grid = tiles × cluster CTAs in clusters of
// `cluster` (2..8) consecutive CTAs, p.seg_launch = cluster.  With `fit` non-null, launch nothing
// and return in fit[0] how many such clusters can be resident at once and in fit[1] the CTAs per SM.
cudaError_t launch_fwd_lane_cluster(bool bf16, const FwdParams& p, const FwdMaps& m, cudaStream_t stream, int cluster,
                                    int* fit = nullptr);
// The cluster-balanced schedule (fwd_lane_cbal.cu): p.grid = Q × cluster CTAs in clusters of
// `cluster` (2..8), p.cbal = cluster; bf16 at lpc 2 or fp32 at lpc 4; per_sm > 0 pads the shared
// memory so that at most per_sm CTAs share an SM.  With `fit` non-null, launch nothing and return in
// fit[0] how many such clusters can be resident at once and in fit[1] the CTAs per SM.
cudaError_t launch_fwd_lane_cbal(bool bf16, int lpc, const FwdParams& p, const FwdMaps& m, cudaStream_t stream,
                                 int cluster, int per_sm, int* fit = nullptr);
// Test instantiations at other chunk lengths (fwd_lane_chunks.cu): whether v (with v.chunk set)
// is one of them, and its launch.
bool chunk_override_ok(const FwdVariant& v);
cudaError_t launch_fwd_lane_chunked(const FwdVariant& v, const FwdParams& p, const FwdMaps& m, cudaStream_t stream);
// Time-split carry pass: slot 0 of p.seg_slots = h0 (or zeros); slot s = exp(A·ΣΔ of segment
// s-1)·slot s-1 + the end state pass A left in slot s, for s = 1 .. p.nseg - 1.
cudaError_t launch_fwd_carry(const FwdParams& p, cudaStream_t stream);

// Unswizzled 3-D TMA descriptor over a [batch, rows, cols] tensor (cols contiguous, element
// strides row_stride and batch_stride) with a [1, box_rows, box_cols] box; elements past the
// ends read as zero.  False when the tensor's alignment or strides rule TMA out.
bool make_tile_map(CUtensorMap* m, const void* base, bool bf16, int64_t cols, int64_t rows, int64_t batch,
                   int64_t row_stride, int64_t batch_stride, int box_cols, int box_rows);

// The current device's error word (kErr* bits), or nullptr if its address cannot be found.
unsigned int* device_error_word();

// The calling thread's current CUDA context (nullptr if there is none or it cannot be had).
CUcontext current_context();

}  // namespace selscan
