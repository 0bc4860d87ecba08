// Kernel argument blocks shared by the host dispatcher and the kernels.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace selscan {

// Forward scan: element strides (channel / state stride is 1), sizes and pointers.
struct FwdParams {
    const void* u;
    const void* delta;
    const void* z;       // nullptr: no gate
    const void* Bm;
    const void* Cm;
    const float* bias;   // nullptr: 0
    const float* A_log;  // [Dm, N]
    const float* Dv;     // nullptr: 0
    void* y;
    float* last_state;   // nullptr: not written; else [batch, Dm, N] contiguous
    int64_t u_b, u_l, d_b, d_l, z_b, z_l, y_b, y_l, B_b, B_l, C_b, C_l;
    int batch, L, Dm, N;
    int nchunks;
    int tiles_per_batch;
    int chunk_steps;     // steps per chunk the host sized the grid and TMA boxes for
    int tile_channels;   // channels per CTA the host sized them for
    int box_channels;    // width of the u/Δ/z TMA boxes the host encoded (0: no TMA)
    unsigned int* err;   // device error word
    // Balanced schedule (ws_flag != nullptr): the grid's CTAs split the batch·tiles·nchunks
    // (tile, chunk) units into equal contiguous ranges; a range that starts inside a tile takes
    // the state at its start from the previous CTA, which publishes it (ws_state, then ws_flag
    // set to epoch) as soon as it has folded the head of that tile.
    float* ws_state;     // [grid][tile_channels][ns] fp32
    unsigned int* ws_flag;   // [grid]
    unsigned int epoch;  // this call's nonzero tag
    int grid;            // CTAs in the launch (0: batch·tiles_per_batch)
    // Cluster-balanced schedule (cbal > 0, no workspace): the grid is clusters of cbal CTAs; cluster
    // q takes the whole tiles [T·q/Q, T·(q+1)/Q) of the T tiles (Q clusters) and splits their
    // (tile, chunk) units into cbal equal contiguous ranges, one per CTA; a tile split between two
    // CTAs of the cluster hands its state over through distributed shared memory.
    int cbal;
    // Initial state h_{-1} [batch, Dm, N] contiguous (nullptr: zeros).
    const float* h0;
    // Checkpoints for the backward pass (the CKPT kernel, one CTA per 32-channel tile, 16 states):
    // the state entering every 16th step, [tiles][ckpt_chunks][2][32][16] fp32 with
    // ckpt_chunks = ceil(L / 32) (the steps past L are identity steps: their entries hold the
    // final state).
    float* ckpt;
    int ckpt_chunks;
    // Time-split schedule (seg_launch > 0): the sequence is cut into segments of seg_chunks
    // chunks; CTA x takes segment x % seg_launch of tile x / seg_launch.  Pass A (state-only
    // kernel) folds segments 0 .. nseg-2 from zero and writes each end state to slot s + 1
    // of seg_slots and its Σ Δ to seg_dsum; the carry kernel turns the slots into the state at
    // every segment's start (slot 0 = h0); pass C folds every segment from its slot.
    int seg_launch;      // segments per tile in this launch
    int seg_chunks;      // chunks per segment
    int nseg;            // segments per tile in the schedule
    float* seg_slots;    // [nseg][batch·Dm·N]
    float* seg_dsum;     // [nseg - 1][batch·Dm]
    int seg_out0;        // pass A writes segment s's end state to slot s + seg_out0 (1 in the time
                         // split; 0 for a segment summary, whose slot 0 is the output)
    // Low-rank time-step projection folded in (dt_rank > 0): `delta` points to dt_low
    // [batch, L, dt_rank] (strides d_b, d_l) and delta_raw[b,t,d] = Σ_k W_dt[d,k] dt_low[b,t,k].
    const float* W_dt;   // [Dm, dt_rank] contiguous
    int dt_rank;
    int dt_pitch;        // floats per staged dt_low row (dt_rank rounded up so that rows fall on different banks)
};

// TMA descriptors for the five streamed tensors (unused by the plain-load variant).
struct FwdMaps {
    CUtensorMap u, delta, z, B, C;
};

// Decode step.
struct StepParams {
    float* state;        // [batch, Dm, N] with strides state_b, state_d (state stride 1)
    const void* x;
    const void* delta;
    const void* z;       // nullptr: no gate
    const void* Bm;      // [batch, N]
    const void* Cm;
    const float* bias;
    const float* A_log;
    const float* Dv;
    void* y;             // [batch, Dm]
    int64_t x_b, d_b, z_b, y_b, B_b, C_b, s_b, s_d;
    int batch, Dm, N;
};

// Decode step over many layers in one launch: the layers share sizes and strides (`common`,
// whose pointers are unused) and each has its own buffers.
constexpr int kStepMaxLayers = 128;
struct StepLayerPtrs {
    float* state;
    const void* x;
    const void* delta;
    const void* z;
    const void* Bm;
    const void* Cm;
    const float* bias;
    const float* A_log;
    const float* Dv;
    void* y;
};
struct StepLayersParams {
    StepParams common;
    unsigned int* err;   // device error word (the staged kernel's bounded waits)
    int n_layers;
    StepLayerPtrs layer[kStepMaxLayers];
};

}  // namespace selscan
