/*
 * libselscan — Mamba selective-scan forward pass and single-token decode update on
 * NVIDIA GB300 (sm_103a).  Plain C ABI: device pointers, sizes, a CUDA stream handle.
 *
 * The operation (sources: "mamba-metal: Apple Silicon で Mamba を動かす", sections
 * "Selective scan の本質", "チャンク間 running prefix" and "O(L) インクリメンタルデコード";
 * the same blog's walkthrough of the official CUDA forward kernel, section
 * "1チャンク内の処理フロー"; SpeechLens docs/kernel-optimization.md, MetalSelectiveScan
 * tensor contract).  For every batch row b, channel d and state n, with h_{-1} = 0:
 *
 *   Δ_t      = softplus(delta_raw[b,t,d] + delta_bias[d])
 *   h_t[n]   = exp(Δ_t · A[d,n]) · h_{t-1}[n] + Δ_t · B[b,t,n] · u[b,t,d],
 *              A[d,n] = -exp(A_log[d,n])
 *   y[b,t,d] = (Σ_n C[b,t,n] · h_t[n] + D[d] · u[b,t,d]) · silu(z[b,t,d])
 *
 * with silu(z) = z · sigmoid(z).  It is evaluated as a chunked associative scan over the
 * pairs (a,b) = (exp(Δ A), Δ B u) with (a2,b2)∘(a1,b1) = (a2 a1, a2 b1 + b2) and a
 * per-state carry across chunks, so any L runs in one launch.
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every buffer.  The library allocates no device or
 *     host memory and never synchronises; work is enqueued on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and runs asynchronously.
 *   - Errors: arguments are validated on the host before anything is enqueued; a
 *     failed check returns an SS_ERR_* code and enqueues nothing.  There is no CPU or
 *     alternative fallback.  A failed launch returns SS_ERR_CUDA.  Faults detected on
 *     the device (a wait that timed out) set bits in a per-device error word, read
 *     with ss_device_error().
 *   - Pointers: every pointer argument must be device-accessible memory of the current
 *     device (cudaMalloc or managed); host pointers are rejected with SS_ERR_INVALID_ARG.
 *   - Types: u, delta_raw, z, B, C and y are `io_dtype` (fp32 or bf16); A_log, D,
 *     delta_bias, last_state and the decode state are always fp32.  Arithmetic and
 *     the recurrent state are fp32 in both cases.
 *   - Thread safety: calls are reentrant.  Process-wide state: the cached driver entry
 *     point used to build TMA descriptors, the per-device error word, and a call counter that
 *     tags ss_fwd_ws hand-overs.
 */
#ifndef SELSCAN_H
#define SELSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SS_OK = 0,
    SS_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, host pointer, aliasing */
    SS_ERR_UNSUPPORTED = 2,   /* N outside 1..16, size beyond the 32-bit grid limits */
    SS_ERR_MISALIGNED = 3,    /* a pointer not aligned to its element size */
    SS_ERR_CUDA = 4           /* a CUDA runtime/driver call or a kernel launch failed */
} ss_status;

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

/*
 * Element strides (not bytes) of the forward tensors.  The channel axis of u,
 * delta_raw, z, y and the state axis of B, C have stride 1.  A NULL strides pointer
 * means: io_dtype = SS_F32 and every tensor contiguous
 * (x_b = L·Dm, x_l = Dm for [batch, L, Dm]; B_b = L·N, B_l = N for [batch, L, N]).
 * Steps of B and C are at least N elements apart, or B_l = C_l = 0: B and C constant over the
 * steps of a batch row, the linear time-invariant case that the blog's walkthrough of the
 * official CUDA kernel (section "主要な最適化テクニック", the kIsVariableB/C branch) specialises.
 * The forward pass then holds each state's B and C in registers instead of staging tiles of
 * them (only one of the two at stride 0 is served by the generic fill).
 */
typedef struct {
    int32_t io_dtype;                       /* ss_dtype */
    int64_t u_b, u_l;                       /* u        [batch, L, Dm] */
    int64_t delta_b, delta_l;               /* delta_raw[batch, L, Dm] */
    int64_t z_b, z_l;                       /* z        [batch, L, Dm] (ignored if z NULL) */
    int64_t y_b, y_l;                       /* y        [batch, L, Dm] */
    int64_t B_b, B_l;                       /* B        [batch, L, N]  */
    int64_t C_b, C_l;                       /* C        [batch, L, N]  */
} ss_fwd_strides;

/*
 * Selective-scan forward pass (prefill / layer scan).
 * Defined by: the recurrence and its left-to-right carry of "mamba-metal: Apple Silicon で
 * Mamba を動かす" (sections "Selective scan の本質" and "チャンク間 running prefix"); the
 * per-chunk steps, i.e. softplus on Δ, the D·u skip, out += h·C per state and the z·sigmoid(z)
 * gate, of the same blog's walkthrough of the official CUDA forward kernel (section
 * "1チャンク内の処理フロー"); the tensor contract of SpeechLens docs/kernel-optimization.md
 * (MetalSelectiveScan: [B, L, D] streams, B and C [B, L, N] shared by every channel, raw A_log
 * turned into -exp(A_log) inside the kernel).  last_state is the prefill-to-decode hand-off of
 * the blog's section "O(L) インクリメンタルデコード".
 *   u, delta_raw  [batch, L, Dm] io_dtype   input activation, pre-softplus time step
 *   delta_bias    [Dm] fp32 or NULL (= 0)   added to delta_raw before softplus
 *   A_log         [Dm, N] fp32 contiguous    A = -exp(A_log), computed in-kernel
 *   B, C          [batch, L, N] io_dtype    input / output state coefficients, shared
 *                                           by all channels of a batch row
 *   D             [Dm] fp32 or NULL (= 0)   skip weight
 *   z             [batch, L, Dm] io_dtype or NULL (no gate)
 *   y             [batch, L, Dm] io_dtype   output; must not overlap any input, and its strides
 *                                           must give every element its own address (no
 *                                           stride-0 or overlapping rows): SS_ERR_INVALID_ARG
 *   last_state    [batch, Dm, N] fp32 contiguous or NULL: h_{L-1}, the state that a
 *                                           following ss_step continues from
 *   batch, L, Dm  >= 0; batch == 0 or Dm == 0 is a no-op; L == 0 writes zeros to
 *                 last_state (if given) and nothing else (ss_fwd_h0: copies h0 there)
 *   N             1..16
 * Returns SS_OK once the work is enqueued.
 */
ss_status ss_fwd(const void* u, const void* delta_raw, const float* delta_bias,
                 const float* A_log, const void* B, const void* C, const float* D,
                 const void* z, void* y, float* last_state, int64_t batch, int64_t L,
                 int64_t Dm, int64_t N, const ss_fwd_strides* strides, void* stream);

/*
 * Forward pass with a caller-provided workspace; same arguments and result as ss_fwd.
 *
 * ss_fwd runs one CTA per tile of channels over the whole sequence; with more tiles than the GPU
 * holds at once, clusters of CTAs instead split their tiles' chunks evenly, handing the state of
 * a tile split between two CTAs over through the cluster's distributed shared memory (bitwise
 * the same results), and with too few tiles to fill the GPU, the CTAs of a cluster fold the time
 * segments of one tile (equal up to rounding).  With a workspace, one of two schedules of the
 * same carry-across-chunks scan ("mamba-metal: Apple Silicon で Mamba を動かす", section
 * "チャンク間 running prefix") runs instead:
 *   - balanced (enough channel tiles to fill the GPU): the (tile, chunk) work is split into
 *     equal contiguous ranges, one per CTA the device can hold at once (a cooperative launch),
 *     so every SM gets the same amount of work; a range that starts inside a tile takes the
 *     state at its start from the CTA before it (the workspace holds one flag and one tile
 *     state per CTA).  Results are bitwise equal to the one-CTA-per-tile schedule's at the
 *     same number of lanes per channel; ss_fwd may split a channel's states over more lanes
 *     (it has fewer CTAs per SM to fill), which sums the C·h terms in another order, so the
 *     two calls then agree up to rounding.
 *   - time-split (too few channel tiles, e.g. one long sequence): each sequence is cut into
 *     segments that run side by side.  A first pass folds every segment but the last from a
 *     zero state; a carry pass combines those end states left to right (the decay over a
 *     segment is exp(A · Σ Δ)); a last pass folds every segment from its carried start.  The
 *     workspace holds one state per (segment, row, state) and one Σ Δ per (segment, row).
 *     Results equal ss_fwd's up to rounding (the carry is composed in another order).
 *   workspace        device memory, 256-byte aligned, at least workspace_bytes =
 *                    ss_fwd_workspace_size(...) bytes, zero-filled before its first use (the
 *                    library never needs it cleared again).  Calls that share a workspace must
 *                    not run concurrently on the device.  A workspace smaller than the size
 *                    query asks for gives the time-split schedule fewer segments (none, i.e.
 *                    ss_fwd's schedule, below two); for the balanced schedule it returns
 *                    SS_ERR_INVALID_ARG.
 *   workspace NULL   behaves exactly like ss_fwd.
 * A misaligned workspace returns SS_ERR_MISALIGNED.  When the arguments cannot use TMA-fed
 * tiles (see ss_fwd_strides) the workspace is not used.
 */
ss_status ss_fwd_ws(const void* u, const void* delta_raw, const float* delta_bias,
                    const float* A_log, const void* B, const void* C, const float* D,
                    const void* z, void* y, float* last_state, int64_t batch, int64_t L,
                    int64_t Dm, int64_t N, const ss_fwd_strides* strides, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Workspace bytes ss_fwd_ws (and ss_fwd_h0) need for these sizes on the current device (0: none,
 * or the sizes are invalid).  Depends on the device's SM count and the kernel's occupancy.
 */
size_t ss_fwd_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype);

/*
 * Forward pass from a given initial state: ss_fwd_ws with h_{-1} = h0 instead of 0.
 * The recurrence continues from a state an earlier call left behind: the carry of
 * "mamba-metal: Apple Silicon で Mamba を動かす" (section "チャンク間 running prefix") handed
 * across calls, so a long sequence can be processed in pieces (chunked prefill: pass the
 * previous piece's last_state as h0) with the same result as one call, up to rounding.
 *   h0               [batch, Dm, N] fp32 contiguous, or NULL (= zeros, i.e. ss_fwd_ws).
 *                    It may be last_state itself (the state is then updated in place); it must
 *                    not overlap last_state otherwise, nor y.  4-byte aligned.
 *   L == 0           last_state (if given) receives a copy of h0 (zeros without one).
 *   workspace        as for ss_fwd_ws, NULL allowed.
 * Other arguments, errors and results as ss_fwd_ws.
 */
ss_status ss_fwd_h0(const void* u, const void* delta_raw, const float* delta_bias,
                    const float* A_log, const void* B, const void* C, const float* D,
                    const void* z, void* y, float* last_state, const float* h0, int64_t batch,
                    int64_t L, int64_t Dm, int64_t N, const ss_fwd_strides* strides,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Summary of one segment of a sequence, for sequence parallelism: the state the segment's steps
 * leave when folded from a zero state, and the sum of their Δ.  Over a segment the pairs
 * (a_t, b_t) compose to (Π a_t, h_end) with Π a_t = exp(A · Σ Δ_t), so a segment is summed up by
 * (h_end, Σ Δ): the aggregate that "mamba-metal: Apple Silicon で Mamba を動かす" (section
 * "チャンク間 running prefix") carries from one chunk to the next, here between parts of a
 * sequence held by different processes.  ss_carry_compose combines the summaries left to right
 * into each segment's entering state; ss_fwd_h0 then runs each segment from it.
 *   u, delta_raw, delta_bias, A_log, B   as for ss_fwd (C, D, z are not needed); the strides
 *                struct's z, y and C fields are ignored
 *   h_end        [batch, Dm, N] fp32 contiguous: h_{L-1} folded from h_{-1} = 0
 *   dsum         [batch, Dm] fp32 contiguous: Σ_t softplus(delta_raw[b,t,d] + delta_bias[d])
 *   L == 0       both outputs zero.
 * Schedule: one CTA per 32-channel tile over the segment (the state-only fold of ss_fwd_ws's
 * time split); the tiles must be TMA-fed (16-byte aligned bases and row strides, B rows of
 * exactly 4, 8 or 16 states), otherwise SS_ERR_UNSUPPORTED (no fallback).  Outputs must not
 * overlap the inputs or each other.  Errors as ss_fwd.
 */
ss_status ss_fwd_summary(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                         const void* B, float* h_end, float* dsum, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                         const ss_fwd_strides* strides, void* stream);

/*
 * Left-to-right composition of segment summaries into entering states (the carry of
 * "mamba-metal: Apple Silicon で Mamba を動かす", section "チャンク間 running prefix", across
 * segments):
 *   H_0 = h0 (zeros if NULL),   H_s = exp(A · dsum[s-1]) · H_{s-1} + slots[s]   (s = 1 .. nseg-1)
 * with A = -exp(A_log), per (b, d, n).
 *   slots   [nseg][batch, Dm, N] fp32 contiguous, in/out: on entry slot s (s >= 1) is the h_end of
 *           segment s-1 (ss_fwd_summary), slot 0 is ignored unless it is h0 itself; on exit slot s
 *           is H_s, the state entering segment s
 *   dsum    [nseg-1][batch, Dm] fp32 contiguous: the dsum of segments 0 .. nseg-2 (NULL if nseg == 1)
 *   h0      [batch, Dm, N] fp32 or NULL; may be slot 0 itself, must not overlap another slot
 *   nseg >= 1.  One thread per (b, d, n) walks the segments in order.  Errors as ss_fwd.
 */
ss_status ss_carry_compose(float* slots, const float* dsum, const float* h0, const float* A_log, int64_t nseg,
                           int64_t batch, int64_t Dm, int64_t N, void* stream);

/*
 * Forward pass with the low-rank time-step projection folded in: the pre-softplus time step is
 *   delta_raw[b,t,d] = Σ_k W_dt[d,k] · dt_low[b,t,k]   (k < dt_rank)
 * computed inside the scan instead of being read as a [batch, L, Dm] tensor.  This is the
 * "dtProj–scan fusion" of SpeechLens kernel-optimization.md (the rank-R delta projection
 * folded into the scan kernel; rejected there on Apple GPUs as slower at high sample rates).
 *   dt_low           [batch, L, dt_rank] fp32, strides strides->delta_b / delta_l (rows at
 *                    least dt_rank apart); 16-byte aligned base and row stride a multiple of
 *                    16 bytes
 *   W_dt             [Dm, dt_rank] fp32 contiguous, 16-byte aligned
 *   dt_rank          4..64, a multiple of 4 (else SS_ERR_UNSUPPORTED)
 *   h0               as ss_fwd_h0 (NULL = zeros)
 * Other arguments as ss_fwd (delta_raw replaced).  fp32 I/O only, and every tensor must allow
 * TMA-fed tiles (16-byte aligned bases and strides, B/C rows of exactly 4, 8 or 16 states):
 * otherwise SS_ERR_UNSUPPORTED, with no fallback.  One CTA per 32-channel tile, 48-step chunks.
 */
ss_status ss_fwd_dtproj(const void* u, const void* dt_low, const float* W_dt, int64_t dt_rank,
                        const float* delta_bias, const float* A_log, const void* B, const void* C,
                        const float* D, const void* z, void* y, float* last_state, const float* h0,
                        int64_t batch, int64_t L, int64_t Dm, int64_t N, const ss_fwd_strides* strides,
                        void* stream);

/*
 * Forward pass on host-resident tensors: ss_fwd's result with the copies to and from the device
 * inside the call.  The work goes in units of a group of batch rows (up to eight groups, one row
 * each when the batch allows) and a piece of the sequence (about 64 MB of inputs; each piece
 * scanned from the state the previous piece of its rows left, as ss_fwd_h0 does), through two
 * device staging slots on three internal streams, so that the copy in of one unit, the scan of
 * another and the copy back of a third overlap.  The result equals one ss_fwd call up to
 * rounding.  No counterpart in the pages: it serves callers whose tensors live in host memory.
 *   u, delta_raw, z, y   [batch, L, Dm] io_dtype, contiguous, HOST memory (pinned memory lets the
 *                        copies run asynchronously; pageable memory works but serialises them)
 *   B, C                 [batch, L, N] io_dtype, contiguous, host memory
 *   A_log [Dm, N], D, delta_bias [Dm] (NULL allowed as for ss_fwd), last_state [batch, Dm, N]
 *                        (or NULL): fp32, contiguous, host memory
 *   workspace            device memory, 256-byte aligned, at least
 *                        ss_fwd_host_workspace_size(...) bytes (staging only; no contents carried
 *                        between calls)
 *   stream               the work starts after everything enqueued on it, and it waits for the
 *                        last copy back: y and last_state are valid on the host once the stream is
 *                        synchronised.  L == 0 synchronises the stream and zeroes last_state.
 * Device pointers where host memory is expected, overlapping outputs or a small workspace return
 * SS_ERR_INVALID_ARG; errors of the scan itself are ss_fwd's.
 */
ss_status ss_fwd_host(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                      const void* B, const void* C, const float* D, const void* z, void* y,
                      float* last_state, int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes ss_fwd_host needs (0: sizes invalid or empty). */
size_t ss_fwd_host_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype);

/* Size of the fixed device array ss_fwd_static uses as its workspace (1 MiB). */
#define SS_STATIC_WORKSPACE_BYTES ((size_t)1 << 20)

/*
 * ss_fwd_ws without a caller-provided workspace, for callers that cannot allocate device
 * memory: a host whose own allocator already owns all device memory and lends none to
 * libraries, a runtime that forbids allocation once it has started (fixed-footprint serving),
 * or a plugin interface that passes the library tensors and a stream but no allocation hook.
 * The pages this library follows have no counterpart of this call; it is a packaging of
 * ss_fwd_ws.
 *   Arguments and results are those of ss_fwd_ws on the same sizes: it runs the schedule
 *   ss_fwd_ws picks (balanced or time-split), so its results are bitwise equal to ss_fwd_ws's,
 *   and equal to ss_fwd's up to rounding (ss_fwd may split a channel's states over a different
 *   number of lanes, which sums the C·h terms in another order).
 *   Workspace: a fixed SS_STATIC_WORKSPACE_BYTES array built into the library's device code;
 *   each device that loads the library holds it until the process exits.  The call allocates
 *   nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *   Sizes that need more than SS_STATIC_WORKSPACE_BYTES return SS_ERR_UNSUPPORTED (use
 *   ss_fwd_ws with your own workspace).  For the balanced schedule that is its
 *   ss_fwd_workspace_size; the time-split schedule takes as many segments as fit in the array
 *   (at least two), as ss_fwd_ws does with a smaller workspace.  Sizes that need no workspace
 *   run as ss_fwd.
 *   The first call on each device (each CUDA context) looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that first call before
 *   any stream capture.  The cache is keyed by the current context, so a context torn down and
 *   created again (cudaDeviceReset) is looked up afresh.
 *   Every call on a device shares the array: calls that overlap on the GPU (e.g. on two
 *   streams) race and give wrong results.  Nothing in it needs clearing between calls.
 */
ss_status ss_fwd_static(const void* u, const void* delta_raw, const float* delta_bias,
                        const float* A_log, const void* B, const void* C, const float* D,
                        const void* z, void* y, float* last_state, int64_t batch, int64_t L,
                        int64_t Dm, int64_t N, const ss_fwd_strides* strides, void* stream);

/*
 * Backward pass: the gradients of ss_fwd_h0's outputs (y and last_state) with respect to every
 * input, for training.  The pages implement no backward pass ("mamba-metal: Apple Silicon で
 * Mamba を動かす", section "残り課題", lists the backward kernel for training as still to do); this
 * is the derivative of the forward definition above, evaluated as the reverse (adjoint) recurrence
 * of the same scan:
 *   dŷ_t = dy_t·silu(z_t),  dz_t = dy_t·ŷ_t·silu'(z_t),  λ_t = C_t dŷ_t + exp(Δ_{t+1}A) λ_{t+1}
 *   (dlast joins at t = L-1); dC_t = Σ_d dŷ_t h_t, dB_t = Σ_d λ_t Δ_t u_t, du_t = D dŷ_t +
 *   Σ_n λ_t Δ_t B_t, ddelta_raw_t = sigmoid(r_t) Σ_n λ_t (A exp(Δ_t A) h_{t-1} + B_t u_t),
 *   dA_log = A Σ_{b,t} λ_t Δ_t exp(Δ_t A) h_{t-1}, dD = Σ dŷ_t u_t, ddelta_bias = Σ ddelta_raw,
 *   dh0 = exp(Δ_0 A) λ_0,  with r = delta_raw + delta_bias.
 *   Inputs: those of ss_fwd_h0 (same strides struct; h0 NULL = zeros); dy [batch, L, Dm] io_dtype
 *   contiguous (the gradient of y); dlast [batch, Dm, N] fp32 or NULL (of last_state).
 *   Outputs (caller-owned, written or zeroed by the call):
 *     du, ddelta_raw, dz   [batch, L, Dm] io_dtype contiguous (dz NULL when z is NULL)
 *     dB, dC               [batch, L, N] fp32 contiguous (sums over channels)
 *     dA_log               [Dm, N] fp32
 *     dD, ddelta_bias      [Dm] fp32 or NULL (not computed)
 *     dh0                  [batch, Dm, N] fp32 or NULL
 *   Outputs must not overlap each other or any input.  The sums (dB, dC, dA_log, dD,
 *   ddelta_bias) are accumulated with atomic adds, so their rounding varies from run to run.
 *   workspace          device memory, 256-byte aligned, ss_bwd_workspace_size(...) bytes (the
 *                      state at every 16th step and, for few channel tiles, the time split's
 *                      per-segment entering states, adjoints and Σ Δ); contents need no
 *                      initialisation.  Calls that share it must not overlap on the device.
 * Schedule: one CTA per 32-channel tile over the whole sequence, or, when the tiles alone cannot
 * fill the GPU (e.g. one long sequence), the sequence cut into segments that run side by side:
 * each segment is folded and its adjoint swept from zero, the entering states are composed left
 * to right and the entering adjoints right to left (the carry of the blog's section "チャンク間
 * running prefix", both ways), then every segment runs both passes from them.  Four launches.
 * Errors as ss_fwd.  Returns SS_OK once the work is enqueued.
 */
ss_status ss_bwd(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                 const void* B, const void* C, const float* D, const void* z, const float* h0,
                 const void* dy, const float* dlast, void* du, void* ddelta_raw, void* dz,
                 float* dB, float* dC, float* dA_log, float* dD, float* ddelta_bias, float* dh0,
                 int64_t batch, int64_t L, int64_t Dm, int64_t N, const ss_fwd_strides* strides,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes ss_bwd needs for these sizes on the current device (0: sizes invalid or
 * empty); the time split's share depends on how many CTAs the device holds at once. */
size_t ss_bwd_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N);

/*
 * Forward pass for training: ss_fwd_h0's results and, besides, the checkpoints ss_bwd_ckpt reads
 * instead of refolding the sequence in a first pass of its own.  Schedule: with a workspace
 * (ss_fwd_workspace_size bytes) the balanced one of ss_fwd_ws where it applies (bf16 I/O, or fp32
 * with at least two 32-channel tiles per SM); when the tiles alone cannot fill the GPU, ss_fwd's
 * single-launch cluster split (no workspace used); else one CTA per 32-channel tile at 4 lanes
 * per channel.  The checkpoints are the state entering every 16th step,
 *   ckpt   [batch·ceil(Dm/32)][ceil(L/32)][2][32][16] fp32, device memory, 16-byte aligned,
 *          ss_fwd_ckpt_size(...) bytes; entries past the last step hold the final state.
 * N must be 16 and every tensor must allow TMA-fed tiles (16-byte aligned bases and strides);
 * time-invariant B/C (step stride 0) are not taken: SS_ERR_UNSUPPORTED.  ckpt must not overlap
 * any other argument; the workspace (NULL allowed) as for ss_fwd_ws.  Other arguments, errors and
 * results as ss_fwd_h0.
 */
ss_status ss_fwd_ckpt(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                      const void* B, const void* C, const float* D, const void* z, void* y, float* last_state,
                      const float* h0, float* ckpt, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                      const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of ss_fwd_ckpt's checkpoints (0: sizes invalid, empty, or N other than 16). */
size_t ss_fwd_ckpt_size(int64_t batch, int64_t L, int64_t Dm, int64_t N);

/*
 * ss_bwd with the forward's checkpoints (ss_fwd_ckpt on the same inputs and h0): the backward
 * then skips its own first pass (the forward fold that writes them), one pass over the inputs
 * fewer.  With the time split (few tiles) the checkpoints also hold every segment's entering
 * state: the local launch sweeps only the adjoint and the forward carry is not run (three
 * launches).  ckpt as ss_fwd_ckpt writes it (an input here: it must not overlap an output); N
 * must be 16.  Other arguments, errors and results as ss_bwd.
 */
ss_status ss_bwd_ckpt(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                      const void* B, const void* C, const float* D, const void* z, const float* h0,
                      const float* ckpt, const void* dy, const float* dlast, void* du, void* ddelta_raw,
                      void* dz, float* dB, float* dC, float* dA_log, float* dD, float* ddelta_bias,
                      float* dh0, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                      const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream);

/* Kernel width of the causal convolution (the Mamba blocks of the pages use 4). */
#define SS_CONV_WIDTH 4

/*
 * Element strides of the convolution's [batch, L, Dm] tensors (channel stride 1).  NULL means
 * io_dtype = SS_F32 and both contiguous.
 */
typedef struct {
    int32_t io_dtype;                       /* x and out: SS_F32 or SS_BF16 */
    int64_t x_b, x_l;                       /* x   [batch, L, Dm] */
    int64_t out_b, out_l;                   /* out [batch, L, Dm] */
} ss_conv_strides;

/*
 * Causal depthwise convolution over the sequence, with optional SiLU: the stage before the
 * scan in a Mamba block ("mamba-metal: Apple Silicon で Mamba を動かす", MambaBlock = in_proj ->
 * conv1d -> SiLU -> ...; SpeechLens docs/kernel-optimization.md, MetalCausalConv1d: depthwise,
 * kernel 4, three zero samples on the causal left edge, output length L), with the sliding
 * window that the blog's section "O(L) インクリメンタルデコード" carries across calls:
 *
 *   out[b,t,d] = act( bias[d] + Σ_{k=0..3} weight[d,k] · e[t + k] ),   e = window_in[b,d,:] ++ x[b,:,d]
 *   window_out[b,d,:] = the last three samples of e
 *
 * act is SiLU when silu != 0, the identity otherwise.  The newest sample meets weight[d,3].
 *   x            [batch, L, Dm] io_dtype
 *   weight       [Dm, 4] fp32 contiguous (a [Dm, 1, 4] depthwise Conv1d weight)
 *   bias         [Dm] fp32 or NULL (= 0)
 *   out          [batch, L, Dm] io_dtype; must not overlap any input or window, every element at
 *                its own address (as y of ss_fwd)
 *   window_in    [batch, Dm, 3] fp32 contiguous or NULL (= the zero left padding): the three
 *                samples before t = 0, oldest first
 *   window_out   [batch, Dm, 3] fp32 contiguous or NULL; may be window_in itself (updated in
 *                place: chunked prefill and decode, L = 1, keep one window buffer)
 *   batch <= 65535, L, Dm >= 0; batch == 0 or Dm == 0 is a no-op; L == 0 copies window_in (or
 *   zeros) to window_out.
 * Errors as ss_fwd.  Returns SS_OK once the work is enqueued.
 */
ss_status ss_conv1d(const void* x, const float* weight, const float* bias, void* out,
                    const float* window_in, float* window_out, int64_t batch, int64_t L,
                    int64_t Dm, int32_t silu, const ss_conv_strides* strides, void* stream);

/*
 * Element strides of the decode tensors.  x, delta_raw, z, y are [batch, Dm] with channel
 * stride 1; B, C are [batch, N] with state stride 1; the state is [batch, Dm, N] with
 * state stride 1.  NULL means io_dtype = SS_F32 and all contiguous.
 */
typedef struct {
    int32_t io_dtype;
    int64_t x_b, delta_b, z_b, y_b, B_b, C_b;
    int64_t state_b, state_d;
} ss_step_strides;

/*
 * Single-token decode update (the O(1)-per-token step of "mamba-metal: Apple Silicon で Mamba
 * を動かす", section "O(L) インクリメンタルデコード": the recurrent state is kept and advanced
 * one token at a time instead of re-scanning the prefix; the update itself is the recurrence of
 * section "Selective scan の本質" at one step, with the softplus, skip and gate of ss_fwd):
 *   Δ = softplus(delta_raw[b,d] + delta_bias[d]);
 *   state[b,d,n] <- exp(Δ·A[d,n])·state[b,d,n] + Δ·x[b,d]·B[b,n]   (in place, fp32)
 *   y[b,d] = (Σ_n C[b,n]·state[b,d,n] + D[d]·x[b,d]) · silu(z[b,d])
 * Arguments as for ss_fwd with L = 1 and the initial state given; y must not overlap any
 * input or the state, and y and the state must each give every element its own address.
 * batch == 0 or Dm == 0 is a no-op.
 */
ss_status ss_step(float* state, const void* x, const void* delta_raw, const float* delta_bias,
                  const float* A_log, const void* B, const void* C, const float* D,
                  const void* z, void* y, int64_t batch, int64_t Dm, int64_t N,
                  const ss_step_strides* strides, void* stream);

/*
 * The buffers of one layer for ss_step_layers: the pointer arguments of one ss_step call, same
 * meaning, types and layout.
 */
typedef struct {
    float* state;
    const void* x;
    const void* delta_raw;
    const float* delta_bias;
    const float* A_log;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    void* y;
} ss_step_layer;

/* Most layers one ss_step_layers call takes. */
#define SS_STEP_MAX_LAYERS 128

/*
 * The decode update of many layers in one launch: for each layer l, exactly what
 * ss_step(layers[l].state, layers[l].x, ..., layers[l].y, batch, Dm, N, strides, stream) does
 * ("mamba-metal: Apple Silicon で Mamba を動かす", section "O(L) インクリメンタルデコード": each
 * layer keeps and advances its own recurrent state).  The layers run at the same time, so this
 * serves layers whose inputs are all ready, e.g. independent models or the states of a stack
 * stepped together; a model whose layer l+1 reads layer l's y calls ss_step per layer.
 *   layers       HOST array of n_layers descriptors (read during the call; the pointers in it are
 *                device memory as for ss_step); the table travels in the kernel's parameters,
 *                so the call allocates nothing
 *   n_layers     0..SS_STEP_MAX_LAYERS (0 is a no-op; more returns SS_ERR_UNSUPPORTED)
 *   batch, Dm, N, strides   shared by every layer, as for ss_step
 * Each layer is validated as ss_step validates its arguments; in addition no layer's y or state
 * may overlap another layer's buffers (SS_ERR_INVALID_ARG).  Results are bitwise equal to the
 * n_layers ss_step calls.  Returns SS_OK once the work is enqueued.
 */
ss_status ss_step_layers(const ss_step_layer* layers, int64_t n_layers, int64_t batch, int64_t Dm, int64_t N,
                         const ss_step_strides* strides, void* stream);

/* Static, human-readable name of a status code. */
const char* ss_status_string(ss_status status);

/*
 * Read (and, if `clear` is non-zero, reset) the device error word of the current
 * device: bit 0 = a kernel gave up waiting for a TMA tile; bit 1 = a kernel was launched
 * with a tile geometry other than its own and did nothing.  Either way that call's outputs
 * are invalid.
 * Synchronises with the device.  Returns SS_ERR_CUDA if the word cannot be read.
 */
ss_status ss_device_error(uint32_t* bits, int clear);

/* Library version as 10000*major + 100*minor + patch. */
int ss_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_H */
