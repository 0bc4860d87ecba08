// Forward pass on host-resident tensors: the work is cut into units of a group of batch rows and
// a piece of the sequence, and each unit's inputs are copied to the device, scanned and its
// outputs copied back on three streams, so that the copies of one unit overlap the copies and
// the scan of the others.  The pieces of a row group run in order, each from the state the
// previous piece left (ss_fwd_h0 with the state updated in place on the device), so units can be
// small: the copy in of the first unit and the copy back of the last, which nothing overlaps, are
// short.  (Copies in on two streams, two units at once, measured slower: 2.24 against 1.87 ms on
// the 130m-shaped layer.)
// Every step of the scan itself is ss_fwd_h0 (selscan_api.cu) on the device copies.
//
// The three streams and their events are created once per device (per CUDA context, on its
// first call) and kept for the life of the process.  Calls on one device enqueue their work one
// at a time (a mutex held while enqueueing, not while the GPU runs it), so a call's waits always
// see its own event records; the GPU work of concurrent calls is then ordered on the shared
// streams.  Ordering: the work starts after everything already enqueued on the caller's stream,
// and the caller's stream waits for the last copy back, so synchronising it makes y and
// last_state valid on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/selscan.h"
#include "host_util.h"
#include "internal.h"

namespace selscan {
namespace {

constexpr int kSlots = 2;          // device staging slots (double buffering)
constexpr int kGroups = 8;         // row groups of ceil(batch / kGroups) rows (8 measured 2% faster than 4)
// A unit's pieces of the sequence: steps for about this many input bytes (whole 64-step chunks).
constexpr int64_t kUnitBytes = int64_t(64) << 20;

// Test hook: steps per piece (0: chosen from kUnitBytes).
std::atomic<int64_t> g_force_host_steps{0};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Staging layout of one slot, of the carried state and of the parameter block, in bytes.
struct HostPlan {
    int64_t rows;                  // batch rows per group
    int64_t groups;
    int64_t steps;                 // steps per piece of the sequence
    int64_t pieces;
    size_t x_bytes, bc_bytes, last_bytes;   // per row: one [steps, Dm] stream, one [steps, N], one [Dm, N] fp32
    size_t slot_bytes;             // u, delta, z, y, B, C of `rows` rows and `steps` steps
    size_t state_bytes;            // [batch, Dm, N] fp32: each row group's state between its pieces
    size_t param_bytes;            // A_log, D, delta_bias
    size_t total;
};

HostPlan host_plan(int64_t batch, int64_t L, int64_t Dm, int64_t N, int64_t es) {
    HostPlan h;
    h.rows = std::max<int64_t>(1, (batch + kGroups - 1) / kGroups);
    h.groups = (batch + h.rows - 1) / h.rows;
    const int64_t per_step = h.rows * (3 * Dm + 2 * N) * es;      // input bytes of one step of a group
    const int64_t forced = g_force_host_steps.load();
    int64_t steps = forced > 0 ? forced : std::max<int64_t>(64, kUnitBytes / std::max<int64_t>(per_step, 1) / 64 * 64);
    h.steps = std::min<int64_t>(steps, L);
    h.pieces = (L + h.steps - 1) / h.steps;
    h.x_bytes = static_cast<size_t>(h.steps * Dm * es);
    h.bc_bytes = static_cast<size_t>(h.steps * N * es);
    h.last_bytes = static_cast<size_t>(Dm * N * 4);
    h.slot_bytes = 4 * up256(h.rows * h.x_bytes) + 2 * up256(h.rows * h.bc_bytes);
    h.state_bytes = up256(static_cast<size_t>(batch) * h.last_bytes);
    h.param_bytes = up256(static_cast<size_t>(Dm * N * 4)) + 2 * up256(static_cast<size_t>(Dm * 4));
    h.total = kSlots * h.slot_bytes + h.state_bytes + h.param_bytes;
    return h;
}

bool host_ptr(const void* q) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

// Streams and events of the copy / scan / copy-back pipeline of one device.
struct Pipeline {
    cudaStream_t s_in = nullptr, s_c = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, params = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
    bool ok = true;
    Pipeline() {
        auto st = [&](cudaStream_t* s) { ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess; };
        auto ev = [&](cudaEvent_t* e) { ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
        st(&s_in); st(&s_c); st(&s_out);
        ev(&start); ev(&params);
        for (int i = 0; i < kSlots; ++i) { ev(&in_done[i]); ev(&comp_done[i]); ev(&out_done[i]); }
    }
    ~Pipeline() {
        for (cudaEvent_t e : {start, params}) if (e) cudaEventDestroy(e);
        for (int i = 0; i < kSlots; ++i)
            for (cudaEvent_t e : {in_done[i], comp_done[i], out_done[i]}) if (e) cudaEventDestroy(e);
        for (cudaStream_t s : {s_in, s_c, s_out}) if (s) cudaStreamDestroy(s);
    }
};

// One pipeline per device, made on the device's first call in a context and remade when the
// context changes (the old handles belonged to a context that is gone and are not touched).
struct PipelineSlot {
    std::mutex mu;
    CUcontext ctx = nullptr;
    Pipeline* pl = nullptr;
};
PipelineSlot g_pipelines[64];

}  // namespace
}  // namespace selscan

using namespace selscan;
using namespace selscan::host;

extern "C" int64_t ss__force_host_steps(int64_t steps) { return g_force_host_steps.exchange(steps > 0 ? steps : 0); }

extern "C" size_t ss_fwd_host_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype) {
    if (batch <= 0 || L <= 0 || Dm <= 0 || N < 1 || N > 16) return 0;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return 0;
    return host_plan(batch, L, Dm, N, io_dtype == SS_BF16 ? 2 : 4).total;
}

extern "C" ss_status ss_fwd_host(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                                 const void* B, const void* C, const float* D, const void* z, void* y,
                                 float* last_state, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                                 int32_t io_dtype, void* workspace, size_t workspace_bytes, void* stream_ptr) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (batch < 0 || L < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return SS_ERR_INVALID_ARG;
    if (batch == 0 || Dm == 0 || L == 0) {
        if (L == 0 && batch > 0 && Dm > 0 && last_state) {
            // no steps: the zero state, written by the host once the stream's earlier work is done
            if (!host_ptr(last_state)) return SS_ERR_INVALID_ARG;
            if (cudaStreamSynchronize(stream) != cudaSuccess) return SS_ERR_CUDA;
            std::memset(last_state, 0, sizeof(float) * batch * Dm * N);
        }
        return SS_OK;
    }
    if (!u || !delta_raw || !A_log || !B || !C || !y) return SS_ERR_INVALID_ARG;
    const int64_t es = io_dtype == SS_BF16 ? 2 : 4;
    const void* io_ptrs[] = {u, delta_raw, B, C, z, y};
    for (const void* q : io_ptrs)
        if (q && !is_aligned(q, es)) return SS_ERR_MISALIGNED;
    const void* f_ptrs[] = {A_log, D, delta_bias, last_state};
    for (const void* q : f_ptrs)
        if (q && !is_aligned(q, 4)) return SS_ERR_MISALIGNED;
    const void* hosts[] = {u, delta_raw, B, C, z, y, A_log, D, delta_bias, last_state};
    for (const void* q : hosts)
        if (q && !host_ptr(q)) return SS_ERR_INVALID_ARG;
    // outputs disjoint from the inputs and each other
    const Range ry = range3(y, 1, batch, L * Dm, 0, L * Dm, es);
    const Range rl = range3(last_state, 1, batch, Dm * N, 0, Dm * N, 4);
    const Range ins[] = {range3(u, 1, batch, L * Dm, 0, L * Dm, es), range3(delta_raw, 1, batch, L * Dm, 0, L * Dm, es),
                         range3(z, 1, batch, L * Dm, 0, L * Dm, es), range3(B, 1, batch, L * N, 0, L * N, es),
                         range3(C, 1, batch, L * N, 0, L * N, es), range3(A_log, 1, 1, Dm * N, 0, 0, 4),
                         range3(D, 1, 1, Dm, 0, 0, 4), range3(delta_bias, 1, 1, Dm, 0, 0, 4)};
    for (const Range& r : ins)
        if (meet(ry, r) || meet(rl, r)) return SS_ERR_INVALID_ARG;
    if (meet(ry, rl)) return SS_ERR_INVALID_ARG;
    const HostPlan h = host_plan(batch, L, Dm, N, es);
    if (!workspace || workspace_bytes < h.total) return SS_ERR_INVALID_ARG;
    if (!is_aligned(workspace, 256)) return SS_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (!dev_ptr(workspace, dev)) return SS_ERR_INVALID_ARG;

    // staging: the parameter block, the carried state, then kSlots slots
    char* ws = static_cast<char*>(workspace);
    float* d_Alog = reinterpret_cast<float*>(ws);
    float* d_D = reinterpret_cast<float*>(ws + up256(static_cast<size_t>(Dm * N * 4)));
    float* d_bias = reinterpret_cast<float*>(ws + up256(static_cast<size_t>(Dm * N * 4)) + up256(static_cast<size_t>(Dm * 4)));
    float* d_state = reinterpret_cast<float*>(ws + h.param_bytes);
    struct Slot { char *u, *d, *z, *y, *B, *C; };
    Slot slot[kSlots];
    for (int i = 0; i < kSlots; ++i) {
        char* base = ws + h.param_bytes + h.state_bytes + i * h.slot_bytes;
        const size_t xs = up256(h.rows * h.x_bytes), bs = up256(h.rows * h.bc_bytes);
        slot[i].u = base;
        slot[i].d = base + xs;
        slot[i].z = base + 2 * xs;
        slot[i].y = base + 3 * xs;
        slot[i].B = base + 4 * xs;
        slot[i].C = base + 4 * xs + bs;
    }

    if (dev < 0 || dev >= 64) return SS_ERR_UNSUPPORTED;
    PipelineSlot& slot_of_dev = g_pipelines[dev];
    std::lock_guard<std::mutex> lock(slot_of_dev.mu);
    const CUcontext cur = current_context();
    if (!slot_of_dev.pl || slot_of_dev.ctx != cur) {
        Pipeline* fresh = new Pipeline();
        if (!fresh->ok) {
            delete fresh;
            return SS_ERR_CUDA;
        }
        slot_of_dev.pl = fresh;
        slot_of_dev.ctx = current_context();
    }
    Pipeline& pl = *slot_of_dev.pl;
    auto chk = [](cudaError_t e) { return e == cudaSuccess; };
    // `nr` rows of `width` bytes, `src_pitch` apart in the source and `dst_pitch` in the destination
    auto copy_rows = [&](cudaStream_t q, void* dst, size_t dst_pitch, const void* src, size_t src_pitch, size_t width,
                         int64_t nr, cudaMemcpyKind kind) {
        if (nr == 1 || (dst_pitch == width && src_pitch == width))
            return chk(cudaMemcpyAsync(dst, src, width * nr, kind, q));
        return chk(cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, width, static_cast<size_t>(nr), kind, q));
    };
    bool ok = chk(cudaEventRecord(pl.start, stream)) && chk(cudaStreamWaitEvent(pl.s_in, pl.start, 0)) &&
              chk(cudaStreamWaitEvent(pl.s_c, pl.start, 0)) && chk(cudaStreamWaitEvent(pl.s_out, pl.start, 0));
    cudaStream_t s0 = pl.s_in;
    auto h2d_flat = [&](void* dst, const void* src, size_t n) {
        return chk(cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s0));
    };
    ok = ok && h2d_flat(d_Alog, A_log, sizeof(float) * Dm * N) && (!D || h2d_flat(d_D, D, sizeof(float) * Dm)) &&
         (!delta_bias || h2d_flat(d_bias, delta_bias, sizeof(float) * Dm)) && chk(cudaEventRecord(pl.params, s0)) &&
         chk(cudaStreamWaitEvent(pl.s_c, pl.params, 0));
    ss_status st = SS_OK;
    const size_t row_x = static_cast<size_t>(L * Dm * es), row_bc = static_cast<size_t>(L * N * es);
    int64_t unit = 0;
    for (int64_t g = 0; ok && st == SS_OK && g < h.groups; ++g) {
        const int64_t r0 = g * h.rows, nr = std::min<int64_t>(h.rows, batch - r0);
        float* state = d_state + r0 * Dm * N;
        for (int64_t piece = 0; ok && st == SS_OK && piece < h.pieces; ++piece, ++unit) {
            const int k = static_cast<int>(unit % kSlots);
            const int64_t t0 = piece * h.steps, nt = std::min<int64_t>(h.steps, L - t0);
            const Slot& s = slot[k];
            const size_t wx = static_cast<size_t>(nt * Dm * es), wbc = static_cast<size_t>(nt * N * es);
            const size_t ox = static_cast<size_t>(t0 * Dm * es), obc = static_cast<size_t>(t0 * N * es);
            // copy in, once the scan that last read this slot is done
            cudaStream_t si = pl.s_in;
            auto in = [&](char* dst, const void* src, size_t row, size_t off, size_t w) {
                return copy_rows(si, dst, w, static_cast<const char*>(src) + r0 * row + off, row, w, nr,
                                 cudaMemcpyHostToDevice);
            };
            if (unit >= kSlots) ok = ok && chk(cudaStreamWaitEvent(si, pl.comp_done[k], 0));
            ok = ok && in(s.u, u, row_x, ox, wx) && in(s.d, delta_raw, row_x, ox, wx) &&
                 (!z || in(s.z, z, row_x, ox, wx)) && in(s.B, B, row_bc, obc, wbc) && in(s.C, C, row_bc, obc, wbc) &&
                 chk(cudaEventRecord(pl.in_done[k], si));
            // scan, once the inputs are in and the copy back of this slot's last outputs is done;
            // from the state the previous piece left (zeros before the first)
            ok = ok && chk(cudaStreamWaitEvent(pl.s_c, pl.in_done[k], 0));
            if (unit >= kSlots) ok = ok && chk(cudaStreamWaitEvent(pl.s_c, pl.out_done[k], 0));
            if (!ok) break;
            ss_fwd_strides fs;
            std::memset(&fs, 0, sizeof(fs));
            fs.io_dtype = io_dtype;
            fs.u_b = fs.delta_b = fs.z_b = fs.y_b = nt * Dm;
            fs.u_l = fs.delta_l = fs.z_l = fs.y_l = Dm;
            fs.B_b = fs.C_b = nt * N;
            fs.B_l = fs.C_l = N;
            st = ss_fwd_h0(s.u, s.d, delta_bias ? d_bias : nullptr, d_Alog, s.B, s.C, D ? d_D : nullptr,
                           z ? s.z : nullptr, s.y, state, piece > 0 ? state : nullptr, nr, nt, Dm, N, &fs, nullptr, 0,
                           pl.s_c);
            ok = ok && st == SS_OK && chk(cudaEventRecord(pl.comp_done[k], pl.s_c));
            // copy back (the last piece's state too)
            const bool last_piece = piece + 1 == h.pieces;
            ok = ok && chk(cudaStreamWaitEvent(pl.s_out, pl.comp_done[k], 0)) &&
                 copy_rows(pl.s_out, static_cast<char*>(y) + r0 * row_x + ox, row_x, s.y, wx, wx, nr,
                           cudaMemcpyDeviceToHost) &&
                 (!last_state || !last_piece ||
                  chk(cudaMemcpyAsync(reinterpret_cast<char*>(last_state) + r0 * h.last_bytes, state, nr * h.last_bytes,
                                      cudaMemcpyDeviceToHost, pl.s_out))) &&
                 chk(cudaEventRecord(pl.out_done[k], pl.s_out));
        }
    }
    // the caller's stream continues after everything enqueued here (also after a failure part
    // way, so that no copy is left running unordered)
    bool joined = true;
    for (cudaStream_t q : {pl.s_in, pl.s_c, pl.s_out}) {
        joined = joined && chk(cudaEventRecord(pl.start, q)) && chk(cudaStreamWaitEvent(stream, pl.start, 0));
    }
    if (st != SS_OK) return st;
    return ok && joined ? SS_OK : SS_ERR_CUDA;
}
