// Forward pass on host-resident tensors: the batch rows are processed in groups, and each
// group's inputs are copied to the device, scanned and its outputs copied back on three
// streams, so that the copies of one group overlap the copies and the scan of the others.
// (Copies in on two streams, two groups at once, measured slower: 2.24 against 1.87 ms on the
// 130m-shaped layer.)
// Every step of the scan itself is ss_fwd (selscan_api.cu) on the device copies.
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

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Staging layout of one slot and of the parameter block, in bytes.
struct HostPlan {
    int64_t rows;                  // batch rows per group
    int64_t groups;
    size_t x_bytes, bc_bytes, last_bytes;   // per row: one [L, Dm] stream, one [L, N], one [Dm, N] fp32
    size_t slot_bytes;             // u, delta, z, y, B, C, last_state of `rows` rows
    size_t param_bytes;            // A_log, D, delta_bias
    size_t total;
};

HostPlan host_plan(int64_t batch, int64_t L, int64_t Dm, int64_t N, int64_t es) {
    HostPlan h;
    h.rows = std::max<int64_t>(1, (batch + kGroups - 1) / kGroups);
    h.groups = (batch + h.rows - 1) / h.rows;
    h.x_bytes = static_cast<size_t>(L * Dm * es);
    h.bc_bytes = static_cast<size_t>(L * N * es);
    h.last_bytes = static_cast<size_t>(Dm * N * 4);
    h.slot_bytes = 4 * up256(h.rows * h.x_bytes) + 2 * up256(h.rows * h.bc_bytes) + up256(h.rows * h.last_bytes);
    h.param_bytes = up256(static_cast<size_t>(Dm * N * 4)) + 2 * up256(static_cast<size_t>(Dm * 4));
    h.total = kSlots * h.slot_bytes + h.param_bytes;
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

    // staging: the parameter block, then kSlots slots
    char* ws = static_cast<char*>(workspace);
    float* d_Alog = reinterpret_cast<float*>(ws);
    float* d_D = reinterpret_cast<float*>(ws + up256(static_cast<size_t>(Dm * N * 4)));
    float* d_bias = reinterpret_cast<float*>(ws + up256(static_cast<size_t>(Dm * N * 4)) + up256(static_cast<size_t>(Dm * 4)));
    struct Slot { char *u, *d, *z, *y, *B, *C; float* last; };
    Slot slot[kSlots];
    for (int i = 0; i < kSlots; ++i) {
        char* base = ws + h.param_bytes + i * h.slot_bytes;
        const size_t xs = up256(h.rows * h.x_bytes), bs = up256(h.rows * h.bc_bytes);
        slot[i].u = base;
        slot[i].d = base + xs;
        slot[i].z = base + 2 * xs;
        slot[i].y = base + 3 * xs;
        slot[i].B = base + 4 * xs;
        slot[i].C = base + 4 * xs + bs;
        slot[i].last = reinterpret_cast<float*>(base + 4 * xs + 2 * bs);
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
    auto h2d_on = [&](cudaStream_t q, void* dst, const void* src, size_t n) {
        return chk(cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, q));
    };
    auto d2h = [&](void* dst, const void* src, size_t n) { return chk(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, pl.s_out)); };
    bool ok = chk(cudaEventRecord(pl.start, stream)) && chk(cudaStreamWaitEvent(pl.s_in, pl.start, 0)) &&
              chk(cudaStreamWaitEvent(pl.s_c, pl.start, 0)) && chk(cudaStreamWaitEvent(pl.s_out, pl.start, 0));
    cudaStream_t s0 = pl.s_in;
    ok = ok && h2d_on(s0, d_Alog, A_log, sizeof(float) * Dm * N) && (!D || h2d_on(s0, d_D, D, sizeof(float) * Dm)) &&
         (!delta_bias || h2d_on(s0, d_bias, delta_bias, sizeof(float) * Dm)) && chk(cudaEventRecord(pl.params, s0)) &&
         chk(cudaStreamWaitEvent(pl.s_c, pl.params, 0));
    ss_status st = SS_OK;
    for (int64_t g = 0; ok && st == SS_OK && g < h.groups; ++g) {
        const int k = static_cast<int>(g % kSlots);
        const int64_t r0 = g * h.rows, nr = std::min<int64_t>(h.rows, batch - r0);
        const Slot& s = slot[k];
        // copy in, once the scan that last read this slot is done
        cudaStream_t si = pl.s_in;
        auto h2d = [&](void* dst, const void* src, size_t n) { return h2d_on(si, dst, src, n); };
        if (g >= kSlots) ok = ok && chk(cudaStreamWaitEvent(si, pl.comp_done[k], 0));
        const char* hu = static_cast<const char*>(u) + r0 * h.x_bytes;
        const char* hd = static_cast<const char*>(delta_raw) + r0 * h.x_bytes;
        ok = ok && h2d(s.u, hu, nr * h.x_bytes) && h2d(s.d, hd, nr * h.x_bytes) &&
             (!z || h2d(s.z, static_cast<const char*>(z) + r0 * h.x_bytes, nr * h.x_bytes)) &&
             h2d(s.B, static_cast<const char*>(B) + r0 * h.bc_bytes, nr * h.bc_bytes) &&
             h2d(s.C, static_cast<const char*>(C) + r0 * h.bc_bytes, nr * h.bc_bytes) &&
             chk(cudaEventRecord(pl.in_done[k], si));
        // scan, once the inputs are in and the copy back of this slot's last outputs is done
        ok = ok && chk(cudaStreamWaitEvent(pl.s_c, pl.in_done[k], 0));
        if (g >= kSlots) ok = ok && chk(cudaStreamWaitEvent(pl.s_c, pl.out_done[k], 0));
        if (!ok) break;
        ss_fwd_strides fs;
        std::memset(&fs, 0, sizeof(fs));
        fs.io_dtype = io_dtype;
        fs.u_b = fs.delta_b = fs.z_b = fs.y_b = L * Dm;
        fs.u_l = fs.delta_l = fs.z_l = fs.y_l = Dm;
        fs.B_b = fs.C_b = L * N;
        fs.B_l = fs.C_l = N;
        st = ss_fwd(s.u, s.d, delta_bias ? d_bias : nullptr, d_Alog, s.B, s.C, D ? d_D : nullptr, z ? s.z : nullptr,
                    s.y, last_state ? s.last : nullptr, nr, L, Dm, N, &fs, pl.s_c);
        ok = ok && st == SS_OK && chk(cudaEventRecord(pl.comp_done[k], pl.s_c));
        // copy back
        ok = ok && chk(cudaStreamWaitEvent(pl.s_out, pl.comp_done[k], 0)) &&
             d2h(static_cast<char*>(y) + r0 * h.x_bytes, s.y, nr * h.x_bytes) &&
             (!last_state || d2h(reinterpret_cast<char*>(last_state) + r0 * h.last_bytes, s.last, nr * h.last_bytes)) &&
             chk(cudaEventRecord(pl.out_done[k], pl.s_out));
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
