// libselscan C ABI: host-side validation, TMA descriptor construction and kernel dispatch.
// Declarations and the full contract are in include/selscan.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/selscan.h"
#include "host_util.h"
#include "internal.h"

namespace selscan {

__device__ unsigned int g_device_error;

// Workspace of ss_fwd_static: a fixed array in the library's device image, so that callers
// that cannot allocate device memory can still run the balanced schedule.  Every device that
// loads the library holds these SS_STATIC_WORKSPACE_BYTES until the process exits.  It needs
// no clearing: each call tags its hand-overs with a fresh call number, so flags left by
// earlier calls never match.  All calls on a device share it.
static __device__ __align__(256) unsigned char g_static_ws[SS_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kVersion = 100;   // 0.1.0

// Test hook overriding the automatic choice of forward kernel: family (-1 auto, 0 state-split
// lane, 1 segment-lane, 2 the lane family's single-launch cluster split where it applies: no
// workspace, TMA-fed, 16 states), lanes per channel of the lane family (0 auto, 1, 2 or 4) and tile fill
// (-1 auto, 0 plain loads, 1 TMA; a forced choice the arguments cannot use is
// SS_ERR_UNSUPPORTED).
std::atomic<int> g_force_family{-1}, g_force_lpc{0}, g_force_tma{-1};
// Test hook: 0 runs ss_fwd_ws with the one-CTA-per-tile schedule (workspace unused).
std::atomic<int> g_force_balanced{1};
// Test hook on the time-split schedule: -1 automatic (with a workspace, for shapes with too
// few channel tiles to fill the GPU), 0 never, n >= 2 always with up to n segments.
std::atomic<int> g_force_nseg{-1};
// Test hook: steps per chunk of the lane kernel (0: its own 64; 16, 32 or 256: the test
// instantiations of one configuration, per tile, which take no workspace schedule).
std::atomic<int> g_force_chunk{0};
// Test hook on the cluster-balanced schedule of ss_fwd without a workspace: -1 automatic (when one
// CTA per tile would need more than one wave), 0 never, 2..8 always where it applies, with
// clusters of that many CTAs.
std::atomic<int> g_force_cbal{-1};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// The calling thread's current CUDA context, through the runtime's driver entry point (the
// library does not link libcuda); nullptr if it cannot be had.
CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    CUcontext c = nullptr;
    if (fn) fn(&c);
    return c;
}

namespace {

// Device address of a __device__ symbol, looked up with the device current and cached per device
// and context: in host code the symbol's name is only a host-side handle, and a context that is
// torn down and created again (cudaDeviceReset) loads the module afresh, at a new address.
// nullptr if the lookup fails.
template <class Sym>
void* symbol_address(const Sym& sym, std::mutex& mu, CUcontext (&ctx)[64], void* (&addr)[64]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    const CUcontext cur = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] && cur && ctx[dev] == cur) return addr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, sym) != cudaSuccess) {   // creates the context if there is none yet
        cudaGetLastError();
        return nullptr;
    }
    ctx[dev] = current_context();
    addr[dev] = p;
    return p;
}

unsigned int* device_error_ptr() {
    static std::mutex mu;
    static CUcontext ctx[64] = {};
    static void* addr[64] = {};
    return static_cast<unsigned int*>(symbol_address(g_device_error, mu, ctx, addr));
}

// Device address of g_static_ws on the current device and context.
void* static_workspace_ptr() {
    static std::mutex mu;
    static CUcontext ctx[64] = {};
    static void* addr[64] = {};
    return symbol_address(g_static_ws, mu, ctx, addr);
}

// Argument checks shared with the other entry points (host_util.h).
using host::Range;
inline bool is_device_pointer(const void* p, int dev) { return host::dev_ptr(p, dev); }
inline bool aligned(const void* p, size_t a) { return host::is_aligned(p, a); }
inline Range span3(const void* p, int64_t n0, int64_t n1, int64_t n2, int64_t s0, int64_t s1, int64_t es) {
    return host::range3(p, n0, n1, n2, s0, s1, es);
}
inline bool overlap(const Range& a, const Range& b) { return host::meet(a, b); }

ss_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SS_OK : SS_ERR_CUDA; }

// 3-D tiled descriptor over a [batch, rows, cols] tensor (cols contiguous) with a box of
// [1, box_rows, box_cols]; rows/channels past the end read as zero.  L2 promotion is 128 bytes:
// 256-byte promotion fetched lines of neighbouring tiles early and re-read them (measured).
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t cols, int64_t rows,
              int64_t batch, int64_t row_stride, int64_t batch_stride, int box_cols, int box_rows,
              bool swizzle) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int64_t es = bf16 ? 2 : 4;
    const int row_bytes = box_cols * static_cast<int>(es);
    CUtensorMapSwizzle sw = !swizzle         ? CU_TENSOR_MAP_SWIZZLE_NONE
                          : row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                          : row_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                             : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (batch <= 1) batch_stride = rows * row_stride;   // any valid stride; never stepped
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride * es),
                             static_cast<cuuint64_t>(batch_stride * es)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Automatic forward-kernel choice (see ss_fwd).
FwdVariant choose_fwd_variant(int64_t batch, int64_t Dm, int64_t N) {
    const int64_t tiles32 = batch * ((Dm + 31) / 32);
    const int64_t want_warps = 1216;   // ~8 warps on each of GB300's 152 SMs
    FwdVariant v;
    v.ns = N <= 4 ? 4 : N <= 8 ? 8 : 16;
    const int max_lpc = v.ns / 4;
    v.lpc = 1;
    while (v.lpc < max_lpc && tiles32 * v.lpc < want_warps) v.lpc *= 2;
    v.family = tiles32 * v.lpc >= want_warps / 2 ? kFamLane : kFamSeg;
    v.tma = true;
    v.balanced = false;
    v.state_only = false;
    v.lti = false;
    v.dtp = false;
    return v;
}

// Lanes per channel for the one-CTA-per-tile schedule: more warps pay there (the 2.8b-shaped
// bf16 layer ran 993 us at 4 lanes against 1027 us at 2), so LPC doubles until about 16 warps
// per SM (2432) rather than 8.  The balanced schedule keeps choose_fwd_variant's choice (at 4
// lanes it measured 995 against 947 us).
int per_tile_lpc(int64_t batch, int64_t Dm, int ns) {
    const int64_t tiles32 = batch * ((Dm + 31) / 32);
    int lpc = 1;
    while (lpc < ns / 4 && tiles32 * lpc < 2432) lpc *= 2;
    return lpc;
}

bool tma_stride_ok(int64_t stride_elems, int64_t es) {
    return stride_elems > 0 && (stride_elems * es) % 16 == 0 && stride_elems * es < (int64_t(1) << 40);
}

}  // namespace

bool make_tile_map(CUtensorMap* m, const void* base, bool bf16, int64_t cols, int64_t rows, int64_t batch,
                   int64_t row_stride, int64_t batch_stride, int box_cols, int box_rows) {
    const int64_t es = bf16 ? 2 : 4;
    return tma_stride_ok(row_stride, es) && (batch <= 1 || tma_stride_ok(batch_stride, es)) &&
           reinterpret_cast<uintptr_t>(base) % 16 == 0 &&
           make_map(m, base, bf16, cols, rows, batch, row_stride, batch_stride, box_cols, box_rows, false);
}

unsigned int* device_error_word() { return device_error_ptr(); }

}  // namespace selscan

using namespace selscan;

extern "C" {

const char* ss_status_string(ss_status s) {
    switch (s) {
        case SS_OK: return "SS_OK";
        case SS_ERR_INVALID_ARG: return "SS_ERR_INVALID_ARG: invalid argument";
        case SS_ERR_UNSUPPORTED: return "SS_ERR_UNSUPPORTED: unsupported size or configuration";
        case SS_ERR_MISALIGNED: return "SS_ERR_MISALIGNED: pointer not aligned to its element type";
        case SS_ERR_CUDA: return "SS_ERR_CUDA: CUDA call or kernel launch failed";
    }
    return "unknown ss_status";
}

int ss_version(void) { return kVersion; }

ss_status ss_device_error(uint32_t* bits, int clear) {
    if (!bits) return SS_ERR_INVALID_ARG;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return SS_ERR_CUDA;
    *bits = v;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return SS_ERR_CUDA;
    }
    return SS_OK;
}

// Internal reporting hook (not part of the public header): the forward kernel ss_fwd would
// launch for these sizes, as "<family>-<lanes>" ("lane-4", "seg-0"), forced choices included.
const char* ss__fwd_kernel_name(int64_t batch, int64_t Dm, int64_t N) {
    if (N < 1 || N > 16) return "unsupported";
    FwdVariant v = choose_fwd_variant(batch, Dm, N);
    if (g_force_family.load() >= 0) v.family = g_force_family.load() == 2 ? kFamSeg : g_force_family.load();
    if (g_force_lpc.load() > 0)
        v.lpc = g_force_lpc.load();
    else if (v.family == kFamLane)
        v.lpc = per_tile_lpc(batch, Dm, v.ns);
    if (v.family == kFamSeg) return "ss_fwd_seg_kernel";
    return v.lpc == 1 ? "ss_fwd_lane_kernel(lpc=1)" : v.lpc == 2 ? "ss_fwd_lane_kernel(lpc=2)"
                                                               : "ss_fwd_lane_kernel(lpc=4)";
}

// Internal test hook (see g_force_chunk): 0 restores the kernels' own chunk length; returns the
// previous setting, or -1 for a length without a test instantiation.
int ss__force_chunk_steps(int steps) {
    if (steps != 0 && steps != 16 && steps != 32 && steps != 256) return -1;
    return g_force_chunk.exchange(steps);
}

// Internal test hook: 0 keeps ss_fwd_ws on the one-CTA-per-tile schedule; 1 (default) lets it
// use the balanced schedule.
int ss__force_balanced(int on) { return g_force_balanced.exchange(on ? 1 : 0); }

// Internal test hook (see g_force_nseg); returns the previous setting.
int ss__force_nseg(int n) { return g_force_nseg.exchange(n < 0 ? -1 : n == 1 ? 0 : n); }

// Internal test hook (see g_force_cbal): -1 automatic, 0 never, 2..8 always with that cluster size;
// returns the previous setting, or -2 for a value it does not take.
int ss__force_cbal(int s) {
    if (s < -1 || s == 1 || s > 8) return -2;
    return g_force_cbal.exchange(s);
}

// Internal test hook (not part of the public header); see g_force_family.
int ss__force_fwd_variant(int family, int lpc, int tma) {
    if (family < -1 || family > 2 || (lpc != 0 && lpc != 1 && lpc != 2 && lpc != 4) || tma < -1 || tma > 1)
        return -1;
    g_force_family.store(family);
    g_force_lpc.store(lpc);
    g_force_tma.store(tma);
    return 0;
}

}  // extern "C"

namespace selscan {
namespace {

std::atomic<unsigned int> g_epoch{0};

unsigned int next_epoch() {
    unsigned int e;
    do {
        e = g_epoch.fetch_add(1) + 1;
    } while (e == 0);
    return e;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace bytes of the balanced schedule for `grid` CTAs of tile width w and ns states.
size_t balanced_ws_bytes(int grid, int w, int ns) {
    return align_up(static_cast<size_t>(grid) * 4, 256) + static_cast<size_t>(grid) * w * ns * 4;
}

// Time-split schedule sizes.  Workspace: the per-segment state slots [nseg][rows·N] fp32,
// then the per-segment Σ Δ [nseg - 1][rows] fp32.
struct SplitPlan {
    int nseg = 0;        // 0: the schedule does not apply
    int seg_chunks = 0;
    size_t bytes = 0;
    size_t off_dsum = 0;
};

size_t split_slot_bytes(int nseg, int64_t rows, int64_t N) {
    return align_up(static_cast<size_t>(nseg) * rows * N * 4, 256);
}

// As many segments as fill the GPU once (tiles × segments <= the CTAs resident together),
// or the forced count; at most one per chunk and 64; fewer if ws_bytes cannot hold them.
SplitPlan split_plan(int64_t tiles_total, int nchunks, int64_t rows, int64_t N, int max_grid,
                     size_t ws_bytes, int forced) {
    SplitPlan pl;
    int64_t want = forced >= 2 ? forced : (tiles_total > 0 ? max_grid / tiles_total : 0);
    want = std::min<int64_t>(std::min<int64_t>(want, nchunks), 64);
    auto bytes = [&](int64_t ns) {
        return split_slot_bytes(static_cast<int>(ns), rows, N) + static_cast<size_t>(ns - 1) * rows * 4;
    };
    while (want >= 2 && bytes(want) > ws_bytes) --want;
    if (want < 2) return pl;
    const int seg_chunks = static_cast<int>((nchunks + want - 1) / want);
    const int nseg = (nchunks + seg_chunks - 1) / seg_chunks;
    if (nseg < 2) return pl;
    pl.nseg = nseg;
    pl.seg_chunks = seg_chunks;
    pl.bytes = bytes(nseg);
    pl.off_dsum = split_slot_bytes(nseg, rows, N);
    return pl;
}

// Grid of the balanced schedule: a whole number of CTAs per SM when there are at least as many
// tiles as SMs, so that every SM gets the same share of the work; never more CTAs than tiles
// (a range must not lie inside one tile) or than fit on the GPU at once (cooperative launch).
int64_t balanced_grid(int64_t tiles_total, int max_grid) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
        const int64_t k = std::min<int64_t>(max_grid / sms, tiles_total / sms);
        if (k >= 1) return k * sms;
    }
    return std::min<int64_t>(tiles_total, max_grid);
}

// fp32 balanced schedule on 32-channel tiles (the per-tile kernel, run balanced) when those tiles
// alone give two CTAs per SM; else 16-channel tiles, twice as many.
bool balanced_w32(int64_t batch, int64_t Dm, int es) {
    if (es != 4) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return false;
    return batch * ((Dm + 31) / 32) >= 2 * static_cast<int64_t>(sms);
}

// The balanced 32-channel fp32 schedule at 4 lanes per channel hands (Δ, Δ·u) over through shared
// memory (the DX4 instantiation, two CTAs per SM) when the grid is two CTAs per SM anyway (fewer
// than three tiles per SM); with more tiles the shuffle form keeps three CTAs per SM.
cudaError_t lane_max_grid(const FwdVariant& v, bool bf16, int* out);

// Cluster-balanced plan for tiles_total channel tiles of nch chunks: the cluster size S (8, 4 or
// 2; force_s > 0: that one), the CTAs per SM K and the cluster count Q.  As in the balanced
// schedule the grid is a whole number K of CTAs per SM (the CTAs an SM holds, at most tiles / SMs;
// fewer tiles than SMs: one) with the shared memory padded so that no SM takes more; Q is at most
// the clusters that then fit at once (a cluster stays within one GPC, so large clusters can leave
// SMs idle) and at most tiles / S, so that every CTA's range spans at least one tile.  Of the sizes
// that fit, the one with the fewest (tile, chunk) units on the busiest CTA,
// ceil(ceil(tiles / Q) · nch / S).  False when none fits.
bool cbal_plan(bool bf16, int lpc, int64_t tiles_total, int64_t nch, int force_s, int* S, int* K, int* Q) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return false;
    // the occupancy queries cost some microseconds a call: plans are kept per device and shape
    struct Entry {
        int dev, lpc, force_s;
        bool bf16;
        int64_t tiles, nch;
        int S, K, Q;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.dev == dev && e.lpc == lpc && e.force_s == force_s && e.bf16 == bf16 && e.tiles == tiles_total &&
                e.nch == nch) {
                if (e.S <= 0) return false;
                *S = e.S;
                *K = e.K;
                *Q = e.Q;
                return true;
            }
    }
    int bs = 0, bk = 0, bq = 0;
    FwdParams dummy;
    std::memset(&dummy, 0, sizeof(dummy));
    FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    int64_t best = -1;
    for (int sz : {8, 4, 2}) {
        if (force_s > 0 && sz != force_s) continue;
        int fit[2] = {0, 0};
        if (launch_fwd_lane_cbal(bf16, lpc, dummy, maps, nullptr, sz, 0, fit) != cudaSuccess || fit[1] <= 0) {
            cudaGetLastError();
            continue;
        }
        const int k = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(fit[1], tiles_total / sms)));
        if (launch_fwd_lane_cbal(bf16, lpc, dummy, maps, nullptr, sz, k, fit) != cudaSuccess || fit[0] <= 0) {
            cudaGetLastError();
            continue;
        }
        const int64_t q = std::min<int64_t>(std::min<int64_t>(static_cast<int64_t>(k) * sms / sz, fit[0]),
                                            tiles_total / sz);
        if (q < 1) continue;
        const int64_t cost = (((tiles_total + q - 1) / q) * nch + sz - 1) / sz;
        if (best < 0 || cost < best) {
            best = cost;
            bs = sz;
            bk = k;
            bq = static_cast<int>(q);
        }
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() >= 64) cache.clear();
        cache.push_back(Entry{dev, lpc, force_s, bf16, tiles_total, nch, best >= 0 ? bs : 0, bk, bq});
    }
    if (best < 0) return false;
    *S = bs;
    *K = bk;
    *Q = bq;
    return true;
}

// Whether ss_fwd without a workspace takes the cluster-balanced schedule for a per-tile lane
// variant v (TMA-fed, 16 states, one CTA per 32-channel tile): when the tiles are more than fit on
// the GPU at once (g_force_cbal: never, or always with a given cluster size).  Sets the schedule's
// lanes per channel (bf16 2, fp32 4; a forced lane count must be that one), S and Q.
bool cbal_choice(const FwdVariant& v, bool bf16, int64_t batch, int64_t Dm, int64_t L, int forced_lpc, int* lpc,
                 int* S, int* K, int* Q) {
    const int fc = g_force_cbal.load();
    if (fc == 0 || v.family != kFamLane || !v.tma || v.lti || v.dtp || v.ns != 16 || v.balanced || v.cluster > 0 ||
        v.ckpt || v.chunk > 0)
        return false;
    const int want = bf16 ? 2 : 4;
    if (forced_lpc > 0 && forced_lpc != want) return false;
    const int64_t tiles_total = batch * ((Dm + 31) / 32);
    const int64_t nch = (L + kLaneT - 1) / kLaneT;
    if (nch > INT32_MAX || tiles_total > INT32_MAX) return false;
    if (fc < 0) {
        int cap = 0;
        if (lane_max_grid(v, bf16, &cap) != cudaSuccess || cap <= 0) return false;
        if (tiles_total <= cap) return false;   // one CTA per tile runs in one wave
    }
    if (!cbal_plan(bf16, want, tiles_total, nch, fc > 0 ? fc : 0, S, K, Q)) return false;
    *lpc = want;
    return true;
}

bool balanced_dx4(const FwdVariant& v, int64_t batch, int64_t Dm) {
    if (!v.w32 || v.lpc != 4 || v.es != 4 || v.ckpt) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return false;
    return batch * ((Dm + 31) / 32) < 3 * static_cast<int64_t>(sms);
}

cudaError_t lane_max_grid(const FwdVariant& v, bool bf16, int* out) {
    FwdParams dummy;
    std::memset(&dummy, 0, sizeof(dummy));
    FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    return v.bcf32 ? launch_fwd_lane_bf16w(v, dummy, maps, nullptr, out)
         : bf16     ? launch_fwd_lane_bf16(v, dummy, maps, nullptr, out)
                    : launch_fwd_lane_f32(v, dummy, maps, nullptr, out);
}

size_t fwd_ws_need(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype, bool* split,
                   bool with_widen = true);

// Bytes of the backward's checkpoints for these sizes (16 states): the state entering every 16th
// step, [batch·ceil(Dm/32)][ceil(L/32)][2][32][16] fp32.
size_t ckpt_bytes(int64_t batch, int64_t L, int64_t Dm) {
    return sizeof(float) * static_cast<size_t>(batch) * static_cast<size_t>((Dm + 31) / 32) *
           static_cast<size_t>((L + 31) / 32) * 2 * 32 * 16;
}

// Bytes of one widened (fp32) copy of bf16 B or C, and whether the workspace schedules widen them
// (bf16 I/O with 16 states).
size_t widen_copy_bytes(int64_t batch, int64_t L, int64_t N) {
    return align_up(sizeof(float) * static_cast<size_t>(batch) * static_cast<size_t>(L) * static_cast<size_t>(N), 256);
}
bool widens_bc(int32_t io_dtype, int64_t N) { return io_dtype == SS_BF16 && N == 16; }

// Segments per cluster of the single-launch time split for these sizes (as many as fill the GPU
// once, at most 8, none empty; 0: it does not fit), and the chunks per segment.
int cluster_plan(bool bf16, int64_t batch, int64_t L, int64_t Dm, int* seg_chunks) {
    const int64_t nch = (L + kLaneT - 1) / kLaneT;
    const int64_t tiles_c = batch * ((Dm + 31) / 32);
    int dev = 0, sms = 0, fit[2] = {0, 0};
    FwdParams probe;
    std::memset(&probe, 0, sizeof(probe));
    FwdMaps none;
    std::memset(&none, 0, sizeof(none));
    int result = 0;
    if (tiles_c > 0 && cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        launch_fwd_lane_cluster(bf16, probe, none, nullptr, 8, fit) == cudaSuccess && fit[1] > 0) {
        int64_t cs = std::min<int64_t>(std::min<int64_t>(static_cast<int64_t>(fit[1]) * sms / tiles_c, 8), nch);
        if (cs >= 2) {
            const int64_t seg = (nch + cs - 1) / cs;
            cs = (nch + seg - 1) / seg;
            int fit_cs[2] = {0, 0};
            if (cs >= 2 && seg <= INT32_MAX &&
                launch_fwd_lane_cluster(bf16, probe, none, nullptr, static_cast<int>(cs), fit_cs) == cudaSuccess &&
                fit_cs[0] > 0) {
                *seg_chunks = static_cast<int>(seg);
                result = static_cast<int>(cs);
            }
        }
    }
    cudaGetLastError();
    return result;
}

ss_status fwd_impl(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                   const void* B, const void* C, const float* D, const void* z, void* y,
                   float* last_state, const float* h0, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                   const ss_fwd_strides* strides, void* workspace, size_t ws_bytes, void* stream_ptr,
                   const float* W_dt = nullptr, int64_t R = 0, float* ckpt = nullptr) {
    // W_dt != nullptr: the low-rank time-step projection is folded in; `delta_raw` is then dt_low
    // [batch, L, R] (strides delta_b, delta_l) and delta_raw[b,t,d] = Σ_k W_dt[d,k] dt_low[b,t,k].
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const bool dtp = W_dt != nullptr;
    if (batch < 0 || L < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (dtp && (R < 4 || R > kDtRankMax || R % 4 != 0)) return SS_ERR_UNSUPPORTED;
    if (ckpt && (N != 16 || dtp)) return SS_ERR_UNSUPPORTED;   // checkpoints: 16 states
    ss_fwd_strides s;
    if (strides) {
        s = *strides;
    } else {
        std::memset(&s, 0, sizeof(s));
        s.io_dtype = SS_F32;
        s.u_b = s.delta_b = s.z_b = s.y_b = L * Dm;
        s.u_l = s.delta_l = s.z_l = s.y_l = Dm;
        s.B_b = s.C_b = L * N;
        s.B_l = s.C_l = N;
    }
    if (s.io_dtype != SS_F32 && s.io_dtype != SS_BF16) return SS_ERR_INVALID_ARG;
    const bool bf16 = s.io_dtype == SS_BF16;
    const int64_t es = bf16 ? 2 : 4;
    if (dtp && bf16) return SS_ERR_UNSUPPORTED;
    if (batch == 0 || Dm == 0) return SS_OK;
    if (!A_log) return SS_ERR_INVALID_ARG;
    if (h0 && !aligned(h0, 4)) return SS_ERR_MISALIGNED;
    const int64_t dcols = dtp ? R : Dm;   // columns of the time-step input
    const Range sh = span3(h0, batch, Dm, N, Dm * N, N, 4);
    const Range sl = span3(last_state, batch, Dm, N, Dm * N, N, 4);
    // h0 may be last_state itself (continue in place) but not overlap it otherwise
    if (h0 && static_cast<const void*>(h0) != static_cast<const void*>(last_state) && overlap(sh, sl))
        return SS_ERR_INVALID_ARG;
    if (L == 0) {
        // no steps: the final state is the initial one
        if (!last_state) return SS_OK;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
        if (!is_device_pointer(last_state, dev)) return SS_ERR_INVALID_ARG;
        const size_t bytes = sizeof(float) * batch * Dm * N;
        if (!h0) return cuda_status(cudaMemsetAsync(last_state, 0, bytes, stream));
        if (!is_device_pointer(h0, dev)) return SS_ERR_INVALID_ARG;
        if (static_cast<const void*>(h0) == static_cast<const void*>(last_state)) return SS_OK;
        return cuda_status(cudaMemcpyAsync(last_state, h0, bytes, cudaMemcpyDeviceToDevice, stream));
    }
    if (!u || !delta_raw || !B || !C || !y) return SS_ERR_INVALID_ARG;
    // strides: non-negative; the batch stride may only be anything when batch == 1
    const int64_t st[] = {s.u_b, s.u_l, s.delta_b, s.delta_l, s.y_b, s.y_l, s.B_b, s.B_l, s.C_b, s.C_l,
                          z ? s.z_b : 0, z ? s.z_l : 0};
    for (int64_t v : st)
        if (v < 0) return SS_ERR_INVALID_ARG;
    if (s.u_l < Dm || s.delta_l < dcols || s.y_l < Dm || (z && s.z_l < Dm)) {
        if (L > 1) return SS_ERR_INVALID_ARG;
    }
    // B, C: rows at least N apart, or step stride 0 (time-invariant, the LTI case)
    if (((s.B_l < N && s.B_l != 0) || (s.C_l < N && s.C_l != 0)) && L > 1) return SS_ERR_INVALID_ARG;
    // every element of y its own word (inputs may share memory, the output may not)
    if (!host::distinct3(batch, s.y_b, L, s.y_l, Dm)) return SS_ERR_INVALID_ARG;
    const bool lti = L > 1 && s.B_l == 0 && s.C_l == 0 && !dtp;
    if (L > INT32_MAX || Dm > INT32_MAX || batch > INT32_MAX) return SS_ERR_UNSUPPORTED;
    // alignment to the element type
    const void* io_ptrs[] = {u, delta_raw, B, C, y, z};
    for (const void* p : io_ptrs)
        if (p && !aligned(p, es)) return SS_ERR_MISALIGNED;
    const void* f_ptrs[] = {A_log, D, delta_bias, last_state, h0};
    for (const void* p : f_ptrs)
        if (p && !aligned(p, 4)) return SS_ERR_MISALIGNED;
    if (dtp && !aligned(W_dt, 16)) return SS_ERR_MISALIGNED;
    if (ckpt && !aligned(ckpt, 16)) return SS_ERR_MISALIGNED;
    // device memory of the current device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    const void* all_ptrs[] = {u, delta_raw, B, C, y, z, A_log, D, delta_bias, last_state, h0, W_dt, ckpt};
    for (const void* p : all_ptrs)
        if (p && !is_device_pointer(p, dev)) return SS_ERR_INVALID_ARG;
    // outputs must not overlap inputs
    const Range sy = span3(y, batch, L, Dm, s.y_b, s.y_l, es);
    if (overlap(sy, sh)) return SS_ERR_INVALID_ARG;
    const Range ins[] = {span3(u, batch, L, Dm, s.u_b, s.u_l, es),
                        span3(delta_raw, batch, L, dcols, s.delta_b, s.delta_l, es),
                        span3(W_dt, 1, Dm, R, 0, R, 4),
                        span3(z, batch, L, Dm, s.z_b, s.z_l, es),
                        span3(B, batch, L, N, s.B_b, s.B_l, es),
                        span3(C, batch, L, N, s.C_b, s.C_l, es),
                        span3(A_log, 1, Dm, N, 0, N, 4),
                        span3(D, 1, 1, Dm, 0, 0, 4),
                        span3(delta_bias, 1, 1, Dm, 0, 0, 4)};
    for (const Range& in : ins)
        if (overlap(sy, in) || overlap(sl, in)) return SS_ERR_INVALID_ARG;
    if (overlap(sy, sl)) return SS_ERR_INVALID_ARG;
    if (ckpt) {
        // the checkpoints are an output too
        const Range sc = span3(ckpt, 1, 1, static_cast<int64_t>(ckpt_bytes(batch, L, Dm) / 4), 0, 0, 4);
        for (const Range& in : ins)
            if (overlap(sc, in)) return SS_ERR_INVALID_ARG;
        if (overlap(sc, sy) || overlap(sc, sl) || overlap(sc, sh)) return SS_ERR_INVALID_ARG;
    }

    // Kernel choice.  The lane family folds each (channel, state) chain sequentially, its
    // parallelism being channels x LPC lanes; LPC grows until there are enough warps to fill
    // the GPU.  With few rows even LPC = 4 is not enough (a long sequence at batch 1) and the
    // segment-lane family, which runs time segments in parallel through the scan, takes over.
    FwdVariant v = choose_fwd_variant(batch, Dm, N);
    v.es = static_cast<int>(es);
    const int max_lpc = v.ns / 4;
    const int ff = g_force_family.load(), fl = g_force_lpc.load(), ft = g_force_tma.load();
    const int fc = dtp ? 0 : g_force_chunk.load();
    if (ff >= 0) v.family = ff == 2 ? kFamSeg : ff;   // 2: the cluster split where it applies, else segment
    if (fc > 0) v.chunk = fc;
    if (dtp) {                           // lane family only, as many lanes per channel as allowed
        if (v.family != kFamLane) v.lpc = max_lpc;
        v.family = kFamLane;
        v.dtp = true;
    }
    if (fl > 0) {
        if (fl > max_lpc) return SS_ERR_UNSUPPORTED;
        v.lpc = fl;
    }
    // TMA fill: B/C rows exactly ns wide and a multiple of 16 bytes, 16-byte aligned bases
    // and row/batch strides.  Time-invariant B/C (LTI) on the lane family: u/Δ/z by TMA, B and
    // C held in registers (no B/C tiles); elsewhere LTI takes the plain-load fill.
    bool tma = lti ? v.family == kFamLane : (N == v.ns) && (N * es) % 16 == 0;
    const void* tma_ptrs[] = {u, delta_raw, lti ? nullptr : B, lti ? nullptr : C, z};
    for (const void* q : tma_ptrs)
        if (q && !aligned(q, 16)) tma = false;
    const int64_t tma_strides[] = {s.u_l, s.delta_l, lti ? s.u_l : s.B_l, lti ? s.u_l : s.C_l, z ? s.z_l : s.u_l};
    for (int64_t v2 : tma_strides)
        if (!tma_stride_ok(v2, es)) tma = false;
    if (batch > 1) {
        const int64_t bstr[] = {s.u_b, s.delta_b, lti ? s.u_b : s.B_b, lti ? s.u_b : s.C_b, z ? s.z_b : s.u_b};
        for (int64_t v2 : bstr)
            if (!tma_stride_ok(v2, es)) tma = false;
    }
    if (ft == 0) tma = false;
    v.lti = lti && tma;

    // bf16 B and C are widened once into the front of the workspace when it holds the full size
    // the size query asks for; the workspace schedules then stage fp32 B/C tiles and need no
    // per-chunk widening (nor its block barriers) inside the scan.
    float* Bw = nullptr;
    float* Cw = nullptr;
    if (widens_bc(s.io_dtype, N) && tma && !lti && !dtp && fc == 0 && workspace) {
        bool need_split = false;
        const size_t one = widen_copy_bytes(batch, L, N);
        const size_t need = fwd_ws_need(batch, L, Dm, N, SS_BF16, &need_split);
        if (need >= 2 * one && ws_bytes >= need) {
            Bw = static_cast<float*>(workspace);
            Cw = reinterpret_cast<float*>(static_cast<char*>(workspace) + one);
            workspace = static_cast<char*>(workspace) + 2 * one;
            ws_bytes -= 2 * one;
        }
    }

    // Time-split schedule (needs a workspace and TMA): when the channel tiles alone cannot
    // fill the GPU, cut the sequence into segments that run side by side (pass A: end states
    // from zero; carry pass; pass C: the fold from each segment's carried start).
    const int fs = g_force_nseg.load();
    SplitPlan plan;
    if (workspace && !ckpt && tma && !lti && !dtp && fc == 0 && fs != 0 && (fs >= 2 || (v.family == kFamSeg && ff < 0))) {
        FwdVariant vs = v;
        vs.family = kFamLane;
        if (fl <= 0) vs.lpc = vs.ns / 4;
        vs.tma = true;
        vs.balanced = false;
        vs.state_only = false;
        int max_grid = 0;
        if (lane_max_grid(vs, bf16, &max_grid) != cudaSuccess || max_grid <= 0) return SS_ERR_CUDA;
        const int64_t tiles_ts = batch * ((Dm + lane_w(vs.lpc, false, 4) - 1) / lane_w(vs.lpc, false, 4));
        const int64_t nch = (L + kLaneT - 1) / kLaneT;
        if (nch <= INT32_MAX && tiles_ts * 64 <= INT32_MAX) {
            plan = split_plan(tiles_ts, static_cast<int>(nch), batch * Dm, N, max_grid, ws_bytes, fs);
            if (plan.nseg >= 2) v = vs;
        }
    }

    // TMA descriptors.  Both kernels read the u/Δ/z tiles through the hardware swizzle (one
    // box per stream, rows of a whole tile's channels); the segment-lane kernel also reads its
    // B/C tiles swizzled, the lane kernel reads them linearly.  A shape the descriptor encoder
    // rejects is served by the plain-load fill.
    // The schedule fixes the tile width (and so the box width): decide it first.  With a
    // workspace, TMA-fed lane kernels that do not take the time split run the balanced one.
    v.balanced = plan.nseg < 2 && workspace != nullptr && v.family == kFamLane && tma && !v.lti && !dtp &&
                 fc == 0 && g_force_balanced.load() != 0;
    if (!v.balanced && plan.nseg < 2 && v.family == kFamLane && fl <= 0) v.lpc = per_tile_lpc(batch, Dm, v.ns);
    v.w32 = v.balanced && balanced_w32(batch, Dm, v.es);
    v.dx4 = !ckpt && balanced_dx4(v, batch, Dm);
    if (ckpt) {
        // the checkpoint-writing kernels (TMA-fed): the balanced schedule where a workspace allows it
        // (bf16 with fp32 B/C tiles at 2 lanes per channel; fp32 on 32-channel tiles at 4), the
        // single-launch time split for few tiles (below), else one CTA per tile at 4 lanes
        if (!tma || lti) return SS_ERR_UNSUPPORTED;
        const bool bal_ok = v.balanced && ((bf16 && Bw && v.lpc == 2) || (!bf16 && v.w32 && v.lpc == 4));
        if (!bal_ok) {
            v.balanced = false;
            v.w32 = false;
            if (v.family != kFamSeg) {
                v.family = kFamLane;
                v.lpc = 4;
            }
        }
        v.ckpt = true;
    }
    FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));

    // Single-launch time split (no workspace): when the channel tiles alone cannot fill the GPU
    // (the segment family's case; family 2 forces it), CTAs that fold the time segments of one
    // tile form a cluster and exchange their segments' summaries through distributed shared
    // memory, so the split needs neither a workspace nor a second launch.
    int cluster_seg_chunks = 0;
    if ((!workspace || ckpt) && tma && !lti && !dtp && fc == 0 && v.ns == 16 && v.family == kFamSeg &&
        (ff < 0 || ff == 2) && (fl <= 0 || fl == 4)) {
        const int cs = cluster_plan(bf16, batch, L, Dm, &cluster_seg_chunks);
        if (cs >= 2) {
            v.family = kFamLane;
            v.lpc = 4;
            v.cluster = cs;
        }
    }
    if (ckpt && v.family == kFamSeg) {   // no cluster split for these sizes: one CTA per tile
        v.family = kFamLane;
        v.lpc = 4;
    }
    if (tma) {
        const FwdGeom g0 = fwd_geometry(v);
        const bool swbc = v.family == kFamSeg;
        const int bw = g0.box_channels, bh = g0.chunk_steps;
        tma = make_map(&maps.u, u, bf16, Dm, L, batch, s.u_l, s.u_b, bw, bh, true) &&
              (dtp ? make_map(&maps.delta, delta_raw, false, R, L, batch, s.delta_l, s.delta_b,
                              dt_pitch(static_cast<int>(R)), bh, false)
                   : make_map(&maps.delta, delta_raw, bf16, Dm, L, batch, s.delta_l, s.delta_b, bw, bh, true)) &&
              (!z || make_map(&maps.z, z, bf16, Dm, L, batch, s.z_l, s.z_b, bw, bh, true)) &&
              (v.lti || (make_map(&maps.B, B, bf16, N, L, batch, s.B_l, s.B_b, v.ns, bh, swbc) &&
                         make_map(&maps.C, C, bf16, N, L, batch, s.C_l, s.C_b, v.ns, bh, swbc)));
    }
    if ((ft == 1 || dtp) && !tma) return SS_ERR_UNSUPPORTED;   // the folded projection is TMA-fed only
    v.tma = tma;
    if (!tma) v.lti = false;
    if (!tma) {                     // descriptors refused: the plain-load fill, per-tile schedule
        plan = SplitPlan();
        v.balanced = false;
        v.w32 = false;
        v.dx4 = false;
    }
    const bool split = plan.nseg >= 2;
    // Cluster-balanced schedule: no workspace, and more channel tiles than one CTA per tile can
    // run at once (a second wave would hold the rest).
    int cbal_q = 0, cbal_k = 0;
    if (!workspace && !split) {
        int lpc_c = 0, s_c = 0, k_c = 0, q_c = 0;
        if (cbal_choice(v, bf16, batch, Dm, L, fl, &lpc_c, &s_c, &k_c, &q_c)) {
            v.lpc = lpc_c;
            v.cbal = s_c;
            cbal_k = k_c;
            cbal_q = q_c;
        }
    }
    v.bcf32 = Bw && tma && v.family == kFamLane && (v.balanced || split);
    if (v.bcf32) {
        const int bh = fwd_geometry(v).chunk_steps;
        if (!make_map(&maps.B, Bw, false, N, L, batch, N, L * N, v.ns, bh, false) ||
            !make_map(&maps.C, Cw, false, N, L, batch, N, L * N, v.ns, bh, false))
            return SS_ERR_CUDA;
    }
    // enqueued once every check of the schedule has passed, right before the scan
    auto widen = [&]() -> cudaError_t {
        return v.bcf32 ? launch_widen_bc(B, C, s.B_b, s.B_l, s.C_b, s.C_l, Bw, Cw, batch, L, static_cast<int>(N), stream)
                       : cudaSuccess;
    };

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.u = u; p.delta = delta_raw; p.z = z; p.Bm = B; p.Cm = C;
    p.bias = delta_bias; p.A_log = A_log; p.Dv = D; p.y = y; p.last_state = last_state; p.h0 = h0;
    p.ckpt = ckpt;
    p.ckpt_chunks = static_cast<int>((L + 31) / 32);
    p.u_b = s.u_b; p.u_l = s.u_l; p.d_b = s.delta_b; p.d_l = s.delta_l;
    p.z_b = s.z_b; p.z_l = s.z_l; p.y_b = s.y_b; p.y_l = s.y_l;
    p.B_b = s.B_b; p.B_l = s.B_l; p.C_b = s.C_b; p.C_l = s.C_l;
    const FwdGeom geo = fwd_geometry(v);
    const int64_t tiles = (Dm + geo.tile_channels - 1) / geo.tile_channels;
    if (batch * tiles > INT32_MAX) return SS_ERR_UNSUPPORTED;
    p.batch = static_cast<int>(batch);
    p.L = static_cast<int>(L);
    p.Dm = static_cast<int>(Dm);
    p.N = static_cast<int>(N);
    p.nchunks = static_cast<int>((L + geo.chunk_steps - 1) / geo.chunk_steps);
    p.tiles_per_batch = static_cast<int>(tiles);
    p.chunk_steps = geo.chunk_steps;
    p.tile_channels = geo.tile_channels;
    p.box_channels = tma ? geo.box_channels : 0;
    p.err = device_error_ptr();
    if (!p.err) return SS_ERR_CUDA;
    if (dtp) {
        p.W_dt = W_dt;
        p.dt_rank = static_cast<int>(R);
        p.dt_pitch = dt_pitch(static_cast<int>(R));
        return cuda_status(launch_fwd_lane_dtp(v, p, maps, stream));
    }
    if (v.balanced) {
        // grid: every CTA resident at once (cooperative launch), never more CTAs than tiles
        int max_grid = 0;
        if (lane_max_grid(v, bf16, &max_grid) != cudaSuccess || max_grid <= 0) return SS_ERR_CUDA;
        const int64_t grid = balanced_grid(batch * tiles, max_grid);
        if (balanced_ws_bytes(static_cast<int>(grid), geo.tile_channels, v.ns) > ws_bytes)
            return SS_ERR_INVALID_ARG;
        if (!aligned(workspace, 256)) return SS_ERR_MISALIGNED;
        if (!is_device_pointer(workspace, dev)) return SS_ERR_INVALID_ARG;
        p.grid = static_cast<int>(grid);
        p.ws_flag = static_cast<unsigned int*>(workspace);
        p.ws_state = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              align_up(static_cast<size_t>(grid) * 4, 256));
        p.epoch = next_epoch();
        const cudaError_t we = widen();
        if (we != cudaSuccess) return cuda_status(we);
    }
    if (split) {
        if (plan.bytes > ws_bytes) return SS_ERR_INVALID_ARG;
        if (!aligned(workspace, 256)) return SS_ERR_MISALIGNED;
        if (!is_device_pointer(workspace, dev)) return SS_ERR_INVALID_ARG;
        const int64_t tiles_total = batch * tiles;
        p.nseg = plan.nseg;
        p.seg_chunks = plan.seg_chunks;
        p.seg_slots = static_cast<float*>(workspace);
        p.seg_dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.off_dsum);
        p.seg_out0 = 1;                   // slot 0 holds h0; segment s ends in slot s + 1
        auto lane = [&](const FwdVariant& vv, const FwdParams& pp) {
            return vv.bcf32 ? launch_fwd_lane_bf16w(vv, pp, maps, stream)
                 : bf16     ? launch_fwd_lane_bf16(vv, pp, maps, stream)
                            : launch_fwd_lane_f32(vv, pp, maps, stream);
        };
        cudaError_t e = widen();
        if (e != cudaSuccess) return cuda_status(e);
        FwdParams pa = p;                 // pass A: segments 0 .. nseg-2 from zero
        pa.seg_launch = plan.nseg - 1;
        pa.grid = static_cast<int>(tiles_total * pa.seg_launch);
        pa.h0 = nullptr;
        pa.last_state = nullptr;
        pa.z = nullptr;                   // pass A reads neither z nor C
        FwdVariant va = v;
        va.state_only = true;
        e = lane(va, pa);
        if (e != cudaSuccess) return cuda_status(e);
        if ((e = launch_fwd_carry(p, stream)) != cudaSuccess) return cuda_status(e);
        FwdParams pc = p;                 // pass C: every segment from its carried start
        pc.seg_launch = plan.nseg;
        pc.grid = static_cast<int>(tiles_total * plan.nseg);
        return cuda_status(lane(v, pc));
    }
    cudaError_t e;
    if (v.cluster > 0) {
        p.seg_launch = v.cluster;
        p.seg_chunks = cluster_seg_chunks;
        p.nseg = v.cluster;
        p.grid = static_cast<int>(batch * tiles * v.cluster);
        return cuda_status(launch_fwd_lane_cluster(bf16, p, maps, stream, v.cluster));
    }
    if (v.cbal > 0) {
        p.cbal = v.cbal;
        p.grid = cbal_q * v.cbal;
        return cuda_status(launch_fwd_lane_cbal(bf16, v.lpc, p, maps, stream, v.cbal, cbal_k));
    }
    if (v.chunk > 0) {
        if (!chunk_override_ok(v)) return SS_ERR_UNSUPPORTED;
        return cuda_status(launch_fwd_lane_chunked(v, p, maps, stream));
    }
    if (v.family == kFamSeg)
        e = launch_fwd_seg(v, bf16, p, maps, stream);
    else if (v.bcf32)
        e = launch_fwd_lane_bf16w(v, p, maps, stream);
    else
        e = bf16 ? launch_fwd_lane_bf16(v, p, maps, stream) : launch_fwd_lane_f32(v, p, maps, stream);
    return cuda_status(e);
}

}  // namespace
}  // namespace selscan

extern "C" {

ss_status ss_fwd(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                 const void* B, const void* C, const float* D, const void* z, void* y,
                 float* last_state, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                 const ss_fwd_strides* strides, void* stream) {
    return fwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, y, last_state, nullptr, batch, L, Dm, N,
                    strides, nullptr, 0, stream);
}

ss_status ss_fwd_dtproj(const void* u, const void* dt_low, const float* W_dt, int64_t dt_rank,
                        const float* delta_bias, const float* A_log, const void* B, const void* C, const float* D,
                        const void* z, void* y, float* last_state, const float* h0, int64_t batch, int64_t L,
                        int64_t Dm, int64_t N, const ss_fwd_strides* strides, void* stream) {
    if (!W_dt || !dt_low) return SS_ERR_INVALID_ARG;
    return fwd_impl(u, dt_low, delta_bias, A_log, B, C, D, z, y, last_state, h0, batch, L, Dm, N, strides,
                    nullptr, 0, stream, W_dt, dt_rank);
}

ss_status ss_fwd_ws(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                    const void* B, const void* C, const float* D, const void* z, void* y,
                    float* last_state, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                    const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, y, last_state, nullptr, batch, L, Dm, N,
                    strides, workspace, workspace_bytes, stream);
}

ss_status ss_fwd_h0(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                    const void* B, const void* C, const float* D, const void* z, void* y,
                    float* last_state, const float* h0, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                    const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, y, last_state, h0, batch, L, Dm, N,
                    strides, workspace, workspace_bytes, stream);
}

ss_status ss_fwd_ckpt(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                      const void* B, const void* C, const float* D, const void* z, void* y, float* last_state,
                      const float* h0, float* ckpt, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                      const ss_fwd_strides* strides, void* workspace, size_t workspace_bytes, void* stream) {
    if (!ckpt && batch > 0 && L > 0 && Dm > 0) return SS_ERR_INVALID_ARG;
    return fwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, y, last_state, h0, batch, L, Dm, N, strides,
                    workspace, workspace_bytes, stream, nullptr, 0, ckpt);
}

size_t ss_fwd_ckpt_size(int64_t batch, int64_t L, int64_t Dm, int64_t N) {
    if (batch <= 0 || L <= 0 || Dm <= 0 || N != 16) return 0;
    return ckpt_bytes(batch, L, Dm);
}

}  // extern "C"

namespace selscan {
namespace {

// Workspace bytes of the schedule ss_fwd_ws picks for these sizes (0: none needed, or invalid
// sizes).  *split tells whether it is the time split, which also runs on less (fewer segments).
// with_widen: count the widened fp32 copies of bf16 B and C that a full-size workspace carries.
size_t fwd_ws_need(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype, bool* split,
                   bool with_widen) {
    *split = false;
    const size_t widen = with_widen && widens_bc(io_dtype, N) ? 2 * widen_copy_bytes(batch, L, N) : 0;
    if (batch <= 0 || L <= 0 || Dm <= 0 || N < 1 || N > 16) return 0;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return 0;
    FwdVariant v = choose_fwd_variant(batch, Dm, N);
    v.es = io_dtype == SS_BF16 ? 2 : 4;
    const int ff = g_force_family.load(), fs = g_force_nseg.load();
    if (ff >= 0) v.family = ff == 2 ? kFamSeg : ff;
    const int fl = g_force_lpc.load() > 0 && g_force_lpc.load() <= v.ns / 4 ? g_force_lpc.load() : 0;
    if (fl) v.lpc = fl;
    if (fs != 0 && (fs >= 2 || (v.family == kFamSeg && ff < 0))) {
        // the time-split schedule
        v.family = kFamLane;
        if (!fl) v.lpc = v.ns / 4;
        v.tma = true;
        int max_grid = 0;
        if (lane_max_grid(v, io_dtype == SS_BF16, &max_grid) != cudaSuccess || max_grid <= 0) return 0;
        const int64_t tiles_ts = batch * ((Dm + lane_w(v.lpc, false, 4) - 1) / lane_w(v.lpc, false, 4));
        const int64_t nch = (L + kLaneT - 1) / kLaneT;
        if (nch > INT32_MAX) return 0;
        const SplitPlan pl = split_plan(tiles_ts, static_cast<int>(nch), batch * Dm, N, max_grid,
                                        static_cast<size_t>(-1), fs);
        *split = pl.nseg >= 2;
        return pl.nseg >= 2 ? pl.bytes + widen : 0;
    }
    if (v.family != kFamLane) return 0;
    v.balanced = true;
    v.tma = true;
    v.bcf32 = widen > 0;
    v.w32 = balanced_w32(batch, Dm, v.es);
    v.dx4 = balanced_dx4(v, batch, Dm);
    const FwdGeom geo = fwd_geometry(v);
    const int64_t tiles = batch * ((Dm + geo.tile_channels - 1) / geo.tile_channels);
    int max_grid = 0;
    if (lane_max_grid(v, io_dtype == SS_BF16, &max_grid) != cudaSuccess || max_grid <= 0) return 0;
    const int64_t grid = balanced_grid(tiles, max_grid);
    return balanced_ws_bytes(static_cast<int>(grid), geo.tile_channels, v.ns) + widen;
}

}  // namespace
}  // namespace selscan

extern "C" {

ss_status ss_fwd_summary(const void* u, const void* delta_raw, const float* delta_bias, const float* A_log,
                         const void* B, float* h_end, float* dsum, int64_t batch, int64_t L, int64_t Dm, int64_t N,
                         const ss_fwd_strides* strides, void* stream_ptr) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (batch < 0 || L < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    ss_fwd_strides s;
    if (strides) {
        s = *strides;
    } else {
        std::memset(&s, 0, sizeof(s));
        s.io_dtype = SS_F32;
        s.u_b = s.delta_b = s.z_b = s.y_b = L * Dm;
        s.u_l = s.delta_l = s.z_l = s.y_l = Dm;
        s.B_b = s.C_b = L * N;
        s.B_l = s.C_l = N;
    }
    if (s.io_dtype != SS_F32 && s.io_dtype != SS_BF16) return SS_ERR_INVALID_ARG;
    const bool bf16 = s.io_dtype == SS_BF16;
    const int64_t es = bf16 ? 2 : 4;
    if (batch == 0 || Dm == 0) return SS_OK;
    if (!A_log || !h_end || !dsum) return SS_ERR_INVALID_ARG;
    if (!aligned(h_end, 4) || !aligned(dsum, 4) || !aligned(A_log, 4)) return SS_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (!is_device_pointer(h_end, dev) || !is_device_pointer(dsum, dev) || !is_device_pointer(A_log, dev))
        return SS_ERR_INVALID_ARG;
    const Range sh = span3(h_end, batch, Dm, N, Dm * N, N, 4);
    const Range sd = span3(dsum, 1, batch, Dm, 0, Dm, 4);
    if (overlap(sh, sd)) return SS_ERR_INVALID_ARG;
    if (L == 0) {   // no steps: the end state from zero is zero, and so is the sum of Δ
        if (cudaMemsetAsync(h_end, 0, sizeof(float) * batch * Dm * N, stream) != cudaSuccess) return SS_ERR_CUDA;
        return cuda_status(cudaMemsetAsync(dsum, 0, sizeof(float) * batch * Dm, stream));
    }
    if (!u || !delta_raw || !B) return SS_ERR_INVALID_ARG;
    const int64_t st[] = {s.u_b, s.u_l, s.delta_b, s.delta_l, s.B_b, s.B_l};
    for (int64_t v : st)
        if (v < 0) return SS_ERR_INVALID_ARG;
    if ((s.u_l < Dm || s.delta_l < Dm || s.B_l < N) && L > 1) return SS_ERR_INVALID_ARG;
    if (L > INT32_MAX || Dm > INT32_MAX || batch > INT32_MAX) return SS_ERR_UNSUPPORTED;
    const void* io_ptrs[] = {u, delta_raw, B};
    for (const void* q : io_ptrs)
        if (!aligned(q, es)) return SS_ERR_MISALIGNED;
    if (delta_bias && !aligned(delta_bias, 4)) return SS_ERR_MISALIGNED;
    const void* ptrs[] = {u, delta_raw, B, delta_bias};
    for (const void* q : ptrs)
        if (q && !is_device_pointer(q, dev)) return SS_ERR_INVALID_ARG;
    const Range ins[] = {span3(u, batch, L, Dm, s.u_b, s.u_l, es), span3(delta_raw, batch, L, Dm, s.delta_b, s.delta_l, es),
                        span3(B, batch, L, N, s.B_b, s.B_l, es), span3(A_log, 1, Dm, N, 0, N, 4),
                        span3(delta_bias, 1, 1, Dm, 0, 0, 4)};
    for (const Range& in : ins)
        if (overlap(sh, in) || overlap(sd, in)) return SS_ERR_INVALID_ARG;

    // The state-only fold (the time split's first pass) over the whole sequence as one segment:
    // one CTA per 32-channel tile, TMA-fed tiles of u, Δ and B (C and z are not read).
    FwdVariant v = choose_fwd_variant(batch, Dm, N);
    v.es = static_cast<int>(es);
    v.family = kFamLane;
    v.lpc = v.ns / 4;
    v.tma = true;
    v.state_only = true;
    v.balanced = false;
    bool tma = N == v.ns && (N * es) % 16 == 0 && aligned(u, 16) && aligned(delta_raw, 16) && aligned(B, 16) &&
               tma_stride_ok(s.u_l, es) && tma_stride_ok(s.delta_l, es) && tma_stride_ok(s.B_l, es);
    if (batch > 1)
        tma = tma && tma_stride_ok(s.u_b, es) && tma_stride_ok(s.delta_b, es) && tma_stride_ok(s.B_b, es);
    const FwdGeom geo = fwd_geometry(v);
    FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    tma = tma && make_map(&maps.u, u, bf16, Dm, L, batch, s.u_l, s.u_b, geo.box_channels, geo.chunk_steps, true) &&
          make_map(&maps.delta, delta_raw, bf16, Dm, L, batch, s.delta_l, s.delta_b, geo.box_channels,
                   geo.chunk_steps, true) &&
          make_map(&maps.B, B, bf16, N, L, batch, s.B_l, s.B_b, v.ns, geo.chunk_steps, false);
    if (!tma) return SS_ERR_UNSUPPORTED;   // the state-only fold is TMA-fed only; no fallback
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.u = u; p.delta = delta_raw; p.Bm = B; p.bias = delta_bias; p.A_log = A_log;
    p.u_b = s.u_b; p.u_l = s.u_l; p.d_b = s.delta_b; p.d_l = s.delta_l; p.B_b = s.B_b; p.B_l = s.B_l;
    const int64_t tiles = (Dm + geo.tile_channels - 1) / geo.tile_channels;
    if (batch * tiles > INT32_MAX) return SS_ERR_UNSUPPORTED;
    p.batch = static_cast<int>(batch);
    p.L = static_cast<int>(L);
    p.Dm = static_cast<int>(Dm);
    p.N = static_cast<int>(N);
    p.nchunks = static_cast<int>((L + geo.chunk_steps - 1) / geo.chunk_steps);
    p.tiles_per_batch = static_cast<int>(tiles);
    p.chunk_steps = geo.chunk_steps;
    p.tile_channels = geo.tile_channels;
    p.box_channels = geo.box_channels;
    p.err = device_error_ptr();
    if (!p.err) return SS_ERR_CUDA;
    p.seg_launch = 1;
    p.seg_chunks = p.nchunks;
    p.nseg = 1;
    p.seg_slots = h_end;
    p.seg_dsum = dsum;
    p.seg_out0 = 0;
    p.grid = static_cast<int>(batch * tiles);
    return cuda_status(bf16 ? launch_fwd_lane_bf16(v, p, maps, stream) : launch_fwd_lane_f32(v, p, maps, stream));
}

ss_status ss_carry_compose(float* slots, const float* dsum, const float* h0, const float* A_log, int64_t nseg,
                           int64_t batch, int64_t Dm, int64_t N, void* stream_ptr) {
    if (nseg < 1 || batch < 0 || Dm < 0) return SS_ERR_INVALID_ARG;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (batch == 0 || Dm == 0) return SS_OK;
    if (!slots || !A_log || (nseg > 1 && !dsum)) return SS_ERR_INVALID_ARG;
    if (batch * Dm * N * nseg > (int64_t(1) << 40) || Dm > INT32_MAX || nseg > INT32_MAX) return SS_ERR_UNSUPPORTED;
    const void* f_ptrs[] = {slots, dsum, h0, A_log};
    for (const void* q : f_ptrs)
        if (q && !aligned(q, 4)) return SS_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    for (const void* q : f_ptrs)
        if (q && !is_device_pointer(q, dev)) return SS_ERR_INVALID_ARG;
    const int64_t rows = batch * Dm;
    const Range ss_ = span3(slots, 1, nseg, rows * N, 0, rows * N, 4);
    const Range ins[] = {span3(nseg > 1 ? dsum : nullptr, 1, nseg - 1, rows, 0, rows, 4),
                        span3(A_log, 1, Dm, N, 0, N, 4)};
    for (const Range& in : ins)
        if (overlap(ss_, in)) return SS_ERR_INVALID_ARG;
    // h0 may be slot 0 itself; it must not overlap any other slot
    if (h0 && h0 != slots && overlap(ss_, span3(h0, 1, 1, rows * N, 0, 0, 4))) return SS_ERR_INVALID_ARG;
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.A_log = A_log;
    p.h0 = h0;
    p.seg_slots = slots;
    p.seg_dsum = const_cast<float*>(dsum);
    p.batch = static_cast<int>(batch);
    p.Dm = static_cast<int>(Dm);
    p.N = static_cast<int>(N);
    p.nseg = static_cast<int>(nseg);
    return cuda_status(launch_fwd_carry(p, static_cast<cudaStream_t>(stream_ptr)));
}

size_t ss_fwd_workspace_size(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype) {
    bool split = false;
    return fwd_ws_need(batch, L, Dm, N, io_dtype, &split);
}

// Internal reporting hook (not part of the public header): the schedule a forward call with
// (with_ws != 0) or without a workspace of ss_fwd_workspace_size bytes makes for these sizes,
// assuming TMA-eligible arguments.  Writes its name into `name` (cap bytes) and returns the
// number of kernel launches per call (0: sizes invalid).
int ss__fwd_plan(int64_t batch, int64_t L, int64_t Dm, int64_t N, int32_t io_dtype, int with_ws,
                 char* name, int cap) {
    auto put = [&](const char* txt) {
        if (name && cap > 0) {
            std::strncpy(name, txt, static_cast<size_t>(cap) - 1);
            name[cap - 1] = '\0';
        }
    };
    if (batch <= 0 || L <= 0 || Dm <= 0 || N < 1 || N > 16) {
        put("none");
        return 0;
    }
    FwdVariant v = choose_fwd_variant(batch, Dm, N);
    v.es = io_dtype == SS_BF16 ? 2 : 4;
    const int ff = g_force_family.load(), fs = g_force_nseg.load();
    if (ff >= 0) v.family = ff == 2 ? kFamSeg : ff;
    const int fl = g_force_lpc.load() > 0 && g_force_lpc.load() <= v.ns / 4 ? g_force_lpc.load() : 0;
    if (fl) v.lpc = fl;
    char buf[96];
    if (with_ws && fs != 0 && (fs >= 2 || (v.family == kFamSeg && ff < 0))) {
        FwdVariant vs = v;
        vs.family = kFamLane;
        if (!fl) vs.lpc = vs.ns / 4;
        int max_grid = 0;
        if (lane_max_grid(vs, io_dtype == SS_BF16, &max_grid) == cudaSuccess && max_grid > 0) {
            const int64_t tiles = batch * ((Dm + lane_w(vs.lpc, false, 4) - 1) / lane_w(vs.lpc, false, 4));
            const int64_t nch = (L + kLaneT - 1) / kLaneT;
            if (nch <= INT32_MAX) {
                const SplitPlan pl = split_plan(tiles, static_cast<int>(nch), batch * Dm, N, max_grid,
                                                static_cast<size_t>(-1), fs);
                if (pl.nseg >= 2) {
                    const bool wide = widens_bc(io_dtype, N);
                    std::snprintf(buf, sizeof(buf), "ss_fwd_lane_kernel(lpc=%d,time-split,nseg=%d%s)", vs.lpc, pl.nseg,
                                  wide ? ",fp32 B/C" : "");
                    put(buf);
                    return wide ? 4 : 3;      // (widening,) pass A, carry, pass C
                }
            }
        }
    }
    if (v.family == kFamSeg) {
        int seg = 0;
        const int cs = !with_ws && N == 16 && (fl <= 0 || fl == 4) ? cluster_plan(io_dtype == SS_BF16, batch, L, Dm, &seg)
                                                                    : 0;
        if (cs >= 2) {
            std::snprintf(buf, sizeof(buf), "ss_fwd_lane_kernel(lpc=4,cluster split,nseg=%d)", cs);
            put(buf);
        } else {
            put("ss_fwd_seg_kernel");
        }
        return 1;
    }
    const bool bal = with_ws && g_force_balanced.load() != 0;
    if (!bal && !fl) v.lpc = per_tile_lpc(batch, Dm, v.ns);
    if (!with_ws && N == 16) {
        FwdVariant vc = v;
        vc.tma = true;
        vc.es = io_dtype == SS_BF16 ? 2 : 4;
        int lc = 0, sc = 0, kc = 0, qc = 0;
        if (cbal_choice(vc, io_dtype == SS_BF16, batch, Dm, L, fl, &lc, &sc, &kc, &qc)) {
            std::snprintf(buf, sizeof(buf), "ss_fwd_lane_kernel(lpc=%d,cluster-balanced,S=%d)", lc, sc);
            put(buf);
            return 1;
        }
    }
    const bool wide = bal && widens_bc(io_dtype, N);
    const bool w32 = bal && balanced_w32(batch, Dm, io_dtype == SS_BF16 ? 2 : 4);
    FwdVariant vd = v;
    vd.w32 = w32;
    vd.es = io_dtype == SS_BF16 ? 2 : 4;
    const bool dx4 = balanced_dx4(vd, batch, Dm);
    std::snprintf(buf, sizeof(buf), "ss_fwd_lane_kernel(lpc=%d%s%s%s%s)", v.lpc, bal ? ",balanced" : "",
                  w32 ? ",32-channel tiles" : "", dx4 ? ",shared-memory hand-over" : "", wide ? ",fp32 B/C" : "");
    put(buf);
    return wide ? 2 : 1;                  // (the B/C widening pass,) the scan
}

ss_status ss_fwd_static(const void* u, const void* delta_raw, const float* delta_bias,
                        const float* A_log, const void* B, const void* C, const float* D,
                        const void* z, void* y, float* last_state, int64_t batch, int64_t L,
                        int64_t Dm, int64_t N, const ss_fwd_strides* strides, void* stream) {
    const int32_t io = strides ? strides->io_dtype : SS_F32;
    bool split = false;
    // the fixed array carries no widened B/C copies: the schedules' own bytes only
    const size_t need = (batch > 0 && L > 0 && Dm > 0) ? fwd_ws_need(batch, L, Dm, N, io, &split, false) : 0;
    // beyond the fixed array: the balanced schedule cannot shrink; the time split takes as many
    // segments as the array holds (fwd_impl's plan), or none below two
    if (need > SS_STATIC_WORKSPACE_BYTES && !split) return SS_ERR_UNSUPPORTED;
    void* ws = nullptr;
    if (need > 0) {
        ws = static_workspace_ptr();
        if (!ws) return SS_ERR_CUDA;
    }
    return fwd_impl(u, delta_raw, delta_bias, A_log, B, C, D, z, y, last_state, nullptr, batch, L, Dm, N,
                    strides, ws, ws ? SS_STATIC_WORKSPACE_BYTES : 0, stream);
}

}  // extern "C"

namespace selscan {
namespace {

// Validated decode-step arguments of one layer.
struct StepCheck {
    ss_status status = SS_OK;
    bool empty = false;      // batch == 0 or Dm == 0: nothing to do
    bool bf16 = false;
    bool vec = false;        // the vector (state quad) path applies
    StepParams p{};
    Range out_y, out_state;  // the bytes the step writes
    Range in[8];             // the bytes it reads
};

StepCheck step_check(float* state, const void* x, const void* delta_raw, const float* delta_bias,
                     const float* A_log, const void* B, const void* C, const float* D, const void* z,
                     void* y, int64_t batch, int64_t Dm, int64_t N, const ss_step_strides* strides) {
    StepCheck r;
    auto fail = [&](ss_status e) { r.status = e; return r; };
    if (batch < 0 || Dm < 0) return fail(SS_ERR_INVALID_ARG);
    if (N < 1 || N > 16) return fail(SS_ERR_UNSUPPORTED);
    ss_step_strides s;
    if (strides) {
        s = *strides;
    } else {
        std::memset(&s, 0, sizeof(s));
        s.io_dtype = SS_F32;
        s.x_b = s.delta_b = s.z_b = s.y_b = Dm;
        s.B_b = s.C_b = N;
        s.state_b = Dm * N;
        s.state_d = N;
    }
    if (s.io_dtype != SS_F32 && s.io_dtype != SS_BF16) return fail(SS_ERR_INVALID_ARG);
    const bool bf16 = s.io_dtype == SS_BF16;
    r.bf16 = bf16;
    const int64_t es = bf16 ? 2 : 4;
    if (batch == 0 || Dm == 0) {
        r.empty = true;
        return r;
    }
    if (!state || !x || !delta_raw || !A_log || !B || !C || !y) return fail(SS_ERR_INVALID_ARG);
    const int64_t st[] = {s.x_b, s.delta_b, s.y_b, s.B_b, s.C_b, s.state_b, s.state_d, z ? s.z_b : 0};
    for (int64_t v : st)
        if (v < 0) return fail(SS_ERR_INVALID_ARG);
    if (batch > 1 && (s.x_b < Dm || s.delta_b < Dm || s.y_b < Dm || (z && s.z_b < Dm) || s.B_b < N ||
                      s.C_b < N))
        return fail(SS_ERR_INVALID_ARG);
    if (Dm > 1 && s.state_d < N) return fail(SS_ERR_INVALID_ARG);
    // y and the state are written: every element its own word
    if (!host::distinct3(1, 0, batch, s.y_b, Dm) || !host::distinct3(batch, s.state_b, Dm, s.state_d, N))
        return fail(SS_ERR_INVALID_ARG);
    if (batch * Dm * 4 > (int64_t(1) << 40) || Dm > INT32_MAX || batch > INT32_MAX)
        return fail(SS_ERR_UNSUPPORTED);
    const void* io_ptrs[] = {x, delta_raw, B, C, y, z};
    for (const void* q : io_ptrs)
        if (q && !aligned(q, es)) return fail(SS_ERR_MISALIGNED);
    const void* f_ptrs[] = {state, A_log, D, delta_bias};
    for (const void* q : f_ptrs)
        if (q && !aligned(q, 4)) return fail(SS_ERR_MISALIGNED);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SS_ERR_CUDA);
    const void* all_ptrs[] = {state, x, delta_raw, B, C, y, z, A_log, D, delta_bias};
    for (const void* q : all_ptrs)
        if (q && !is_device_pointer(q, dev)) return fail(SS_ERR_INVALID_ARG);
    r.out_y = span3(y, 1, batch, Dm, 0, s.y_b, es);
    r.out_state = span3(state, batch, Dm, N, s.state_b, s.state_d, 4);
    const Range ins[] = {span3(x, 1, batch, Dm, 0, s.x_b, es),
                        span3(delta_raw, 1, batch, Dm, 0, s.delta_b, es),
                        span3(z, 1, batch, Dm, 0, s.z_b, es),
                        span3(B, 1, batch, N, 0, s.B_b, es),
                        span3(C, 1, batch, N, 0, s.C_b, es),
                        span3(A_log, 1, Dm, N, 0, N, 4),
                        span3(D, 1, 1, Dm, 0, 0, 4),
                        span3(delta_bias, 1, 1, Dm, 0, 0, 4)};
    for (int i = 0; i < 8; ++i) {
        r.in[i] = ins[i];
        if (overlap(r.out_y, ins[i]) || overlap(r.out_state, ins[i])) return fail(SS_ERR_INVALID_ARG);
    }
    if (overlap(r.out_y, r.out_state)) return fail(SS_ERR_INVALID_ARG);

    StepParams& p = r.p;
    p.state = state; p.x = x; p.delta = delta_raw; p.z = z; p.Bm = B; p.Cm = C;
    p.bias = delta_bias; p.A_log = A_log; p.Dv = D; p.y = y;
    p.x_b = s.x_b; p.d_b = s.delta_b; p.z_b = s.z_b; p.y_b = s.y_b;
    p.B_b = s.B_b; p.C_b = s.C_b; p.s_b = s.state_b; p.s_d = s.state_d;
    p.batch = static_cast<int>(batch);
    p.Dm = static_cast<int>(Dm);
    p.N = static_cast<int>(N);
    // vector path: whole state quads, 16-byte aligned state and A_log rows, B/C quads aligned
    r.vec = (N % 4 == 0) && aligned(state, 16) && aligned(A_log, 16) &&
            (s.state_d % 4 == 0 || Dm == 1) && (s.state_b % 4 == 0 || batch == 1) &&
            aligned(B, 4 * es) && aligned(C, 4 * es) && (s.B_b % 4 == 0 || batch == 1) &&
            (s.C_b % 4 == 0 || batch == 1);
    return r;
}

}  // namespace
}  // namespace selscan

extern "C" {

ss_status ss_step(float* state, const void* x, const void* delta_raw, const float* delta_bias,
                  const float* A_log, const void* B, const void* C, const float* D, const void* z,
                  void* y, int64_t batch, int64_t Dm, int64_t N, const ss_step_strides* strides,
                  void* stream_ptr) {
    const StepCheck c = step_check(state, x, delta_raw, delta_bias, A_log, B, C, D, z, y, batch, Dm, N, strides);
    if (c.status != SS_OK || c.empty) return c.status;
    return cuda_status(launch_step(c.p, c.bf16, c.vec, static_cast<cudaStream_t>(stream_ptr)));
}

ss_status ss_step_layers(const ss_step_layer* layers, int64_t n_layers, int64_t batch, int64_t Dm, int64_t N,
                         const ss_step_strides* strides, void* stream_ptr) {
    if (n_layers < 0) return SS_ERR_INVALID_ARG;
    if (n_layers > kStepMaxLayers) return SS_ERR_UNSUPPORTED;
    if (n_layers == 0) return SS_OK;
    if (!layers) return SS_ERR_INVALID_ARG;
    static_assert(sizeof(StepLayersParams) <= 32000, "kernel parameter block too large");
    StepLayersParams q;
    std::memset(&q, 0, sizeof(q));
    q.n_layers = static_cast<int>(n_layers);
    q.err = device_error_ptr();
    std::vector<StepCheck> cs;
    cs.reserve(static_cast<size_t>(n_layers));
    bool vec = true;
    for (int64_t l = 0; l < n_layers; ++l) {
        const ss_step_layer& L = layers[l];
        cs.push_back(step_check(L.state, L.x, L.delta_raw, L.delta_bias, L.A_log, L.B, L.C, L.D, L.z, L.y, batch,
                                Dm, N, strides));
        const StepCheck& c = cs.back();
        if (c.status != SS_OK) return c.status;
        if (c.empty) return SS_OK;          // sizes are shared: every layer is empty
        vec = vec && c.vec;
        if (l == 0) q.common = c.p;
        StepLayerPtrs& P = q.layer[l];
        P.state = L.state; P.x = L.x; P.delta = L.delta_raw; P.z = L.z; P.Bm = L.B; P.Cm = L.C;
        P.bias = L.delta_bias; P.A_log = L.A_log; P.Dv = L.D; P.y = L.y;
    }
    // the layers run at the same time: what one writes must not meet what another reads or writes
    for (int64_t a = 0; a < n_layers; ++a)
        for (int64_t b = 0; b < n_layers; ++b) {
            if (a == b) continue;
            const StepCheck& A = cs[static_cast<size_t>(a)];
            const StepCheck& Bc = cs[static_cast<size_t>(b)];
            if (overlap(A.out_y, Bc.out_y) || overlap(A.out_y, Bc.out_state) || overlap(A.out_state, Bc.out_state))
                return SS_ERR_INVALID_ARG;
            for (const Range& in : Bc.in)
                if (overlap(A.out_y, in) || overlap(A.out_state, in)) return SS_ERR_INVALID_ARG;
        }
    return cuda_status(launch_step_layers(q, cs[0].bf16, vec, static_cast<cudaStream_t>(stream_ptr)));
}

}  // extern "C"
