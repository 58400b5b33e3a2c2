// mk_api.cu -- host side of the C ABI declared in include/mk.h: argument
// validation, the per-(device, stream) workspace cache, TMA tensor maps, the
// role split between dispatch and compute CTAs, and error reporting.
//
// The split follows the mKernel design note that the number of SMs given to
// each CTA role is set from the tensor shapes ("UC Berkeley presenta mKernel
// ...", edge.aivizor.me, para. 3; lefilia.fr, para. 2): here it is the share
// of the gather's HBM time in the path's total time.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "mk.h"
#include "mk_common.h"

namespace mk {
cudaError_t launch_fused(const Params& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                         const CUtensorMap& y, int grid, cudaStream_t st);
cudaError_t launch_unfused(const Params& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                           const CUtensorMap& y, int grid, cudaStream_t st);
cudaError_t launch_ep(const Params& p, const CUtensorMap* a, const CUtensorMap& b, const CUtensorMap& b3, int grid,
                      cudaStream_t st);
cudaError_t set_kernel_attributes();
cudaError_t fused_max_blocks_per_sm(int* n);
cudaError_t read_and_clear_error(uint32_t out[4], cudaStream_t st);
void noalloc_forget_scratch();
}  // namespace mk

using namespace mk;

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultSpinNs = 2000000000LL;

struct DevInfo {
    bool ready = false;
    mk_status_t status = MK_OK;
    int sms = 0;
    int max_blocks = 0;
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuStreamWaitValue32_v11070 g_wait_value = nullptr;
thread_local mk_launch_info_t g_last_info{};
uint32_t g_last_err[4] = {0, 0, 0, 0};

struct WsEntry {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws;
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws_ep;  // expert-parallel layout (zeroed whole)

struct HostStage {
    void* ptr = nullptr;
    size_t bytes = 0;
    cudaStream_t copy = nullptr;     // streams finished result chunks to the host
    cudaEvent_t copied = nullptr;    // recorded on `copy` after the last chunk
    cudaEvent_t computed = nullptr;  // recorded on the caller's stream after the kernel (fallback)
    uint32_t* flags = nullptr;       // chunk flags: plain device memory (the driver's stream waits
                                     // do not accept stream-ordered pool memory)
    uint32_t seq = 0;                // calls made with this stage (chunk flags hold it)
};
std::map<std::pair<int, cudaStream_t>, HostStage> g_host_stage;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mk_status_t device_info(int* dev_out, DevInfo** info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return MK_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            d.status = MK_ERR_UNSUPPORTED;
        } else if (set_kernel_attributes() != cudaSuccess || fused_max_blocks_per_sm(&d.max_blocks) != cudaSuccess) {
            return MK_ERR_CUDA;
        } else if (d.max_blocks < 1) {
            d.status = MK_ERR_UNSUPPORTED;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return MK_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            // stream waits on a value in memory (optional: without them the host
            // entry point copies the results after the kernel instead)
            void* wf = nullptr;
            cudaDriverEntryPointQueryResult wq{};
            if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &wf, 11070, cudaEnableDefault, &wq) ==
                    cudaSuccess &&
                wq == cudaDriverEntryPointSuccess)
                g_wait_value = reinterpret_cast<PFN_cuStreamWaitValue32_v11070>(wf);
        }
        d.ready = true;
    }
    *dev_out = dev;
    *info = &d;
    return d.status;
}

mk_status_t validate_sizes(int T, int H, int E, int k, int F) {
    if (T < 0 || E < 1 || k < 1 || k > E || k > MAX_K) return MK_ERR_INVALID_ARG;
    if (E > MAX_E) return MK_ERR_UNSUPPORTED;
    if (H < 64 || F < 64 || H % 64 != 0 || F % 64 != 0) return MK_ERR_INVALID_ARG;
    if (H > 32768 || F > 32768) return MK_ERR_UNSUPPORTED;
    if (int64_t(T) * k >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    if (int64_t(E) * H >= (int64_t(1) << 31)) return MK_ERR_UNSUPPORTED;
    return MK_OK;
}

mk_config_t config_or_default(const mk_config_t* cfg) {
    mk_config_t c;
    mk_config_default(&c);
    if (cfg) c = *cfg;
    return c;
}

int grid_for(const DevInfo& d, const mk_config_t& c) {
    int grid = d.sms * (d.max_blocks > 0 ? d.max_blocks : 1);
    grid = grid > d.sms ? d.sms : grid;  // one CTA per SM: each holds ~200 KB smem and 512 TMEM columns
    if (c.grid_ctas > 0 && c.grid_ctas < grid) grid = c.grid_ctas;
    if (grid > MAX_GRID) grid = MAX_GRID;
    return grid;
}

// Role split from the shapes: the dispatch role gets the gather's share of
// the path's estimated time (row bytes moved at HBM rate vs. the FLOPs at
// tensor rate), and at least as many CTAs as the first wave of work items
// (one per compute CTA) needs gather units, for evenly loaded experts, so
// that every unit of those tiles is taken in the gather's first round; at
// most half of the grid.  Dispatch CTAs join the compute role once the
// gather queue is empty, so the gather's total CTA time is the same for any
// split; a larger one fills the first tiles sooner.  (One SM's bulk copies
// from HBM run at about 33 GB/s, so the gather's rate grows with its CTAs.)
// The gather's share of the path's estimated time, in CTAs of the grid.
int gather_share(int grid, int T, int H, int F, int k) {
    const double rows = double(T) * k;
    const double gather_s = rows * H * 4.0 / 6.0e12;
    const double gemm_s = 2.0 * rows * H * double(F) / 1.8e15;
    return int(std::ceil(grid * gather_s / (gather_s + gemm_s)));
}

int dispatch_split(int grid, int T, int H, int F, int E, int k, int tile_rows, int nb, int slots) {
    const double rows = double(T) * k;
    int d = gather_share(grid, T, H, F, k);
    // gather units of the tiles the first `grid` work items use
    const double rows_e = rows / E;
    const double tiles_e = std::ceil(rows_e / tile_rows);
    const double items_e = tiles_e * nb;
    const double experts_first = std::min(double(E), std::ceil(grid / std::max(items_e, 1.0)));
    const double units_first =
        experts_first * tiles_e * std::ceil(std::min(double(tile_rows), rows_e) / std::max(slots, 1));
    if (d < units_first) d = int(units_first);
    if (d < 4) d = 4;
    if (d > grid / 2) d = grid / 2;
    if (d < 1) d = 1;
    return d;
}

// Average expert rows fill at least two 128-row tiles.
bool wide_shape(int T, int E, int k) { return int64_t(T) * k >= int64_t(2 * BM) * E; }

// Where the GEMM's token rows come from.  STAGED: the dispatch role copies
// them into expert-contiguous tiles and flags each tile.  DIRECT: the GEMM's
// producer warps copy them from x themselves (no staging rows in the
// workspace, no gather role).  Dispatch-only always stages (it measures the
// gather).  AUTO: DIRECT for fine-grained routing (k >= 4) on wide tiles,
// where staging would copy T*k rows of x (0.9-1.1 GB on the skewed and
// imbalanced workloads) and direct rows measured 13-15% faster on GB300,
// and for problems with under 1 MiB of rows to stage; STAGED otherwise (the
// Mixtral-like layer, k = 2, runs 6% faster staged).
int resolve_gather(const mk_config_t& c, int T, int H, int E, int k) {
    if (c.mode == MK_MODE_DISPATCH_ONLY) return MK_GATHER_STAGED;
    if (c.gather != MK_GATHER_AUTO) return c.gather;
    // the injected fault withholds a staged tile's arrival count
    if (c.debug_fault != MK_FAULT_NONE) return MK_GATHER_STAGED;
    if (c.mma_pair == MK_MMA_PAIR || c.mma_pair == MK_MMA_SINGLE) return MK_GATHER_STAGED;
    const bool fits = uint64_t(T) * uint64_t(H) * 2 < (uint64_t(1) << 32);  // 32-bit row offsets into x
    // Under 1 MiB of rows to stage the gather is pure latency before the
    // first tile (measured on GB300, the tiny layer: 0.028-0.029 ms direct
    // against 0.030-0.032 staged).
    const bool small = uint64_t(T) * uint64_t(k) * uint64_t(H) * 2 < (uint64_t(1) << 20);
    return ((k >= 4 && wide_shape(T, E, k)) || small) && fits ? MK_GATHER_DIRECT : MK_GATHER_STAGED;
}

// Tile height.  AUTO: 256-row tiles on one SM (WIDE) when the average expert
// holds at least two 128-row tiles; 128-row tiles otherwise.  Measured on
// GB300: WIDE is 5-14% faster on the Mixtral-like, skewed and imbalanced
// workloads (plain and gated FFN) with staged rows, 15-23% with direct rows,
// and 2% slower on decode (4 rows per expert).  SM pairs only when asked.
int resolve_pair(const mk_config_t& c, int T, int E, int k) {
    if (c.mma_pair != MK_MMA_AUTO) return c.mma_pair;
    if (c.mode == MK_MODE_DISPATCH_ONLY) return MK_MMA_SINGLE;
    return wide_shape(T, E, k) ? MK_MMA_WIDE : MK_MMA_SINGLE;
}

// Work order within an expert: whole expert weight reused through L2 when it
// is small (N-group = all N-blocks, tiles outer); otherwise groups of
// N-blocks whose weight slices total ~8 MB.
// N-blocks per group of the work order, chosen so the weight slices one
// group streams stay in L2 while all its tiles use them.  `sharers` groups
// stream at the same time (the ranks of the expert-parallel simulation, each
// on its own experts), so they share a budget of 16 MB.  Measured on GB300
// (Mixtral-like layer, 2 MB per slice): groups of 4 N-blocks 0.636 ms, 8:
// 0.640, 16: 0.640, 28: 0.655, all 56: 0.670.
int n_group_for(int H, int F, int nb, int sharers = 1) {
    const double w_bytes = double(H) * F * 2.0;
    if (w_bytes <= 32.0 * 1024 * 1024 / sharers) return nb;
    const double budget = sharers == 1 ? 8.0 * 1024 * 1024 : 16.0 * 1024 * 1024 / sharers;
    int g = int(budget / (double(H) * BN * 2.0));
    if (g < 1) g = 1;
    if (g > nb) g = nb;
    return g;
}

CUresult encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// The library's workspace for (device, stream), grown on demand.  The new
// buffer's bookkeeping part (everything before the staging rows) is zeroed.
mk_status_t cached_workspace(int dev, cudaStream_t st, size_t need, size_t zero_bytes, void** out, bool ep = false) {
    std::lock_guard<std::mutex> lock(g_mu);
    WsEntry& w = ep ? g_ws_ep[{dev, st}] : g_ws[{dev, st}];
    if (w.bytes < need) {
        if (w.ptr && cudaFreeAsync(w.ptr, st) != cudaSuccess) return MK_ERR_CUDA;
        w.ptr = nullptr;
        w.bytes = 0;
        size_t grow = need + need / 4;
        if (cudaMallocAsync(&w.ptr, grow, st) != cudaSuccess) {
            w.ptr = nullptr;
            return MK_ERR_CUDA;
        }
        if (cudaMemsetAsync(w.ptr, 0, ep ? grow : zero_bytes, st) != cudaSuccess) return MK_ERR_CUDA;
        w.bytes = grow;
    }
    *out = w.ptr;
    return MK_OK;
}

}  // namespace

extern "C" {

void mk_config_default(mk_config_t* cfg) {
    if (!cfg) return;
    std::memset(cfg, 0, sizeof(*cfg));
    cfg->mode = MK_MODE_FUSED;
    cfg->out_dtype = MK_OUT_BF16;
}

int mk_version(void) { return 100; }

const char* mk_status_string(mk_status_t s) {
    switch (s) {
        case MK_OK: return "MK_OK";
        case MK_ERR_INVALID_ARG: return "MK_ERR_INVALID_ARG";
        case MK_ERR_UNSUPPORTED: return "MK_ERR_UNSUPPORTED";
        case MK_ERR_CUDA: return "MK_ERR_CUDA";
        case MK_ERR_TIMEOUT: return "MK_ERR_TIMEOUT";
        case MK_ERR_DEVICE_FAULT: return "MK_ERR_DEVICE_FAULT";
        case MK_ERR_NOT_IMPLEMENTED: return "MK_ERR_NOT_IMPLEMENTED";
        case MK_ERR_WORKSPACE: return "MK_ERR_WORKSPACE";
    }
    return "MK_ERR_UNKNOWN";
}

size_t mk_workspace_size(int T, int H, int F, int E, int k, const mk_config_t* cfg) {
    (void)cfg;
    if (validate_sizes(T, H, E, k, F) != MK_OK) return 0;
    const mk_config_t c = config_or_default(cfg);
    return ws_layout(T, H, E, k, resolve_gather(c, T, H, E, k) == MK_GATHER_STAGED).total;
}

}  // extern "C"

namespace {

// Streamed results: chunk counters and flags in device memory, rows per
// chunk, and this call's sequence number (see Params::stream_done).
struct StreamOut {
    uint32_t* done;
    uint32_t* flag;
    int rows;
    uint32_t seq;
};

// The whole path; with combine_out it also combines each token's expert
// rows (gated sum) into combine_out[T,F].  With `so` (fused single-SM path
// only, else MK_ERR_UNSUPPORTED) the kernel also raises each result chunk's
// flag as it completes.
mk_status_t run_path(const void* x, const float* logits, int T, int H, int E, int k, const void* W, const void* W3,
                     int F, void* y_sorted, int32_t* src_index, int32_t* expert_offsets, float* gate_w,
                     void* combine_out, void* stream, const mk_config_t* cfg_in, void* workspace, size_t ws_bytes,
                     const StreamOut* so = nullptr) {
    g_last_info = mk_launch_info_t{};
    mk_status_t s = validate_sizes(T, H, E, k, F);
    if (s != MK_OK) return s;
    const mk_config_t c = config_or_default(cfg_in);
    for (int i = 0; i < 4; ++i)
        if (c.reserved[i] != 0) return MK_ERR_INVALID_ARG;
    if (c.mma_pair < MK_MMA_AUTO || c.mma_pair > MK_MMA_WIDE) return MK_ERR_INVALID_ARG;
    if (c.gather < MK_GATHER_AUTO || c.gather > MK_GATHER_GATHER4) return MK_ERR_INVALID_ARG;
    if (c.mode < MK_MODE_FUSED || c.mode > MK_MODE_DISPATCH_ONLY) return MK_ERR_INVALID_ARG;
    if (c.out_dtype != MK_OUT_BF16 && c.out_dtype != MK_OUT_F32) return MK_ERR_INVALID_ARG;
    if (c.debug_fault != MK_FAULT_NONE && c.debug_fault != MK_FAULT_DROP_TILE_FLAG) return MK_ERR_INVALID_ARG;
    if (c.dispatch_ctas < 0 || c.grid_ctas < 0 || c.n_group < 0 || c.spin_limit_ns < 0) return MK_ERR_INVALID_ARG;
    if (!expert_offsets || !aligned(expert_offsets, 4)) return MK_ERR_INVALID_ARG;
    if (T > 0) {
        if (!x || !logits || !W || !src_index || !gate_w) return MK_ERR_INVALID_ARG;
        if (!y_sorted && c.mode != MK_MODE_DISPATCH_ONLY) return MK_ERR_INVALID_ARG;
        if (!aligned(x, 16) || !aligned(W, 16) || !aligned(logits, 4) || !aligned(src_index, 4) ||
            !aligned(gate_w, 4))
            return MK_ERR_INVALID_ARG;
        if (y_sorted && !aligned(y_sorted, 16)) return MK_ERR_INVALID_ARG;
        if (combine_out && (!aligned(combine_out, 16) || c.mode == MK_MODE_DISPATCH_ONLY)) return MK_ERR_INVALID_ARG;
        if (W3 && !aligned(W3, 16)) return MK_ERR_INVALID_ARG;
    }
    int dev = 0;
    DevInfo* d = nullptr;
    if ((s = device_info(&dev, &d)) != MK_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (T == 0) {
        g_last_info.launches = 0;
        return cudaMemsetAsync(expert_offsets, 0, size_t(E + 1) * 4, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }

    const int gather = resolve_gather(c, T, H, E, k);
    const bool direct = gather != MK_GATHER_STAGED;  // rows straight from x: cp.async or TMA gather4
    const bool gather4 = gather == MK_GATHER_GATHER4;
    const int mma = resolve_pair(c, T, E, k);
    const bool pair = mma == MK_MMA_PAIR, wide = mma == MK_MMA_WIDE;
    if (pair && W3) return MK_ERR_UNSUPPORTED;  // the gated FFN runs on single-SM tiles
    if (direct && pair) return MK_ERR_UNSUPPORTED;  // SM pairs load staged rows only
    // direct rows are addressed with 32-bit byte offsets into x
    if (direct && uint64_t(T) * uint64_t(H) * 2 >= (uint64_t(1) << 32)) return MK_ERR_UNSUPPORTED;
    int grid = grid_for(*d, c);
    if (pair) grid &= ~1;  // whole clusters of two
    if (grid < (pair ? 2 : 1)) return MK_ERR_UNSUPPORTED;
    const int rows = T * k;
    const int route_lanes = route_lanes_for(T, E, grid, aligned(logits, 16));
    const int route_chunk = ROUTE_CHUNK / route_lanes;
    const int nch = (T + route_chunk - 1) / route_chunk;
    if (nch > grid * MAX_CHUNKS_PER_CTA) return MK_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(T, H, E, k, !direct);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (ws) {
        if (ws_bytes < L.total || !aligned(ws, 256)) return MK_ERR_WORKSPACE;
    } else {
        void* p = nullptr;
        if ((s = cached_workspace(dev, st, L.total, L.xs, &p)) != MK_OK) return s;
        ws = static_cast<uint8_t*>(p);
    }

    Params p{};
    p.x = static_cast<const uint16_t*>(x);
    p.logits = logits;
    p.W = static_cast<const uint16_t*>(W);
    p.y = y_sorted;
    p.src_index = src_index;
    p.expert_offsets = expert_offsets;
    p.gate_w = gate_w;
    p.T = T;
    p.H = H;
    p.F = F;
    p.E = E;
    p.k = k;
    p.out_f32 = c.out_dtype == MK_OUT_F32;
    p.y_v8 = aligned(y_sorted, 32) ? 1 : 0;
    p.rows = rows;
    p.nch = nch;
    p.route_lanes = route_lanes;
    p.route_chunk = route_chunk;
    p.gated = W3 ? 1 : 0;
    p.W3 = static_cast<const uint16_t*>(W3);
    const int bnw = W3 ? BN / 2 : BN;  // gated: 128 columns of each projection per item
    p.nb = (F + bnw - 1) / bnw;
    p.kblocks = H / BK;
    p.n_group = c.n_group > 0 ? (c.n_group < p.nb ? c.n_group : p.nb) : n_group_for(H, F, p.nb);
    p.mode = c.mode;
    p.compute = c.mode != MK_MODE_DISPATCH_ONLY;
    p.direct = direct ? 1 : 0;
    p.gather4 = gather4 ? 1 : 0;
    {
        int slots = int((SM_STAGE_END) / (size_t(H) * 2));
        p.gather_slots = slots > MAX_GATHER_SLOTS ? MAX_GATHER_SLOTS : slots;
        // several gathering warps only where tiles are whole: with a few rows
        // per expert (decode) smaller units would mostly be empty
        p.gather_warps = wide_shape(T, E, k) ? std::min(GATHER_WARPS, p.gather_slots) : 1;
    }
    if (c.mode == MK_MODE_DISPATCH_ONLY) {
        p.dispatch_ctas = grid;
    } else if (direct) {
        p.dispatch_ctas = 0;  // rows go straight into the GEMM's shared memory: no gather role
    } else {
        p.dispatch_ctas = c.dispatch_ctas > 0 ? c.dispatch_ctas
                                              : dispatch_split(grid, T, H, F, E, k, pair ? PAIR_TILE_M
                                                                                       : wide ? WIDE_TILE_M : BM,
                                                               p.nb, p.gather_slots);
        if (p.dispatch_ctas > grid) p.dispatch_ctas = grid;
        if (pair) p.dispatch_ctas = (p.dispatch_ctas + 1) & ~1;  // both CTAs of a cluster share a role
        if (p.dispatch_ctas > grid) p.dispatch_ctas = grid;
    }
    p.pair = pair ? 1 : 0;
    p.wide = wide ? 1 : 0;
    p.tile_rows = pair ? PAIR_TILE_M : wide ? WIDE_TILE_M : BM;
    p.debug_drop_tile = c.debug_fault == MK_FAULT_DROP_TILE_FLAG ? 0 : -1;
    // measured on GB300: issuing L2 prefetches from the producer thread slows
    // the loads behind them, so it is off unless asked for
    p.l2_prefetch = c.l2_prefetch > 0 ? c.l2_prefetch : 0;
    p.trace = c.trace ? 1 : 0;
    p.spin_limit_ns = c.spin_limit_ns > 0 ? c.spin_limit_ns : kDefaultSpinNs;
    p.ctl = reinterpret_cast<Ctl*>(ws + L.ctl);
    p.counts = reinterpret_cast<int32_t*>(ws + L.counts);
    p.topk_idx = reinterpret_cast<int32_t*>(ws + L.topk_idx);
    p.topk_gate = reinterpret_cast<float*>(ws + L.topk_gate);
    p.lrank = reinterpret_cast<int32_t*>(ws + L.lrank);
    p.bases = reinterpret_cast<int32_t*>(ws + L.bases);
    p.totals = reinterpret_cast<int32_t*>(ws + L.totals);
    p.dist_scan = int64_t(nch) * E > DIST_SCAN_COUNTS ? 1 : 0;
    p.row_of = reinterpret_cast<int32_t*>(ws + L.row_of);
    p.combine_out = combine_out;
    p.ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    p.xs = reinterpret_cast<uint16_t*>(ws + L.xs);
    p.trace_buf = reinterpret_cast<unsigned long long*>(ws + L.trace);
    p.max_tiles = (rows + p.tile_rows - 1) / p.tile_rows + E;
    p.ranks = 1;  // routing chunks over [0, T)
    p.ep_t0[1] = T;
    p.ep_c0[1] = nch;
    if (so) {
        if (c.mode != MK_MODE_FUSED || pair || so->rows < 1) return MK_ERR_UNSUPPORTED;
        p.stream_done = so->done;
        p.stream_flag = so->flag;
        p.stream_rows = so->rows;
        p.stream_seq = so->seq;
    }

    CUtensorMap tmA, tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    const uint32_t kbox = BK;  // boxes hold one stage's rows of K
    // A: the staging rows (staged); with TMA gather4, x itself in boxes one row
    // high; encoded over x and unused with cp.async rows
    if (encode_2d(&tmA, direct ? x : static_cast<const void*>(p.xs), uint64_t(H), uint64_t(direct ? T : rows),
                  uint64_t(H) * 2, kbox, gather4 ? 1 : BM) != CUDA_SUCCESS)
        return MK_ERR_CUDA;
    if (encode_2d(&tmB, W, uint64_t(F), uint64_t(E) * H, uint64_t(F) * 2, 64, kbox) != CUDA_SUCCESS)
        return MK_ERR_CUDA;
    CUtensorMap tmB3 = tmB;
    if (W3 && encode_2d(&tmB3, W3, uint64_t(F), uint64_t(E) * H, uint64_t(F) * 2, 64, kbox) != CUDA_SUCCESS)
        return MK_ERR_CUDA;
    // bf16 results in whole 32-row groups go out as tensor stores of 32 x 64
    // boxes (not with f32 output, nor with streamed results, whose chunk
    // counts follow per-row stores)
    CUtensorMap tmY;
    std::memset(&tmY, 0, sizeof(tmY));
    p.y_tma = 0;
    if (c.mode != MK_MODE_DISPATCH_ONLY && !p.out_f32 && !so) {
        if (encode_2d(&tmY, y_sorted, uint64_t(F), uint64_t(rows), uint64_t(F) * 2, EPI_BOX_COLS, EPI_BOX_ROWS) !=
            CUDA_SUCCESS)
            return MK_ERR_CUDA;
        p.y_tma = 1;
    }

    if (p.trace && cudaMemsetAsync(p.trace_buf, 0, size_t(grid) * TRACE_SLOTS * 8, st) != cudaSuccess)
        return MK_ERR_CUDA;

    cudaError_t err;
    if (c.mode == MK_MODE_UNFUSED) {
        err = launch_unfused(p, tmA, tmB, tmB3, tmY, grid, st);
        g_last_info.launches = combine_out ? 5 : 4;
    } else {
        err = launch_fused(p, tmA, tmB, tmB3, tmY, grid, st);
        g_last_info.launches = 1;
    }
    g_last_info.grid_ctas = grid;
    g_last_info.dispatch_ctas = c.mode == MK_MODE_UNFUSED ? 0 : p.dispatch_ctas;
    g_last_info.n_group = p.n_group;
    g_last_info.mma_pair = mma;
    g_last_info.gather = gather;
    g_last_info.route_lanes = route_lanes;
    g_last_info.route_chunks = nch;
    g_last_info.workspace_bytes = int64_t(L.total);
    if (getenv("MK_LOG"))
        fprintf(stderr, "[mk] T=%d H=%d F=%d E=%d k=%d mode=%d grid=%d dispatch=%d n_group=%d slots=%d ws=%zu\n", T, H,
                F, E, k, c.mode, grid, p.dispatch_ctas, p.n_group, p.gather_slots, L.total);
    return err == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

// Expert parallelism simulated with `ranks` logical ranks in one launch.
mk_status_t run_ep(const void* x, const float* logits, int T, int H, int E, int k, const void* W, const void* W3,
                   int F, int ranks,
                   void* y_tok, int32_t* src_index, int32_t* expert_offsets, float* gate_w, void* out, void* stream,
                   const mk_config_t* cfg_in, void* workspace, size_t ws_bytes) {
    g_last_info = mk_launch_info_t{};
    mk_status_t s = validate_sizes(T, H, E, k, F);
    if (s != MK_OK) return s;
    if (ranks < 1 || ranks > MAX_RANKS || E % ranks != 0) return MK_ERR_INVALID_ARG;
    const mk_config_t c = config_or_default(cfg_in);
    for (int i = 0; i < 4; ++i)
        if (c.reserved[i] != 0) return MK_ERR_INVALID_ARG;
    if (c.mma_pair < MK_MMA_AUTO || c.mma_pair > MK_MMA_WIDE) return MK_ERR_INVALID_ARG;
    if (c.gather < MK_GATHER_AUTO || c.gather > MK_GATHER_GATHER4) return MK_ERR_INVALID_ARG;
    if (c.mode < MK_MODE_FUSED || c.mode > MK_MODE_DISPATCH_ONLY) return MK_ERR_INVALID_ARG;
    if (c.out_dtype != MK_OUT_BF16 && c.out_dtype != MK_OUT_F32) return MK_ERR_INVALID_ARG;
    if (c.debug_fault != MK_FAULT_NONE && c.debug_fault != MK_FAULT_DROP_TILE_FLAG) return MK_ERR_INVALID_ARG;
    if (c.dispatch_ctas < 0 || c.grid_ctas < 0 || c.n_group < 0 || c.spin_limit_ns < 0) return MK_ERR_INVALID_ARG;
    // one fused launch, staged rows, tiles on one SM (128-row or wide)
    if (c.mode != MK_MODE_FUSED || c.gather == MK_GATHER_DIRECT || c.gather == MK_GATHER_GATHER4 ||
        c.mma_pair == MK_MMA_PAIR)
        return MK_ERR_UNSUPPORTED;
    const bool wide = resolve_pair(c, T, E, k) == MK_MMA_WIDE;
    if (!expert_offsets || !aligned(expert_offsets, 4)) return MK_ERR_INVALID_ARG;
    if (T > 0) {
        if (!x || !logits || !W || !y_tok || !src_index || !gate_w) return MK_ERR_INVALID_ARG;
        if (W3 && !aligned(W3, 16)) return MK_ERR_INVALID_ARG;
        if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y_tok, 16) || !aligned(logits, 4) ||
            !aligned(src_index, 4) || !aligned(gate_w, 4))
            return MK_ERR_INVALID_ARG;
        if (out && !aligned(out, 16)) return MK_ERR_INVALID_ARG;
    }
    int dev = 0;
    DevInfo* d = nullptr;
    if ((s = device_info(&dev, &d)) != MK_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        g_last_info.launches = 0;
        return cudaMemsetAsync(expert_offsets, 0, size_t(E + 1) * 4, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }

    int grid = grid_for(*d, c);
    grid -= grid % ranks;  // whole ranks
    const int cpr = grid / ranks;
    if (cpr < 1) return MK_ERR_UNSUPPORTED;
    const EpLayout L = ep_layout(T, H, E, k, ranks);
    for (int r = 0; r < ranks; ++r) {
        const int nt = ep_token0(T, ranks, r + 1) - ep_token0(T, ranks, r);
        if ((nt + ROUTE_CHUNK - 1) / ROUTE_CHUNK > cpr * MAX_CHUNKS_PER_CTA) return MK_ERR_UNSUPPORTED;
    }
    const int bnw = W3 ? BN / 2 : BN;  // gated: 128 columns of each projection per item
    const int nb = (F + bnw - 1) / bnw;
    // completion counts: a rank's (row, N-block) results in 32 bits
    if (uint64_t(T) * uint64_t(k) * uint64_t(nb) >= (uint64_t(1) << 32)) return MK_ERR_UNSUPPORTED;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (ws) {
        if (ws_bytes < L.total || !aligned(ws, 256)) return MK_ERR_WORKSPACE;
    } else {
        void* pw = nullptr;
        if ((s = cached_workspace(dev, st, L.total, L.total, &pw, true)) != MK_OK) return s;
        ws = static_cast<uint8_t*>(pw);
    }

    Params p{};
    p.x = static_cast<const uint16_t*>(x);
    p.logits = logits;
    p.W = static_cast<const uint16_t*>(W);
    p.W3 = static_cast<const uint16_t*>(W3);
    p.gated = W3 ? 1 : 0;
    p.y = y_tok;
    p.src_index = src_index;
    p.expert_offsets = expert_offsets;
    p.gate_w = gate_w;
    p.T = T;
    p.H = H;
    p.F = F;
    p.E = E;
    p.k = k;
    p.out_f32 = c.out_dtype == MK_OUT_F32;
    p.y_v8 = aligned(y_tok, 32) ? 1 : 0;
    p.rows = T * k;
    p.nch = L.nch;
    p.route_lanes = 1;  // each rank's chunks keep a lane per token
    p.route_chunk = ROUTE_CHUNK;
    p.nb = nb;
    p.kblocks = H / BK;
    // ranks stream their own experts' weights at once, so they share L2
    p.n_group = c.n_group > 0 ? (c.n_group < nb ? c.n_group : nb) : n_group_for(H, F, nb, ranks);
    p.mode = MK_MODE_FUSED;
    p.compute = 1;
    p.wide = wide ? 1 : 0;
    p.tile_rows = wide ? WIDE_TILE_M : BM;
    {
        int slots = int((SM_STAGE_END) / (size_t(H) * 2));
        p.gather_slots = slots > MAX_GATHER_SLOTS ? MAX_GATHER_SLOTS : slots;
        p.gather_warps = 1;  // the expert-parallel send role copies with one warp
    }
    p.debug_drop_tile = c.debug_fault == MK_FAULT_DROP_TILE_FLAG ? 0 : -1;
    p.spin_limit_ns = c.spin_limit_ns > 0 ? c.spin_limit_ns : kDefaultSpinNs;
    p.ctl = reinterpret_cast<Ctl*>(ws + L.ctl);
    p.topk_idx = reinterpret_cast<int32_t*>(ws + L.topk_idx);
    p.topk_gate = reinterpret_cast<float*>(ws + L.topk_gate);
    p.lrank = reinterpret_cast<int32_t*>(ws + L.lrank);
    p.row_of = reinterpret_cast<int32_t*>(ws + L.row_of);
    p.combine_out = out;
    p.trace_buf = reinterpret_cast<unsigned long long*>(ws + L.trace);
    p.ranks = ranks;
    int c0 = 0;
    for (int r = 0; r <= ranks; ++r) {
        p.ep_t0[r] = ep_token0(T, ranks, r);
        p.ep_c0[r] = c0;
        if (r < ranks) c0 += (ep_token0(T, ranks, r + 1) - ep_token0(T, ranks, r) + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    }
    p.ep = 1;
    p.ep_cpr = cpr;
    {
        // Every tile waits for the rows of all R sources, so each rank's send
        // role must be quick: about 64 sending CTAs in all (at most half of a
        // rank's) measured best or near it on GB300 for R = 2..8; they join
        // the GEMM once their rows are out.
        int want = c.dispatch_ctas > 0 ? c.dispatch_ctas : std::max(4, std::min(grid / 2, gather_share(grid, T, H, F, k)));
        if (c.dispatch_ctas <= 0 && ranks > 1 && want < 64) want = 64;
        int per = (want + ranks - 1) / ranks;
        if (c.dispatch_ctas <= 0 && ranks > 1 && per > cpr / 2) per = cpr / 2;
        p.ep_dispatch = per < 1 ? 1 : (per > cpr ? cpr : per);
    }
    p.ep_tile_cap = L.tile_cap;
    p.ep_cap_rows = int(L.cap_rows);
    CUtensorMap tmA[MAX_RANKS], tmB;
    std::memset(tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    const uint32_t kbox = BK;  // boxes hold one stage's rows of K
    for (int r = 0; r < ranks; ++r) {
        uint8_t* base = ws + L.rank_base[r];
        p.ep_ctl[r] = reinterpret_cast<EpCtl*>(ws + L.ep_ctl) + r;
        p.ep_counts[r] = reinterpret_cast<int32_t*>(base + L.counts_off);
        p.ep_ready[r] = reinterpret_cast<uint32_t*>(base + L.ready_off);
        p.ep_recv[r] = reinterpret_cast<uint16_t*>(base + L.recv_off);
        if (encode_2d(&tmA[r], p.ep_recv[r], uint64_t(H), uint64_t(L.cap_rows), uint64_t(H) * 2, kbox, BM) !=
            CUDA_SUCCESS)
            return MK_ERR_CUDA;
    }
    if (encode_2d(&tmB, W, uint64_t(F), uint64_t(E) * H, uint64_t(F) * 2, 64, kbox) != CUDA_SUCCESS)
        return MK_ERR_CUDA;
    CUtensorMap tmB3 = tmB;
    if (W3 && encode_2d(&tmB3, W3, uint64_t(F), uint64_t(E) * H, uint64_t(F) * 2, 64, kbox) != CUDA_SUCCESS)
        return MK_ERR_CUDA;

    const cudaError_t err = launch_ep(p, tmA, tmB, tmB3, grid, st);
    g_last_info.launches = 1;
    g_last_info.grid_ctas = grid;
    g_last_info.dispatch_ctas = p.ep_dispatch * ranks;
    g_last_info.n_group = p.n_group;
    g_last_info.mma_pair = wide ? MK_MMA_WIDE : MK_MMA_SINGLE;
    g_last_info.gather = MK_GATHER_STAGED;
    g_last_info.route_lanes = 1;
    g_last_info.route_chunks = L.nch;
    g_last_info.workspace_bytes = int64_t(L.total);
    return err == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // namespace

extern "C" {

mk_status_t mk_moe_ep_sim(const void* x, const float* logits, int T, int H, int E, int k, const void* W, int F,
                          int ranks, void* y_tok, int32_t* src_index, int32_t* expert_offsets, float* gate_w,
                          void* out, void* stream, const mk_config_t* cfg, void* workspace, size_t ws_bytes) {
    return run_ep(x, logits, T, H, E, k, W, nullptr, F, ranks, y_tok, src_index, expert_offsets, gate_w, out, stream,
                  cfg, workspace, ws_bytes);
}

mk_status_t mk_moe_ep_sim_gated(const void* x, const float* logits, int T, int H, int E, int k, const void* W1,
                                const void* W3, int F, int ranks, void* h_tok, int32_t* src_index,
                                int32_t* expert_offsets, float* gate_w, void* out, void* stream,
                                const mk_config_t* cfg, void* workspace, size_t ws_bytes) {
    if (T > 0 && !W3) return MK_ERR_INVALID_ARG;
    return run_ep(x, logits, T, H, E, k, W1, T > 0 ? W3 : nullptr, F, ranks, h_tok, src_index, expert_offsets,
                  gate_w, out, stream, cfg, workspace, ws_bytes);
}

size_t mk_ep_workspace_size(int T, int H, int F, int E, int k, int ranks) {
    if (validate_sizes(T, H, E, k, F) != MK_OK || ranks < 1 || ranks > MAX_RANKS || E % ranks != 0) return 0;
    return ep_layout(T, H, E, k, ranks).total;
}

mk_status_t mk_moe_dispatch_gemm_ex(const void* x, const float* logits, int T, int H, int E, int k, const void* W,
                                    int F, void* y_sorted, int32_t* src_index, int32_t* expert_offsets,
                                    float* gate_w, void* stream, const mk_config_t* cfg, void* workspace,
                                    size_t ws_bytes) {
    return run_path(x, logits, T, H, E, k, W, nullptr, F, y_sorted, src_index, expert_offsets, gate_w, nullptr,
                    stream, cfg, workspace, ws_bytes);
}

mk_status_t mk_moe_dispatch_gated(const void* x, const float* logits, int T, int H, int E, int k, const void* W1,
                                  const void* W3, int F, void* h_sorted, int32_t* src_index, int32_t* expert_offsets,
                                  float* gate_w, void* stream, const mk_config_t* cfg, void* workspace,
                                  size_t ws_bytes) {
    if (T > 0 && !W3) return MK_ERR_INVALID_ARG;
    return run_path(x, logits, T, H, E, k, W1, T > 0 ? W3 : nullptr, F, h_sorted, src_index, expert_offsets, gate_w,
                    nullptr, stream, cfg, workspace, ws_bytes);
}

mk_status_t mk_moe_dispatch_gemm_combine(const void* x, const float* logits, int T, int H, int E, int k,
                                         const void* W, int F, void* y_sorted, int32_t* src_index,
                                         int32_t* expert_offsets, float* gate_w, void* out, void* stream,
                                         const mk_config_t* cfg, void* workspace, size_t ws_bytes) {
    if (T > 0 && !out) return MK_ERR_INVALID_ARG;
    return run_path(x, logits, T, H, E, k, W, nullptr, F, y_sorted, src_index, expert_offsets, gate_w, out, stream,
                    cfg, workspace, ws_bytes);
}

mk_status_t mk_moe_dispatch_gemm(const void* x, const float* logits, int T, int H, int E, int k, const void* W, int F,
                                 void* y_sorted, int32_t* src_index, int32_t* expert_offsets, float* gate_w,
                                 void* stream) {
    return mk_moe_dispatch_gemm_ex(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w, stream,
                                   nullptr, nullptr, 0);
}

mk_status_t mk_moe_dispatch_gemm_host(const void* x_host, const float* logits_host, int T, int H, int E, int k,
                                      const void* W, int F, void* y_sorted_host, int32_t* src_index_host,
                                      int32_t* expert_offsets_host, float* gate_w_host, void* stream,
                                      const mk_config_t* cfg) {
    mk_status_t s = validate_sizes(T, H, E, k, F);
    if (s != MK_OK) return s;
    mk_config_t c = config_or_default(cfg);
    if (!expert_offsets_host) return MK_ERR_INVALID_ARG;
    if (T > 0 && (!x_host || !logits_host || !W || !y_sorted_host || !src_index_host || !gate_w_host))
        return MK_ERR_INVALID_ARG;
    int dev = 0;
    DevInfo* d = nullptr;
    if ((s = device_info(&dev, &d)) != MK_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t rows = size_t(T) * k;
    const size_t row_bytes = size_t(F) * (c.out_dtype == MK_OUT_F32 ? 4 : 2);
    const size_t ybytes = rows * row_bytes;
    // The results go back in chunks of sorted rows as the kernel completes
    // them, on a second stream, so the copy overlaps the GEMM (the host link,
    // not the GPU, bounds this call).  The fused single-SM path raises the
    // chunk flags; other configurations copy after the kernel.
    const bool streamed = T > 0 && g_wait_value && c.mode == MK_MODE_FUSED && c.mma_pair != MK_MMA_PAIR;
    if (!streamed && getenv("MK_LOG"))
        fprintf(stderr, "[mk] host entry: results copied after the kernel (stream waits %s)\n",
                g_wait_value ? "available" : "unavailable");
    // The copy can start only once the first chunk is complete in all its
    // N-blocks.  Unless the caller fixed the work order, take each expert's
    // tiles one after the other (all N-blocks of a tile together), so the
    // sorted rows complete in order from the first wave of items on; the
    // kernel is a little slower that way, but it stays well ahead of the
    // host link.  Measured on GB300 (Mixtral-like layer, 235 MB of results):
    // the call takes 1.565 ms instead of 1.622.
    if (streamed && c.n_group == 0) c.n_group = 1 << 20;  // clamped to the N-blocks per tile
    // Chunks are whole 256-row tiles (a multiple of either tile height), at
    // most 64 of them.  Copies grow: one chunk, one, two, four, ... so the
    // first leaves early and the later ones run at the link's full rate.
    constexpr int kMaxChunks = 64;
    const size_t per = (rows + kMaxChunks - 1) / kMaxChunks;
    const int srows = int((per + 255) / 256 * 256);
    const int nchunks = int((rows + srows - 1) / srows);  // <= kMaxChunks
    const size_t o_x = 0, o_l = ws_align(o_x + size_t(T) * H * 2), o_y = ws_align(o_l + size_t(T) * E * 4),
                 o_s = ws_align(o_y + ybytes), o_o = ws_align(o_s + rows * 4), o_g = ws_align(o_o + size_t(E + 1) * 4),
                 o_done = ws_align(o_g + rows * 4), total = ws_align(o_done + size_t(nchunks) * 4);
    uint8_t* base = nullptr;
    HostStage* hs = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        HostStage& h = g_host_stage[{dev, st}];
        if (h.bytes < total) {
            if (h.ptr && cudaFreeAsync(h.ptr, st) != cudaSuccess) return MK_ERR_CUDA;
            h.ptr = nullptr;
            h.bytes = 0;
            if (cudaMallocAsync(&h.ptr, total, st) != cudaSuccess) return MK_ERR_CUDA;
            h.bytes = total;

        }
        if (streamed && !h.copy) {
            if (cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&h.copied, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h.computed, cudaEventDisableTiming) != cudaSuccess ||
                cudaMalloc(&h.flags, kMaxChunks * sizeof(uint32_t)) != cudaSuccess ||
                cudaMemset(h.flags, 0, kMaxChunks * sizeof(uint32_t)) != cudaSuccess)  // below every sequence number
                return MK_ERR_CUDA;
        }
        base = static_cast<uint8_t*>(h.ptr);
        hs = &h;
    }
    if (T > 0) {
        if (cudaMemcpyAsync(base + o_x, x_host, size_t(T) * H * 2, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(base + o_l, logits_host, size_t(T) * E * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return MK_ERR_CUDA;
    }
    StreamOut so{reinterpret_cast<uint32_t*>(base + o_done), hs->flags, srows, 0u};
    if (streamed) so.seq = ++hs->seq;
    s = run_path(base + o_x, reinterpret_cast<const float*>(base + o_l), T, H, E, k, W, nullptr, F, base + o_y,
                 reinterpret_cast<int32_t*>(base + o_s), reinterpret_cast<int32_t*>(base + o_o),
                 reinterpret_cast<float*>(base + o_g), nullptr, stream, &c, nullptr, 0, streamed ? &so : nullptr);
    if (s != MK_OK) return s;
    if (streamed) {
        // chunk i is copied once the kernel has raised its flag to this call's
        // number (the last CTA out raises every flag, even if the call gave up).
        // If the driver refuses a wait, the remaining chunks wait for the whole
        // kernel instead.
        bool waits = true;
        int wait_err = 0;
        int ncopies = 0;
        for (int i = 0, g = 1; i < nchunks; ++ncopies) {
            const int i_end = std::min(nchunks, i + g);
            const size_t r0 = size_t(i) * srows, r1 = std::min(rows, size_t(i_end) * srows);
            for (; i < i_end; ++i) {
                CUresult wr = CUDA_SUCCESS;
                if (waits && (wr = g_wait_value(hs->copy, reinterpret_cast<CUdeviceptr>(so.flag + i), so.seq,
                                                CU_STREAM_WAIT_VALUE_GEQ)) != CUDA_SUCCESS) {
                    waits = false;
                    wait_err = int(wr);
                    if (cudaEventRecord(hs->computed, st) != cudaSuccess ||
                        cudaStreamWaitEvent(hs->copy, hs->computed, 0) != cudaSuccess)
                        return MK_ERR_CUDA;
                }
            }
            if (cudaMemcpyAsync(static_cast<uint8_t*>(y_sorted_host) + r0 * row_bytes, base + o_y + r0 * row_bytes,
                                (r1 - r0) * row_bytes, cudaMemcpyDeviceToHost, hs->copy) != cudaSuccess)
                return MK_ERR_CUDA;
            if (ncopies > 0) g *= 2;
        }
        if (getenv("MK_LOG"))
            fprintf(stderr, "[mk] host entry: %d result chunks of %d rows streamed in %d copies, stream waits %s (%d)\n",
                    nchunks, srows, ncopies, waits ? "used" : "refused, copies follow the kernel", wait_err);
    }
    // the small outputs follow the kernel on `stream`, beside the streamed rows
    if (cudaMemcpyAsync(expert_offsets_host, base + o_o, size_t(E + 1) * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MK_ERR_CUDA;
    if (T > 0) {
        if ((!streamed && cudaMemcpyAsync(y_sorted_host, base + o_y, ybytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
            cudaMemcpyAsync(src_index_host, base + o_s, rows * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaMemcpyAsync(gate_w_host, base + o_g, rows * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return MK_ERR_CUDA;
    }
    if (streamed &&
        (cudaEventRecord(hs->copied, hs->copy) != cudaSuccess || cudaStreamWaitEvent(st, hs->copied, 0) != cudaSuccess))
        return MK_ERR_CUDA;
    return mk_get_status(stream);
}

mk_status_t mk_get_status(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the read of the error word is ordered after all of the stream's work,
    // and synchronises with it
    uint32_t e[4] = {0, 0, 0, 0};
    if (read_and_clear_error(e, st) != cudaSuccess) return MK_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MK_ERR_CUDA;
    if (e[0] == ERR_NONE) return MK_OK;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        std::memcpy(g_last_err, e, sizeof(e));
    }
    return e[0] == ERR_TIMEOUT ? MK_ERR_TIMEOUT : MK_ERR_DEVICE_FAULT;
}

void mk_last_error_detail(int32_t* site, int32_t* cta, int32_t* info) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (site) *site = int32_t(g_last_err[1]);
    if (cta) *cta = int32_t(g_last_err[2]);
    if (info) *info = int32_t(g_last_err[3]);
}

void mk_last_launch_info(mk_launch_info_t* info) {
    if (info) *info = g_last_info;
}

mk_status_t mk_read_trace(void* stream, const void* workspace, int T, int H, int E, int k, uint64_t* out, size_t n) {
    if (!out) return MK_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    if (!ws) {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_ws.find({dev, st});
        if (it == g_ws.end()) return MK_ERR_INVALID_ARG;
        ws = static_cast<const uint8_t*>(it->second.ptr);
    }
    const WsLayout L = ws_layout(T, H, E, k);
    const size_t want = size_t(MAX_GRID) * TRACE_SLOTS;
    const size_t cnt = n < want ? n : want;
    if (cudaMemcpyAsync(out, ws + L.trace, cnt * 8, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MK_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

void mk_release_workspace(void) {
    noalloc_forget_scratch();  // the allocation-free entry point looks its array up again
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    // streams may be gone by now: synchronise the device, then free
    for (auto& kv : g_ws) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        cudaFree(kv.second.ptr);
    }
    g_ws.clear();
    for (auto& kv : g_ws_ep) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        cudaFree(kv.second.ptr);
    }
    g_ws_ep.clear();
    for (auto& kv : g_host_stage) {
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        if (kv.second.ptr) cudaFree(kv.second.ptr);
        if (kv.second.copy) cudaStreamDestroy(kv.second.copy);
        if (kv.second.copied) cudaEventDestroy(kv.second.copied);
        if (kv.second.computed) cudaEventDestroy(kv.second.computed);
        if (kv.second.flags) cudaFree(kv.second.flags);
    }
    g_host_stage.clear();
    cudaSetDevice(cur);
}

}  // extern "C"
