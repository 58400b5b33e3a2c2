// mk_common.h -- constants and parameter blocks shared by the host launcher
// and the device code of the MoE dispatch + expert-GEMM library.
#pragma once

#include <cstddef>
#include <cstdint>

namespace mk {

// Tile shape of the expert GEMM: one CTA computes a BM x BN block of
// y_sorted with tcgen05.mma (M = 128, N = 256, K = 16 per instruction),
// K staged through shared memory BK = 64 bf16 (one 128-byte swizzle row).
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;            // 16 KiB
constexpr int B_CHUNK_BYTES = BK * 64 * 2;            //  8 KiB: 64 rows of K x 64 columns of N
constexpr int B_STAGE_BYTES = BK * BN * 2;            // 32 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;                     // two fp32 accumulators
constexpr int EPI_WARP_END = 6;                       // warps 2..5: epilogue (TMEM lane quads 2, 3, 0, 1)
// Direct gather: warp 0 and warps 6.. copy the A rows.  Two beat one by 4-12%
// on GB300; four do not help (nine warps cap registers at 168 and spill).
constexpr int COPY_WARPS = 2;
constexpr int NWARPS = EPI_WARP_END + COPY_WARPS - 1; // producer, MMA, 4 x epilogue, copy helpers
constexpr int COPY_ROWS = BM / COPY_WARPS;            // A rows per copy warp and stage
static_assert(COPY_ROWS % 8 == 0, "each copy warp owns whole 8-row swizzle atoms");
constexpr int NTHREADS = NWARPS * 32;
constexpr int ROUTE_CHUNK = NWARPS * 32;              // tokens per routing chunk (lane per token)
constexpr int MAX_ROUTE_LANES = 8;                    // lanes sharing one token's experts (E >= 64)
constexpr int MAX_E = 256;
constexpr int MAX_K = 8;
constexpr int MAX_CHUNKS_PER_CTA = 16;
constexpr int MAX_GATHER_SLOTS = 32;
// Gathering warps per dispatch CTA when experts fill whole tiles: each takes
// units of gather_slots / GATHER_WARPS rows, so the CTAs' gather ends more
// evenly.  Measured on GB300 (Mixtral-like layer): dispatch alone 45.7 ->
// 44.0 us, the fused launch -0.7%, with 2 warps instead of 1.
constexpr int GATHER_WARPS = 2;
constexpr int TRACE_SLOTS = 16;

// CTA-pair variant (cta_group::2): a 256 x 256 tile per pair of SMs; each
// CTA stages its 128 rows of A and 128 of B's 256 columns, so a stage is
// 32 KiB and six fit where four single-CTA stages did.
constexpr int PAIR_TILE_M = 2 * BM;
constexpr int PSTAGES = 6;
constexpr int PA_STAGE_BYTES = BM * BK * 2;                // 16 KiB (own 128 rows)
constexpr int PB_STAGE_BYTES = BK * (BN / 2) * 2;          // 16 KiB (own 128 columns)
constexpr int SM_PA = 0;
constexpr int SM_PB = SM_PA + PSTAGES * PA_STAGE_BYTES;    // 96 KiB

// Wide variant (one SM, 256-row tiles, two accumulators sharing each B
// stage): a stage holds 2 x 16 KiB of A and 32 KiB of B, so three fit.
// (Six stages of 32 rows of K, the same bytes in finer steps, measured 17%
// slower on GB300: per row of K the MMA warp waited longer, not shorter.)
constexpr int WIDE_TILE_M = 2 * BM;
static_assert((BM & (BM - 1)) == 0 && (WIDE_TILE_M & (WIDE_TILE_M - 1)) == 0 && (PAIR_TILE_M & (PAIR_TILE_M - 1)) == 0,
              "tile rows are powers of two (the tile tables count tiles with a shift)");
constexpr int WSTAGES = 3;
// Two-accumulator items issue their last K-block's MMAs accumulator by
// accumulator, so the epilogue drains the first while the second finishes.
constexpr bool WIDE_EARLY_HALF = true;

constexpr int MAX_STAGES = PSTAGES > STAGES ? (PSTAGES > WSTAGES ? PSTAGES : WSTAGES)
                                             : (STAGES > WSTAGES ? STAGES : WSTAGES);

// Dynamic shared memory map (offsets from a 1024-byte aligned base).
constexpr int SM_A = 0;
constexpr int SM_B = SM_A + STAGES * A_STAGE_BYTES;           // 64 KiB
constexpr int SM_STAGE_END = SM_B + STAGES * B_STAGE_BYTES;   // 192 KiB
// Epilogue output buffers: one 32-row x 64-column bf16 box (4 KiB, 128-byte
// swizzle) per epilogue warp, the source of its tensor stores.
constexpr int EPI_BOX_COLS = 64;
constexpr int EPI_BOX_ROWS = 32;
constexpr int EPI_BUF_BYTES = EPI_BOX_COLS * EPI_BOX_ROWS * 2;
constexpr int SM_EPI = SM_STAGE_END;
// Whole boxes leave the buffer by one TMA store (true) or by coalesced
// 16-byte stores of the warp after a transpose in the buffer (false).
constexpr bool EPI_TMA_STORE = true;
constexpr int SM_CTRL = SM_EPI + 4 * EPI_BUF_BYTES;           // 208 KiB
constexpr int SM_CTRL_BYTES = 8192;
constexpr int SMEM_BYTES = SM_CTRL + SM_CTRL_BYTES + 1024;    // + alignment slack
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory of one CTA on sm_103");

// Routing scratch aliases the stage area (routing ends before the GEMM).
constexpr int RT_LOGIT_STRIDE = 65;                           // 64 experts per pass + 1 pad
constexpr int RT_LOGITS = 0;
constexpr int RT_LOGITS_BYTES = NWARPS * 32 * RT_LOGIT_STRIDE * 4;
constexpr int RT_IDX = RT_LOGITS + RT_LOGITS_BYTES;
constexpr int RT_LRANK = RT_IDX + NWARPS * 32 * MAX_K * 4;
constexpr int RT_WCNT = RT_LRANK + NWARPS * 32 * MAX_K * 4;
constexpr int RT_WCNT_END = RT_WCNT + NWARPS * MAX_E * 4;
// The bases of a CTA's own chunks sit at the end of the stage area: the
// scan copies the whole count table to [0, RT_BASES) once the routing
// scratch is dead, so up to RT_BASES / 4 counts are scanned in shared memory.
constexpr int RT_BASES = SM_STAGE_END - MAX_CHUNKS_PER_CTA * MAX_E * 4;
static_assert(RT_WCNT_END <= RT_BASES, "routing scratch must fit below the chunk bases");
static_assert(RT_BASES / 4 >= 152 * MAX_E, "one chunk per SM of every expert's counts fits in shared memory");
static_assert(SM_PB + PSTAGES * PB_STAGE_BYTES <= SM_STAGE_END, "pair stages must fit in the stage area");

// Control block at the head of the workspace.  The kernels leave it ready
// for the next call: the last CTA to exit zeroes the counters and the abort
// word.  Tile arrival counts are cleared by the fused kernel itself.
struct Ctl {
    uint32_t epoch;
    uint32_t exit_count;
    uint32_t bar_routed;     // CTAs whose routing chunks are written
    uint32_t bar_scattered;  // CTAs whose src_index / gate_w scatter is written
    uint32_t next_tile;      // gather queue (dispatch role)
    uint32_t next_item;      // GEMM work queue (compute role)
    uint32_t abort;          // 1 once any CTA of this call gave up
    uint32_t tiles_done;     // tiles the dispatch role has gathered and flagged
    uint32_t bar_computed;   // CTAs done with the GEMM (combine barrier)
    uint32_t bar_scanned;    // CTAs whose expert columns are scanned (distributed scan)
    uint32_t pad[54];
};
static_assert(sizeof(Ctl) == 256, "control block is 256 bytes");

// Expert-parallel simulation: R logical ranks inside one GPU.  Each rank
// owns a region of the workspace (its "device memory") and this control
// block; other ranks touch them only through the exchange: count rows and
// their flags, received rows and their arrival counts, returned results and
// their completion count.
constexpr int MAX_RANKS = 8;
struct EpCtl {
    uint32_t routed;                // this rank's CTAs whose count rows are sent
    uint32_t scattered;             // this rank's CTAs whose receive metadata is written
    uint32_t next_send;             // this rank's send queue (as a source)
    uint32_t next_item;             // work queue over this rank's experts
    uint32_t ret_done;              // (row, N-block) results stored into this rank's return rows
    uint32_t cnt_flag[MAX_RANKS];   // source r's count rows are in this rank's table copy
    uint32_t pad[64 - 5 - MAX_RANKS];
};
static_assert(sizeof(EpCtl) == 256, "rank control block is 256 bytes");

enum Mode : int { MODE_FUSED = 0, MODE_UNFUSED = 1, MODE_DISPATCH_ONLY = 2 };

// Error sites recorded with a device error (mk_last_error_detail()).
enum Site : int {
    SITE_BAR_ROUTED = 1,
    SITE_BAR_SCATTERED = 2,
    SITE_GATHER_LOAD = 3,
    SITE_TILE_READY = 4,
    SITE_STAGE_EMPTY = 5,
    SITE_STAGE_FULL = 6,
    SITE_ACC_EMPTY = 7,
    SITE_ACC_FULL = 8,
    SITE_INFO_FULL = 9,
    SITE_INFO_EMPTY = 10,
    SITE_DEST_RANGE = 11,
    SITE_ROW_TOTAL = 12,
    SITE_DRAIN = 13,
    SITE_BAR_COMPUTED = 14,
    SITE_EP_COUNTS = 15,
    SITE_EP_SCATTERED = 16,
    SITE_EP_RETURNED = 17,
    SITE_PAIR_ALIGN = 18,
    SITE_PAIR_CLUSTER = 19,
    SITE_BAR_SCANNED = 20,
};

enum ErrCode : uint32_t { ERR_NONE = 0, ERR_TIMEOUT = 1, ERR_FAULT = 2 };

struct Params {
    // problem (device pointers)
    const uint16_t* x;       // [T,H] bf16
    const float* logits;     // [T,E]
    const uint16_t* W;       // [E,H,F] bf16 (the gate projection W1 when gated)
    const uint16_t* W3;      // [E,H,F] bf16 up projection (gated only)
    void* y;                 // [T*k,F] bf16 or f32
    int32_t* src_index;      // [T*k]
    int32_t* expert_offsets; // [E+1]
    float* gate_w;           // [T*k]
    int T, H, F, E, k;
    int out_f32;
    int y_v8;                // y is 32-byte aligned: results go out as 256-bit stores
    int y_tma;               // whole 32-row groups go out as tensor stores (tmY: bf16 y_sorted)
    // derived sizes
    int rows;                // T*k
    int nch;                 // routing chunks
    int route_lanes;         // lanes sharing each token's experts in routing: 1, 2, 4 or 8
    int route_chunk;         // tokens per routing chunk: ROUTE_CHUNK / route_lanes
    int nb;                  // N-blocks per expert, ceil(F / BN)
    int kblocks;             // H / BK
    int n_group;             // N-blocks per group in the work order
    int dispatch_ctas;       // CTAs [0, dispatch_ctas) take the dispatch role
    int gather_slots;        // rows in flight per dispatch CTA
    int gather_warps;        // warps of a dispatch CTA that gather, gather_slots / gather_warps slots each
    int mode;
    int compute;             // 0: dispatch only
    int debug_drop_tile;     // tile whose flag is withheld (-1: none)
    int l2_prefetch;         // W k-blocks prefetched into L2 ahead of the TMA loads (0: off)
    int pair;                // 1: 2-SM MMA (cluster of 2 CTAs per 256-row tile)
    int wide;                // 1: 256-row tiles on one SM, two accumulators sharing each B stage
    int gated;               // 1: y = silu(x.W1) * (x.W3), 128-column N-blocks
    int direct;              // 1: the GEMM's producer copies token rows from x (no staging rows)
    int gather4;             // with direct: rows arrive by TMA tile::gather4 (tmA maps x, one-row box),
                             // not by the copy warps' cp.async
    int tile_rows;           // rows per tile: 128, or 256 with pair or wide
    int dist_scan;           // 1: each CTA scans whole expert columns of the count table
                             // (bases, totals), a barrier, then every CTA reads the totals
    int trace;
    long long spin_limit_ns;
    // workspace
    Ctl* ctl;
    int32_t* counts;         // [nch][E]
    int32_t* topk_idx;       // [T*k]
    float* topk_gate;        // [T*k]
    int32_t* lrank;          // [T*k]
    int32_t* bases;          // [nch][E] rows of earlier chunks per expert (unfused path,
                             // distributed scan)
    int32_t* totals;         // [E] rows per expert (distributed scan)
    int32_t* row_of;         // [T*k] sorted row of each (t, j)
    void* combine_out;       // [T,F] (y_sorted's dtype) or null: no combine
    uint32_t* ready;         // [max_tiles] rows of each tile gathered so far (staged rows)
    uint16_t* xs;            // [T*k,H] bf16 staging
    unsigned long long* trace_buf;  // [grid][TRACE_SLOTS]
    int max_tiles;
    // Streamed results (host-buffer entry point, fused single-SM path): sorted
    // rows [c*stream_rows, (c+1)*stream_rows) form chunk c.  Once every row of
    // the chunk is stored for every N-block, stream_flag[c] = stream_seq, and a
    // copy stream waiting on that value starts copying the chunk to the host.
    uint32_t* stream_done;   // [chunks] (row, N-block) results stored; cleared per call (null: off)
    uint32_t* stream_flag;   // [chunks] sequence number of the call that completed the chunk
    int stream_rows;
    uint32_t stream_seq;
    // token ranges of the routing chunks: rank r's tokens [ep_t0[r], ep_t0[r+1])
    // are split into the chunks [ep_c0[r], ep_c0[r+1]) (one rank, [0, T), when
    // not simulating expert parallelism)
    int ranks;
    int ep_t0[MAX_RANKS + 1];
    int ep_c0[MAX_RANKS + 1];
    // expert-parallel simulation (ep = 1): rank r also owns the experts
    // [r*E/R, (r+1)*E/R) and the CTAs [r*ep_cpr, (r+1)*ep_cpr), the first
    // ep_dispatch of which send before they compute
    int ep;
    int ep_cpr;
    int ep_dispatch;
    int ep_tile_cap;                 // tile counters per rank
    int ep_cap_rows;                 // receive rows per rank
    EpCtl* ep_ctl[MAX_RANKS];
    int32_t* ep_counts[MAX_RANKS];   // each rank's copy of the count table [nch][E]
    uint32_t* ep_ready[MAX_RANKS];   // rows arrived per tile of the rank's experts
    uint16_t* ep_recv[MAX_RANKS];    // received rows [cap][H] bf16 (the GEMM's A operand)
};

// Workspace carve-up, shared by the size query and the launcher.
struct WsLayout {
    size_t ctl, counts, topk_idx, topk_gate, lrank, row_of, bases, totals, ready, trace, xs, total;
};

inline size_t ws_align(size_t v) { return (v + 255) & ~size_t(255); }

constexpr int MAX_GRID = 1024;

// Lanes per token for routing.  With E = 64, 128 or 256 experts a token's
// experts are split over S lanes (S * 32 or S * 64 experts, read with
// 16-byte loads), so a chunk holds ROUTE_CHUNK / S tokens and S times as
// many CTAs route.  S is the largest split whose chunks still number at
// most one per CTA (routing time is per chunk).  S = 1 (a lane per token)
// for other expert counts, for logits that are not 16-byte aligned, or
// when no split passes.  Large count tables (chunks x E) are scanned by
// columns across the CTAs (DIST_SCAN_COUNTS), so the table size sets no
// limit here.
inline int route_lanes_for(int T, int E, int grid, bool logits_16b) {
    if (!logits_16b) return 1;
    int S = E == 64 ? 2 : E == 128 ? 4 : E == 256 ? MAX_ROUTE_LANES : 1;
    while (S > 1 && (int64_t(T) + ROUTE_CHUNK / S - 1) / (ROUTE_CHUNK / S) > grid) S >>= 1;
    if (S > 1 && E / S > 64) S = 1;  // a lane scans 32 or 64 experts
    return S;
}

// Count tables of more than this many entries are scanned by columns, each
// CTA one expert at a time (a second grid barrier, but no CTA reads the
// whole table); smaller ones by every CTA from a copy in shared memory.
constexpr int DIST_SCAN_COUNTS = 4096;

// Routing chunks of a call: with S > 1 there are at most `grid` of them.
inline size_t route_chunks_bound(int T) {
    const size_t whole = (size_t(T) + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    const size_t split = (size_t(T) + ROUTE_CHUNK / MAX_ROUTE_LANES - 1) / (ROUTE_CHUNK / MAX_ROUTE_LANES);
    const size_t capped = split < size_t(MAX_GRID) ? split : size_t(MAX_GRID);
    return whole > capped ? whole : capped;
}

inline WsLayout ws_layout(int T, int H, int E, int k, bool staging = true, int grid = MAX_GRID) {
    WsLayout L{};
    const size_t rows = size_t(T) * k;
    const size_t nch = route_chunks_bound(T);
    const size_t max_tiles = (rows + BM - 1) / BM + E;
    size_t o = 0;
    L.ctl = o;        o = ws_align(o + sizeof(Ctl));
    L.counts = o;     o = ws_align(o + nch * E * 4);
    L.topk_idx = o;   o = ws_align(o + rows * 4);
    L.topk_gate = o;  o = ws_align(o + rows * 4);
    L.lrank = o;      o = ws_align(o + rows * 4);
    L.row_of = o;     o = ws_align(o + rows * 4);
    L.bases = o;      o = ws_align(o + nch * E * 4);
    L.totals = o;     o = ws_align(o + size_t(E) * 4);
    L.ready = o;      o = ws_align(o + max_tiles * 4);
    L.trace = o;      o = ws_align(o + size_t(grid) * TRACE_SLOTS * 8);
    L.xs = o;         o = ws_align(o + (staging ? rows * size_t(H) * 2 : 0));
    L.total = o;
    return L;
}

// Expert-parallel workspace: a head (control block, the ranks' control
// blocks, routing results of the ranks' own tokens, trace) and one region
// per rank.  The rank control blocks sit at fixed offsets whatever the
// sizes, so a cached workspace reused with other sizes or rank counts still
// finds them zeroed (the last CTA of every call leaves them so).  A rank
// receives at most T * min(k, E/R) rows: every token brings at most one row
// per expert, and each of the rank's E/R experts is one of its k.
struct EpLayout {
    size_t ctl, ep_ctl, topk_idx, topk_gate, lrank, row_of, trace;
    size_t rank_base[MAX_RANKS], rank_bytes;
    size_t counts_off, ready_off, recv_off;  // inside a rank region
    int nch, tile_cap;
    size_t cap_rows;
    size_t total;
};

inline int ep_token0(int T, int R, int r) { return int((int64_t(T) * r) / R); }

inline EpLayout ep_layout(int T, int H, int E, int k, int R, int grid = MAX_GRID) {
    EpLayout L{};
    const size_t rows = size_t(T) * k;
    int nch = 0;
    for (int r = 0; r < R; ++r) nch += (ep_token0(T, R, r + 1) - ep_token0(T, R, r) + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    L.nch = nch;
    L.cap_rows = size_t(T) * size_t(k < E / R ? k : E / R);
    L.tile_cap = int((L.cap_rows + BM - 1) / BM) + E / R;
    size_t o = 0;
    L.ctl = o;        o = ws_align(o + sizeof(Ctl));
    L.ep_ctl = o;     o = ws_align(o + MAX_RANKS * sizeof(EpCtl));
    L.topk_idx = o;   o = ws_align(o + rows * 4);
    L.topk_gate = o;  o = ws_align(o + rows * 4);
    L.lrank = o;      o = ws_align(o + rows * 4);
    L.row_of = o;     o = ws_align(o + rows * 4);
    L.trace = o;      o = ws_align(o + size_t(grid) * TRACE_SLOTS * 8);
    size_t q = 0;
    L.counts_off = q; q = ws_align(q + size_t(nch) * E * 4);
    L.ready_off = q;  q = ws_align(q + size_t(L.tile_cap) * 4);
    L.recv_off = q;   q = ws_align(q + L.cap_rows * size_t(H) * 2);
    L.rank_bytes = q;
    for (int r = 0; r < R; ++r) {
        L.rank_base[r] = o;
        o += q;
    }
    L.total = o;
    return L;
}

}  // namespace mk
