/*
 * mk.h -- C ABI of the GB300 (sm_103a) MoE token dispatch + expert GEMM.
 *
 * What the operation is.  The mKernel write-ups name "MoE Dispatch+GEMM" as
 * one of five fused persistent kernels: tokens are routed dynamically to
 * experts and each expert's dense product runs as soon as its tile of tokens
 * has arrived, inside one kernel ("mKernel: UCCL fuses NVLink, RDMA and
 * compute into one persistent CUDA kernel", zubnet.ai, paras. 1-2;
 * "UC Berkeley presenta mKernel ...", edge.aivizor.me, para. 3;
 * "mKernel : une bibliotheque de noyaux fusionnes ...", lefilia.fr,
 * paras. 1 and 3).  The pages print none of the steps, so this header
 * states the contract the library implements:
 *
 *   1. Router top-k.  For token t, the k experts with the largest logits,
 *      in descending order, ties to the lower expert id; -inf is a legal
 *      logit (NaN and +inf are outside the contract: results unspecified,
 *      no fault).
 *   2. Gates.  gate[t,j] = softmax over the k chosen logits (fp32 expf);
 *      a -inf logit gets 0; if all k chosen are -inf every gate is 0.
 *   3. expert_offsets[e] = number of (t,j) routed to experts < e
 *      (exclusive scan of the per-expert histogram); expert_offsets[E] = T*k.
 *   4. Sorted rows: every (t,j) pair, ordered by (expert, t, j).  For sorted
 *      row r: src_index[r] = t*k + j, gate_w[r] = gate[t,j].
 *   5. y_sorted[r,:] = x[t,:] . W[e,:,:] with fp32 accumulation, stored as
 *      bf16 (round-to-nearest-even) or, with MK_OUT_F32, as fp32.  Rows are
 *      not scaled by the gate.
 *
 * Layouts (all row-major, caller-owned, device memory unless stated):
 *   x[T,H] bf16, logits[T,E] f32, W[E,H,F] bf16 (F contiguous)   -- read only
 *   y_sorted[T*k,F] bf16 (or f32), src_index[T*k] i32,
 *   expert_offsets[E+1] i32, gate_w[T*k] f32                     -- written
 *   bf16 travels as 16-bit storage (void*); the library never frees caller
 *   memory.
 *
 * Limits (checked synchronously, no launch on failure -> MK_ERR_INVALID_ARG
 * or MK_ERR_UNSUPPORTED): T >= 0; 1 <= k <= min(E, 8); 1 <= E <= 256;
 * H and F multiples of 64 in [64, 32768]; T*k < 2^31; x, W, y_sorted 16-byte
 * aligned, the other arrays 4-byte aligned; the current device must be
 * sm_103 (compute capability 10.3).  T == 0 is valid: expert_offsets is set
 * to zeros and nothing else is written.
 *
 * Asynchrony.  Calls enqueue work on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and return without synchronising.  A fault or a
 * bounded wait that ran out inside the kernel is recorded in a per-device
 * error word; mk_get_status() synchronises the stream and reports it.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer      */
    MK_ERR_UNSUPPORTED = 2,   /* wrong device, or shape beyond the limits  */
    MK_ERR_CUDA = 3,          /* a CUDA runtime call failed                */
    MK_ERR_TIMEOUT = 4,       /* a bounded device wait ran out             */
    MK_ERR_DEVICE_FAULT = 5,  /* the kernel detected an inconsistent state */
    MK_ERR_NOT_IMPLEMENTED = 6,
    MK_ERR_WORKSPACE = 7      /* caller workspace too small or misaligned  */
} mk_status_t;

/* Execution modes. */
enum {
    MK_MODE_FUSED = 0,         /* one persistent launch: dispatch and compute roles overlap per tile */
    MK_MODE_UNFUSED = 1,       /* the same steps as four launches (route, scan, gather, GEMM)       */
    MK_MODE_DISPATCH_ONLY = 2  /* routing + gather only (y_sorted untouched); measures dispatch      */
};

enum { MK_OUT_BF16 = 0, MK_OUT_F32 = 1 };

/* Host-side fault injection (never a device trap): withhold the arrival of
 * one tile's rows (its readiness never completes) so the compute role's
 * bounded wait runs out.  It acts on staged rows: with the fault set, AUTO
 * row sources resolve to MK_GATHER_STAGED. */
enum { MK_FAULT_NONE = 0, MK_FAULT_DROP_TILE_FLAG = 1 };

typedef struct mk_config {
    int32_t mode;           /* MK_MODE_*                                        */
    int32_t out_dtype;      /* MK_OUT_BF16 or MK_OUT_F32                         */
    int32_t dispatch_ctas;  /* CTAs in the dispatch role; 0 = shape heuristic    */
    int32_t grid_ctas;      /* persistent grid size; 0 = one CTA per SM          */
    int32_t n_group;        /* N-blocks per group in the work order; 0 = auto    */
    int32_t debug_fault;    /* MK_FAULT_*                                        */
    int64_t spin_limit_ns;  /* bound on every device wait; 0 = 2 s               */
    int32_t trace;          /* 1 = record per-CTA %globaltimer phase stamps      */
    int32_t l2_prefetch;    /* W K-blocks prefetched into L2 ahead of use;
                               <= 0 = off (the default)                          */
    int32_t mma_pair;       /* MK_MMA_*: one SM per 128-row tile, an SM pair
                               (cta_group::2) per 256-row tile, or one SM per
                               256-row tile with two accumulators (WIDE)     */
    int32_t gather;         /* MK_GATHER_*: where the GEMM's token rows come from */
    int32_t reserved[4];    /* must be zero                                     */
} mk_config_t;

/* Token rows for the GEMM.  STAGED: dispatch CTAs copy them into
 * expert-contiguous tiles in the workspace, in units of up to 32 rows, and
 * add each unit's rows to its tile's arrival count; compute CTAs wait until
 * a tile's count reaches its rows and load whole tiles.  DIRECT: the GEMM's
 * producer warp copies each tile's rows straight from x into its
 * shared-memory stages (16-byte cp.async), so there is no staging copy, no
 * gather role, and the workspace holds no staging rows (T*k*H*2 bytes
 * less); 128-row or wide tiles (not SM pairs), and T*H*2 < 4 GiB.  GATHER4:
 * as DIRECT, but the rows arrive by TMA tile::gather4 (four token rows per
 * instruction, one instruction per lane of the producer warp) instead of
 * cp.async; same tiles and limits.  AUTO: DIRECT when k >= 4 and
 * T*k >= 256*E (wide tiles), or when the staged rows would take under
 * 1 MiB (T*k*H*2 < 2^20), with cfg.mma_pair AUTO or WIDE and
 * T*H*2 < 4 GiB; STAGED otherwise.  The expert-parallel entry points stage
 * rows (DIRECT and GATHER4 return MK_ERR_UNSUPPORTED there). */
enum { MK_GATHER_AUTO = 0, MK_GATHER_STAGED = 1, MK_GATHER_DIRECT = 2, MK_GATHER_GATHER4 = 3 };

/* Expert GEMM tile.  SINGLE: each CTA runs a 128 x 256 tile alone.  PAIR: a
 * cluster of two CTAs (two SMs) runs a 256 x 256 tile with the 2-SM tensor
 * core instruction; each SM stages half the operands, so the same shared
 * memory holds six stages instead of four.  WIDE: each CTA runs a 256 x 256
 * tile alone, as two 128-row accumulators that share every staged block of
 * the weights (three stages of 64 KiB; an expert's last tile of at most 128
 * rows uses one accumulator); with any MK_GATHER_* form.  AUTO: WIDE when
 * T*k >= 256*E (two or more 128-row tiles per expert on average), SINGLE
 * otherwise. */
enum { MK_MMA_AUTO = 0, MK_MMA_SINGLE = 1, MK_MMA_PAIR = 2, MK_MMA_WIDE = 3 };

/* Per-launch facts, for tests and the benchmark. */
typedef struct mk_launch_info {
    int32_t grid_ctas;      /* CTAs launched by the persistent kernel */
    int32_t dispatch_ctas;  /* of which in the dispatch role          */
    int32_t launches;       /* kernels launched by the last call      */
    int32_t n_group;
    int64_t workspace_bytes;
    int32_t mma_pair;       /* MK_MMA_SINGLE, MK_MMA_PAIR or MK_MMA_WIDE as resolved */
    int32_t gather;         /* MK_GATHER_STAGED, _DIRECT or _GATHER4 as resolved */
    int32_t route_lanes;    /* lanes sharing each token's experts in routing (1, 2, 4, 8) */
    int32_t route_chunks;   /* routing chunks (224 / route_lanes tokens each) */
} mk_launch_info_t;

/* Fill `cfg` with the defaults (fused, bf16 output, heuristic split). */
void mk_config_default(mk_config_t* cfg);

/* The fused path with default configuration and the library's
 * per-(device, stream) workspace cache.  Device pointers; see above. */
mk_status_t mk_moe_dispatch_gemm(const void* x, const float* logits, int T, int H, int E, int k,
                                 const void* W, int F, void* y_sorted, int32_t* src_index,
                                 int32_t* expert_offsets, float* gate_w, void* stream);

/* As mk_moe_dispatch_gemm with an explicit configuration (NULL = defaults)
 * and an optional caller workspace.  With workspace == NULL the library's
 * cache is used (grown with cudaMallocAsync on `stream`).  A caller
 * workspace must hold mk_workspace_size() bytes, be 256-byte aligned, and be
 * zero-filled before its first use (the kernels leave it ready for the next
 * call).  One workspace serves one stream at a time. */
mk_status_t mk_moe_dispatch_gemm_ex(const void* x, const float* logits, int T, int H, int E, int k,
                                    const void* W, int F, void* y_sorted, int32_t* src_index,
                                    int32_t* expert_offsets, float* gate_w, void* stream,
                                    const mk_config_t* cfg, void* workspace, size_t ws_bytes);

/* The path plus the combine that completes an MoE layer: after the expert
 * products, out[t,:] = sum_j gate[t,j] * y_sorted[row of (t,j), :] (fp32,
 * slots in order, no atomics), in y_sorted's dtype (bf16, or f32 with
 * MK_OUT_F32).  The pages name the operation "MoE Dispatch+GEMM" and route
 * each token to experts ("mKernel : une bibliotheque ...", lefilia.fr,
 * para. 3); this weighted sum of a token's expert outputs is the textbook
 * step that follows.  out[T,F]: device, caller-owned, 16-byte aligned.
 * Fused mode combines inside the same persistent launch after a grid
 * barrier; unfused mode adds a fifth launch.  y_sorted and the other outputs
 * are written as by mk_moe_dispatch_gemm_ex.  Not valid with
 * MK_MODE_DISPATCH_ONLY. */
mk_status_t mk_moe_dispatch_gemm_combine(const void* x, const float* logits, int T, int H, int E, int k,
                                         const void* W, int F, void* y_sorted, int32_t* src_index,
                                         int32_t* expert_offsets, float* gate_w, void* out, void* stream,
                                         const mk_config_t* cfg, void* workspace, size_t ws_bytes);

/* Gated expert FFN (SwiGLU, the Mixtral / DeepSeek expert shape; both model
 * families are named in "mKernel : une bibliotheque de noyaux fusionnes
 * ...", lefilia.fr, para. 3): the same dispatch, then for sorted row r of
 * token t routed to expert e,
 *   h_sorted[r,:] = silu(x[t,:] . W1[e]) * (x[t,:] . W3[e]),  silu(a) = a / (1 + e^-a),
 * both products accumulated in fp32 in the same tensor-core pass (the A tile
 * is shared; 128 columns of each projection per work item) and the SwiGLU
 * applied in the epilogue (fp32, fast exponential and divide) before
 * rounding to bf16 (or f32 with MK_OUT_F32).  W1, W3: [E,H,F] bf16, device,
 * 16-byte aligned.  Runs on tiles of one SM, 128-row or wide (MK_MMA_PAIR
 * returns MK_ERR_UNSUPPORTED).  Other
 * arguments and outputs as for mk_moe_dispatch_gemm_ex. */
mk_status_t mk_moe_dispatch_gated(const void* x, const float* logits, int T, int H, int E, int k, const void* W1,
                                  const void* W3, int F, void* h_sorted, int32_t* src_index,
                                  int32_t* expert_offsets, float* gate_w, void* stream, const mk_config_t* cfg,
                                  void* workspace, size_t ws_bytes);

/* Expert parallelism simulated on one GPU.  The pages run MoE
 * Dispatch+GEMM across GPUs, tokens travelling to the GPU that holds their
 * expert ("mKernel: UCCL fuses NVLink, RDMA, compute ...", zubnet.ai, para.
 * 2; "mKernel : une bibliotheque ...", lefilia.fr, paras. 2-3).  Here
 * `ranks` logical ranks share one launch, each with its own region of the
 * workspace standing for its device memory.  Rank r owns the tokens
 * [floor(r*T/R), floor((r+1)*T/R)) and the experts [r*E/R, (r+1)*E/R)
 * (R = ranks, 1..8, dividing E).  Each rank routes its own tokens, sends
 * its per-expert count rows to every rank (a flag per source), sends each
 * routed row to the rank of its expert (a count of arrived rows per tile:
 * the GEMM starts a tile once every source's rows are in), runs the expert
 * GEMM for its own experts, and stores every result back into the sending
 * rank's rows; with `out`, each rank then combines its own tokens once all
 * their results are back.
 *
 * Outputs (device, caller-owned, written):
 *   y_tok[T*k,F]: the product x[t].W[e] of entry (t, j) at row t*k + j
 *     (token-major: the sending ranks' return rows, rank r's being rows
 *     [T0(r)*k, T0(r+1)*k)); bf16, or f32 with MK_OUT_F32.  Not gate-scaled.
 *   src_index[T*k], gate_w[T*k], expert_offsets[E+1]: the ranks' receive
 *     buffers one after another, which is exactly the sorted order of
 *     mk_moe_dispatch_gemm (rank q's rows are [expert_offsets[q*E/R],
 *     expert_offsets[(q+1)*E/R])).
 *   out[T,F] (optional, may be NULL): sum_j gate[t,j] * y_tok[t*k+j], fp32
 *     in slot order, in y_tok's dtype.
 * Supported: MK_MODE_FUSED, staged rows, tiles of one SM (128-row or
 * wide, resolved as for the single-device call); other choices
 * return MK_ERR_UNSUPPORTED.  cfg.trace records nothing here.  workspace:
 * NULL (library cache, zeroed when allocated) or mk_ep_workspace_size()
 * bytes, 256-byte aligned, zero-filled before its first use, and used by
 * this entry point only (the others write over its control blocks).  Every rank may
 * receive up to T*min(k, E/R) rows, so the workspace holds that many
 * H-wide rows per rank.  Errors as for mk_moe_dispatch_gemm_ex. */
mk_status_t mk_moe_ep_sim(const void* x, const float* logits, int T, int H, int E, int k, const void* W, int F,
                          int ranks, void* y_tok, int32_t* src_index, int32_t* expert_offsets, float* gate_w,
                          void* out, void* stream, const mk_config_t* cfg, void* workspace, size_t ws_bytes);

/* The gated (SwiGLU) expert FFN of mk_moe_dispatch_gated under the same
 * expert-parallel simulation: each rank computes
 * h = silu(x[t].W1[e]) * (x[t].W3[e]) for the rows it received and returns
 * them to the sending ranks (h_tok[t*k + j]); with `out`, each rank combines
 * its own tokens' h rows.  W1, W3: [E,H,F] bf16, device, 16-byte aligned.
 * Other arguments, outputs and errors as for mk_moe_ep_sim; the workspace
 * is the same size. */
mk_status_t mk_moe_ep_sim_gated(const void* x, const float* logits, int T, int H, int E, int k, const void* W1,
                                const void* W3, int F, int ranks, void* h_tok, int32_t* src_index,
                                int32_t* expert_offsets, float* gate_w, void* out, void* stream,
                                const mk_config_t* cfg, void* workspace, size_t ws_bytes);

/* Workspace bytes mk_moe_ep_sim needs (0 for invalid sizes). */
size_t mk_ep_workspace_size(int T, int H, int F, int E, int k, int ranks);

/* End-to-end variant: x, logits and the four outputs are HOST buffers
 * (pinned memory gives asynchronous copies); W stays on the device (expert
 * weights are resident).  Copies the inputs in, runs the fused path, copies
 * the outputs back, and synchronises `stream` before returning, so the host
 * buffers are ready on return.  With the fused single-SM path, y_sorted goes
 * back in chunks of sorted rows (whole 256-row tiles, at most 64 chunks)
 * while the kernel still runs: the kernel raises a flag per finished chunk
 * and a second, library-owned stream waits on the flags and copies the rows,
 * in copies of 1, 1, 2, 4, ... chunks; other configurations copy after the
 * kernel.  With cfg->n_group = 0 this call orders the work tile by tile
 * (all N-blocks of a tile together), so rows complete in order.  Device staging comes from the library cache.  The library's
 * stream and chunk flags belong to (device, stream); calls on one stream run
 * one after another. */
mk_status_t mk_moe_dispatch_gemm_host(const void* x_host, const float* logits_host, int T, int H, int E,
                                      int k, const void* W, int F, void* y_sorted_host,
                                      int32_t* src_index_host, int32_t* expert_offsets_host,
                                      float* gate_w_host, void* stream, const mk_config_t* cfg);

/* Size of the fixed device array that mk_moe_dispatch_gemm_noalloc works in. */
#define MK_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Allocation-free variant of mk_moe_dispatch_gemm_ex (the pages have no
 * counterpart: it serves callers of this library that may not allocate
 * device memory while they run it -- a host framework that owns the whole
 * device-memory budget through its own allocator, or a latency-critical
 * decode loop where cudaMalloc and its possible device-wide synchronisation
 * are not allowed).  Same arguments and outputs as the allocating path; the
 * caller still passes every input and output.  Instead of a workspace it
 * uses one static device array of MK_NOALLOC_SCRATCH_BYTES (64 MiB), which
 * each GPU where it is set up keeps until the process exits.  Calls whose
 * mk_workspace_size() exceeds that return MK_ERR_WORKSPACE and launch
 * nothing (it fits decode-sized batches: about T*k*H*2 bytes of staged rows
 * plus small tables).  No cudaMalloc, cudaFree or allocating library call
 * is made.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture.  After a device reset
 * (cudaDeviceReset), call mk_release_workspace() before the next call: it
 * drops the kept addresses (the array may sit elsewhere in the new context)
 * as well as the workspace cache.  Every call on a device shares the array
 * and finds the previous call's contents there (the call clears what must
 * start at zero), so calls that overlap on the GPU -- on different streams,
 * or from different threads -- race: serialise them.  cfg->trace must be 0
 * (MK_ERR_UNSUPPORTED otherwise): phase stamps would land in the array,
 * where mk_read_trace cannot reach them. */
mk_status_t mk_moe_dispatch_gemm_noalloc(const void* x, const float* logits, int T, int H, int E, int k,
                                         const void* W, int F, void* y_sorted, int32_t* src_index,
                                         int32_t* expert_offsets, float* gate_w, void* stream,
                                         const mk_config_t* cfg);

/* Bytes of workspace a call with these sizes needs (0 on invalid sizes). */
size_t mk_workspace_size(int T, int H, int F, int E, int k, const mk_config_t* cfg);

/* Synchronise `stream`, then return and clear the device error word
 * (MK_ERR_TIMEOUT / MK_ERR_DEVICE_FAULT), or MK_ERR_CUDA if the stream holds
 * a CUDA error.  MK_OK when nothing was recorded. */
mk_status_t mk_get_status(void* stream);

/* Detail of the last recorded device error: site code and CTA (or -1). */
void mk_last_error_detail(int32_t* site, int32_t* cta, int32_t* info);

/* Facts about the last call on this thread (grid, role split, launches). */
void mk_last_launch_info(mk_launch_info_t* info);

/* Copy the phase stamps of the last traced call (cfg.trace = 1) made with
 * these sizes on `stream` to the host: up to n uint64 values, 16 per CTA
 * (%globaltimer ns; 0 = phase not reached).  `workspace` is the caller
 * workspace that call used, or NULL for the library cache of `stream`.
 * Synchronises `stream`.  Slots of the fused single-SM kernel: 0 CTA start,
 * 1 its routing chunks done, 2 routing barrier passed, 3 scan and scatter
 * done, 4 scatter barrier passed (dispatch CTAs), 5 gather done (dispatch
 * CTAs), 6 GEMM role start, 7 GEMM role end, 8 combine barrier passed,
 * 9 combine done, 10 first full stage reaches the tensor core, 11 last MMA
 * completed, 15 CTA exit. */
mk_status_t mk_read_trace(void* stream, const void* workspace, int T, int H, int E, int k, uint64_t* out,
                          size_t n);

/* Free the library's workspace cache on every device (synchronises), and
 * forget the device addresses mk_moe_dispatch_gemm_noalloc looked up. */
void mk_release_workspace(void);

/* Static string for a status code. */
const char* mk_status_string(mk_status_t s);

/* Library ABI version (major * 100 + minor). */
int mk_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
