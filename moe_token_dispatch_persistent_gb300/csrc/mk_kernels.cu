// mk_kernels.cu -- device code of the MoE dispatch + expert GEMM for sm_103a.
//
// One persistent kernel (mk_fused_kernel) runs the whole path.  Its CTAs
// take roles, as the mKernel write-ups describe for their fused kernels
// (CTAs specialise into compute and communication roles, with the number of
// SMs per role set from the tensor shapes; "UC Berkeley presenta mKernel
// ...", edge.aivizor.me, para. 3; lefilia.fr, para. 2), and a tile that has
// landed feeds the GEMM while the next one is still being moved (zubnet.ai,
// para. 2).  On one GPU the "communication" role is the gather of token rows
// from x into expert-contiguous tiles in HBM:
//
//   phase R  (all CTAs)    router top-k + gates per token (a lane per token,
//                           or 2-8 lanes sharing a token's experts when
//                           E = 64, 128, 256), per-chunk histogram and
//                           stable in-chunk ranks
//   barrier               every chunk's counts are in
//   phase S  (all CTAs)    per-expert totals, exclusive scan -> offsets,
//                           tile and work-item tables (each CTA, in smem);
//                           scatter src_index / gate_w of the CTA's chunks
//   dispatch role          pull-gather: units of up to 32 rows of a tile
//                           taken in GEMM consumption order, rows moved with
//                           1-D bulk copies through shared memory, each
//                           unit's row count added to its tile's arrival
//                           count (release); then the CTA joins compute
//   compute role           TMA producer warp -> mbarrier ring -> MMA warp
//                           (tcgen05.mma 128x256x16, fp32 in TMEM; both
//                           loops run on whole warps, one elected lane
//                           issues) -> 4 epilogue warps (tcgen05.ld,
//                           bf16/f32 stores of the tile's valid rows); with
//                           streamed results each finished chunk of rows
//                           raises a flag for a copy stream.  Tiles of 128
//                           rows (4 stages, double-buffered accumulators) or
//                           wide tiles of 256 rows (3 stages; two
//                           accumulators share each weight stage)
//   phase C  (optional)    after a grid barrier, the weighted sum of each
//                           token's k rows (the MoE layer's combine)
//
// Variants of the same pipeline: the gated FFN (W1 and W3 columns side by
// side in one N = 256 product, SwiGLU in the epilogue); rows copied straight
// from x by two copy warps instead of staged by the dispatch role (on 128-row
// or wide tiles); SM pairs (cta_group::2, 256-row tiles); and mk_ep_kernel, which runs R
// logical ranks of an expert-parallel layer in one launch.  The same device
// functions also run as four or five separate launches (route, scan,
// push-gather, GEMM, combine): the host-driven baseline the fused kernel is
// measured against.
//
// Every wait is bounded (spin_limit_ns, %globaltimer); a wait that runs out
// records a timeout in the device error word, raises the call's abort flag
// so the other CTAs stop waiting, drains its own in-flight copies and MMAs,
// frees TMEM and returns.  Nothing traps.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstddef>

#include "mk_common.h"
#include "mk_ptx.cuh"

namespace mk {

struct DevError {
    uint32_t code, site, cta, info;
};
__device__ DevError g_error;

// ------------------------------------------------------------ waiting ------

struct WaitCtx {
    const uint32_t* abort;
    uint32_t abort_val;
    long long limit_ns;
};

__device__ __noinline__ void record_error(uint32_t code, uint32_t site, uint32_t info) {
    if (atomicCAS(&g_error.code, 0u, code) == 0u) {
        g_error.site = site;
        g_error.cta = blockIdx.x;
        g_error.info = info;
        __threadfence();
    }
}

__device__ __forceinline__ bool aborted(const WaitCtx& w) {
    return w.abort != nullptr && ld_relaxed_u32(w.abort) == w.abort_val;
}

__device__ __forceinline__ void raise_abort(const WaitCtx& w) {
    if (w.abort != nullptr) st_relaxed_u32(const_cast<uint32_t*>(w.abort), w.abort_val);
}

// Bounded wait on an mbarrier phase.  False: timed out (recorded) or the call
// was aborted elsewhere.
__device__ __forceinline__ bool wait_mbar(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++n & 63u) == 0u) {
            if (aborted(w)) return false;
            if ((long long)(globaltimer() - t0) > w.limit_ns) {
                record_error(ERR_TIMEOUT, site, parity);
                raise_abort(w);
                return false;
            }
        }
    }
    return true;
}

// Bounded wait for *p >= target (acquire).
__device__ __forceinline__ bool wait_geq(const uint32_t* p, uint32_t target, const WaitCtx& w, int site) {
    if (ld_acquire_u32(p) >= target) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (ld_acquire_u32(p) < target) {
        __nanosleep(64);
        if ((++n & 15u) == 0u) {
            if (aborted(w)) return false;
            if ((long long)(globaltimer() - t0) > w.limit_ns) {
                record_error(ERR_TIMEOUT, site, target);
                raise_abort(w);
                return false;
            }
        }
    }
    return true;
}

// Bounded wait for *p == v (acquire).
__device__ __forceinline__ bool wait_eq(const uint32_t* p, uint32_t v, const WaitCtx& w, int site) {
    if (ld_acquire_u32(p) == v) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (ld_acquire_u32(p) != v) {
        __nanosleep(32);
        if ((++n & 15u) == 0u) {
            if (aborted(w)) return false;
            if ((long long)(globaltimer() - t0) > w.limit_ns) {
                record_error(ERR_TIMEOUT, site, v);
                raise_abort(w);
                return false;
            }
        }
    }
    return true;
}

// The same waits taken by every lane of a warp; the result is the same on
// every lane (a lane that timed out makes the whole warp give up).
__device__ __forceinline__ bool warp_wait_mbar(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, wait_mbar(bar, parity, w, site));
}
__device__ __forceinline__ bool warp_wait_geq(const uint32_t* p, uint32_t target, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, wait_geq(p, target, w, site));
}
__device__ __forceinline__ bool warp_wait_eq(const uint32_t* p, uint32_t v, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, wait_eq(p, v, w, site));
}

__device__ __forceinline__ void stamp(const Params& p, int slot) {
    if (p.trace && threadIdx.x == 0) p.trace_buf[blockIdx.x * TRACE_SLOTS + slot] = globaltimer();
}

// ------------------------------------------------------ shared control -----

struct alignas(16) Info {  // 16-byte aligned: sent to the peer CTA with one v4 store
    int e, row0, nrows, nbk;
};

struct CtrlSmem {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t info_full[4];
    uint64_t info_empty[4];
    uint64_t drain;
    uint64_t gbar[MAX_GATHER_SLOTS];
    Info info[4];
    uint32_t tmem_base;
    int32_t bcast[8];
    int32_t offs[MAX_E + 1];
    int32_t tile_start[MAX_E + 1];
    int32_t item_start[MAX_E + 1];
    int32_t tot[MAX_E];
    int32_t ep_pre[MAX_E];  // expert parallel: rows of each expert sent by earlier ranks
    int32_t ep_cnt[MAX_E];  //                  and by this CTA's rank
};
static_assert(sizeof(CtrlSmem) <= SM_CTRL_BYTES, "control smem too large");
static_assert(offsetof(CtrlSmem, info) % 16 == 0, "info slots must allow 16-byte stores");

__device__ __forceinline__ uint8_t* smem_base() {
    extern __shared__ uint8_t smem_raw[];
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ CtrlSmem* ctrl() { return reinterpret_cast<CtrlSmem*>(smem_base() + SM_CTRL); }

// ------------------------------------------------------------ phase R ------

// Tokens [t0, t1) of routing chunk c: rank r's tokens [ep_t0[r], ep_t0[r+1])
// are cut into chunks of route_chunk tokens from the rank's first token (one
// rank: chunk c covers [c*route_chunk, ...)).  Chunks in id order cover the
// tokens in order, so the sorted order does not depend on where chunks begin.
__device__ __forceinline__ void chunk_tokens(const Params& p, int c, int& t0, int& t1) {
    int r = 0;
    while (r + 1 < p.ranks && p.ep_c0[r + 1] <= c) ++r;
    t0 = p.ep_t0[r] + (c - p.ep_c0[r]) * p.route_chunk;
    t1 = min(t0 + p.route_chunk, p.ep_t0[r + 1]);
}

// Key order of the router: (value desc, expert id asc).
__device__ __forceinline__ bool beats(float v, int e, float u, int f) { return v > u || (v == u && e < f); }

// Sorted insertion of (v, e) into a best-first list of MAX_K entries.
__device__ __forceinline__ void topk_insert(float v, int e, float (&vals)[MAX_K], int (&ids)[MAX_K]) {
    if (beats(v, e, vals[MAX_K - 1], ids[MAX_K - 1])) {
        bool b[MAX_K];
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) b[j] = beats(v, e, vals[j], ids[j]);
#pragma unroll
        for (int j = MAX_K - 1; j >= 0; --j) {
            if (b[j]) {
                const bool prev = (j > 0) && b[j - 1];
                vals[j] = prev ? vals[j - 1] : v;
                ids[j] = prev ? ids[j - 1] : e;
            }
        }
    }
}

// Keep the best MAX_K of this lane's list and that of lane ^ d (both
// best-first, from disjoint experts): entry j against the partner's entry
// MAX_K-1-j gives the best MAX_K as a bitonic sequence, which three
// compare-exchange rounds sort.  Both lanes end with the same list.
__device__ __forceinline__ void topk_merge_xor(int d, float (&vals)[MAX_K], int (&ids)[MAX_K]) {
    float pv[MAX_K];
    int pi[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
        pv[j] = __shfl_xor_sync(0xffffffffu, vals[j], d);
        pi[j] = __shfl_xor_sync(0xffffffffu, ids[j], d);
    }
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
        if (beats(pv[MAX_K - 1 - j], pi[MAX_K - 1 - j], vals[j], ids[j])) {
            vals[j] = pv[MAX_K - 1 - j];
            ids[j] = pi[MAX_K - 1 - j];
        }
    }
#pragma unroll
    for (int h = MAX_K / 2; h > 0; h >>= 1) {
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            if ((j & h) == 0 && beats(vals[j + h], ids[j + h], vals[j], ids[j])) {
                const float tv = vals[j];
                const int ti = ids[j];
                vals[j] = vals[j + h];
                ids[j] = ids[j + h];
                vals[j + h] = tv;
                ids[j + h] = ti;
            }
        }
    }
}

// Route one chunk with S = p.route_lanes > 1 lanes sharing each token
// (E = S * NPL, NPL = 32 or 64; a warp routes 32/S tokens, a chunk
// NWARPS*32/S).  The warp's 32/S logits rows are one contiguous block of
// 32 * NPL floats, read with 16-byte loads and laid out in shared memory as
// 32 segments of NPL (+1 pad) floats, segment (token g, part s) at lane
// g * S + s.  Each lane keeps the best MAX_K of its NPL experts, and log2(S)
// merges give every lane of the token the best MAX_K of all E.  The best
// MAX_K under the key (value desc, id asc) is unique, so the lists equal
// those of a lane per token.  One copy of the code serves every S (runtime).
// Single-device launches only: the expert-parallel kernel routes with a lane
// per token, so the count row goes to the one count table.
__device__ void route_chunk_split(const Params& p, int c) {
    uint8_t* s = smem_base();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.route_lanes, E = p.E, k = p.k;
    const int lgS = __ffs(S) - 1;
    const int TPW = 32 >> lgS;     // tokens per warp
    const int NPL = E >> lgS;      // experts per lane: 32 or 64
    const int NV = NPL >> 2;       // 16-byte loads per lane: 8 or 16
    float* slog = reinterpret_cast<float*>(s + RT_LOGITS) + warp * 32 * RT_LOGIT_STRIDE;
    int* sidx = reinterpret_cast<int*>(s + RT_IDX) + warp * 32 * MAX_K;
    int* slr = reinterpret_cast<int*>(s + RT_LRANK) + warp * 32 * MAX_K;
    int* wcnt = reinterpret_cast<int*>(s + RT_WCNT);
    int tc0, T;  // the chunk's tokens [tc0, T)
    chunk_tokens(p, c, tc0, T);
    const int tbase = tc0 + warp * TPW;
    const int g = lane >> lgS, sub = lane & (S - 1);  // token of the lane in the warp, part of its experts
    const int t = tbase + g;

    for (int e = lane; e < E; e += 32) wcnt[warp * MAX_E + e] = 0;

    const int nvalid = max(0, min(TPW, T - tbase)) * S * NV;  // float4s of the warp's valid rows
    const float4* blk = reinterpret_cast<const float4*>(p.logits + size_t(tbase) * E);
    float4 q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int f = i * 32 + lane;
        q[i] = (i < NV && f < nvalid) ? __ldg(blk + f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (i < NV) {
            const int f = (i * 32 + lane) * 4;  // first float of the load in the warp's block
            float* d = slog + (f / NPL) * (NPL + 1) + f % NPL;
            d[0] = q[i].x;
            d[1] = q[i].y;
            d[2] = q[i].z;
            d[3] = q[i].w;
        }
    }
    __syncwarp();

    float vals[MAX_K];
    int ids[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
        vals[j] = -INFINITY;
        ids[j] = 0x7fffffff;
    }
    if (t < T) {
        const float* seg = slog + lane * (NPL + 1);
        const int e0 = sub * NPL;
#pragma unroll 4
        for (int i = 0; i < NPL; ++i) topk_insert(seg[i], e0 + i, vals, ids);
    }
    for (int d = 1; d < S; d <<= 1) topk_merge_xor(d, vals, ids);

    if (sub == 0 && t < T) {
        // ids outside [0, E) only survive for NaN rows (outside the contract)
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) ids[j] = min(max(ids[j], 0), E - 1);
        const float l0 = vals[0];
        float gv[MAX_K];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            gv[j] = 0.f;
            if (j < k && l0 != -INFINITY) {
                gv[j] = expf(vals[j] - l0);
                sum += gv[j];
            }
        }
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            if (j < k) {
                const float gj = (l0 == -INFINITY) ? 0.f : gv[j] / sum;
                p.topk_idx[size_t(t) * k + j] = ids[j];
                p.topk_gate[size_t(t) * k + j] = gj;
                sidx[g * MAX_K + j] = ids[j];
            }
        }
    }
    __syncwarp();

    // In-warp stable ranks over the warp's TPW tokens, 32/k per pass.
    const int G = 32 / k;
    const uint32_t lt = lanemask_lt();
    for (int it = 0; it * G < TPW; ++it) {
        const int gg = lane / k, j = lane - (lane / k) * k;
        const int tok = it * G + gg;
        const bool valid = (lane < G * k) && (tok < TPW) && (tbase + tok < T);
        const int e = valid ? sidx[tok * MAX_K + j] : -(lane + 1);
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int before = __popc(peers & lt);
        const int base = valid ? wcnt[warp * MAX_E + e] : 0;
        __syncwarp();
        if (valid && before == 0) wcnt[warp * MAX_E + e] = base + __popc(peers);
        __syncwarp();
        if (valid) slr[tok * MAX_K + j] = base + before;
    }
    __syncthreads();

    // Chunk counts and per-warp exclusive bases.
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) {
            const int v = wcnt[w * MAX_E + e];
            wcnt[w * MAX_E + e] = run;
            run += v;
        }
        p.counts[size_t(c) * E + e] = run;
    }
    __syncthreads();
    if (lane < TPW && tbase + lane < T) {
        const int tt = tbase + lane;
        for (int j = 0; j < k; ++j) {
            const int e = sidx[lane * MAX_K + j];
            p.lrank[size_t(tt) * k + j] = slr[lane * MAX_K + j] + wcnt[warp * MAX_E + e];
        }
    }
    __syncthreads();
}

// Route one chunk of ROUTE_CHUNK tokens, a lane per token: top-k + gates,
// per-chunk histogram, and each (t, j)'s rank among the chunk's entries of
// the same expert in (t, j) order.  Whole CTA.  The chunk's count row goes
// to the count table, or, simulating expert parallelism, to every rank's
// copy of it (the all-gather of the counts).
__device__ void route_chunk_lane(const Params& p, int c) {
    uint8_t* s = smem_base();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* slog = reinterpret_cast<float*>(s + RT_LOGITS) + warp * 32 * RT_LOGIT_STRIDE;
    int* sidx = reinterpret_cast<int*>(s + RT_IDX) + warp * 32 * MAX_K;
    int* slr = reinterpret_cast<int*>(s + RT_LRANK) + warp * 32 * MAX_K;
    int* wcnt = reinterpret_cast<int*>(s + RT_WCNT);
    const int E = p.E, k = p.k;
    int tc0, T;  // the chunk's tokens [tc0, T)
    chunk_tokens(p, c, tc0, T);
    const int tbase = tc0 + warp * 32;
    const int t = tbase + lane;

    for (int e = lane; e < E; e += 32) wcnt[warp * MAX_E + e] = 0;

    float vals[MAX_K];
    int ids[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
        vals[j] = -INFINITY;
        ids[j] = 0x7fffffff;
    }
    for (int e0 = 0; e0 < E; e0 += 64) {
        const int ne = min(64, E - e0);
        // All 32 rows' loads are issued before the first store to shared
        // memory (explicit registers), so their latencies overlap.
        float r0[32], r1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int ti = tbase + i;
            const float* row = p.logits + size_t(ti < T ? ti : 0) * E + e0;
            r0[i] = (ti < T && lane < ne) ? __ldg(row + lane) : 0.f;
            r1[i] = (ti < T && lane + 32 < ne) ? __ldg(row + lane + 32) : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            slog[i * RT_LOGIT_STRIDE + lane] = r0[i];
            slog[i * RT_LOGIT_STRIDE + lane + 32] = r1[i];
        }
        __syncwarp();
        if (t < T) {
            // the sorted insertion of topk_insert, written out in place
#pragma unroll 4
            for (int ee = 0; ee < ne; ++ee) {
                const float v = slog[lane * RT_LOGIT_STRIDE + ee];
                const int e = e0 + ee;
                if (beats(v, e, vals[MAX_K - 1], ids[MAX_K - 1])) {
                    // sorted insertion of (v, e) into the 8-entry list
                    bool b[MAX_K];
#pragma unroll
                    for (int j = 0; j < MAX_K; ++j) b[j] = beats(v, e, vals[j], ids[j]);
#pragma unroll
                    for (int j = MAX_K - 1; j >= 0; --j) {
                        if (b[j]) {
                            const bool prev = (j > 0) && b[j - 1];
                            vals[j] = prev ? vals[j - 1] : v;
                            ids[j] = prev ? ids[j - 1] : e;
                        }
                    }
                }
            }
        }
    }

    if (t < T) {
        // ids outside [0, E) only survive for NaN rows (outside the contract)
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) ids[j] = min(max(ids[j], 0), E - 1);
        const float l0 = vals[0];
        float g[MAX_K];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            g[j] = 0.f;
            if (j < k && l0 != -INFINITY) {
                g[j] = expf(vals[j] - l0);
                sum += g[j];
            }
        }
#pragma unroll
        for (int j = 0; j < MAX_K; ++j) {
            if (j < k) {
                const float gj = (l0 == -INFINITY) ? 0.f : g[j] / sum;
                p.topk_idx[size_t(t) * k + j] = ids[j];
                p.topk_gate[size_t(t) * k + j] = gj;
                sidx[lane * MAX_K + j] = ids[j];
            }
        }
    }
    __syncwarp();

    // In-warp stable ranks: lanes hold (token, slot) entries in (t, j) order,
    // 32/k tokens per pass; equal experts are found with match.any.
    const int G = 32 / k;
    const uint32_t lt = lanemask_lt();
    for (int it = 0; it * G < 32; ++it) {
        const int g = lane / k, j = lane - (lane / k) * k;
        const int tok = it * G + g;
        const bool valid = (lane < G * k) && (tok < 32) && (tbase + tok < T);
        const int e = valid ? sidx[tok * MAX_K + j] : -(lane + 1);
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int before = __popc(peers & lt);
        const int base = valid ? wcnt[warp * MAX_E + e] : 0;
        __syncwarp();
        if (valid && before == 0) wcnt[warp * MAX_E + e] = base + __popc(peers);
        __syncwarp();
        if (valid) slr[tok * MAX_K + j] = base + before;
    }
    __syncthreads();

    // Chunk counts and per-warp exclusive bases.
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) {
            const int v = wcnt[w * MAX_E + e];
            wcnt[w * MAX_E + e] = run;
            run += v;
        }
        if (p.ep) {
            for (int q = 0; q < p.ranks; ++q) p.ep_counts[q][size_t(c) * E + e] = run;
        } else {
            p.counts[size_t(c) * E + e] = run;
        }
    }
    __syncthreads();
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = sidx[lane * MAX_K + j];
            p.lrank[size_t(t) * k + j] = slr[lane * MAX_K + j] + wcnt[warp * MAX_E + e];
        }
    }
    __syncthreads();
}

// The routing form the host chose (route_lanes_for).  Measured on GB300:
// each extra copy of the routing code in this kernel slowed the lane-per-
// token path by up to 2 µs, so the split form is one runtime-generic copy
// and the lane path comes first.
__device__ void route_chunk(const Params& p, int c) {
    if (p.route_lanes <= 1) route_chunk_lane(p, c);
    else route_chunk_split(p, c);
}

// ------------------------------------------------------------ phase S ------

// Exclusive scans of per-expert totals into offsets, tile starts and item
// starts (warp 0; E <= 256, 8 experts per lane).
__device__ void build_tables(const Params& p, CtrlSmem* cs) {
    if ((threadIdx.x >> 5) != 0) return;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    // One warp runs this on every CTA's critical path: tiles are 128 or 256
    // rows, so a shift instead of an integer division (about 1 µs here)
    const int tsh = __ffs(p.tile_rows) - 1;
    int lo[8], lt[8], li[8];
    int so = 0, st = 0, si = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        const int v = (e < E) ? cs->tot[e] : 0;
        const int nt = (v + p.tile_rows - 1) >> tsh;
        lo[i] = so;
        lt[i] = st;
        li[i] = si;
        so += v;
        st += nt;
        si += nt * p.nb;
    }
    int io = so, it = st, ii = si;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, io, o);
        const int b = __shfl_up_sync(0xffffffffu, it, o);
        const int c = __shfl_up_sync(0xffffffffu, ii, o);
        if (lane >= o) {
            io += a;
            it += b;
            ii += c;
        }
    }
    const int eo = io - so, et = it - st, ei = ii - si;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        if (e < E) {
            cs->offs[e] = eo + lo[i];
            cs->tile_start[e] = et + lt[i];
            cs->item_start[e] = ei + li[i];
        }
    }
    if (lane == 31) {
        cs->offs[E] = io;
        cs->tile_start[E] = it;
        cs->item_start[E] = ii;
    }
}

// Totals from the full counts table; for the CTA's own chunks (c_first,
// c_first + c_stride, ... below c_end) the column prefix (rows of earlier
// chunks) is kept in smem as the chunk's bases.  With src_rank >= 0 the
// per-expert rows of the chunks before that rank's (ep_pre) and of its own
// chunks (ep_cnt) are kept too: where its rows sit inside each expert.
__device__ void scan_counts(const Params& p, CtrlSmem* cs, const int32_t* counts, bool keep_bases, int c_first,
                            int c_stride, int c_end, int src_rank) {
    int* sbase = reinterpret_cast<int*>(smem_base() + RT_BASES);
    int* scnt = reinterpret_cast<int*>(smem_base());  // routing scratch is dead by now
    const int E = p.E, nch = p.nch;
    const int total = nch * E;
    const bool in_smem = total <= RT_BASES / 4;
    if (in_smem) {
        // copy the counts table to shared memory with 16-byte cp.async (L2
        // only: the rows come from other CTAs), all of a thread's copies in
        // flight at once.  The last piece may read up to 12 bytes of the
        // table's padding (its workspace region is 256-byte aligned and
        // sized), which nothing uses.
        const int n16 = (total + 3) / 4;
        const uint32_t dst = smem_u32(scnt);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(counts);
        for (int i = threadIdx.x; i < n16; i += NTHREADS) cp_async_16_u32(dst + uint32_t(i) * 16u, src + size_t(i) * 16);
        cp_async_wait_all();
        __syncthreads();
    }
    const int s_lo = src_rank >= 0 ? p.ep_c0[src_rank] : 0;
    const int s_hi = src_rank >= 0 ? p.ep_c0[src_rank + 1] : 0;
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        int run = 0, m = 0, pre = 0, upto = 0;
        int mine = c_first;
        for (int c = 0; c < nch; ++c) {
            if (keep_bases && c == mine && c < c_end) {
                sbase[m * MAX_E + e] = run;
                ++m;
                mine += c_stride;
            }
            if (c == s_lo) pre = run;
            if (c == s_hi) upto = run;
            run += in_smem ? scnt[c * E + e] : __ldcg(counts + size_t(c) * E + e);
        }
        cs->tot[e] = run;
        if (src_rank >= 0) {
            if (s_lo >= nch) pre = run;
            if (s_hi >= nch) upto = run;
            cs->ep_pre[e] = pre;
            cs->ep_cnt[e] = upto - pre;
        }
    }
    __syncthreads();
    build_tables(p, cs);
    __syncthreads();
    if (keep_bases) {
        int m = 0;
        for (int c = c_first; c < c_end; c += c_stride, ++m)
            for (int e = threadIdx.x; e < E; e += NTHREADS) sbase[m * MAX_E + e] += cs->offs[e];
    }
    __syncthreads();
}

// Distributed scan, step 1 (CTA b): for the experts e = b, b + grid, ... the
// exclusive prefix over chunks of count[c][e] goes to bases[c][e] and the
// column total to totals[e].  Thread i holds the consecutive chunks
// [i*per, (i+1)*per): a pass over them for its sum, a block-wide exclusive
// scan of the sums (warp shuffles, then the warps' totals), a second pass
// writing the prefixes.
__device__ void scan_columns(const Params& p) {
    int* wsum = reinterpret_cast<int*>(smem_base());  // per-warp sums (routing scratch is dead)
    const int nch = p.nch, E = p.E;
    const int per = (nch + NTHREADS - 1) / NTHREADS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = threadIdx.x * per;
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        int sum = 0;
        for (int i = 0; i < per; ++i) {
            const int c = c0 + i;
            if (c < nch) sum += __ldcg(p.counts + size_t(c) * E + e);
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += wsum[w];
        for (int i = 0; i < per; ++i) {
            const int c = c0 + i;
            if (c < nch) {
                p.bases[size_t(c) * E + e] = run;
                run += __ldcg(p.counts + size_t(c) * E + e);
            }
        }
        if (threadIdx.x == NTHREADS - 1) p.totals[e] = run;  // the last thread's run covers every chunk
        __syncthreads();
    }
}

// Distributed scan, step 2 (after the barrier): the totals give every CTA
// its offset, tile and item tables; the bases of its own chunks (c_first,
// c_first + c_stride, ... below c_end) are offs[e] + bases[c][e], kept in
// shared memory as scan_counts keeps them.
__device__ void scan_from_columns(const Params& p, CtrlSmem* cs, int c_first, int c_stride, int c_end) {
    int* sbase = reinterpret_cast<int*>(smem_base() + RT_BASES);
    const int E = p.E;
    for (int e = threadIdx.x; e < E; e += NTHREADS) cs->tot[e] = __ldcg(p.totals + e);
    __syncthreads();
    build_tables(p, cs);
    __syncthreads();
    int m = 0;
    for (int c = c_first; c < c_end; c += c_stride, ++m)
        for (int e = threadIdx.x; e < E; e += NTHREADS)
            sbase[m * MAX_E + e] = cs->offs[e] + __ldcg(p.bases + size_t(c) * E + e);
    __syncthreads();
}

// Scatter src_index / gate_w for (t, j) entries of chunk c (bases in smem).
__device__ void scatter_chunk(const Params& p, int c, const int* cbase, const WaitCtx& w) {
    const int k = p.k;
    int t0, t1;
    chunk_tokens(p, c, t0, t1);
    const int n = (t1 - t0) * k;
    constexpr int U = 4;  // entries per thread per batch: loads issued before the stores
    for (int i0 = threadIdx.x; i0 < n; i0 += NTHREADS * U) {
        int e[U], lr[U];
        float g[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * NTHREADS;
            const int q = t0 * k + (i < n ? i : 0);
            e[u] = __ldcg(p.topk_idx + q);
            lr[u] = __ldcg(p.lrank + q);
            g[u] = __ldcg(p.topk_gate + q);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * NTHREADS;
            if (i >= n) continue;
            const int q = t0 * k + i;
            const int dest = cbase[min(max(e[u], 0), p.E - 1)] + lr[u];
            if (dest < 0 || dest >= p.rows) {
                record_error(ERR_FAULT, SITE_DEST_RANGE, uint32_t(dest));
                raise_abort(w);
                continue;
            }
            p.src_index[dest] = q;
            p.gate_w[dest] = g[u];
            p.row_of[q] = dest;
        }
    }
}

// ------------------------------------------------------------- gather ------

__device__ __forceinline__ int find_expert(const int32_t* starts, int E, int v) {
    // largest e with starts[e] <= v (starts[0] = 0 <= v < starts[E])
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (starts[mid] <= v) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Dispatch role (the first p.gather_warps warps, each on its own share of
// the slots): pull gather units from the queue in GEMM consumption order.
// A unit is up to gather_slots / gather_warps rows of one tile, one row per
// slot lane, so several dispatch CTAs fill a tile at once and its
// first items start soon after the scan.  Each lane moves its row
// x[src] -> smem -> xs[row] with bulk copies and closes one bulk group per
// unit (empty when it had no row).  The loop is software-pipelined: while a
// unit's loads are in flight the next unit is claimed and its sources are
// read.  Units of the tiles that the first wave of work items needs (items
// [0, grid)) are published as soon as their stores complete: those tiles
// gate the GEMM's start.  Later units are published one unit behind, their
// stores completing while the next unit's loads are in flight.  Publishing
// adds the unit's rows to the tile's arrival count (release); the unit that
// completes a tile also counts it in tiles_done.
__device__ __forceinline__ void publish_unit(const Params& p, int tile, int n, int trows) {
    if (tile == p.debug_drop_tile) return;  // host-side fault injection: this tile never completes
    // the release orders this thread's earlier writes (and, through the
    // proxy fence the caller executed, the completed bulk stores) before it
    const uint32_t before = atom_add_acq_rel_u32(p.ready + tile, uint32_t(n));
    // once tiles_done reaches the tile count, one acquire of it stands in for
    // every tile's arrival count
    if (before + uint32_t(n) == uint32_t(trows)) atom_add_acq_rel_u32(&p.ctl->tiles_done, 1u);
}

__device__ __forceinline__ void decode_item(const Params& p, const CtrlSmem* cs, int item, Info& inf, int& gtile);

// The TMA producers (staged rows, SM pairs) take their next work item from
// the queue this many K-blocks before the end of the current one's loads:
// early enough that the atomic and the decode are hidden, late enough that
// near the end of the queue an item goes to a CTA that is about to be free,
// not to one that still has a whole item ahead of it.  Measured on GB300:
// -1.0% on the Mixtral-like layer and -1.2% on decode against claiming at
// the start of the current item.  The direct-row producers keep claiming at
// the item's start: the late claim cost them 1% on the skewed layer.
constexpr int CLAIM_LEAD = 4;

// Geometry of gather unit u and the source token of this lane's row in it.
struct GatherUnit {
    int tile, row, n, trows, src_t;  // tile; this lane's sorted row; rows in the unit; rows in the tile
};

__device__ __forceinline__ GatherUnit gather_unit(const Params& p, const CtrlSmem* cs, int u, int unit, int upt,
                                                  int lane) {
    GatherUnit g{-1, 0, 0, 0, -1};
    g.tile = u / upt;
    const int e = find_expert(cs->tile_start, p.E, g.tile);
    const int row0 = cs->offs[e] + (g.tile - cs->tile_start[e]) * p.tile_rows;
    g.trows = min(p.tile_rows, cs->offs[e + 1] - row0);
    const int r0 = (u - g.tile * upt) * unit;
    g.n = max(0, min(unit, g.trows - r0));
    g.row = row0 + r0 + lane;
    if (lane < g.n) g.src_t = __ldcg(p.src_index + g.row) / p.k;
    return g;
}

__device__ void gather_role(const Params& p, CtrlSmem* cs, const WaitCtx& w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = p.gather_warps;  // each gathering warp runs this loop on its own slots
    if (warp >= gw) return;
    uint8_t* s = smem_base();
    const uint32_t row_bytes = uint32_t(p.H) * 2u;
    const int unit = p.gather_slots / gw;             // rows per unit: one per slot lane
    const int upt = (p.tile_rows + unit - 1) / unit;  // units per tile
    const int nunits = cs->tile_start[p.E] * upt;
    const int sl = min(warp * unit + lane, p.gather_slots - 1);  // this lane's slot (lanes >= unit never copy)
    uint8_t* slot = s + size_t(sl) * row_bytes;
    // tiles [0, urgent] hold the rows of the first wave of work items; worked
    // out while the first unit's loads are in flight (it is first needed once
    // they have landed)
    int urgent = -1;
    bool urgent_known = false;
    uint32_t ph = 0;
    bool ok = true;
    int pend_tile = -1, pend_n = 0, pend_rows = 0;    // the unit whose stores may still be in flight
    int u = 0;
    if (lane == 0) u = int(atom_add_relaxed_u32(&p.ctl->next_tile, 1u));
    u = __shfl_sync(0xffffffffu, u, 0);
    GatherUnit cur{-1, 0, 0, 0, -1};
    if (u < nunits) cur = gather_unit(p, cs, u, unit, upt, lane);
    for (;;) {
        const bool have = ok && u < nunits && !aborted(w);
        // claim the next unit now: its atomic and source reads overlap this unit's copies
        int un = 0;
        if (have && lane == 0) un = int(atom_add_relaxed_u32(&p.ctl->next_tile, 1u));
        bool issued = false;
        if (have && lane < cur.n) {
            if (cur.src_t < 0 || cur.src_t >= p.T) {
                record_error(ERR_FAULT, SITE_DEST_RANGE, uint32_t(cur.row));
                raise_abort(w);
                ok = false;
            } else {
                bulk_wait_read<0>();  // the slot's previous store has read it
                mbar_arrive_expect_tx(&cs->gbar[sl], row_bytes);
                bulk_load(slot, p.x + size_t(cur.src_t) * p.H, row_bytes, &cs->gbar[sl]);
                issued = true;
            }
        }
        un = __shfl_sync(0xffffffffu, un, 0);
        GatherUnit nxt{-1, 0, 0, 0, -1};
        if (have && un < nunits) nxt = gather_unit(p, cs, un, unit, upt, lane);
        if (!urgent_known) {
            const int nfirst = min(int(gridDim.x), cs->item_start[p.E]);
            for (int i = lane; i < nfirst; i += 32) {
                Info inf;
                int gt;
                decode_item(p, cs, i, inf, gt);
                urgent = max(urgent, gt);
            }
            urgent = __reduce_max_sync(0xffffffffu, urgent);
            urgent_known = true;
        }
        if (issued) {
            if (!wait_mbar(&cs->gbar[sl], ph, w, SITE_GATHER_LOAD)) {
                ok = false;
                // the load is in flight: give it a short, bounded chance to land
                WaitCtx shortw{nullptr, 0u, 2000000LL};
                wait_mbar(&cs->gbar[sl], ph, shortw, SITE_DRAIN);
            }
            ph ^= 1u;
            if (ok) bulk_store(p.xs + size_t(cur.row) * p.H, slot, row_bytes);
        }
        bulk_commit();  // this unit's group (empty without a row)
        ok = __all_sync(0xffffffffu, ok);
        if (have && cur.n > 0 && cur.tile <= urgent) {
            // a unit of the first wave's tiles: publish it without waiting for
            // the next one (and the one before it, if still pending)
            bulk_wait<0>();
            fence_proxy_async();
            __syncwarp();
            if (lane == 0 && ok) {
                if (pend_tile >= 0) publish_unit(p, pend_tile, pend_n, pend_rows);
                publish_unit(p, cur.tile, cur.n, cur.trows);
            }
            pend_tile = -1;
        } else {
            if (pend_tile >= 0) {
                // the previous unit's group is complete once at most this one is pending
                bulk_wait<1>();
                fence_proxy_async();
                __syncwarp();
                if (lane == 0 && ok) publish_unit(p, pend_tile, pend_n, pend_rows);
            }
            pend_tile = (have && cur.n > 0) ? cur.tile : -1;
            pend_n = cur.n;
            pend_rows = cur.trows;
        }
        if (!have) break;
        u = un;
        cur = nxt;
    }
    bulk_wait_all();
}

// Expert-parallel send role of source rank `src` (warp 0): the rank walks
// the destination tiles (tile i of every rank before tile i + 1 of any, so
// each destination's first tiles fill first) and, for each tile that holds
// rows of its own tokens, copies those rows x -> smem -> the destination's
// receive buffer with 1-D bulk copies, then adds their number to the tile's
// arrival count (release).  Inside one expert the rows of a source are one
// contiguous range (sorted by token), so a tile takes one range per source;
// the tile is complete when its count reaches its row count.
__device__ void send_role(const Params& p, CtrlSmem* cs, int src, const WaitCtx& w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp != 0) return;
    uint8_t* s = smem_base();
    const uint32_t row_bytes = uint32_t(p.H) * 2u;
    const int nslot = p.gather_slots;
    const int R = p.ranks, epr = p.E / R;
    int max_tiles = 0;
    for (int q = 0; q < R; ++q)
        max_tiles = max(max_tiles, cs->tile_start[(q + 1) * epr] - cs->tile_start[q * epr]);
    const int t_lo = p.ep_t0[src], t_hi = p.ep_t0[src + 1];
    uint32_t ph = 0;
    bool ok = true;
    while (ok) {
        int sq = 0;
        if (lane == 0) sq = int(atom_add_relaxed_u32(&p.ep_ctl[src]->next_send, 1u));
        sq = __shfl_sync(0xffffffffu, sq, 0);
        if (sq >= R * max_tiles) break;
        const int q = sq % R, i = sq / R;
        const int tile_lo = cs->tile_start[q * epr];
        const int tile = tile_lo + i;
        if (tile >= cs->tile_start[(q + 1) * epr]) continue;
        const int e = find_expert(cs->tile_start, p.E, tile);
        const int row0 = cs->offs[e] + (tile - cs->tile_start[e]) * p.tile_rows;
        const int row1 = min(row0 + p.tile_rows, cs->offs[e + 1]);
        const int lo = max(row0, cs->offs[e] + cs->ep_pre[e]);
        const int hi = min(row1, cs->offs[e] + cs->ep_pre[e] + cs->ep_cnt[e]);
        if (lo >= hi) continue;
        uint16_t* recv = p.ep_recv[q];
        const int recv0 = cs->offs[q * epr];  // first sorted row of rank q
        if (lane < nslot) {
            uint8_t* slot = s + size_t(lane) * row_bytes;
            for (int r = lo + lane; r < hi && ok; r += nslot) {
                const int src_t = __ldcg(p.src_index + r) / p.k;
                if (src_t < t_lo || src_t >= t_hi) {
                    record_error(ERR_FAULT, SITE_DEST_RANGE, uint32_t(r));
                    raise_abort(w);
                    ok = false;
                    break;
                }
                bulk_wait_read<0>();
                mbar_arrive_expect_tx(&cs->gbar[lane], row_bytes);
                bulk_load(slot, p.x + size_t(src_t) * p.H, row_bytes, &cs->gbar[lane]);
                if (!wait_mbar(&cs->gbar[lane], ph, w, SITE_GATHER_LOAD)) {
                    ok = false;
                    WaitCtx shortw{nullptr, 0u, 2000000LL};
                    wait_mbar(&cs->gbar[lane], ph, shortw, SITE_DRAIN);
                }
                ph ^= 1u;
                if (ok) {
                    bulk_store(recv + size_t(r - recv0) * p.H, slot, row_bytes);
                    bulk_commit();
                }
            }
            bulk_wait_all();
            fence_proxy_async();
        }
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0 && ok && tile != p.debug_drop_tile) {
            __threadfence();
            atom_add_acq_rel_u32(p.ep_ready[q] + (tile - tile_lo), uint32_t(hi - lo));
        }
        if (aborted(w)) break;
    }
    bulk_wait_all();
}

// Unfused path: push-gather of chunk c (every entry to its destination row).
__device__ void push_gather_chunk(const Params& p, int c, CtrlSmem* cs, uint32_t& ph, const WaitCtx& w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp != 0) return;
    uint8_t* s = smem_base();
    const uint32_t row_bytes = uint32_t(p.H) * 2u;
    const int nslot = p.gather_slots;
    const int k = p.k;
    int t0, t1;
    chunk_tokens(p, c, t0, t1);
    const int n = (t1 - t0) * k;
    if (lane < nslot) {
        uint8_t* slot = s + size_t(lane) * row_bytes;
        for (int i = lane; i < n; i += nslot) {
            const int q = t0 * k + i;
            const int e = __ldcg(p.topk_idx + q);
            const int dest = __ldcg(p.bases + size_t(c) * p.E + e) + __ldcg(p.lrank + q);
            if (dest < 0 || dest >= p.rows) {
                record_error(ERR_FAULT, SITE_DEST_RANGE, uint32_t(dest));
                continue;
            }
            p.src_index[dest] = q;
            p.gate_w[dest] = __ldcg(p.topk_gate + q);
            p.row_of[q] = dest;
            bulk_wait_read<0>();
            mbar_arrive_expect_tx(&cs->gbar[lane], row_bytes);
            bulk_load(slot, p.x + size_t(q / k) * p.H, row_bytes, &cs->gbar[lane]);
            if (!wait_mbar(&cs->gbar[lane], ph, w, SITE_GATHER_LOAD)) {
                WaitCtx shortw{nullptr, 0u, 2000000LL};
                wait_mbar(&cs->gbar[lane], ph, shortw, SITE_DRAIN);
                ph ^= 1u;
                break;
            }
            ph ^= 1u;
            bulk_store(p.xs + size_t(dest) * p.H, slot, row_bytes);
            bulk_commit();
        }
        bulk_wait_all();
    }
}

// ------------------------------------------------------------ compute ------

__device__ __forceinline__ void decode_item(const Params& p, const CtrlSmem* cs, int item, Info& inf, int& gtile) {
    const int e = find_expert(cs->item_start, p.E, item);
    const int local = item - cs->item_start[e];
    const int nt = cs->tile_start[e + 1] - cs->tile_start[e];
    const int NB = p.nb, G = p.n_group;
    const int full = NB / G;
    int t_in, nbk;
    if (local < full * nt * G) {
        const int g = local / (nt * G);
        const int r = local - g * (nt * G);
        t_in = r / G;
        nbk = g * G + (r - t_in * G);
    } else {
        const int l2 = local - full * nt * G;
        const int Gl = NB - full * G;
        t_in = l2 / Gl;
        nbk = full * G + (l2 - t_in * Gl);
    }
    inf.e = e;
    inf.row0 = cs->offs[e] + t_in * p.tile_rows;
    inf.nrows = min(p.tile_rows, cs->offs[e + 1] - inf.row0);
    inf.nbk = nbk;
    gtile = cs->tile_start[e] + t_in;
}

constexpr uint32_t IDESC = umma_idesc_bf16(BM, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);
// Gated FFN: 128 output columns per item; the item's B stage holds those
// columns of both projections (gate W1, up W3) side by side.
constexpr int GATED_BN = BN / 2;

// One thread's 32 consecutive fp32 results of row `row`, columns [col, col+32),
// stored as bf16 (round to nearest even) or f32.  Each lane writes its own
// row, so a warp instruction touches 32 rows: with a 32-byte aligned y every
// store fills whole 32-byte sectors (256-bit stores; a 16-byte store writes
// half a sector, and the epilogue then costs about 6% of the kernel).
__device__ __forceinline__ void store_row32(const Params& p, size_t row, int col, const uint32_t (&r)[32]) {
    if (p.out_f32) {
        float* dst = static_cast<float*>(p.y) + row * p.F + col;
        if (p.y_v8) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_global_v8(dst + 8 * v, r[8 * v], r[8 * v + 1], r[8 * v + 2], r[8 * v + 3], r[8 * v + 4],
                             r[8 * v + 5], r[8 * v + 6], r[8 * v + 7]);
        } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int v = 0; v < 8; ++v) d4[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        }
    } else {
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
            pk[u] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint16_t* dst = static_cast<uint16_t*>(p.y) + row * p.F + col;
        if (p.y_v8) {
            st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
            st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int v = 0; v < 4; ++v) d4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
    }
}

// Shared-memory stage geometry of the two single-SM tile forms, 64 rows of
// K per stage.  128-row tiles: four stages of one A block and one B block.
// Wide (256-row) tiles: three stages of two A blocks and one B block.  A
// rows are K-major in the 128-byte swizzle (one row = 64 bf16 = one swizzle
// span); B is N-major, 64-column chunks in the 128-byte swizzle.
template <bool WIDE>
struct StageGeo {
    static constexpr int KB = BK;                      // K per stage
    static constexpr int NST = WIDE ? WSTAGES : STAGES;
    static constexpr int ABLK = BM * KB * 2;           // one 128-row A block
    static constexpr int ASB = (WIDE ? 2 : 1) * ABLK;  // A bytes of a stage
    static constexpr int BCH = KB * 64 * 2;            // one 64-column B chunk
    static constexpr int BSB = KB * BN * 2;            // B bytes of a stage
    static constexpr int SMB = NST * ASB;              // B stages follow the A stages
    static_assert(SMB + NST * BSB <= SM_STAGE_END, "stages must fit in the stage area");
    static_assert(NST <= MAX_STAGES, "one full/empty barrier pair per stage");
    static_assert(BSB / 2 == (GATED_BN / 64) * BCH, "gated: W3 chunks follow the W1 chunks directly");
};

// Descriptor of a 128-row A block at `addr` (K offset already added):
// K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t a_desc(uint32_t addr) { return umma_desc_sw128(addr, 16, 1024); }

// Epilogue of 32 whole rows (TMEM lanes of this warp, all inside the tile)
// through shared memory.  Per 64-column chunk the warp reads its
// accumulator columns (for the gated FFN: the W1 and W3 halves, SwiGLU
// applied), rounds them to bf16 and writes its 32 rows into its own 4 KiB
// buffer in the 128-byte swizzle (lane = row, chunk c of row r at
// r*128 + ((c ^ (r % 8)) * 16): conflict-free).  With EPI_TMA_STORE one lane
// stores the 32 x 64 box with one TMA store (the buffer is rewritten once
// that store has read it); otherwise the warp reads the box back with 8
// lanes per row and writes four whole 128-byte lines per store
// instruction.  Either way the per-row stores of the plain epilogue (32
// rows, 32 bytes each, per warp instruction) become whole lines.
__device__ __forceinline__ void epi_rows_box(const Params& p, const CUtensorMap* tmY, uint8_t* buf, uint32_t tbase,
                                             int n0, int row_first) {
    const int lane = threadIdx.x & 31;
    const int nchunks = (p.gated ? GATED_BN : BN) / EPI_BOX_COLS;
#pragma unroll 1
    for (int c64 = 0; c64 < nchunks; ++c64) {
        const int col = n0 + c64 * EPI_BOX_COLS;
        if (col >= p.F) break;
        uint32_t pk[32];
        if (p.gated) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32], r3[32];
                tmem_ld_32x32b_x32(tbase + c64 * 64 + h * 32, r);
                tmem_ld_32x32b_x32(tbase + GATED_BN + c64 * 64 + h * 32, r3);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    // SwiGLU as in the per-row epilogue: silu(a) * b, fast intrinsics
                    const float a0 = __uint_as_float(r[2 * u]), a1 = __uint_as_float(r[2 * u + 1]);
                    const float v0 = __fdividef(a0, 1.f + __expf(-a0)) * __uint_as_float(r3[2 * u]);
                    const float v1 = __fdividef(a1, 1.f + __expf(-a1)) * __uint_as_float(r3[2 * u + 1]);
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
                    pk[16 * h + u] = *reinterpret_cast<const uint32_t*>(&b2);
                }
            }
        } else {
            uint32_t r[32], r2[32];
            tmem_ld_32x32b_x32(tbase + c64 * 64, r);
            tmem_ld_32x32b_x32(tbase + c64 * 64 + 32, r2);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const __nv_bfloat162 b0 = __floats2bfloat162_rn(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
                const __nv_bfloat162 b1 =
                    __floats2bfloat162_rn(__uint_as_float(r2[2 * u]), __uint_as_float(r2[2 * u + 1]));
                pk[u] = *reinterpret_cast<const uint32_t*>(&b0);
                pk[16 + u] = *reinterpret_cast<const uint32_t*>(&b1);
            }
        }
        const uint32_t rowaddr = smem_u32(buf) + uint32_t(lane) * 128u;
        if constexpr (EPI_TMA_STORE) {
            if (lane == 0) bulk_wait_read<0>();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(rowaddr + ((uint32_t(c) ^ uint32_t(lane & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                             pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_shared();  // the generic writes before the tensor store reads them
            __syncwarp();
            if (lane == 0) {
                tma_store_2d_hint(tmY, buf, col, row_first, l2_policy_evict_first());  // results are not read again
                bulk_commit();
            }
        } else {
            // transpose through the buffer: lane = row on the way in; on the way
            // out 8 lanes cover one row's 128 bytes, so a warp store writes four
            // whole lines
            __syncwarp();  // the previous box has been read out of the buffer
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(rowaddr + ((uint32_t(c) ^ uint32_t(lane & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                             pk[4 * c + 2], pk[4 * c + 3]);
            __syncwarp();
            const int c = lane & 7, rq = lane >> 3;
            uint16_t* ybase = static_cast<uint16_t*>(p.y) + size_t(row_first) * p.F + col + c * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + rq;  // r % 8 = rq + 4 * (i & 1)
                uint32_t v0, v1, v2, v3;
                ld_shared_v4(smem_u32(buf) + uint32_t(r) * 128u + ((uint32_t(c) ^ uint32_t(r & 7)) << 4), v0, v1, v2,
                             v3);
                *reinterpret_cast<uint4*>(ybase + size_t(r) * p.F) = make_uint4(v0, v1, v2, v3);
            }
        }
    }
}

// Direct-gather producer: COPY_WARPS warps (warp 0, the leader, and warps
// 6..), no staging rows, no tile flags.  Per item the leader's lane 0 takes a
// work item from the queue and publishes it; the helpers read it from the
// same info slot.  Per K-block the leader arms the stage with the TMA bytes
// of B (W boxes, as in the staged path), and every copy warp copies its
// COPY_ROWS token rows of the tile straight from x with 16-byte cp.async
// into the 128-byte-swizzled layout the MMA reads: lane (c = lane % 8,
// rq = lane / 8) copies chunk c of rows 4i + rq of the warp's slice, so each
// warp instruction reads four whole 128-byte lines, and chunk c of row r
// lands at r*128 + ((c ^ (r % 8)) * 16).  Each lane then arms an asynchronous
// arrival on the stage's full barrier that fires once its copies have landed
// (1 + 32 * COPY_WARPS arrivals per phase); the MMA thread orders those
// generic-proxy writes before the tensor core's reads with a proxy fence.
// One warp alone cannot issue the copies as fast as the tensor core consumes
// them, hence several.
//
// WIDE (256-row tiles): each copy warp fills one whole 128-row A block of
// the stage; a tile of at most 128 rows needs only the first.
template <bool WIDE>
__device__ void producer_direct(const Params& p, const CUtensorMap* tmB, const CUtensorMap* tmB3, CtrlSmem* cs,
                                const int cw, const WaitCtx& wp) {
    static_assert(!WIDE || COPY_WARPS == 2, "wide tiles: one 128-row block per copy warp");
    using G = StageGeo<WIDE>;
    constexpr int NST = G::NST, ASB = G::ASB, SMB = G::SMB;
    constexpr int ROWS = WIDE ? BM : COPY_ROWS;  // A rows this warp copies per stage
    constexpr int CPR = G::KB * 2 / 16;          // 16-byte chunks per row and stage: 8
    constexpr int RPI = 32 / CPR;                // rows per warp instruction: 4
    static_assert(CPR == 8, "one A row of a stage is one 128-byte swizzle span");
    const int kblocks = p.H / G::KB;
    const int lane = threadIdx.x & 31;
    const bool leader = cw == 0;
    uint8_t* s = smem_base();
    const int total_items = cs->item_start[p.E];
    const uint64_t wpol = l2_policy_evict_last();  // weight slices: the other tiles of the group read them next
    uint32_t stage = 0, phase = 0;
    uint32_t issued_par = 0, issued_any = 0;
    bool ok = true;
    uint32_t next = 0;
    if (leader && lane == 0) next = atom_add_relaxed_u32(&p.ctl->next_item, 1u);
    for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
        int go = 1;  // 1: an item to run, 0: queue empty, -1: gave up
        Info inf{0, 0, 0, 0};
        if (lane == 0) {
            if (leader) {
                const int item = int(next);
                int gtile = 0;
                if (!wait_mbar(&cs->info_empty[slot], iph ^ 1u, wp, SITE_INFO_EMPTY)) {
                    go = -1;
                } else if (item >= total_items) {
                    cs->info[slot].e = -1;
                    mbar_arrive(&cs->info_full[slot]);
                    go = 0;
                } else {
                    next = atom_add_relaxed_u32(&p.ctl->next_item, 1u);  // claimed one item ahead
                    decode_item(p, cs, item, inf, gtile);
                    cs->info[slot] = inf;
                    mbar_arrive(&cs->info_full[slot]);
                }
            } else if (!wait_mbar(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) {
                go = -1;
            } else {
                inf = cs->info[slot];
                mbar_arrive(&cs->info_empty[slot]);
                go = inf.e < 0 ? 0 : 1;
            }
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (go <= 0) {
            ok = go == 0;
            break;
        }
        inf.e = __shfl_sync(0xffffffffu, inf.e, 0);
        inf.row0 = __shfl_sync(0xffffffffu, inf.row0, 0);
        inf.nrows = __shfl_sync(0xffffffffu, inf.nrows, 0);
        inf.nbk = __shfl_sync(0xffffffffu, inf.nbk, 0);
        // byte offset in x of the tile rows this lane copies (rows past the
        // tile repeat its first row; their products are never stored)
        uint32_t rowoff[ROWS / RPI];
#pragma unroll
        for (int i = 0; i < ROWS / RPI; ++i) {
            const int r = cw * ROWS + RPI * i + lane / CPR;
            const int q = __ldcg(p.src_index + inf.row0 + (r < inf.nrows ? r : 0));
            rowoff[i] = uint32_t(min(max(q / p.k, 0), p.T - 1)) * uint32_t(p.H) * 2u;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
            if (!warp_wait_mbar(&cs->empty[stage], phase ^ 1u, wp, SITE_STAGE_EMPTY)) {
                ok = false;
                break;
            }
            if (leader) mbar_arrive_expect_tx_elect(&cs->full[stage], G::BSB);
            __syncwarp();  // the expect-tx before this warp's copies arrive
            uint64_t* fb = &cs->full[stage];
            uint8_t* a = s + stage * ASB + cw * ROWS * 128;
            if (!WIDE || cw * ROWS < inf.nrows) {
                const int c = lane % CPR, rq = lane / CPR;
                const uint8_t* src = reinterpret_cast<const uint8_t*>(p.x) + kb * (G::KB * 2) + c * 16;
                // 128-byte swizzle: chunk c of row r at r*128 + ((c ^ (r % 8)) * 16)
                const uint32_t d0 = smem_u32(a) + rq * 128 + ((c ^ rq) << 4);             // rows 4i + rq, i even
                const uint32_t d1 = smem_u32(a) + (4 + rq) * 128 + ((c ^ (4 + rq)) << 4);  // i odd: row % 8 = 4 + rq
#pragma unroll
                for (int i = 0; i < ROWS / RPI; ++i)
                    cp_async_16_u32(((i & 1) ? d1 - 512 : d0) + 512 * i, src + rowoff[i]);
            }
            cp_async_mbar_arrive_noinc(fb);  // fires once this lane's copies (if any) have landed
            if (leader) {
                uint8_t* b = s + SMB + stage * G::BSB;
                const int ncol = p.F;
                if (p.gated) {
#pragma unroll
                    for (int q = 0; q < GATED_BN / 64; ++q) {
                        const int col = inf.nbk * GATED_BN + q * 64;
                        const int cc = col < ncol ? col : ncol;
                        tma_load_2d_elect_hint(b + q * G::BCH, tmB, cc, inf.e * p.H + kb * G::KB, fb, wpol);
                        tma_load_2d_elect_hint(b + G::BSB / 2 + q * G::BCH, tmB3, cc, inf.e * p.H + kb * G::KB, fb, wpol);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < BN / 64; ++q) {
                        const int col = inf.nbk * BN + q * 64;
                        tma_load_2d_elect_hint(b + q * G::BCH, tmB, col < ncol ? col : ncol, inf.e * p.H + kb * G::KB,
                                          fb, wpol);
                    }
                }
                issued_any |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == NST) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
    }
    cp_async_wait_all();  // no copy of this warp outlives the role
    if (!ok && leader && lane == 0) {
        WaitCtx shortw{nullptr, 0u, 5000000LL};
        for (int st = 0; st < NST; ++st)
            if (issued_any & (1u << st)) wait_mbar(&cs->full[st], (issued_par >> st) & 1u, shortw, SITE_DRAIN);
    }
    __syncwarp();
}

// TMA-gather producer (rows straight from x, one warp): per K-block each
// lane issues one tile::gather4 per 128-row A block of the stage for rows
// 4*lane .. 4*lane+3 of that block, so the warp lands the whole block in
// the A stage's swizzled layout (the tensor map over x has a one-row box of
// one stage's K, and its swizzle is the A stage's); an elected lane loads
// the weight chunks as in the staged path.  All of a stage's bytes complete
// on its full barrier (one arrival: the expect-tx), and the tensor core
// reads what the async proxy wrote, so no proxy fence is needed.  Rows past
// the tile's end repeat its first row; their products are never stored.
template <bool WIDE>
__device__ void producer_gather4(const Params& p, const CUtensorMap* tmX, const CUtensorMap* tmB,
                                 const CUtensorMap* tmB3, CtrlSmem* cs, const WaitCtx& wp) {
    using G = StageGeo<WIDE>;
    constexpr int NBLK = WIDE ? 2 : 1;  // 128-row A blocks per stage
    constexpr int RB = G::KB * 2;       // bytes of one A row in a stage
    static_assert(BM == 4 * 32, "a warp's gather4 loads cover one 128-row block");
    const int lane = threadIdx.x & 31;
    uint8_t* s = smem_base();
    const int total_items = cs->item_start[p.E];
    const int kblocks = p.H / G::KB;
    const uint64_t wpol = l2_policy_evict_last();  // weight slices: the other tiles of the group read them next
    uint32_t stage = 0, phase = 0;
    uint32_t issued_par = 0, issued_any = 0;
    bool ok = true;
    uint32_t next = 0;
    if (lane == 0) next = atom_add_relaxed_u32(&p.ctl->next_item, 1u);
    next = __shfl_sync(0xffffffffu, next, 0);
    for (uint32_t it = 0; ok; ++it) {
        const int item = int(next);
        const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
        if (!warp_wait_mbar(&cs->info_empty[slot], iph ^ 1u, wp, SITE_INFO_EMPTY)) {
            ok = false;
            break;
        }
        if (item >= total_items) {
            if (lane == 0) {
                cs->info[slot].e = -1;
                mbar_arrive(&cs->info_full[slot]);
            }
            break;
        }
        uint32_t ahead = 0;
        if (lane == 0) ahead = atom_add_relaxed_u32(&p.ctl->next_item, 1u);  // claimed one item ahead
        Info inf;
        int gtile;
        decode_item(p, cs, item, inf, gtile);
        if (lane == 0) {
            cs->info[slot] = inf;
            mbar_arrive(&cs->info_full[slot]);
        }
        const int nblk = (WIDE && inf.nrows > BM) ? 2 : 1;
        // token of each of this lane's rows: block bl, rows bl*128 + 4*lane + q
        int tok[NBLK][4];
#pragma unroll
        for (int bl = 0; bl < NBLK; ++bl)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = bl * BM + 4 * lane + q;
                const int sidx = __ldcg(p.src_index + inf.row0 + (r < inf.nrows ? r : 0));
                tok[bl][q] = min(max(sidx / p.k, 0), p.T - 1);
            }
        const int ncol = p.F;
        for (int kb = 0; kb < kblocks; ++kb) {
            if (!warp_wait_mbar(&cs->empty[stage], phase ^ 1u, wp, SITE_STAGE_EMPTY)) {
                ok = false;
                break;
            }
            uint64_t* fb = &cs->full[stage];
            mbar_arrive_expect_tx_elect(fb, nblk * G::ABLK + G::BSB);
            __syncwarp();  // the expect-tx before any of the stage's copies
            uint8_t* a = s + stage * G::ASB;
#pragma unroll
            for (int bl = 0; bl < NBLK; ++bl)
                if (bl < nblk)
                    tma_gather4(a + bl * G::ABLK + lane * 4 * RB, tmX, kb * G::KB, tok[bl][0], tok[bl][1], tok[bl][2],
                                tok[bl][3], fb);
            uint8_t* b = s + G::SMB + stage * G::BSB;
            if (p.gated) {
#pragma unroll
                for (int q = 0; q < GATED_BN / 64; ++q) {
                    const int col = inf.nbk * GATED_BN + q * 64;
                    const int c = col < ncol ? col : ncol;
                    tma_load_2d_elect_hint(b + q * G::BCH, tmB, c, inf.e * p.H + kb * G::KB, fb, wpol);
                    tma_load_2d_elect_hint(b + G::BSB / 2 + q * G::BCH, tmB3, c, inf.e * p.H + kb * G::KB, fb, wpol);
                }
            } else {
#pragma unroll
                for (int q = 0; q < BN / 64; ++q) {
                    const int col = inf.nbk * BN + q * 64;
                    tma_load_2d_elect_hint(b + q * G::BCH, tmB, col < ncol ? col : ncol, inf.e * p.H + kb * G::KB, fb, wpol);
                }
            }
            issued_any |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == G::NST) {
                stage = 0;
                phase ^= 1u;
            }
        }
        next = __shfl_sync(0xffffffffu, ahead, 0);
    }
    if (!ok && lane == 0) {
        // let every issued tensor load land before the CTA can exit
        WaitCtx shortw{nullptr, 0u, 5000000LL};
        for (int st = 0; st < G::NST; ++st)
            if (issued_any & (1u << st)) wait_mbar(&cs->full[st], (issued_par >> st) & 1u, shortw, SITE_DRAIN);
    }
    __syncwarp();
}

// Where a compute role takes its work: items [lo, hi) of the work order,
// claimed through the counter `next`; the A operand's tensor map starts at
// sorted row a_row0.  With `arrived` (expert parallel) tile g is ready once
// arrived[g - tile_lo] reaches its row count.
struct WorkQueue {
    uint32_t* next;
    int lo, hi;
    int a_row0;
    const uint32_t* arrived;
    int tile_lo;
};

// The single-device queue: every work item, A operand over all sorted rows.
__device__ __forceinline__ WorkQueue whole_queue(const Params& p, const CtrlSmem* cs) {
    return WorkQueue{&p.ctl->next_item, 0, cs->item_start[p.E], 0, nullptr, 0};
}

// Sending rank of token t (expert parallel).
__device__ __forceinline__ int rank_of_token(const Params& p, int t) {
    int r = 0;
    while (r + 1 < p.ranks && p.ep_t0[r + 1] <= t) ++r;
    return r;
}

// Warp-specialised expert GEMM over work items (tile, N-block) taken from the
// queue until it is empty.  wait_ready: spin on the tile's flag first.
//
// WIDE: 256-row tiles on one SM.  Each stage holds the tile's two 128-row A
// blocks and one B block; two 128 x 256 accumulators (all 512 TMEM columns)
// share that B block, so a stage carries 64 KiB for 1024 cycles of MMA
// instead of 48 KiB for 512.  With TMEM full, the accumulators are
// single-buffered: the epilogue frees the first as soon as it has read it,
// and the next item's MMAs start on that one while the second is read (see
// the MMA issuer).  A tile of at most 128 rows (an expert's last) uses one
// accumulator and loads one A block.
template <bool WIDE>
__device__ void compute_role(const Params& p, const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmB3,
                             const CUtensorMap* tmY, CtrlSmem* cs, const WorkQueue& wq,
                             bool wait_ready, uint32_t flag, const WaitCtx& w) {
    using G = StageGeo<WIDE>;
    constexpr int NST = G::NST, ASB = G::ASB, SMA = 0, SMB = G::SMB;
    constexpr uint32_t NACC = WIDE ? 1u : 2u;  // accumulator buffers
    const int kblocks = p.H / G::KB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* s = smem_base();
    // Waits inside the pipeline only stall because something upstream (a
    // tile flag, a barrier) stalls: they get twice the limit, so the wait
    // that times out and is recorded is the one at the root.
    const WaitCtx wp{w.abort, w.abort_val, w.limit_ns * 2};

    if (p.direct && p.gather4 && (warp == 0 || warp >= EPI_WARP_END)) {
        if (warp == 0) producer_gather4<WIDE>(p, tmA, tmB, tmB3, cs, wp);  // the copy helpers idle
    } else if (p.direct && (warp == 0 || warp >= EPI_WARP_END)) {
        producer_direct<WIDE>(p, tmB, tmB3, cs, warp == 0 ? 0 : warp - EPI_WARP_END + 1, wp);
    } else if (warp == 0) {
        // ---------------- TMA producer: the whole warp runs the loop, one elected lane issues ----------------
        // Weight slices are read by the other tiles of the same work-order
        // group soon after (evict-last); results are never read again
        // (evict-first in the epilogue).  Measured on GB300: -0.6% on the
        // Mixtral-like layer against the default policy.
        const uint64_t wpol = l2_policy_evict_last();
        uint32_t stage = 0, phase = 0;
        uint32_t issued_par = 0, issued_any = 0;  // per-stage bit: parity of the last issue
        bool ok = true;
        uint32_t next = 0;
        if (lane == 0) next = atom_add_relaxed_u32(wq.next, 1u);
        next = __shfl_sync(0xffffffffu, next, 0);
        const int ntiles = cs->tile_start[p.E];
        for (uint32_t it = 0; ok; ++it) {
            const int item = wq.lo + int(next);
            const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
            if (!warp_wait_mbar(&cs->info_empty[slot], iph ^ 1u, wp, SITE_INFO_EMPTY)) {
                ok = false;
                break;
            }
            if (item >= wq.hi) {
                if (lane == 0) {
                    cs->info[slot].e = -1;
                    mbar_arrive(&cs->info_full[slot]);
                }
                break;
            }
            uint32_t ahead = 0;  // the next item, claimed CLAIM_LEAD K-blocks before this one's end
            Info inf;
            int gtile;
            decode_item(p, cs, item, inf, gtile);
            const int pf = p.l2_prefetch;
            if (pf > 0) {
                // the first k-blocks of this item's weight slice head for L2 now
                const int n0 = min(pf, kblocks);
                for (int kb = 0; kb < n0; ++kb)
#pragma unroll
                    for (int q = 0; q < BN / 64; ++q) {
                        const int col = inf.nbk * BN + q * 64;
                        if (col < p.F) tma_prefetch_l2_2d_elect(tmB, col, inf.e * p.H + kb * G::KB);
                    }
            }
            if (lane == 0) {
                cs->info[slot] = inf;
                mbar_arrive(&cs->info_full[slot]);
            }
            const int ncol = p.F;
            const bool two = WIDE && inf.nrows > BM;  // second 128-row A block
            const uint32_t stage_bytes = (two ? 2 : 1) * G::ABLK + G::BSB;
            // this item's weight boxes of K-block kb into B stage b
            auto load_b = [&](int kb, uint8_t* b, uint64_t* fb) {
                if (p.gated) {
                    // 128 columns of W1 into the first half of the B stage, of W3 into the second
#pragma unroll
                    for (int q = 0; q < GATED_BN / 64; ++q) {
                        const int col = inf.nbk * GATED_BN + q * 64;
                        const int c = col < ncol ? col : ncol;
                        tma_load_2d_elect_hint(b + q * G::BCH, tmB, c, inf.e * p.H + kb * G::KB, fb, wpol);
                        tma_load_2d_elect_hint(b + G::BSB / 2 + q * G::BCH, tmB3, c, inf.e * p.H + kb * G::KB, fb, wpol);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < BN / 64; ++q) {
                        const int col = inf.nbk * BN + q * 64;
                        // chunks past F read as zeros (out of bounds fill)
                        tma_load_2d_elect_hint(b + q * G::BCH, tmB, col < ncol ? col : ncol, inf.e * p.H + kb * G::KB,
                                          fb, wpol);
                    }
                }
            };
            // The CTA's first item finds every stage free: its first weight
            // boxes (which do not depend on the gather) go out before the wait
            // for the tile's rows, and the rows follow into the same stages.
            int pre = 0;
            if (it == 0 && (wq.arrived || wait_ready)) {
                pre = min(NST, kblocks);
                for (int kb = 0; kb < pre; ++kb) {
                    mbar_arrive_expect_tx_elect(&cs->full[kb], stage_bytes);
                    load_b(kb, s + SMB + kb * G::BSB, &cs->full[kb]);
                    issued_any |= 1u << kb;  // stage kb, phase 0: the first use of every stage
                }
            }
            if (wq.arrived) {
                // every source's rows of this tile have landed
                if (!warp_wait_geq(wq.arrived + (gtile - wq.tile_lo), uint32_t(inf.nrows), w, SITE_TILE_READY)) {
                    ok = false;
                    break;
                }
                fence_proxy_async();
            } else if (wait_ready) {
                // one acquire per item until every tile is known to be in;
                // before that, the tile's arrival count reaches its rows
                if (__all_sync(0xffffffffu, ld_acquire_u32(&p.ctl->tiles_done) >= uint32_t(ntiles))) {
                    wait_ready = false;
                } else if (!warp_wait_geq(p.ready + gtile, uint32_t(inf.nrows), w, SITE_TILE_READY)) {
                    ok = false;
                    break;
                }
                fence_proxy_async();
            }
            const int kclaim = max(0, kblocks - CLAIM_LEAD);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (kb == kclaim && lane == 0) ahead = atom_add_relaxed_u32(wq.next, 1u);
                uint64_t* fb = &cs->full[stage];
                if (kb >= pre) {
                    if (!warp_wait_mbar(&cs->empty[stage], phase ^ 1u, wp, SITE_STAGE_EMPTY)) {
                        ok = false;
                        break;
                    }
                    if (pf > 0 && kb + pf < kblocks) {
#pragma unroll
                        for (int q = 0; q < BN / 64; ++q) {
                            const int col = inf.nbk * BN + q * 64;
                            if (col < ncol) tma_prefetch_l2_2d_elect(tmB, col, inf.e * p.H + (kb + pf) * G::KB);
                        }
                    }
                    mbar_arrive_expect_tx_elect(fb, stage_bytes);
                    load_b(kb, s + SMB + stage * G::BSB, fb);
                }
                uint8_t* a = s + SMA + stage * ASB;
                tma_load_2d_elect(a, tmA, kb * G::KB, inf.row0 - wq.a_row0, fb);
                if (two) tma_load_2d_elect(a + G::ABLK, tmA, kb * G::KB, inf.row0 - wq.a_row0 + BM, fb);
                issued_any |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == NST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            next = __shfl_sync(0xffffffffu, ahead, 0);
        }
        if (!ok) {
            // let every issued tensor load land before the CTA can exit
            WaitCtx shortw{nullptr, 0u, 5000000LL};
            for (int st = 0; st < NST; ++st)
                if (issued_any & (1u << st)) wait_mbar(&cs->full[st], (issued_par >> st) & 1u, shortw, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp runs the loop, one elected lane issues ----------------
        // WIDE: the epilogue frees the two accumulators one after the other
        // (acc_empty[1]: rows 0-127 drained; acc_empty[0]: the whole tile).
        // An item starts once the first is free; while the second is still
        // being drained, its K-blocks run on the first accumulator alone, up
        // to a full ring of stages, and the second accumulator's MMAs of those
        // K-blocks follow, in order, once it is free.  Each accumulator still
        // sums its K-blocks in ascending order, so results are unchanged.
        uint32_t stage = 0, phase = 0, acc = 0, accph = 0, e0ph = 0;
        bool issued = false;
        for (uint32_t it = 0;; ++it) {
            const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
            if (!warp_wait_mbar(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) break;
            const int e = cs->info[slot].e;
            const bool two = WIDE && cs->info[slot].nrows > BM;
            __syncwarp();
            if (lane == 0) mbar_arrive(&cs->info_empty[slot]);
            if (e < 0) break;
            if (WIDE) {
                if (!warp_wait_mbar(&cs->acc_empty[1], e0ph ^ 1u, wp, SITE_ACC_EMPTY)) break;
                e0ph ^= 1u;
            } else if (!warp_wait_mbar(&cs->acc_empty[acc], accph ^ 1u, wp, SITE_ACC_EMPTY)) {
                break;
            }
            tc_fence_after();
            // WIDE: rows 0-127 in TMEM columns [0, 256), rows 128-255 in [256, 512)
            const uint32_t d = cs->tmem_base + acc * BN;
            bool ok = true;
            bool second_free = false;             // two: the second accumulator may be written
            int kb_lo = 0;                        // two: first K-block without its second-accumulator MMAs
            uint32_t st_lo = stage;               // ... and its stage
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!warp_wait_mbar(&cs->full[stage], phase, wp, SITE_STAGE_FULL)) {
                    ok = false;
                    break;
                }
                // direct rows were written by cp.async (generic proxy): order
                // them before the tensor core reads the stage
                if (p.direct && !p.gather4) fence_proxy_async_shared();
                tc_fence_after();
                // trace: this CTA's first full stage reaches the tensor core
                if (!issued && p.trace && lane == 0) p.trace_buf[blockIdx.x * TRACE_SLOTS + 10] = globaltimer();
                const uint32_t a0 = smem_u32(s + SMA + stage * ASB);
                const uint32_t b0 = smem_u32(s + SMB + stage * G::BSB);
#pragma unroll
                for (int kk = 0; kk < G::KB / 16; ++kk) {
                    // A: K-major, 128B swizzle, 8-row groups 1024 B apart; +32 B per K=16
                    const uint64_t ad = a_desc(a0 + kk * 32);
                    // B: N-major, 128B swizzle; 64-column chunks 8 KiB apart (LBO),
                    // 8-row K groups 1024 B apart (SBO); +2 KiB per K=16
                    // Gated: the stage holds 128 columns of W1 then the same 128
                    // of W3 as four consecutive 64-column chunks, so one N = 256
                    // product leaves A.W1 in accumulator columns [0, 128) and
                    // A.W3 in [128, 256).
                    const uint64_t bd = umma_desc_sw128(b0 + kk * 2048, G::BCH, 1024);
                    tc_mma_f16_elect(d, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
                }
                issued = true;
                if (two) {
                    const bool last = kb == kblocks - 1;
                    // last K-block: the first accumulator's MMAs are all issued,
                    // so its epilogue may start (acc_full[1], unused by wide tiles
                    // otherwise) while the tensor core runs the second's last MMAs
                    if (WIDE_EARLY_HALF && last) tc_commit_elect(&cs->acc_full[1]);
                    if (!second_free) {
                        if (last || kb - kb_lo + 1 == NST) {
                            // no stage left to run ahead on: wait for the second accumulator
                            if (!warp_wait_mbar(&cs->acc_empty[0], accph ^ 1u, wp, SITE_ACC_EMPTY)) {
                                ok = false;
                                break;
                            }
                            second_free = true;
                        } else {
                            second_free = __all_sync(0xffffffffu, mbar_try_wait(&cs->acc_empty[0], accph ^ 1u));
                        }
                        if (second_free) tc_fence_after();
                    }
                    if (second_free) {
                        for (; kb_lo <= kb; ++kb_lo) {
                            // the second A block of each K-block not yet issued, same B chunk
                            const uint32_t a1 = smem_u32(s + SMA + st_lo * ASB) + G::ABLK;
                            const uint32_t b1 = smem_u32(s + SMB + st_lo * G::BSB);
#pragma unroll
                            for (int kk = 0; kk < G::KB / 16; ++kk)
                                tc_mma_f16_elect(d + BN, a_desc(a1 + kk * 32),
                                                 umma_desc_sw128(b1 + kk * 2048, G::BCH, 1024), IDESC,
                                                 (kb_lo | kk) != 0 ? 1u : 0u);
                            tc_commit_elect(&cs->empty[st_lo]);
                            if (++st_lo == NST) st_lo = 0;
                        }
                    }
                } else {
                    tc_commit_elect(&cs->empty[stage]);
                }
                if (++stage == NST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (WIDE && !two) {
                // one-accumulator item: keep in step with the epilogue's
                // release of the second accumulator (long done by now)
                if (!warp_wait_mbar(&cs->acc_empty[0], accph ^ 1u, wp, SITE_ACC_EMPTY)) break;
            }
            tc_commit_elect(&cs->acc_full[acc]);
            if (++acc == NACC) {
                acc = 0;
                accph ^= 1u;
            }
        }
        if (issued) {
            // every MMA this warp issued has completed before TMEM is freed
            tc_commit_elect(&cs->drain);
            WaitCtx shortw{nullptr, 0u, 5000000LL};
            warp_wait_mbar(&cs->drain, 0u, shortw, SITE_DRAIN);
            // trace: this CTA's last MMA has completed
            if (p.trace && lane == 0) p.trace_buf[blockIdx.x * TRACE_SLOTS + 11] = globaltimer();
        }
        __syncwarp();
    } else if (warp < EPI_WARP_END) {
        // ---------------- epilogue: warps 2..5 ----------------
        const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad + 32)
        uint32_t acc = 0, accph = 0, h0ph = 0;
        bool ok = true;
        for (uint32_t it = 0; ok; ++it) {
            const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
            if (!wait_mbar(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) break;
            const Info inf = cs->info[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&cs->info_empty[slot]);
            if (inf.e < 0) break;
            // WIDE: the tile's second 128 rows come from the second accumulator
            const int halves = (WIDE && inf.nrows > BM) ? 2 : 1;
            // with two accumulators the first may be drained before the second is done
            const bool early = WIDE_EARLY_HALF && halves == 2;
            if (early) {
                if (!wait_mbar(&cs->acc_full[1], h0ph, wp, SITE_ACC_FULL)) break;
                h0ph ^= 1u;
            } else if (!wait_mbar(&cs->acc_full[acc], accph, wp, SITE_ACC_FULL)) {
                break;
            }
            tc_fence_after();
            for (int half = 0; half < halves; ++half) {
                if (early && half == 1) {
                    if (!wait_mbar(&cs->acc_full[acc], accph, wp, SITE_ACC_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const int rloc = half * BM + quad * 32 + lane;
                const bool rowok = rloc < inf.nrows;
                // expert parallel: the result goes back to the sending rank, into
                // its return rows in (t, j) order
                const int ep_q = (p.ep && rowok) ? __ldcg(p.src_index + inf.row0 + rloc) : -1;
                const size_t row = p.ep ? size_t(ep_q < 0 ? 0 : ep_q) : size_t(inf.row0) + rloc;
                const uint32_t tbase = cs->tmem_base + (uint32_t(quad * 32) << 16) + (acc + half) * BN;
                if (tmY != nullptr && p.y_tma && half * BM + quad * 32 + 32 <= inf.nrows) {
                    // all 32 rows of this warp lie in the tile: tensor stores
                    epi_rows_box(p, tmY, s + SM_EPI + (warp - 2) * EPI_BUF_BYTES, tbase,
                                 inf.nbk * (p.gated ? GATED_BN : BN), inf.row0 + half * BM + quad * 32);
                } else if (p.gated) {
                    const int n0 = inf.nbk * GATED_BN;
#pragma unroll 1
                    for (int cc = 0; cc < GATED_BN / 32; ++cc) {
                        const int col = n0 + cc * 32;
                        if (col >= p.F) break;
                        uint32_t r[32], r3[32];
                        tmem_ld_32x32b_x32(tbase + cc * 32, r);
                        tmem_ld_32x32b_x32(tbase + GATED_BN + cc * 32, r3);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            // SwiGLU: silu(a) * b, silu(a) = a / (1 + e^-a).  The fast
                            // exponential and divide intrinsics (a few ulp for the
                            // accumulator values that occur) keep the epilogue short,
                            // which matters on wide tiles, where it is not overlapped.
                            const float a = __uint_as_float(r[i]);
                            r[i] = __float_as_uint(__fdividef(a, 1.f + __expf(-a)) * __uint_as_float(r3[i]));
                        }
                        if (rowok) store_row32(p, row, col, r);
                    }
                } else {
                    const int n0 = inf.nbk * BN;
#pragma unroll 1
                    for (int cc = 0; cc < BN / 32; ++cc) {
                        const int col = n0 + cc * 32;
                        if (col >= p.F) break;
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(tbase + cc * 32, r);
                        tmem_ld_wait();
                        if (rowok) store_row32(p, row, col, r);
                    }
                }
                if (p.ep) {
                    // one count per (warp, sending rank): this item's rows are stored
                    const int src = ep_q >= 0 ? rank_of_token(p, ep_q / p.k) : -1;
                    __threadfence();  // this lane's stores before the count that publishes them
                    __syncwarp();
                    const uint32_t peers = __match_any_sync(0xffffffffu, src);
                    if (src >= 0 && lane == __ffs(peers) - 1)
                        atom_add_acq_rel_u32(&p.ep_ctl[src]->ret_done, uint32_t(__popc(peers)));
                }
                if (p.stream_done) {
                    // streamed results: count this item's stored rows per chunk; the
                    // warp that completes a chunk raises its flag for the copy stream
                    const int c = rowok ? int(row / uint32_t(p.stream_rows)) : -1;
                    __threadfence();  // this lane's stores before the count that publishes them
                    __syncwarp();
                    const uint32_t peers = __match_any_sync(0xffffffffu, c);
                    if (c >= 0 && lane == __ffs(peers) - 1) {
                        const uint32_t n = uint32_t(__popc(peers));
                        const uint32_t target =
                            uint32_t(min(p.rows - c * p.stream_rows, p.stream_rows)) * uint32_t(p.nb);
                        if (atom_add_acq_rel_u32(&p.stream_done[c], n) + n == target) {
                            __threadfence_system();
                            st_release_sys_u32(&p.stream_flag[c], p.stream_seq);
                        }
                    }
                }
                if (WIDE && half == 0) {
                    // the first accumulator is drained: the next item's MMAs may start
                    tc_fence_before();
                    mbar_arrive(&cs->acc_empty[1]);
                }
            }
            if (!ok) break;
            tc_fence_before();
            mbar_arrive(&cs->acc_empty[acc]);
            if (++acc == NACC) {
                acc = 0;
                accph ^= 1u;
            }
        }
        if (lane == 0) {
            // this warp's tensor stores have landed (visible to the combine
            // and to later kernels) before the role ends
            if (EPI_TMA_STORE) {
                bulk_wait_all();
                fence_proxy_async();
            }
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------ combine ------

// out[t,:] = sum_j gate[t,j] * y[row of (t,j), :], fp32 in slot order
// (deterministic, no atomics), stored in y's dtype.  y is y_sorted (row of
// (t, j) from row_of) or, expert parallel, the token-major return rows (row
// t*k + j).  Tokens t_first, t_first + stride, ... below t_end.
//
// The pass is bound by load latency: a token's K rows are only a few hundred
// 16-byte vectors, fewer than the CTA's threads can keep in flight.  So the
// CTA first stages the row indices and gates of a batch of its tokens in
// shared memory and then treats the batch's (token, vector) pairs as one flat
// range: every thread issues 16 independent 16-byte loads (U = 16/K vectors
// of K rows, from any tokens) before it accumulates and stores.
constexpr int COMBINE_BATCH = 256;  // tokens whose metadata is staged at once
constexpr int COMBINE_SMEM = COMBINE_BATCH * MAX_K * 8;
static_assert(COMBINE_SMEM <= SM_STAGE_END, "combine metadata must fit in the (idle) stage area");

template <int K>
__device__ void combine_tokens_k(const Params& p, int t_first, int t_end, int stride) {
    constexpr int U = 16 / K;  // 16-byte vectors per thread per pass
    const int F = p.F;
    const bool f32 = p.out_f32 != 0;
    const int nvec = f32 ? F / 4 : F / 8;
    const int ntok = t_first < t_end ? (t_end - t_first + stride - 1) / stride : 0;
    int* srow = reinterpret_cast<int*>(smem_base());                 // [batch][K] row of (t, j)
    float* sg = reinterpret_cast<float*>(smem_base() + COMBINE_BATCH * MAX_K * 4);  // [batch][K] gate
    for (int i0 = 0; i0 < ntok; i0 += COMBINE_BATCH) {
        const int nb = min(COMBINE_BATCH, ntok - i0);
        __syncthreads();  // the previous batch's metadata is no longer read
        for (int q = threadIdx.x; q < nb * K; q += NTHREADS) {
            const int i = q / K, j = q - (q / K) * K;
            const size_t tj = size_t(t_first + (i0 + i) * stride) * K + j;
            // in range even if an error path left a row unrecorded
            srow[q] = p.ep ? int(tj) : min(max(__ldcg(p.row_of + tj), 0), p.rows - 1);
            sg[q] = __ldcg(p.topk_gate + tj);
        }
        __syncthreads();
        const int units = nb * nvec;
        // (token, vector) of this thread's first unit, advanced by steps of
        // NTHREADS vectors instead of a division per unit
        int tk = threadIdx.x / nvec, vc = threadIdx.x - (threadIdx.x / nvec) * nvec;
        for (int f0 = threadIdx.x; f0 < units; f0 += U * NTHREADS) {
            uint4 buf[U][K];
            int tok[U], vec[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * NTHREADS;
                tok[u] = f < units ? tk : 0;
                vec[u] = vc;
                vc += NTHREADS;
                while (vc >= nvec) {
                    vc -= nvec;
                    ++tk;
                }
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const size_t off = size_t(srow[tok[u] * K + j]) * F;
                    const uint4* src = f32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(p.y) + off)
                                           : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.y) + off);
                    buf[u][j] = f < units ? __ldcg(src + vec[u]) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (f0 + u * NTHREADS >= units) break;
                const float* g = sg + tok[u] * K;
                const size_t t = size_t(t_first + (i0 + tok[u]) * stride);
                if (f32) {
                    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        a[0] += g[j] * __uint_as_float(buf[u][j].x);
                        a[1] += g[j] * __uint_as_float(buf[u][j].y);
                        a[2] += g[j] * __uint_as_float(buf[u][j].z);
                        a[3] += g[j] * __uint_as_float(buf[u][j].w);
                    }
                    reinterpret_cast<uint4*>(static_cast<float*>(p.combine_out) + t * F)[vec[u]] =
                        make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                   __float_as_uint(a[3]));
                } else {
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        const uint32_t w4[4] = {buf[u][j].x, buf[u][j].y, buf[u][j].z, buf[u][j].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 fv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[q]));
                            a[2 * q] += g[j] * fv.x;
                            a[2 * q + 1] += g[j] * fv.y;
                        }
                    }
                    uint32_t pk[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * q], a[2 * q + 1]);
                        pk[q] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.combine_out) + t * F)[vec[u]] =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        }
    }
}

__device__ void combine_tokens(const Params& p, int t_first, int t_end, int stride) {
    switch (p.k) {
        case 1: combine_tokens_k<1>(p, t_first, t_end, stride); break;
        case 2: combine_tokens_k<2>(p, t_first, t_end, stride); break;
        case 3: combine_tokens_k<3>(p, t_first, t_end, stride); break;
        case 4: combine_tokens_k<4>(p, t_first, t_end, stride); break;
        case 5: combine_tokens_k<5>(p, t_first, t_end, stride); break;
        case 6: combine_tokens_k<6>(p, t_first, t_end, stride); break;
        case 7: combine_tokens_k<7>(p, t_first, t_end, stride); break;
        default: combine_tokens_k<8>(p, t_first, t_end, stride); break;
    }
}

// ----------------------------------------------------------- CTA setup -----

// Bounded wait with cluster-scope acquire (arrivals may come from the peer CTA
// or from the pair's tensor core).
__device__ __forceinline__ bool wait_mbar_cl(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (!mbar_try_wait_cluster(bar, parity)) {
        if ((++n & 63u) == 0u) {
            if (aborted(w)) return false;
            if ((long long)(globaltimer() - t0) > w.limit_ns) {
                record_error(ERR_TIMEOUT, site, parity);
                raise_abort(w);
                return false;
            }
        }
    }
    return true;
}

__device__ __forceinline__ bool warp_wait_mbar_cl(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, wait_mbar_cl(bar, parity, w, site));
}

constexpr uint32_t IDESC_PAIR = umma_idesc_bf16(PAIR_TILE_M, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);

// CTA-pair compute role (cluster of two CTAs, cta_group::2): one 256 x 256
// tile per pair.  Rank 0 (the leader) takes work items from the queue and
// writes each item's description into both CTAs' shared memory; both CTAs'
// producers load their own 128 rows of A and their own 128 of B's columns
// into their 6-stage rings, the bytes of both counted on the leader's full
// barrier; one leader thread issues the 2-SM MMAs, whose commits release the
// stage and hand over the accumulator in both CTAs at once (multicast); each
// CTA's epilogue drains its own 128 TMEM lanes (rows rank*128 + ...) and
// tells the leader (remote arrive) when the accumulator is free again.
__device__ void compute_role_pair(const Params& p, const CUtensorMap* tmA, const CUtensorMap* tmB, CtrlSmem* cs,
                                  bool wait_ready, uint32_t flag, const WaitCtx& w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    uint8_t* s = smem_base();
    const WaitCtx wp{w.abort, w.abort_val, w.limit_ns * 2};
    const int total_items = cs->item_start[p.E];
    // Self-check: the swizzled stages need a 1024-byte aligned base, the work
    // records sent to the peer 16-byte slots.  A miss is recorded and the
    // role is skipped (the call then times out) instead of faulting.
    if ((smem_u32(s) & 1023u) != 0u || (mapa_shared(smem_u32(&cs->info[0]), 1) & 15u) != 0u) {
        if (threadIdx.x == 0) {
            record_error(ERR_FAULT, SITE_PAIR_ALIGN, smem_u32(s));
            raise_abort(w);
        }
        return;
    }

    if (warp == 0) {
        // ---------------- producer (both CTAs): the whole warp runs the loop, one elected lane issues ----------------
        uint32_t stage = 0, phase = 0;
        uint32_t issued_par = 0, issued_any = 0;
        bool ok = true;
        uint32_t next = 0;
        if (leader && lane == 0) next = atom_add_relaxed_u32(&p.ctl->next_item, 1u);
        next = __shfl_sync(0xffffffffu, next, 0);
        const int ntiles = cs->tile_start[p.E];
        const uint32_t full_leader = mapa_shared(smem_u32(&cs->full[0]), 0);
        for (uint32_t it = 0; ok; ++it) {
            const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
            Info inf{-1, 0, 0, 0};
            int gtile = 0;
            uint32_t ahead = 0;
            if (leader) {
                const int item = int(next);
                if (!warp_wait_mbar_cl(&cs->info_empty[slot], iph ^ 1u, wp, SITE_INFO_EMPTY)) {
                    ok = false;
                    break;
                }
                if (item < total_items) decode_item(p, cs, item, inf, gtile);
                const uint32_t peer_info = mapa_shared(smem_u32(&cs->info[slot]), 1);
                if (peer_info & 15u) {  // self-check: a 16-byte store needs a 16-byte slot
                    if (lane == 0) {
                        record_error(ERR_FAULT, SITE_PAIR_ALIGN, peer_info);
                        raise_abort(w);
                    }
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    cs->info[slot] = inf;
                    st_cluster_v4(peer_info, inf.e, inf.row0, inf.nrows, inf.nbk);
                    mbar_arrive(&cs->info_full[slot]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&cs->info_full[slot]), 1));
                }
            } else {
                if (!warp_wait_mbar_cl(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) {
                    ok = false;
                    break;
                }
                inf = cs->info[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&cs->info_empty[slot]), 0));
                if (inf.e >= 0) gtile = cs->tile_start[inf.e] + (inf.row0 - cs->offs[inf.e]) / p.tile_rows;
            }
            if (inf.e < 0) break;
            if (wait_ready) {
                if (__all_sync(0xffffffffu, ld_acquire_u32(&p.ctl->tiles_done) >= uint32_t(ntiles))) {
                    wait_ready = false;
                } else if (!warp_wait_geq(p.ready + gtile, uint32_t(inf.nrows), w, SITE_TILE_READY)) {
                    ok = false;
                    break;
                }
                fence_proxy_async();
            }
            const int arow = inf.row0 + int(rank) * BM;
            const int kclaim = max(0, p.kblocks - CLAIM_LEAD);
            for (int kb = 0; kb < p.kblocks; ++kb) {
                // the leader takes the next item CLAIM_LEAD K-blocks before this one's end
                if (kb == kclaim && leader && lane == 0) ahead = atom_add_relaxed_u32(&p.ctl->next_item, 1u);
                if (!warp_wait_mbar_cl(&cs->empty[stage], phase ^ 1u, wp, SITE_STAGE_EMPTY)) {
                    ok = false;
                    break;
                }
                if (leader) mbar_arrive_expect_tx_elect(&cs->full[stage], 2 * (PA_STAGE_BYTES + PB_STAGE_BYTES));
                const uint32_t fb = full_leader + stage * uint32_t(sizeof(uint64_t));
                tma_load_2d_pair_elect(s + SM_PA + stage * PA_STAGE_BYTES, tmA, kb * BK, arow, fb);
                uint8_t* b = s + SM_PB + stage * PB_STAGE_BYTES;
#pragma unroll
                for (int q = 0; q < BN / 128; ++q) {
                    const int col = inf.nbk * BN + int(rank) * (BN / 2) + q * 64;
                    tma_load_2d_pair_elect(b + q * B_CHUNK_BYTES, tmB, col < p.F ? col : p.F, inf.e * p.H + kb * BK,
                                           fb);
                }
                issued_any |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (leader) next = __shfl_sync(0xffffffffu, ahead, 0);
        }
        if (!ok && leader && lane == 0) {
            WaitCtx shortw{nullptr, 0u, 5000000LL};
            for (int st = 0; st < PSTAGES; ++st)
                if (issued_any & (1u << st)) wait_mbar_cl(&cs->full[st], (issued_par >> st) & 1u, shortw, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader) {
            // ---------------- 2-SM MMA issuer (leader's warp 1; one elected lane issues) ----------------
            uint32_t stage = 0, phase = 0, acc = 0, accph = 0;
            bool issued = false;
            for (uint32_t it = 0;; ++it) {
                const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
                if (!warp_wait_mbar_cl(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) break;
                const int e = cs->info[slot].e;
                __syncwarp();
                if (lane == 0) mbar_arrive(&cs->info_empty[slot]);
                if (e < 0) break;
                if (!warp_wait_mbar_cl(&cs->acc_empty[acc], accph ^ 1u, wp, SITE_ACC_EMPTY)) break;
                tc_fence_after();
                const uint32_t d = cs->tmem_base + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!warp_wait_mbar_cl(&cs->full[stage], phase, wp, SITE_STAGE_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(s + SM_PA + stage * PA_STAGE_BYTES);
                    const uint32_t b0 = smem_u32(s + SM_PB + stage * PB_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // the peer's rows / columns sit at the same offsets in its shared memory
                        const uint64_t ad = umma_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = umma_desc_sw128(b0 + kk * 2048, B_CHUNK_BYTES, 1024);
                        tc_mma_f16_pair_elect(d, ad, bd, IDESC_PAIR, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit_pair_multicast_elect(&cs->empty[stage], 0x3);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_multicast_elect(&cs->acc_full[acc], 0x3);
                acc ^= 1u;
                if (acc == 0) accph ^= 1u;
            }
            if (issued) {
                tc_commit_pair_elect(&cs->drain);
                WaitCtx shortw{nullptr, 0u, 5000000LL};
                warp_wait_mbar_cl(&cs->drain, 0u, shortw, SITE_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp < EPI_WARP_END) {
        // ---------------- epilogue: warps 2..5 of both CTAs ----------------
        const int quad = warp & 3;
        const uint32_t info_empty_leader = mapa_shared(smem_u32(&cs->info_empty[0]), 0);
        const uint32_t acc_empty_leader = mapa_shared(smem_u32(&cs->acc_empty[0]), 0);
        uint32_t acc = 0, accph = 0;
        for (uint32_t it = 0;; ++it) {
            const uint32_t slot = it & 3u, iph = (it >> 2) & 1u;
            if (!wait_mbar_cl(&cs->info_full[slot], iph, wp, SITE_INFO_FULL)) break;
            const Info inf = cs->info[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(info_empty_leader + slot * uint32_t(sizeof(uint64_t)));
            if (inf.e < 0) break;
            if (!wait_mbar_cl(&cs->acc_full[acc], accph, wp, SITE_ACC_FULL)) break;
            tc_fence_after();
            const int rloc = int(rank) * BM + quad * 32 + lane;
            const bool rowok = rloc < inf.nrows;
            const size_t row = size_t(inf.row0) + rloc;
            const int n0 = inf.nbk * BN;
            const uint32_t tbase = cs->tmem_base + (uint32_t(quad * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                const int col = n0 + cc * 32;
                if (col >= p.F) break;
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + cc * 32, r);
                tmem_ld_wait();
                if (rowok) store_row32(p, row, col, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader + acc * uint32_t(sizeof(uint64_t)));
            acc ^= 1u;
            if (acc == 0) accph ^= 1u;
        }
    }
}

// Barrier arrival counts.  Single CTA: the producer's expect-tx, one commit,
// 128 epilogue threads, the MMA thread + 4 epilogue warps.  Direct rows by
// cp.async (copy_warps) add one cp.async arrival per copy lane to each full
// barrier and one info_empty arrival per copy helper warp; rows by TMA
// gather4 add none.  Pair: acc_empty
// gets one arrival per epilogue warp of both CTAs (8) and info_empty the
// leader's MMA thread and 4 epilogue warps plus the peer's producer and 4
// epilogue warps (10); those two live in the leader only.
template <int PAIR>
__device__ void cta_setup(CtrlSmem* cs, bool with_tmem, bool copy_warps) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < MAX_STAGES; ++i) {
            mbar_init(&cs->full[i], copy_warps ? 1 + 32 * COPY_WARPS : 1);
            mbar_init(&cs->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&cs->acc_full[i], 1);
            mbar_init(&cs->acc_empty[i], PAIR ? 8 : 128);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&cs->info_full[i], 1);
            mbar_init(&cs->info_empty[i], PAIR ? 10 : 1 + 4 + (copy_warps ? COPY_WARPS - 1 : 0));
        }
        mbar_init(&cs->drain, 1);
        for (int i = 0; i < MAX_GATHER_SLOTS; ++i) mbar_init(&cs->gbar[i], 1);
        fence_barrier_init();
    }
    if (PAIR) cluster_sync();  // peer running and its barriers initialised before any remote use
    if (with_tmem && warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(&cs->tmem_base, TMEM_COLS);  // collective with the peer's warp 1
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&cs->tmem_base, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ void cta_exit(const Params& p);

template <int PAIR>
__device__ void cta_teardown(const Params& p, CtrlSmem* cs, bool with_tmem) {
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs done with the pair's MMAs before the collective free
    if (with_tmem && (threadIdx.x >> 5) == 1) {
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(cs->tmem_base, TMEM_COLS);
        else tmem_dealloc(cs->tmem_base, TMEM_COLS);
    }
    if (PAIR) cluster_sync();  // neither CTA leaves while the other may touch its shared memory
    cta_exit(p);
}

// Exit bookkeeping of every CTA; the last one out leaves the control blocks
// ready for the next call.
__device__ void cta_exit(const Params& p) {
    if (threadIdx.x == 0) {
        if (p.trace) p.trace_buf[blockIdx.x * TRACE_SLOTS + 15] = globaltimer();
        const uint32_t old = atom_add_acq_rel_u32(&p.ctl->exit_count, 1u);
        if (old == gridDim.x - 1) {
            // last CTA out: leave the control block ready for the next call
            Ctl* c = p.ctl;
            c->bar_routed = 0;
            c->bar_scattered = 0;
            c->next_tile = 0;
            c->next_item = 0;
            c->tiles_done = 0;
            c->bar_computed = 0;
            c->bar_scanned = 0;
            c->abort = 0;
            c->epoch = c->epoch + 1u;  // calls completed on this workspace
            if (p.stream_flag) {
                // a call that gave up still releases every chunk: the copy
                // stream never waits past the end of the call
                __threadfence_system();
                const int nchunks = (p.rows + p.stream_rows - 1) / p.stream_rows;
                for (int i = 0; i < nchunks; ++i) st_release_sys_u32(&p.stream_flag[i], p.stream_seq);
            }
            if (p.ep) {
                for (int r = 0; r < p.ranks; ++r) {
                    EpCtl* q = p.ep_ctl[r];
                    q->routed = 0;
                    q->scattered = 0;
                    q->next_send = 0;
                    q->next_item = 0;
                    q->ret_done = 0;
                    for (int s = 0; s < MAX_RANKS; ++s) q->cnt_flag[s] = 0;
                }
            }
            c->exit_count = 0;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------- kernels -----

// Self-check of the SM-pair kernels: every pair-specific step (peer shared
// memory, pair TMEM allocation, pair MMAs) assumes a cluster of exactly two
// CTAs.  Launched any other way, the CTA records the fact and only does its
// exit bookkeeping.
__device__ bool in_cta_pair(const Params& p, const WaitCtx& w) {
    const uint32_t n = cluster_nctarank();
    if (n == 2u) return true;
    if (threadIdx.x == 0) {
        record_error(ERR_FAULT, SITE_PAIR_CLUSTER, n);
        raise_abort(w);
    }
    cta_exit(p);
    return false;
}

template <int PAIR>
__global__ void __launch_bounds__(NTHREADS, 1)
    mk_fused_kernel(const Params p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmY) {
    CtrlSmem* cs = ctrl();
    const uint32_t flag = 1u;  // tile ready / call aborted
    const WaitCtx w{&p.ctl->abort, flag, p.spin_limit_ns};
    const bool is_dispatch = int(blockIdx.x) < p.dispatch_ctas;
    stamp(p, 0);
    if (threadIdx.x == 0 && p.compute) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (PAIR && !in_cta_pair(p, w)) return;
    cta_setup<PAIR>(cs, p.compute != 0, p.direct != 0 && p.gather4 == 0);

    // This call's tile arrival counts start at 0.  Cleared before the routing
    // barrier; they grow only after it, so no stale value is ever seen.
    for (int i = blockIdx.x * NTHREADS + threadIdx.x; i < p.max_tiles; i += gridDim.x * NTHREADS) p.ready[i] = 0u;
    if (p.stream_done) {
        const int nchunks = (p.rows + p.stream_rows - 1) / p.stream_rows;
        for (int i = blockIdx.x * NTHREADS + threadIdx.x; i < nchunks; i += gridDim.x * NTHREADS) p.stream_done[i] = 0u;
    }

    // phase R
    for (int c = blockIdx.x; c < p.nch; c += gridDim.x) route_chunk(p, c);
    stamp(p, 1);
    bool ok = true;
    if (threadIdx.x == 0) {
        __threadfence();
        atom_add_acq_rel_u32(&p.ctl->bar_routed, 1u);
        ok = wait_geq(&p.ctl->bar_routed, gridDim.x, w, SITE_BAR_ROUTED);
        cs->bcast[0] = ok;
    }
    __syncthreads();
    ok = cs->bcast[0] != 0;
    stamp(p, 2);

    if (ok && p.dist_scan) {
        // phase S on a large count table: columns across the CTAs, then a barrier
        scan_columns(p);
        if (threadIdx.x == 0) {
            __threadfence();
            atom_add_acq_rel_u32(&p.ctl->bar_scanned, 1u);
            ok = wait_geq(&p.ctl->bar_scanned, gridDim.x, w, SITE_BAR_SCANNED);
            cs->bcast[0] = ok;
        }
        __syncthreads();
        ok = cs->bcast[0] != 0;
    }
    if (ok) {
        // phase S
        if (p.dist_scan) scan_from_columns(p, cs, blockIdx.x, gridDim.x, p.nch);
        else scan_counts(p, cs, p.counts, true, blockIdx.x, gridDim.x, p.nch, -1);
        if (blockIdx.x == 0)
            for (int e = threadIdx.x; e <= p.E; e += NTHREADS) p.expert_offsets[e] = cs->offs[e];
        if (threadIdx.x == 0 && cs->offs[p.E] != p.rows) {
            record_error(ERR_FAULT, SITE_ROW_TOTAL, uint32_t(cs->offs[p.E]));
            raise_abort(w);
        }
        const int* sbase = reinterpret_cast<const int*>(smem_base() + RT_BASES);
        int m = 0;
        for (int c = blockIdx.x; c < p.nch; c += gridDim.x, ++m) scatter_chunk(p, c, sbase + m * MAX_E, w);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atom_add_acq_rel_u32(&p.ctl->bar_scattered, 1u);
        }
        stamp(p, 3);

        if (is_dispatch) {
            if (threadIdx.x == 0) cs->bcast[1] = wait_geq(&p.ctl->bar_scattered, gridDim.x, w, SITE_BAR_SCATTERED);
            fence_proxy_async_shared();  // generic smem use (routing) before bulk copies into it
            __syncthreads();
            stamp(p, 4);
            if (cs->bcast[1]) gather_role(p, cs, w);
            __syncthreads();
            stamp(p, 5);
        }
        if (threadIdx.x == 0) {
            bool go = p.compute && !aborted(w);
            // direct rows: the producers read src_index rows that every CTA scattered
            if (go && p.direct) go = wait_geq(&p.ctl->bar_scattered, gridDim.x, w, SITE_BAR_SCATTERED);
            cs->bcast[2] = go;
        }
        fence_proxy_async_shared();  // generic/bulk smem use before TMA writes into it
        __syncthreads();
        if (cs->bcast[2]) {
            stamp(p, 6);
            if constexpr (PAIR) compute_role_pair(p, &tmA, &tmB, cs, true, flag, w);
            else if (p.wide) compute_role<true>(p, &tmA, &tmB, &tmB3, &tmY, cs, whole_queue(p, cs), !p.direct, flag, w);
            else compute_role<false>(p, &tmA, &tmB, &tmB3, &tmY, cs, whole_queue(p, cs), !p.direct, flag, w);
            stamp(p, 7);
        }
    }
    if (p.combine_out) {
        // every CTA's expert rows are written before any token is combined
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atom_add_acq_rel_u32(&p.ctl->bar_computed, 1u);
            cs->bcast[3] = ok && !aborted(w) && wait_geq(&p.ctl->bar_computed, gridDim.x, w, SITE_BAR_COMPUTED);
        }
        __syncthreads();
        stamp(p, 8);
        if (cs->bcast[3]) combine_tokens(p, blockIdx.x, p.T, gridDim.x);
        stamp(p, 9);
    }
    cta_teardown<PAIR>(p, cs, p.compute != 0);
}

// Expert-parallel simulation: R logical ranks in one cooperative launch
// (ranks that wait on one another must be resident together), the CTAs
// [r*cpr, (r+1)*cpr) playing rank r.  Each rank routes its own tokens and
// sends its count rows to every rank (a flag per source at each
// destination); once it holds every rank's rows it scans its copy of the
// table, writes the receive metadata of its own rows, sends the rows to the
// ranks that own their experts (arrival counts per tile), runs the GEMM on
// its own experts' tiles as they complete, stores every result back into
// the sending rank's return rows (a completion count per sending rank), and
// finally combines its own tokens once all their results are back.
struct EpMaps {
    CUtensorMap a[MAX_RANKS];  // A operand of each rank: its received rows
};

__global__ void __launch_bounds__(NTHREADS, 1)
    mk_ep_kernel(const Params p, const __grid_constant__ EpMaps maps, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmB3) {
    CtrlSmem* cs = ctrl();
    const uint32_t flag = 1u;
    const WaitCtx w{&p.ctl->abort, flag, p.spin_limit_ns};
    const int R = p.ranks, cpr = p.ep_cpr, epr = p.E / R;
    const int rank = int(blockIdx.x) / cpr, b = int(blockIdx.x) - rank * cpr;
    EpCtl* me = p.ep_ctl[rank];
    stamp(p, 0);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&maps.a[rank]);
        tma_prefetch_desc(&tmB);
    }
    cta_setup<0>(cs, true, false);
    // This rank's arrival counts start at 0: sources add to them only once
    // they hold this rank's count rows, which it sends after this.
    for (int i = b * NTHREADS + threadIdx.x; i < p.ep_tile_cap; i += cpr * NTHREADS) p.ep_ready[rank][i] = 0u;

    // phase R: own tokens; each chunk's count row goes to every rank
    for (int c = p.ep_c0[rank] + b; c < p.ep_c0[rank + 1]; c += cpr) route_chunk(p, c);
    stamp(p, 1);
    bool ok = true;
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t before = atom_add_acq_rel_u32(&me->routed, 1u);
        if (before == uint32_t(cpr - 1))  // the rank's last CTA raises its flag at every rank
            for (int q = 0; q < R; ++q) st_release_u32(&p.ep_ctl[q]->cnt_flag[rank], 1u);
        for (int s = 0; s < R && ok; ++s) ok = wait_eq(&me->cnt_flag[s], 1u, w, SITE_EP_COUNTS);
        cs->bcast[0] = ok;
    }
    __syncthreads();
    ok = cs->bcast[0] != 0;
    stamp(p, 2);

    if (ok) {
        // phase S on this rank's copy of the table
        scan_counts(p, cs, p.ep_counts[rank], true, p.ep_c0[rank] + b, cpr, p.ep_c0[rank + 1], rank);
        if (blockIdx.x == 0)
            for (int e = threadIdx.x; e <= p.E; e += NTHREADS) p.expert_offsets[e] = cs->offs[e];
        if (threadIdx.x == 0 && cs->offs[p.E] != p.rows) {
            record_error(ERR_FAULT, SITE_ROW_TOTAL, uint32_t(cs->offs[p.E]));
            raise_abort(w);
        }
        // Every rank's rows fit its receive buffer (T*min(k, E/R) rows; only
        // repeated experts in one token, from logits outside the contract,
        // could exceed it).  Every CTA holds the same tables, so all agree.
        bool fits = true;
        for (int q = 0; q < R; ++q)
            if (cs->offs[(q + 1) * epr] - cs->offs[q * epr] > p.ep_cap_rows) fits = false;
        if (!fits) {
            if (threadIdx.x == 0) {
                record_error(ERR_FAULT, SITE_DEST_RANGE, uint32_t(cs->offs[p.E]));
                raise_abort(w);
            }
            cta_teardown<0>(p, cs, true);
            return;
        }
        // receive metadata of the rank's own rows, written at their destinations
        const int* sbase = reinterpret_cast<const int*>(smem_base() + RT_BASES);
        int m = 0;
        for (int c = p.ep_c0[rank] + b; c < p.ep_c0[rank + 1]; c += cpr, ++m)
            scatter_chunk(p, c, sbase + m * MAX_E, w);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atom_add_acq_rel_u32(&me->scattered, 1u);
        }
        stamp(p, 3);
        if (b < p.ep_dispatch) {
            // the send role reads the metadata every CTA of its rank wrote
            if (threadIdx.x == 0) cs->bcast[1] = wait_geq(&me->scattered, uint32_t(cpr), w, SITE_EP_SCATTERED);
            fence_proxy_async_shared();  // generic smem use (routing) before bulk copies into it
            __syncthreads();
            stamp(p, 4);
            if (cs->bcast[1]) send_role(p, cs, rank, w);
            __syncthreads();
            stamp(p, 5);
        }
        if (threadIdx.x == 0) cs->bcast[2] = !aborted(w);
        fence_proxy_async_shared();  // generic/bulk smem use before TMA writes into it
        __syncthreads();
        if (cs->bcast[2]) {
            stamp(p, 6);
            const int e0 = rank * epr, e1 = e0 + epr;
            const WorkQueue wq{&me->next_item, cs->item_start[e0], cs->item_start[e1], cs->offs[e0],
                               p.ep_ready[rank], cs->tile_start[e0]};
            if (p.wide) compute_role<true>(p, &maps.a[rank], &tmB, &tmB3, nullptr, cs, wq, false, flag, w);
            else compute_role<false>(p, &maps.a[rank], &tmB, &tmB3, nullptr, cs, wq, false, flag, w);
            stamp(p, 7);
        }
        if (p.combine_out) {
            // reduce: every result row of the rank's tokens is back
            __syncthreads();
            if (threadIdx.x == 0) {
                const uint32_t need = uint32_t(p.ep_t0[rank + 1] - p.ep_t0[rank]) * uint32_t(p.k) * uint32_t(p.nb);
                cs->bcast[3] = !aborted(w) && wait_geq(&me->ret_done, need, w, SITE_EP_RETURNED);
            }
            __syncthreads();
            stamp(p, 8);
            if (cs->bcast[3]) combine_tokens(p, p.ep_t0[rank] + b, p.ep_t0[rank + 1], cpr);
            stamp(p, 9);
        }
    }
    cta_teardown<0>(p, cs, true);
}

// Unfused baseline, launch 1: routing per chunk.
__global__ void __launch_bounds__(NTHREADS, 1) mk_route_kernel(const Params p) {
    route_chunk(p, blockIdx.x);
}

// Unfused baseline, launch 2: offsets and per-chunk bases (one CTA).
__global__ void __launch_bounds__(NTHREADS, 1) mk_scan_kernel(const Params p) {
    CtrlSmem* cs = ctrl();
    const int E = p.E;
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        int run = 0;
        for (int c = 0; c < p.nch; ++c) run += p.counts[size_t(c) * E + e];
        cs->tot[e] = run;
    }
    __syncthreads();
    build_tables(p, cs);
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += NTHREADS) p.expert_offsets[e] = cs->offs[e];
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        int run = cs->offs[e];
        for (int c = 0; c < p.nch; ++c) {
            const int v = p.counts[size_t(c) * E + e];
            p.bases[size_t(c) * E + e] = run;
            run += v;
        }
    }
}

// Unfused baseline, launch 3: scatter + push-gather per chunk.
__global__ void __launch_bounds__(NTHREADS, 1) mk_gather_kernel(const Params p) {
    CtrlSmem* cs = ctrl();
    if (threadIdx.x == 0) {
        for (int i = 0; i < MAX_GATHER_SLOTS; ++i) mbar_init(&cs->gbar[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const WaitCtx w{nullptr, 0u, p.spin_limit_ns};
    if (p.direct) {
        // rows are copied by the GEMM itself: only src_index / gate_w / row_of here
        scatter_chunk(p, blockIdx.x, p.bases + size_t(blockIdx.x) * p.E, w);
        return;
    }
    uint32_t ph = 0;
    push_gather_chunk(p, blockIdx.x, cs, ph, w);
}

// Unfused baseline, launch 5 (with a combine): tokens over the grid.
__global__ void __launch_bounds__(NTHREADS, 1) mk_combine_kernel(const Params p) {
    combine_tokens(p, blockIdx.x, p.T, gridDim.x);
}

// Unfused baseline, launch 4: persistent expert GEMM over all tiles.
template <int PAIR>
__global__ void __launch_bounds__(NTHREADS, 1)
    mk_gemm_kernel(const Params p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmY) {
    CtrlSmem* cs = ctrl();
    const uint32_t flag = 1u;
    const WaitCtx w{&p.ctl->abort, flag, p.spin_limit_ns};
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (PAIR && !in_cta_pair(p, w)) return;
    cta_setup<PAIR>(cs, true, p.direct != 0 && p.gather4 == 0);
    for (int e = threadIdx.x; e < p.E; e += NTHREADS) cs->tot[e] = p.expert_offsets[e + 1] - p.expert_offsets[e];
    __syncthreads();
    build_tables(p, cs);
    __syncthreads();
    if constexpr (PAIR) compute_role_pair(p, &tmA, &tmB, cs, false, flag, w);
    else if (p.wide) compute_role<true>(p, &tmA, &tmB, &tmB3, &tmY, cs, whole_queue(p, cs), false, flag, w);
    else compute_role<false>(p, &tmA, &tmB, &tmB3, &tmY, cs, whole_queue(p, cs), false, flag, w);
    cta_teardown<PAIR>(p, cs, true);
}

// ---------------------------------------------------------- host hooks -----

// The persistent kernels wait on each other, so every CTA must be resident:
// a cooperative launch guarantees it or fails.  The pair kernel also needs
// clusters of two; if the driver refuses the cooperative attribute together
// with clusters, it is launched without it after an occupancy check that
// every cluster fits at once.
cudaError_t launch_fused(const Params& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                         const CUtensorMap& y, int grid, cudaStream_t st) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    if (!p.pair) {
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, mk_fused_kernel<0>, p, a, b, b3, y);
    }
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, mk_fused_kernel<1>, p, a, b, b3, y);
    if (err == cudaSuccess) return err;
    (void)cudaGetLastError();
    cfg.attrs = attr + 1;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, mk_fused_kernel<1>, &cfg)) != cudaSuccess) return err;
    if (2 * clusters < grid) return cudaErrorCooperativeLaunchTooLarge;
    return cudaLaunchKernelEx(&cfg, mk_fused_kernel<1>, p, a, b, b3, y);
}

cudaError_t launch_ep(const Params& p, const CUtensorMap* a, const CUtensorMap& b, const CUtensorMap& b3, int grid,
                      cudaStream_t st) {
    EpMaps maps{};
    for (int r = 0; r < p.ranks; ++r) maps.a[r] = a[r];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mk_ep_kernel, p, maps, b, b3);
}

cudaError_t launch_unfused(const Params& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                           const CUtensorMap& y, int grid, cudaStream_t st) {
    mk_route_kernel<<<p.nch, NTHREADS, SMEM_BYTES, st>>>(p);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    mk_scan_kernel<<<1, NTHREADS, SMEM_BYTES, st>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    mk_gather_kernel<<<p.nch, NTHREADS, SMEM_BYTES, st>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (!p.pair) {
        mk_gemm_kernel<0><<<grid, NTHREADS, SMEM_BYTES, st>>>(p, a, b, b3, y);
        if ((err = cudaGetLastError()) != cudaSuccess || !p.combine_out) return err;
        mk_combine_kernel<<<grid, NTHREADS, COMBINE_SMEM + 1024, st>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((err = cudaLaunchKernelEx(&cfg, mk_gemm_kernel<1>, p, a, b, b3, y)) != cudaSuccess || !p.combine_out) return err;
    mk_combine_kernel<<<grid, NTHREADS, COMBINE_SMEM + 1024, st>>>(p);
    return cudaGetLastError();
}

cudaError_t set_kernel_attributes() {
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(mk_fused_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    if ((err = cudaFuncSetAttribute(mk_ep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)))
        return err;
    return cudaFuncSetAttribute(mk_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t fused_max_blocks_per_sm(int* n) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, mk_fused_kernel<0>, NTHREADS, SMEM_BYTES);
}

cudaError_t read_and_clear_error(uint32_t out[4], cudaStream_t st) {
    DevError e{};
    cudaError_t err = cudaMemcpyFromSymbolAsync(&e, g_error, sizeof(e), 0, cudaMemcpyDeviceToHost, st);
    if (err != cudaSuccess) return err;
    if ((err = cudaStreamSynchronize(st)) != cudaSuccess) return err;
    out[0] = e.code;
    out[1] = e.site;
    out[2] = e.cta;
    out[3] = e.info;
    if (e.code != 0) {
        DevError z{};
        if ((err = cudaMemcpyToSymbolAsync(g_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st))) return err;
        err = cudaStreamSynchronize(st);
    }
    return err;
}

}  // namespace mk
